// Host side of the C ABI declared in include/gqa_decode.h: argument checks,
// split planning, TMA tensor-map encoding and the decode / combine launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gqa_decode.h"
#include "combine_kernel.cuh"
#include "decode_kernel.cuh"
#include "decode_launch.h"
#include "plan.cuh"

namespace gqa {

// Device error word of this library: bits of kErrTimeout / kErrBadSeqlen,
// set by the kernels (through the address each decode launch is given) and
// read and cleared by gqa_decode_get_error().
__device__ unsigned int g_gqa_error_bits = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kWsAlign = 256;

struct DeviceState {
  int sm_count = 0;
  unsigned attr_done = 0;          // one bit per kernel instantiation
  unsigned int* err_word = nullptr;  // device address of g_gqa_error_bits
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && v[0] != '0';
}

unsigned long long wait_timeout_ns() {
  const char* v = std::getenv("GQA_WAIT_TIMEOUT_MS");
  if (v != nullptr) {
    const long long ms = std::atoll(v);
    if (ms > 0) return static_cast<unsigned long long>(ms) * 1000000ull;
  }
  return 1000000000ull;  // one second: decode launches take microseconds
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

gqa_status_t current_device(int* dev, DeviceState** st) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[*dev];
  if (s.sm_count == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess || n <= 0)
      return GQA_ERR_CUDA;
    s.sm_count = n;
  }
  *st = &s;
  return GQA_OK;
}

// Device address of the error word on the current device (looked up once
// per device, with it current: a __device__ name in host code is only a
// host-side stand-in).
gqa_status_t error_word(DeviceState* st, unsigned int** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->err_word == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gqa_error_bits) != cudaSuccess || p == nullptr) return GQA_ERR_CUDA;
    st->err_word = static_cast<unsigned int*>(p);
  }
  *out = st->err_word;
  return GQA_OK;
}

#ifdef GQA_TRACE
unsigned long long* g_trace_buf = nullptr;  // attached by gqa_trace_attach (trace builds)
#endif

// Sets the dynamic shared memory limit of a kernel once per device.
gqa_status_t ensure_smem_attr(DeviceState* st, unsigned bit, const void* fn, int bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->attr_done & (1u << bit)) return GQA_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return GQA_ERR_CUDA;
  st->attr_done |= 1u << bit;
  return GQA_OK;
}

gqa_status_t check_desc(const gqa_desc_t* d) {
  if (d == nullptr) return GQA_ERR_INVALID_ARG;
  if (d->batch < 0 || d->q_tokens < 1 || d->q_heads < 1 || d->kv_heads < 1 || d->max_seqlen < 1)
    return GQA_ERR_INVALID_ARG;
  if (d->q_heads % d->kv_heads != 0) return GQA_ERR_INVALID_ARG;
  if (d->out_dtype != GQA_DTYPE_BF16 && d->out_dtype != GQA_DTYPE_FP32 && d->out_dtype != GQA_DTYPE_FP16)
    return GQA_ERR_INVALID_ARG;
  if (d->in_dtype != GQA_DTYPE_BF16 && d->in_dtype != GQA_DTYPE_FP16) return GQA_ERR_INVALID_ARG;
  // a 16-bit output has the inputs' type (fp32 goes with either)
  if (d->out_dtype != GQA_DTYPE_FP32 && d->out_dtype != d->in_dtype) return GQA_ERR_UNSUPPORTED;
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return GQA_ERR_INVALID_ARG;
  if (d->reduction != GQA_REDUCE_AUTO && d->reduction != GQA_REDUCE_COMBINE && d->reduction != GQA_REDUCE_CLUSTER)
    return GQA_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return GQA_ERR_UNSUPPORTED;
  const long long g = d->q_heads / d->kv_heads;
  if (static_cast<long long>(d->q_tokens) * g > GQA_MAX_QROWS) return GQA_ERR_UNSUPPORTED;
  if (d->q_heads > 65535 || d->max_seqlen > (1 << 30)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

struct HostPlan {
  PlanParams pp;
  int num_slots;      // partial slots per row (0: the decode writes final outputs only)
  bool combine;       // a combine launch follows
  bool use_n_pieces;  // combine reads per-pair piece counts (balanced plan)
  int cluster_k;      // > 1: the k splits of a pair form a cluster and merge in it
  gqa_status_t status;  // GQA_ERR_UNSUPPORTED: an in-cluster merge was asked for and cannot be done
};

// Largest power of two <= x, for 1 <= x (capped at kMaxClusterK).
int pow2_floor_k(long long x) {
  int k = 1;
  while (2LL * k <= x && k < kMaxClusterK) k *= 2;
  return k;
}

// Automatic split count for the fixed-splits plan, from a load model that
// assumes every sequence is max_seqlen long: the busiest CTA's blocks plus
// the partial traffic spread over the GPU.
int auto_splits(long long pairs, int nblk, int rows_per_pair, int head_dim, int sm) {
  double best = 1e300;
  int best_s = 1;
  for (int S = 1; S <= GQA_MAX_SPLITS && S <= (nblk > 0 ? nblk : 1); S *= 2) {
    const long long items = pairs * S;
    const long long waves = (items + sm - 1) / sm;
    const int per_item = (nblk + S - 1) / S;
    const double kv = static_cast<double>(waves) * per_item * kBlockN * head_dim * 4.0;
    const double part = S > 1 ? static_cast<double>(items) * rows_per_pair * head_dim * 8.0 / sm : 0.0;
    const double cost = kv + part;
    if (cost < best * 0.98) { best = cost; best_s = S; }
  }
  return best_s;
}

// Item units X of the balanced plan: a work item's fixed cost in blocks, by
// the kernel's column count.  Per-CTA traces on GB300 put a CTA's time at
// about a + b * blocks + c * items with c / b ~1.5 (16 query columns) to ~2
// (32).  Timed on GB300 (per call): 16 columns, X = 1 / 2 / 3: Llama-8B
// shape 25.78 / 25.89 / 25.93 us, ragged 137.52 / 137.68 / 137.58 us;
// 32 columns (speculative shape): 17.97 / 17.60 / 17.60 us.
constexpr int kItemUnits16 = 1;
constexpr int kItemUnits32 = 3;

// Cluster size of the in-cluster merge ("Building a Faster GQA Decode Kernel
// for Blackwell SM100", section "Reducing inside a thread block cluster":
// the KV splits of one batch entry and head group form a cluster; the page's
// automatic selection takes it for at most four splits, or eight with at
// most 64 CTAs).  Returns 0 when the kernel-reduction plans (combine launch)
// are to be used, else the number k >= 1 of splits per pair, and -1 for a
// forced in-cluster merge that cannot be done (a split count that is not a
// power of two <= 8).
//
// The automatic choice keeps the page's limits and adds what a sweep on
// GB300 showed (CUDA graphs, pool > L2, per call, cluster minus the best
// combine plan): grids of 128 CTAs with k = 2 gained 0.3-0.8 us and a
// library-chosen split count gained up to 1.5 us where the balanced plan cuts
// few pairs very finely; every grid below 64 CTAs lost 0.3-1.1 us (a cluster
// of 4 CTAs: 7.82 against 7.14 us), explicit split counts 4 and 8 lost
// 0.3-1.1 us against the fixed-split plan, and 16 clusters of 8 took twice
// as long (they do not all fit on the GPU at once).
int cluster_splits(const gqa_desc_t* d, int num_splits, int sm, bool force_partial) {
  if (force_partial || d->reduction == GQA_REDUCE_COMBINE) return 0;
  const bool forced = d->reduction == GQA_REDUCE_CLUSTER;
  const long long pairs = static_cast<long long>(d->batch) * d->kv_heads;
  const int nblk_cap = num_blocks(d->max_seqlen);
  if (num_splits == 0) {
    // the whole-CTAs-per-pair shape of the automatic plan, k a power of two
    const long long per_pair = pairs > 0 ? sm / pairs : 0;
    const long long lim = per_pair < nblk_cap ? per_pair : nblk_cap;
    const int k = lim >= 1 ? pow2_floor_k(lim) : 1;
    if (forced) return k;
    // Only where a cluster CTA streams at most 3 blocks more than a CTA of
    // the automatic balanced plan (k whole CTAs per pair, or one per block):
    // one long pair, say, is spread over every SM there, not over 8.
    const long long bal_ctas = per_pair * pairs < pairs * nblk_cap ? per_pair * pairs : pairs * nblk_cap;
    const long long extra = (nblk_cap + k - 1) / k - (pairs * nblk_cap + bal_ctas - 1) / bal_ctas;
    const bool short_seqs = nblk_cap <= 32 * k;
    return (k >= 2 && short_seqs && extra <= 3 && (k <= 4 || pairs * k <= 64) && k * pairs >= 64) ? k : 0;
  }
  const bool pow2 = (num_splits & (num_splits - 1)) == 0;
  if (forced) return (pow2 && num_splits <= kMaxClusterK) ? num_splits : -1;
  return (num_splits == 2 && pairs * 2 >= 128) ? 2 : 0;
}

HostPlan make_plan(const gqa_desc_t* d, int num_splits, int sm, bool force_partial) {
  HostPlan hp;
  std::memset(&hp, 0, sizeof hp);
  hp.status = GQA_OK;
  PlanParams& pp = hp.pp;
  pp.batch = d->batch;
  pp.kv_heads = d->kv_heads;
  pp.max_seqlen = d->max_seqlen;
  const int nblk_cap = num_blocks(d->max_seqlen);
  const long long pairs = static_cast<long long>(d->batch) * d->kv_heads;
  const int rows_per_pair = d->q_tokens * (d->q_heads / d->kv_heads);
  const int item_units = rows_per_pair <= 16 ? kItemUnits16 : kItemUnits32;
  const int ck = cluster_splits(d, num_splits, sm, force_partial);
  if (ck < 0) {
    hp.status = GQA_ERR_UNSUPPORTED;
    return hp;
  }
  if (ck >= 1) {
    // Fixed splits, k per pair, dealt so that the CTAs of one cluster take
    // the k pieces of the same pairs: a persistent grid of up to #SMs / k
    // clusters, cluster q walking pairs q, q + clusters, ...  (CTA q*k + j
    // holds piece j).  The pieces meet in the cluster's shared memory; no
    // partials reach global memory and no combine launch follows.
    pp.mode = PLAN_SPLITS;
    pp.num_splits = ck;
    pp.min_blocks = 1;
    pp.force_partial = ck > 1 ? 1 : 0;
    long long clusters = sm / ck;
    if (clusters < 1) clusters = 1;
    if (clusters > pairs) clusters = pairs > 0 ? pairs : 1;
    pp.num_ctas = static_cast<int>(clusters * ck);
    hp.num_slots = 0;
    hp.combine = false;
    hp.use_n_pieces = false;
    hp.cluster_k = ck;
    return hp;
  }
  // the balanced plan keeps per-sequence unit prefix sums in int32
  const bool pre_fits = static_cast<long long>(d->batch) * pair_units(nblk_cap, item_units) <= 0x7fffffffLL;
  if (num_splits == 0 && d->batch <= kMaxSmemB && pre_fits) {
    pp.mode = PLAN_BALANCED;
    // Short sequences with room for k >= 2 CTAs per (batch, KV head) pair
    // (at most 32 blocks per CTA): the grid is k CTAs per pair and items cost
    // no units, so equal lengths give every CTA one item of the same size and
    // every pair k pieces (unequal lengths are still cut into equal ranges).
    // Measured on GB300 against all SMs with X item units: Llama-8B shape
    // 25.80 -> 25.18 us per call, speculative 17.71 -> 17.45 us.  Longer
    // sequences keep every SM: the ragged long-context workload measured
    // 137.5 us on 152 CTAs and 139.4 us on 128.
    const long long per_pair = pairs > 0 ? sm / pairs : 0;
    const bool whole = per_pair >= 2 && nblk_cap <= 32 * per_pair;
    const long long ctas = whole ? per_pair * pairs : sm;
    pp.item_units = whole ? 0 : item_units;
    long long units_cap = pairs * pair_units(nblk_cap, pp.item_units);
    if (units_cap < 1) units_cap = 1;
    pp.num_ctas = static_cast<int>(units_cap < ctas ? units_cap : ctas);
    pp.num_splits = 0;
    pp.min_blocks = 1;
    const int slots = pp.num_ctas < nblk_cap ? pp.num_ctas : nblk_cap;
    hp.num_slots = slots >= 2 ? slots : 0;
    hp.combine = hp.num_slots >= 2;
    hp.use_n_pieces = true;
    return hp;
  }
  pp.mode = PLAN_SPLITS;
  pp.num_splits = num_splits > 0 ? num_splits : auto_splits(pairs, nblk_cap, rows_per_pair, d->head_dim, sm);
  pp.min_blocks = 1;
  pp.force_partial = force_partial ? 1 : 0;
  long long items = pairs * pp.num_splits;
  if (items < 1) items = 1;
  pp.num_ctas = static_cast<int>(items < sm ? items : sm);
  hp.num_slots = (pp.num_splits == 1 && !force_partial) ? 0 : pp.num_splits;
  hp.combine = pp.num_splits > 1 && !force_partial;
  hp.use_n_pieces = false;
  return hp;
}

struct WsLayout {
  size_t o_off, lse_off, np_off, total;
};

WsLayout ws_layout(const gqa_desc_t* d, const HostPlan& hp) {
  WsLayout w{0, 0, 0, 0};
  if (!hp.combine) return w;
  const size_t rows = static_cast<size_t>(d->batch) * d->q_tokens * d->q_heads;
  const size_t slots = static_cast<size_t>(hp.num_slots);
  w.o_off = 0;
  w.lse_off = round_up(slots * rows * d->head_dim * sizeof(float), kWsAlign);
  w.np_off = w.lse_off + round_up(slots * rows * sizeof(float), kWsAlign);
  w.total = w.np_off + round_up(static_cast<size_t>(d->batch) * d->kv_heads * 4 * sizeof(int32_t), kWsAlign);
  return w;
}

// Tensor maps of recent (q, k_cache, v_cache) pointer and shape combinations.
// A map is a pure function of its key (base address, dims, strides, type), so
// an entry stays valid for any buffer that later occupies the same address
// with the same shape; nothing needs invalidating.  Saves the three
// cuTensorMapEncodeTiled calls of an eager decode call that repeats its
// buffers (a decode loop over one KV cache).
struct MapKey {
  const void* q;
  const void* k;
  const void* v;
  int batch, q_tokens, q_heads, kv_heads, head_dim, max_seqlen, in_dtype;
  bool operator==(const MapKey& o) const {
    return q == o.q && k == o.k && v == o.v && batch == o.batch && q_tokens == o.q_tokens &&
           q_heads == o.q_heads && kv_heads == o.kv_heads && head_dim == o.head_dim &&
           max_seqlen == o.max_seqlen && in_dtype == o.in_dtype;
  }
};
struct MapEntry {
  MapKey key;
  bool valid;
  CUtensorMap tm_q, tm_k, tm_v;
};
constexpr int kMapCacheEntries = 64;
std::mutex g_map_mu;
MapEntry g_map_cache[kMapCacheEntries];
unsigned g_map_next = 0;

gqa_status_t encode_maps_uncached(const gqa_desc_t* d, const void* q, const void* k, const void* v,
                                  DecodeParams* p);

gqa_status_t encode_maps(const gqa_desc_t* d, const void* q, const void* k, const void* v, DecodeParams* p) {
  const MapKey key{q, k, v, d->batch, d->q_tokens, d->q_heads, d->kv_heads, d->head_dim, d->max_seqlen,
                   d->in_dtype};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < kMapCacheEntries; ++i) {
      const MapEntry& e = g_map_cache[i];
      if (e.valid && e.key == key) {
        p->tm_q = e.tm_q;
        p->tm_k = e.tm_k;
        p->tm_v = e.tm_v;
        return GQA_OK;
      }
    }
  }
  const gqa_status_t rc = encode_maps_uncached(d, q, k, v, p);
  if (rc != GQA_OK) return rc;
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry& e = g_map_cache[g_map_next++ % kMapCacheEntries];
  e.key = key;
  e.tm_q = p->tm_q;
  e.tm_k = p->tm_k;
  e.tm_v = p->tm_v;
  e.valid = true;
  return GQA_OK;
}

gqa_status_t encode_maps_uncached(const gqa_desc_t* d, const void* q, const void* k, const void* v,
                                  DecodeParams* p) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return GQA_ERR_CUDA;
  const cuuint64_t D = static_cast<cuuint64_t>(d->head_dim);
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const int G = d->q_heads / d->kv_heads;
  const CUtensorMapDataType in_type =
      d->in_dtype == GQA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {
    const cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(d->q_heads), static_cast<cuuint64_t>(d->q_tokens),
                                static_cast<cuuint64_t>(d->batch)};
    const cuuint64_t strides[3] = {D * 2, D * 2 * d->q_heads, D * 2 * d->q_heads * d->q_tokens};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(d->q_tokens), 1};
    if (enc(&p->tm_q, in_type, 4, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GQA_ERR_INVALID_ARG;
  }
  const cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(d->kv_heads), static_cast<cuuint64_t>(d->max_seqlen),
                              static_cast<cuuint64_t>(d->batch)};
  const cuuint64_t strides[3] = {D * 2, D * 2 * d->kv_heads, D * 2 * d->kv_heads * d->max_seqlen};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kBlockN), 1};
  CUtensorMap* maps[2] = {&p->tm_k, &p->tm_v};
  const void* ptrs[2] = {k, v};
  for (int i = 0; i < 2; ++i) {
    if (enc(maps[i], in_type, 4, const_cast<void*>(ptrs[i]), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GQA_ERR_INVALID_ARG;
  }
  return GQA_OK;
}

cudaLaunchAttribute pdl_attr(bool on) {
  cudaLaunchAttribute a;
  std::memset(&a, 0, sizeof a);
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = on ? 1 : 0;
  return a;
}

KernelRef decode_kernel_ref(int head_dim, int np, bool f16, bool cluster) {
  if (head_dim == 64) return cluster ? decode_kernel_ref_64_1(np, f16) : decode_kernel_ref_64_0(np, f16);
  if (head_dim == 256) return cluster ? decode_kernel_ref_256_1(np, f16) : decode_kernel_ref_256_0(np, f16);
  return cluster ? decode_kernel_ref_128_1(np, f16) : decode_kernel_ref_128_0(np, f16);
}

gqa_status_t launch_decode(DeviceState* st, DecodeParams& p, bool in_f16, cudaStream_t s) {
  const int np = p.nq * p.G <= 16 ? 16 : 32;
  const bool cluster = p.cluster_k > 1;
  const KernelRef k = decode_kernel_ref(p.head_dim, np, in_f16, cluster);
  // one attribute bit per instantiation: head_dim x columns x input type x merge mode
  const unsigned bit = (p.head_dim == 64 ? 0u : p.head_dim == 128 ? 1u : 2u) * 8u + (np == 16 ? 0u : 4u) +
                       (in_f16 ? 2u : 0u) + (cluster ? 1u : 0u);
  gqa_status_t rc = ensure_smem_attr(st, bit, k.fn, k.smem_bytes);
  if (rc != GQA_OK) return rc;
  if ((rc = error_word(st, &p.err_word)) != GQA_OK) return rc;
#ifdef GQA_TRACE
  p.trace_buf = g_trace_buf;
#endif
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(p.plan.num_ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(k.threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(k.smem_bytes);
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0] = pdl_attr(!env_flag("GQA_DISABLE_PDL"));
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cluster) {
    std::memset(&attrs[1], 0, sizeof attrs[1]);
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = static_cast<unsigned>(p.cluster_k);
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

gqa_status_t launch_combine(const CombineParams& c, int head_dim, cudaStream_t s) {
  if (c.rows == 0) return GQA_OK;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  const long long rows_per_cta = kCombineThreads / 32;
  const long long grid = (c.rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr = pdl_attr(!env_flag("GQA_DISABLE_PDL"));
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = head_dim == 64    ? cudaLaunchKernelEx(&cfg, gqa_combine_kernel<64>, c)
                  : head_dim == 256 ? cudaLaunchKernelEx(&cfg, gqa_combine_kernel<256>, c)
                                    : cudaLaunchKernelEx(&cfg, gqa_combine_kernel<128>, c);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status_t check_inputs(const void* q, const void* k, const void* v, const int32_t* seqlens) {
  if (q == nullptr || k == nullptr || v == nullptr || seqlens == nullptr) return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(seqlens, 4)) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

// Common front half of gqa_decode_attn / gqa_decode_splitkv.
gqa_status_t prepare_decode(const gqa_desc_t* d, const void* q, const void* k, const void* v,
                            const int32_t* seqlens, const HostPlan& hp, DecodeParams* p) {
  std::memset(p, 0, sizeof *p);
  gqa_status_t rc = encode_maps(d, q, k, v, p);
  if (rc != GQA_OK) return rc;
  p->seqlens = seqlens;
  p->plan = hp.pp;
  p->nq = d->q_tokens;
  p->Hq = d->q_heads;
  p->G = d->q_heads / d->kv_heads;
  p->head_dim = d->head_dim;
  p->out_dtype = d->out_dtype;
  p->causal = d->causal != 0;
  const float scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(d->head_dim));
  p->scale_log2 = scale * 1.4426950408889634f;
  p->lse_bulk = (p->G % 4) == 0;  // LSE rows of G floats: 16-byte multiples
  p->cluster_k = hp.cluster_k > 1 ? hp.cluster_k : 0;
  p->timeout_ns = wait_timeout_ns();
  return GQA_OK;
}

__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on this barrier: the wait must give up on its own.
  const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, nullptr, timeout_ns);
  if (!ok && threadIdx.x == 0) atomicOr(&g_gqa_error_bits, kErrTimeout);
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" {

size_t gqa_decode_workspace_size(const gqa_desc_t* desc, int num_splits) {
  if (check_desc(desc) != GQA_OK || num_splits < 0 || num_splits > GQA_MAX_SPLITS) return 0;
  int dev = 0;
  DeviceState* st = nullptr;
  if (current_device(&dev, &st) != GQA_OK) return 0;
  const HostPlan hp = make_plan(desc, num_splits, st->sm_count, false);
  if (hp.status != GQA_OK) return 0;
  return ws_layout(desc, hp).total;
}

}  // extern "C"

namespace gqa {
namespace {

enum AttnPart : int { ATTN_BOTH = 3, ATTN_SPLIT = 1, ATTN_MERGE = 2 };

gqa_status_t attn_impl(const gqa_desc_t* desc, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* seqlens, void* out, float* lse, int num_splits, void* workspace,
                       size_t workspace_bytes, cudaStream_t s, int parts) {
  gqa_status_t rc = check_desc(desc);
  if (rc != GQA_OK) return rc;
  if (num_splits < 0 || num_splits > GQA_MAX_SPLITS) return GQA_ERR_INVALID_ARG;
  if (desc->batch == 0) return GQA_OK;  // nothing to compute; pointers may be null
  if ((parts & ATTN_SPLIT) && (rc = check_inputs(q, k_cache, v_cache, seqlens)) != GQA_OK) return rc;
  if (out == nullptr || !aligned(out, 16) || (lse != nullptr && !aligned(lse, 4))) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  if ((rc = current_device(&dev, &st)) != GQA_OK) return rc;
  const HostPlan hp = make_plan(desc, num_splits, st->sm_count, false);
  if (hp.status != GQA_OK) return hp.status;
  const WsLayout wl = ws_layout(desc, hp);
  if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total || !aligned(workspace, kWsAlign)))
    return GQA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* o_part = hp.combine ? reinterpret_cast<float*>(ws + wl.o_off) : nullptr;
  float* lse_part = hp.combine ? reinterpret_cast<float*>(ws + wl.lse_off) : nullptr;
  int32_t* n_pieces = (hp.combine && hp.use_n_pieces) ? reinterpret_cast<int32_t*>(ws + wl.np_off) : nullptr;
  if (parts & ATTN_SPLIT) {
    DecodeParams p;
    if ((rc = prepare_decode(desc, q, k_cache, v_cache, seqlens, hp, &p)) != GQA_OK) return rc;
    p.out = out;
    p.lse = lse;
    if (lse != nullptr && !aligned(lse, 16)) p.lse_bulk = 0;
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.n_pieces = n_pieces;
    const size_t rows = static_cast<size_t>(desc->batch) * desc->q_tokens * desc->q_heads;
    p.out_bytes = rows * desc->head_dim * (desc->out_dtype == GQA_DTYPE_FP32 ? 4u : 2u);
    p.lse_bytes = lse != nullptr ? rows * 4u : 0u;
    p.o_part_bytes = hp.combine ? wl.lse_off - wl.o_off : 0u;
    p.lse_part_bytes = hp.combine ? wl.np_off - wl.lse_off : 0u;
    p.n_pieces_bytes = (hp.combine && hp.use_n_pieces) ? wl.total - wl.np_off : 0u;
    if ((rc = launch_decode(st, p, desc->in_dtype == GQA_DTYPE_FP16, s)) != GQA_OK) return rc;
  }
  if (!(parts & ATTN_MERGE) || !hp.combine) return GQA_OK;
  CombineParams c;
  std::memset(&c, 0, sizeof c);
  c.o_part = o_part;
  c.lse_part = lse_part;
  c.n_pieces = n_pieces;
  c.out = out;
  c.lse = lse;
  c.rows = static_cast<long long>(desc->batch) * desc->q_tokens * desc->q_heads;
  c.num_splits = hp.num_slots;
  c.out_dtype = desc->out_dtype;
  c.nq = desc->q_tokens;
  c.Hq = desc->q_heads;
  c.G = desc->q_heads / desc->kv_heads;
  c.kv_heads = desc->kv_heads;
  return launch_combine(c, desc->head_dim, s);
}

}  // namespace
}  // namespace gqa

extern "C" {

gqa_status_t gqa_decode_attn(const gqa_desc_t* desc, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* seqlens, void* out, float* lse, int num_splits, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return attn_impl(desc, q, k_cache, v_cache, seqlens, out, lse, num_splits, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), ATTN_BOTH);
}

gqa_status_t gqa_decode_attn_split(const gqa_desc_t* desc, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* seqlens, void* out, float* lse,
                                   int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_impl(desc, q, k_cache, v_cache, seqlens, out, lse, num_splits, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), ATTN_SPLIT);
}

gqa_status_t gqa_decode_attn_merge(const gqa_desc_t* desc, void* out, float* lse, int num_splits, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return attn_impl(desc, nullptr, nullptr, nullptr, nullptr, out, lse, num_splits, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), ATTN_MERGE);
}

}  // extern "C"

namespace gqa {
namespace {

// Library-owned workspace for gqa_decode_attn_static_workspace.  It lives in
// the module's global memory, so every GPU that loads this library holds
// GQA_STATIC_WORKSPACE_BYTES of it until the process exits.
static __device__ __align__(256) unsigned char g_static_workspace[GQA_STATIC_WORKSPACE_BYTES];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device.  The name of a
// __device__ array in host code is only a host-side stand-in, so the address
// is looked up once per device, with that device current.
gqa_status_t static_workspace_ptr(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return GQA_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

extern "C" {

gqa_status_t gqa_decode_attn_static_workspace(const gqa_desc_t* desc, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* seqlens, void* out, float* lse,
                                              int num_splits, void* stream) {
  gqa_status_t rc = check_desc(desc);
  if (rc != GQA_OK) return rc;
  if (num_splits < 0 || num_splits > GQA_MAX_SPLITS) return GQA_ERR_INVALID_ARG;
  if (desc->batch == 0) return GQA_OK;
  int dev = 0;
  DeviceState* st = nullptr;
  if ((rc = current_device(&dev, &st)) != GQA_OK) return rc;
  const HostPlan hp = make_plan(desc, num_splits, st->sm_count, false);
  if (hp.status != GQA_OK) return hp.status;
  const size_t need = ws_layout(desc, hp).total;
  if (need > GQA_STATIC_WORKSPACE_BYTES) return GQA_ERR_WORKSPACE;  // larger than the static array
  void* ws = nullptr;
  if ((rc = static_workspace_ptr(dev, &ws)) != GQA_OK) return rc;
  return gqa_decode_attn(desc, q, k_cache, v_cache, seqlens, out, lse, num_splits, ws, GQA_STATIC_WORKSPACE_BYTES,
                         stream);
}

gqa_status_t gqa_decode_splitkv(const gqa_desc_t* desc, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* seqlens, int num_splits, float* o_part, float* lse_part,
                                void* stream) {
  gqa_status_t rc = check_desc(desc);
  if (rc != GQA_OK) return rc;
  if (num_splits < 1 || num_splits > GQA_MAX_SPLITS) return GQA_ERR_INVALID_ARG;
  if (desc->batch == 0) return GQA_OK;
  if ((rc = check_inputs(q, k_cache, v_cache, seqlens)) != GQA_OK) return rc;
  // Both partial buffers must be 16-byte aligned: the kernel writes their
  // rows with bulk async copies, which need 16-byte aligned addresses.
  if (o_part == nullptr || lse_part == nullptr || !aligned(o_part, 16) || !aligned(lse_part, 16))
    return GQA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  if ((rc = current_device(&dev, &st)) != GQA_OK) return rc;
  const HostPlan hp = make_plan(desc, num_splits, st->sm_count, true);
  DecodeParams p;
  if ((rc = prepare_decode(desc, q, k_cache, v_cache, seqlens, hp, &p)) != GQA_OK) return rc;
  p.o_part = o_part;
  p.lse_part = lse_part;
  const size_t rows = static_cast<size_t>(desc->batch) * desc->q_tokens * desc->q_heads;
  p.o_part_bytes = static_cast<size_t>(num_splits) * rows * desc->head_dim * 4u;
  p.lse_part_bytes = static_cast<size_t>(num_splits) * rows * 4u;
  return launch_decode(st, p, desc->in_dtype == GQA_DTYPE_FP16, static_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_decode_combine(const float* o_part, const float* lse_part, int num_splits, int64_t rows,
                                int head_dim, void* out, int out_dtype, float* lse, void* stream) {
  if (num_splits < 1 || num_splits > GQA_MAX_SPLITS || rows < 0) return GQA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return GQA_ERR_UNSUPPORTED;
  if (out_dtype != GQA_DTYPE_BF16 && out_dtype != GQA_DTYPE_FP32 && out_dtype != GQA_DTYPE_FP16)
    return GQA_ERR_INVALID_ARG;
  if (rows == 0) return GQA_OK;
  if (o_part == nullptr || lse_part == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(out, 16) || (lse != nullptr && !aligned(lse, 4)))
    return GQA_ERR_INVALID_ARG;
  CombineParams c;
  std::memset(&c, 0, sizeof c);
  c.o_part = o_part;
  c.lse_part = lse_part;
  c.out = out;
  c.lse = lse;
  c.rows = rows;
  c.num_splits = num_splits;
  c.out_dtype = out_dtype;
  c.nq = c.Hq = c.G = c.kv_heads = 1;
  return launch_combine(c, head_dim, static_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_decode_get_error(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpyFromSymbol(&bits, g_gqa_error_bits, sizeof bits) != cudaSuccess) return GQA_ERR_CUDA;
  if (clear && bits != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_gqa_error_bits, &zero, sizeof zero) != cudaSuccess) return GQA_ERR_CUDA;
  }
  if (bits & kErrTimeout) return GQA_ERR_TIMEOUT;
  if (bits & kErrBounds) return GQA_ERR_BOUNDS;
  if (bits & kErrBadSeqlen) return GQA_ERR_BAD_SEQLEN;
  return GQA_OK;
}

const char* gqa_status_string(gqa_status_t status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported shape";
    case GQA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GQA_ERR_CUDA: return "CUDA runtime error";
    case GQA_ERR_TIMEOUT: return "a kernel wait timed out";
    case GQA_ERR_BAD_SEQLEN: return "sequence length out of range (clamped)";
    case GQA_ERR_BOUNDS: return "a write or tile outside its buffer was caught (debug build)";
  }
  return "unknown status";
}

gqa_status_t gqa_decode_plan(const gqa_desc_t* desc, const int32_t* seqlens_host, int num_splits, int sm_count,
                             int* num_ctas, int* plan_mode, int* num_slots, int32_t* items, int64_t max_items,
                             int64_t* num_items) {
  gqa_status_t rc = check_desc(desc);
  if (rc != GQA_OK) return rc;
  if (num_splits < 0 || num_splits > GQA_MAX_SPLITS) return GQA_ERR_INVALID_ARG;
  if (desc->batch > 0 && seqlens_host == nullptr) return GQA_ERR_INVALID_ARG;
  if (sm_count <= 0) {
    int dev = 0;
    DeviceState* st = nullptr;
    if ((rc = current_device(&dev, &st)) != GQA_OK) return rc;
    sm_count = st->sm_count;
  }
  const HostPlan hp = make_plan(desc, num_splits, sm_count, false);
  if (hp.status != GQA_OK) return hp.status;
  if (num_ctas) *num_ctas = hp.pp.num_ctas;
  if (plan_mode) *plan_mode = hp.cluster_k > 1 ? 2 : hp.pp.mode;
  if (num_slots) *num_slots = hp.combine ? hp.num_slots : 0;
  const int B = desc->batch;
  std::vector<int32_t> clamped(static_cast<size_t>(B > 0 ? B : 1)), pre(static_cast<size_t>(B) + 1, 0);
  for (int b = 0; b < B; ++b) {
    clamped[b] = clamp_len(seqlens_host[b], desc->max_seqlen);
    pre[b + 1] = pre[b] + (hp.pp.mode == PLAN_BALANCED ? pair_units(num_blocks(clamped[b]), hp.pp.item_units)
                                                        : num_blocks(clamped[b]));
  }
  int64_t n = 0;
  if (desc->batch > 0) {
    for (int c = 0; c < hp.pp.num_ctas; ++c) {
      WorkIter it;
      it.init(hp.pp, seqlens_host, clamped.data(), pre.data(), c);
      WorkItem w;
      while (it.next(w)) {
        if (items != nullptr && n < max_items) {
          int32_t* r = items + 8 * n;
          r[0] = c; r[1] = w.b; r[2] = w.h; r[3] = w.blk_begin; r[4] = w.blk_end;
          r[5] = w.slot; r[6] = w.first_piece; r[7] = w.n_pieces;
        }
        ++n;
      }
    }
  }
  if (num_items) *num_items = n;
  return GQA_OK;
}

#ifdef GQA_TRACE
// Trace builds only: attaches a device buffer of grid x TR_EVENTS x
// kTraceBlocks uint64 for the decode kernel's event stamps (NULL detaches).
gqa_status_t gqa_trace_attach(void* device_buffer) {
  g_trace_buf = static_cast<unsigned long long*>(device_buffer);  // used by the following launches
  return GQA_OK;
}
#endif

gqa_status_t gqa_decode_selftest_timeout(unsigned int timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return GQA_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * timeout_us);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // extern "C"
