// Split-KV GQA decode kernel for sm_103a (TMA + tcgen05 + TMEM).
//
// One persistent CTA per SM walks the work items of plan.cuh.  Per 128-position
// KV block of one (batch, KV head) pair it computes, with the operands swapped
// so that KV positions fill the MMA M dimension and the query-head group fills
// N ("Building a Faster GQA Decode Kernel for Blackwell SM100", section
// "Starting with the simple pipeline"):
//
//     S^T[128 x N] = K_blk[128 x d] Q^T[d x N]          (TMEM, fp32)
//     P^T          = exp2(S^T * scale*log2e - m)       (online softmax)
//     O^T[d x N]  += V_blk^T[d x 128] P^T[128 x N]     (TMEM, fp32)
//
// N = nq*G padded to 16 or 32; column n is query token n / G, head n % G of
// the group (the PackGQA row order of "Flash Attention 4 - warp-role
// choreography and the edges", section "Edge 2 - GQA").
//
// Warp roles (96 + 128 N/8 threads: 352 for N = 16, 608 for N = 32):
//   warp 0      TMA producer: Q per item, then K/V tiles into an mbarrier ring
//               in the order K0 K1 V0 K2 V1 ... (the page's split-local order),
//               so the score MMA of block i+1 can run while block i's softmax
//               is in flight;
//   warp 1      score-MMA issuer (one thread): QK(i+1) goes into the other of
//               two S slots while block i is in the softmax (the S/P
//               ping-pong of "Optimization diaries: S/P ping-pong for
//               FlashAttention-4 decode"); owns the TMEM allocation;
//   warp 2      value-MMA issuer (one thread), as the KQ / VP MMA warps of
//               the CUTLASS kernel ("Building a Faster GQA Decode Kernel for
//               Blackwell SM100", section "Starting with the simple
//               pipeline");
//   warps 3..   N/8 softmax / correction / epilogue warpgroups of 8 columns
//               each.  A warp reads its 32 TMEM lanes (KV positions) of S^T
//               with 16x256b loads: lane i holds positions i/4 + 8j of two
//               columns.  It releases the S slot as soon as the scores are in
//               registers, masks, votes on whether any column's max moved by
//               more than the rescale threshold (8 in log2 units, "Flash
//               Attention 4 - warp-role choreography and the edges", section
//               "The correction"), and only then reduces the column max and
//               rescales O in TMEM (thread r: row r of O^T).  P^T goes to
//               shared memory, as the K-major B operand of the PV MMA, in one
//               transposed stmatrix per thread; the denominators are summed
//               per lane in registers and reduced once per item.
//
// head_dim 64 uses M = 128 for the PV MMA by stacking the two 64-position
// halves of the block along M: A = [V_lo^T ; V_hi^T] (128 x 64), B =
// [P_lo ; P_hi] (2N x 64).  Lanes 0..63 x columns [0, N) then hold the first
// half's contribution and lanes 64..127 x columns [N, 2N) the second's; the
// cross quadrants are discarded and the epilogue adds the two halves.
//
// head_dim 256 streams each block as two ring tiles of 128 positions x 128
// elements, its d-halves (K lo, K hi, V lo, V hi).  The score MMA accumulates
// S^T over both K halves before it commits, and the value issuer runs one
// M = 128 chain per V half into a TMEM accumulator of its own.  The epilogue
// then writes O rows r and r + 128.
//
// Merging the splits (DecodeParams / plan mode): either each CTA writes fp32
// partials and an LSE per row for the combine kernel, or (CLUSTER) the k
// splits of a pair run as the k CTAs of one thread-block cluster.  In the
// cluster case the CTAs exchange their normalised rows and LSEs through
// distributed shared memory and merge them in fixed split order, with no
// second launch ("Building a Faster GQA Decode Kernel for Blackwell SM100",
// section "Reducing inside a thread block cluster").
//
// Every wait is bounded.  A wait that times out sets the device error word,
// raises a CTA-wide abort flag and the roles leave their loops in step (the
// softmax warps decide uniformly, at their exchange barriers), wait for their
// own copies and MMAs in flight and free TMEM before returning.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "plan.cuh"
#include "sm103_ptx.cuh"

namespace gqa {

enum : unsigned { kErrTimeout = 1u, kErrBadSeqlen = 2u, kErrBounds = 4u };

// Optional per-CTA event trace (compile with -DGQA_TRACE): clock64 stamps of
// each role's per-block steps, written to the buffer the host attaches with
// gqa_trace_attach() (DecodeParams::trace_buf).  Compiled out otherwise.
enum TraceEvent : int {
  TR_START = 0, TR_SETUP = 1,
  TR_PROD_WAIT = 2, TR_PROD_K = 3, TR_PROD_V = 4, TR_PROD_PLAN = 5, TR_PROD_Q = 6, TR_LENS = 7,
  TR_MMA_K = 8, TR_MMA_QK = 9, TR_MMA_P = 10, TR_MMA_V = 11, TR_MMA_PV = 12, TR_ITER = 13, TR_PROD_T0 = 14,
  TR_SM_S = 16, TR_SM_LD = 17, TR_SM_X = 18, TR_SM_PE = 19, TR_SM_PF = 20, TR_SM_E0 = 21, TR_SM_E1 = 22,
  // epilogue of the last item (one softmax thread of warpgroup 0 that holds
  // an output row), in this order from TR_EP_L
  TR_EP_L = 23, TR_EP_PV = 24, TR_EP_O = 25, TR_EP_CW = 26, TR_EP_SENT = 27, TR_EP_FULL = 28,
  TR_EP_MERGED = 29, TR_EP_EXIT = 30,
  TR_END = 31, TR_EVENTS = 32
};
constexpr int kTraceBlocks = 64;
constexpr int kTraceEpStamps = TR_EP_EXIT - TR_EP_L + 2;  // + the merge's compute, written as event 15
constexpr int kTraceEpComputed = kTraceEpStamps - 1;
#ifdef GQA_TRACE
__device__ __forceinline__ void trace_event(unsigned long long* buf, int ev, uint32_t idx) {
  if (buf == nullptr) return;
  const uint32_t i = idx < static_cast<uint32_t>(kTraceBlocks) ? idx : kTraceBlocks - 1;
  buf[(static_cast<size_t>(blockIdx.x) * TR_EVENTS + ev) * kTraceBlocks + i] = clock64();
}
// The buffer address is read once per thread (GQA_TRACE_SETUP) so that an
// event costs a clock read and a store, not a dependent global load.
#define GQA_TRACE_SETUP() unsigned long long* const gqa_trace_buf_ = p.trace_buf
#define GQA_TRACE_EVENT(ev, idx) ::gqa::trace_event(gqa_trace_buf_, (ev), (idx))
#define GQA_TRACE_VALUE(ev, idx, v) \
  do { if (gqa_trace_buf_ != nullptr) gqa_trace_buf_[(static_cast<size_t>(blockIdx.x) * ::gqa::TR_EVENTS + (ev)) * ::gqa::kTraceBlocks + (idx)] = (v); } while (0)
// Stamps kept in shared memory and written at the end (GQA_TRACE_FLUSH): a
// global store of a stamp would otherwise hold up a later release fence.
#define GQA_TRACE_STAMPS(arr, n) __shared__ unsigned long long arr[n]
#define GQA_TRACE_STAMP(arr, i) ((arr)[i] = clock64())
#define GQA_TRACE_FLUSH(arr, n, ev0) \
  do { for (int i_ = 0; i_ < (n); ++i_) GQA_TRACE_VALUE(i_ + 1 < (n) ? (ev0) + i_ : 15, 0, (arr)[i_]); } while (0)
#else
#define GQA_TRACE_SETUP() ((void)0)
#define GQA_TRACE_EVENT(ev, idx) ((void)(idx))  // index evaluated in both builds
#define GQA_TRACE_VALUE(ev, idx, v) ((void)0)
#define GQA_TRACE_STAMPS(arr, n) ((void)0)
#define GQA_TRACE_STAMP(arr, i) ((void)0)
#define GQA_TRACE_FLUSH(arr, n, ev0) ((void)0)
#endif

// output element types (the values of gqa_dtype_t)
constexpr int kOutBF16 = 0, kOutF32 = 1, kOutF16 = 2;

constexpr int kSoftmaxThread0 = 96;  // first thread of the (first) softmax warpgroup
constexpr int kMaxSmemB = 512;       // sequences whose lengths are staged in shared memory
constexpr int kMaxListItems = 128;   // work items of one CTA kept as a list in shared memory
constexpr float kRescaleThreshold = 8.0f;
// -max of a column whose max is still -inf: larger than any scaled score can
// make up for, so a visible score votes for a rescale (which replaces it)
constexpr float kNoMax = 1.2676506e30f;  // 2^100
constexpr uint32_t kTmemCols = 128;
constexpr int kMaxClusterK = 8;  // CTAs of an in-cluster merge: a power of two, the portable cluster size
constexpr uint32_t kSCol0 = 0, kSCol1 = 32, kOCol = 64;

struct DecodeParams {
  CUtensorMap tm_q;  // q [B, nq, Hq, d] bf16 or fp16, box {64, G, nq, 1}
  CUtensorMap tm_k;  // k_cache [B, S_max, Hkv, d] bf16 or fp16, box {64, 1, 128, 1}
  CUtensorMap tm_v;  // v_cache, same
  const int32_t* seqlens;
  void* out;          // [B, nq, Hq, d] bf16, fp16 or fp32
  float* lse;         // [B, nq, Hq] or null
  float* o_part;      // [slots, B*nq*Hq, d]
  float* lse_part;    // [slots, B*nq*Hq]
  int32_t* n_pieces;  // [B*Hkv] (PLAN_BALANCED)
  PlanParams plan;
  int nq, Hq, G, head_dim;
  int out_dtype;      // 0 bf16, 1 fp32, 2 fp16 (gqa_dtype_t); 16-bit outputs have the input type
  int causal;
  float scale_log2;   // softmax scale * log2(e)
  int lse_bulk;       // LSE rows may be written by 16-byte bulk copies (G % 4 == 0, aligned)
  int cluster_k;      // > 1: the CTAs of a k-cluster hold the k pieces of a pair and merge them in
                      // distributed shared memory (fixed splits, k = plan.num_splits)
  unsigned long long timeout_ns;
  unsigned int* err_word;            // the library's device error word (kErrTimeout | kErrBadSeqlen | kErrBounds)
  unsigned long long* trace_buf;     // -DGQA_TRACE builds: [grid][TR_EVENTS][kTraceBlocks] stamps, or null
  // byte extents of the buffers the kernel writes, checked by -DGQA_DEBUG builds
  unsigned long long out_bytes, lse_bytes, o_part_bytes, lse_part_bytes, n_pieces_bytes;
};

template <int HEAD_DIM, int NPAD>
struct DecodeCfg {
  static constexpr int kChunks = HEAD_DIM / 64;            // 128-byte swizzle atoms along d
  // A ring tile holds 128 positions x at most 128 elements of d: head_dim 256
  // streams each K or V block as two d-halves (two tiles), so that the ring
  // keeps 32 KB stages.  S^T accumulates over both K halves; O^T is two
  // M = 128 accumulators, one per V half.
  static constexpr int kTileDim = HEAD_DIM < 128 ? HEAD_DIM : 128;
  static constexpr int kTileChunks = kTileDim / 64;
  static constexpr int kTilesPerBlock = HEAD_DIM / kTileDim;
  static constexpr int kSlotBytes = kBlockN * kTileDim * 2;  // one K or V tile
  static constexpr int kQBytes = kChunks * NPAD * 128;       // one Q buffer
  static constexpr int kPBytes = 2 * NPAD * 128;             // one P buffer (two 64-position atoms)
  // TMEM columns of O: head_dim 64 stacks two position halves, 256 has two d-halves
  static constexpr int kOWidth = HEAD_DIM == 128 ? NPAD : 2 * NPAD;
  static constexpr int kPvN = HEAD_DIM == 64 ? 2 * NPAD : NPAD;  // N of one value MMA
  // Q and output staging buffers: two each (the next item's Q loads, and the
  // previous item's rows leave, while this item runs); one each where two do
  // not fit beside a 4-stage ring (head_dim 256 with 32 columns)
  static constexpr int kBufs = (HEAD_DIM == 256 && NPAD == 32) ? 1 : 2;
  // Softmax warpgroups, 8 columns each: every warpgroup keeps the running
  // max and sums, the O columns and the P rows of its own columns, so that
  // more warps hide the softmax's latencies.  With 32 columns the softmax is
  // the slower side of the pipeline in steady state; with 16 its per-item
  // work (first block, epilogue) still sits on the critical path.  Measured
  // on GB300: four warpgroups beat two of 16 columns, and two beat one of 16.
  // Warps: producer, score-MMA issuer, value-MMA issuer, then 4 * kWGs
  // softmax warps.
  static constexpr int kWGs = NPAD / 8;
  static constexpr int kNC = NPAD / kWGs;  // columns per softmax warpgroup
  static constexpr int kThreads = 96 + 128 * kWGs;
  // fixed part of shared memory after the ring
  static constexpr int kXchgBytes = kWGs * 2 * (4 * 4 + 4 * kNC * 4);
  // head_dim 64 with several warpgroups: scratch for the epilogue's exchange of
  // the stacked half-blocks (one warpgroup uses the P buffers, which the
  // other may already be refilling)
  static constexpr int kXoBytes = (kWGs > 1 && HEAD_DIM == 64) ? NPAD * 64 * 4 : 0;
  static constexpr int kListBytes = 16 + kMaxListItems * static_cast<int>(sizeof(WorkItem));
  static constexpr int kMiscBytes =
      (512 + kXchgBytes + 4 * kMaxSmemB + 4 * (kMaxSmemB + 1) + 64 + kListBytes + 127) / 128 * 128;
  // output staging, two buffers: one item's rows (fp32 worst case), its LSEs
  // (in-cluster merge: those of every CTA of the cluster), its piece count
  static constexpr int kOutBytes = (NPAD * HEAD_DIM * 4 + kMaxClusterK * NPAD * 4 + 16 + 127) / 128 * 128;
  // in-cluster merge: this CTA's merged columns of an item (at most half of
  // d, fp32, per row), then the merged LSEs
  static constexpr int kFinBytes = (NPAD * HEAD_DIM * 2 + NPAD * 4 + 127) / 128 * 128;
  static constexpr int kFixedBytes =
      kBufs * kQBytes + 2 * kPBytes + kMiscBytes + kBufs * kOutBytes + kXoBytes + kFinBytes;
  static constexpr int kSmemBudget = 227 * 1024 - 1024;  // minus alignment slack
  static constexpr int kStagesRaw = (kSmemBudget - kFixedBytes) / kSlotBytes;
  // Four stages (two K, two V blocks) per SM keep enough bytes in flight
  // for the whole GPU (152 x 64-128 KB, about twice the bandwidth-latency
  // product); deeper rings were measured slower: the extra queueing made the
  // per-SM bandwidth less even and the slowest CTA later.
  static constexpr int kStages = kStagesRaw > 4 ? 4 : kStagesRaw;
  // K and V have rings of their own (K: stages [0, kStagesK), V: the rest),
  // each consumed in order by one issuer.  A parity wait on a stage is only
  // sound when the waiter has itself seen the stage's previous phase complete;
  // with one shared ring the previous tile of a stage can belong to the other
  // consumer and still be in flight, and the wait would pass a phase early.
  static constexpr int kStagesK = (kStages + 1) / 2;
  static constexpr int kStagesV = kStages / 2;
  static constexpr int kRingBytes = kStages * kSlotBytes;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kFixedBytes;
  static_assert(kStages >= 4 && kStagesV >= 2, "ring too shallow");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory over budget");
  static_assert(kOWidth <= 64 && NPAD <= 32, "TMEM column plan");
  static_assert(kMiscBytes % 128 == 0 && (kBufs * kQBytes + 2 * kPBytes) % 128 == 0, "staging alignment");
  // K and V rings of whole blocks' tiles
  static_assert(kStagesK % kTilesPerBlock == 0 && kStagesV % kTilesPerBlock == 0, "ring of whole blocks");
};

namespace detail {

// Softmax thread layout: with 16x256b TMEM loads, lane i of a warp holds
// the scores of positions i / 4 + 8 j (j = 0..3) of the warp's 32 TMEM lanes
// for two columns, 2 (i % 4) and 2 (i % 4) + 1 of its warpgroup's eight.
// Reduces a and b over the 8 lanes that hold the same two columns; every
// one of them ends with the result.
template <bool IS_MAX>
__device__ __forceinline__ void quad_reduce(float& a, float& b) {
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    const float ra = __shfl_xor_sync(0xffffffffu, a, off);
    const float rb = __shfl_xor_sync(0xffffffffu, b, off);
    a = IS_MAX ? fmaxf(a, ra) : a + ra;
    b = IS_MAX ? fmaxf(b, rb) : b + rb;
  }
}

__device__ __forceinline__ void set_error(unsigned int* word, unsigned bits, volatile int* abort_flag) {
  atomicOr(word, bits);
  if (abort_flag != nullptr) *abort_flag = 1;
}

// -DGQA_DEBUG builds: whether the write [dst, dst + len) lies inside the
// buffer [base, base + bytes); a write that would not is skipped by the
// caller and recorded in the error word (kErrBounds).  Other builds: true.
__device__ __forceinline__ bool write_ok(unsigned int* word, const void* base, unsigned long long bytes,
                                         const void* dst, unsigned long long len) {
#ifdef GQA_DEBUG
  const unsigned long long b = reinterpret_cast<unsigned long long>(base);
  const unsigned long long d = reinterpret_cast<unsigned long long>(dst);
  if (base == nullptr || d < b || d + len > b + bytes) {
    atomicOr(word, kErrBounds);
    return false;
  }
#else
  (void)word; (void)base; (void)bytes; (void)dst; (void)len;
#endif
  return true;
}

// -DGQA_DEBUG builds: records (kErrBounds) a TMA tile origin outside its
// tensor.  The load is still issued -- its barrier expects the bytes, and a
// tiled load outside the tensor reads the fill value, it does not fault.
__device__ __forceinline__ void check_coord(unsigned int* word, bool ok) {
#ifdef GQA_DEBUG
  if (!ok) atomicOr(word, kErrBounds);
#else
  (void)word; (void)ok;
#endif
}

}  // namespace detail

// Work items of one CTA: read from the shared-memory list the producer warp
// built, or (list overflow) walked with the plan iterator.
struct ItemSource {
  const WorkItem* list;
  int count, k;
  WorkIter iter;
  __device__ __forceinline__ void init(const int32_t* hdr, const WorkItem* items, const PlanParams& plan,
                                       const int32_t* raw, const int32_t* clamped, const int32_t* pre) {
    list = items;
    count = hdr[0];
    k = 0;
    if (count < 0) iter.init(plan, raw, clamped, pre, blockIdx.x);
  }
  __device__ __forceinline__ bool next(WorkItem& it) {
    if (count >= 0) {
      if (k >= count) return false;
      it = list[k++];
      return true;
    }
    return iter.next(it);
  }
  // Whether next() would return another item (the walk is not advanced).
  __device__ __forceinline__ bool has_next() const {
    if (count >= 0) return k < count;
    WorkIter copy = iter;
    WorkItem w;
    return copy.next(w);
  }
};

// IN_F16: q, k, v (and P) are fp16; otherwise bf16.  CLUSTER: the launch
// is a grid of clusters of p.cluster_k CTAs that merge their split partials
// in distributed shared memory.  A compile-time choice: the merge's code,
// present but unused, measurably slows the other plans' softmax loop (1.3 us
// per call on the 32-column speculative shape).
template <int HEAD_DIM, int NPAD, bool IN_F16, bool CLUSTER>
__global__ void __launch_bounds__(DecodeCfg<HEAD_DIM, NPAD>::kThreads, 1)
gqa_decode_kernel(const __grid_constant__ DecodeParams p) {
  using Cfg = DecodeCfg<HEAD_DIM, NPAD>;
  constexpr int NS = Cfg::kStages;
  constexpr uint32_t NSK = Cfg::kStagesK, NSV = Cfg::kStagesV;  // K ring, then V ring
  constexpr int KCH = Cfg::kChunks;
  constexpr int kThreads = Cfg::kThreads;
  constexpr int NWG = Cfg::kWGs;  // softmax warpgroups
  constexpr int NC = Cfg::kNC;    // columns per softmax warpgroup
  constexpr int CW = NC < 16 ? NC : 16;  // columns per TMEM load
  static_assert(NC == 8, "softmax lane layout: eight columns per warpgroup");
  constexpr int kLogD = HEAD_DIM == 64 ? 6 : (HEAD_DIM == 128 ? 7 : 8);
  static_assert((1 << kLogD) == HEAD_DIM, "head_dim 64, 128 or 256");
  GQA_TRACE_SETUP();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  constexpr uint32_t NB = Cfg::kBufs;                    // Q / output staging buffers
  constexpr int TPB = Cfg::kTilesPerBlock;               // ring tiles per K or V block
  constexpr int TCH = Cfg::kTileChunks;                  // 64-element chunks per tile
  uint8_t* qbuf = ring + Cfg::kRingBytes;                // NB x kQBytes
  uint8_t* pbuf = qbuf + NB * Cfg::kQBytes;              // 2 x kPBytes
  uint8_t* misc = pbuf + 2 * Cfg::kPBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(misc);     // 64 barrier words max
  // per softmax warpgroup: flags [2][4], then values [2][4][NC]
  auto xflags_of = [&](int w) { return reinterpret_cast<uint32_t*>(misc + 512 + w * (Cfg::kXchgBytes / NWG)); };
  auto xvals_of = [&](int w) { return reinterpret_cast<float*>(misc + 512 + w * (Cfg::kXchgBytes / NWG) + 32); };
  int32_t* s_len = reinterpret_cast<int32_t*>(misc + 512 + Cfg::kXchgBytes);  // [kMaxSmemB]
  int32_t* s_pre = s_len + kMaxSmemB;                                   // [kMaxSmemB + 1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_pre + kMaxSmemB + 1);
  // work-item list: [0] count (-1: too many, walk the iterator)
  int32_t* list_hdr = reinterpret_cast<int32_t*>(misc + 512 + Cfg::kXchgBytes + 4 * kMaxSmemB + 4 * (kMaxSmemB + 1) + 64);
  WorkItem* list_items = reinterpret_cast<WorkItem*>(list_hdr + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // output staging buffer ob: rows, then 32 LSEs, then the piece count
  auto obuf_of = [&](int ob) -> uint8_t* { return misc + Cfg::kMiscBytes + ob * Cfg::kOutBytes; };
  auto lse_of = [&](int ob) -> float* { return reinterpret_cast<float*>(obuf_of(ob) + NPAD * HEAD_DIM * 4); };
  auto np_of = [&](int ob) -> int32_t* { return reinterpret_cast<int32_t*>(lse_of(ob) + kMaxClusterK * NPAD); };
  float* xo_buf = reinterpret_cast<float*>(obuf_of(0) + NB * Cfg::kOutBytes);  // kXoBytes
  uint8_t* fin_buf = obuf_of(0) + NB * Cfg::kOutBytes + Cfg::kXoBytes;         // kFinBytes
  constexpr bool cluster_merge = CLUSTER;

  // barrier indices
  const uint32_t bar_base = ptx::smem_u32(bar);
  auto BAR = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
  const int RING_FULL = 0, RING_EMPTY = NS, Q_FULL = 2 * NS, Q_EMPTY = 2 * NS + 2,
            S_FULL = 2 * NS + 4, S_EMPTY = 2 * NS + 6, P_FULL = 2 * NS + 8, P_EMPTY = 2 * NS + 10,
            DRAIN = 2 * NS + 12;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PlanParams plan = p.plan;  // by value: iterators read it from registers
  const int B = plan.batch;
  const bool lens_in_smem = B <= kMaxSmemB;

  // ---------------------------------------------------------------- set-up
  // Right after the grid dependency the producer warp finds its first item
  // and starts streaming, walking the plan's iterator itself: with the
  // balanced plan after staging the clamped lengths and their unit prefix
  // sums (PRE_READY), which that plan's items need; with split items straight
  // from its sequence's length in global memory, while warp 2 stages the
  // lengths.  Warp 2 expands the same plan into the shared item list the
  // other roles read (PLAN_READY), and the rest allocate TMEM and zero the
  // padding of the MMA operand buffers.
  const int PLAN_READY = DRAIN + 2, OUT_FULL = DRAIN + 3, OUT_EMPTY = DRAIN + 5, PRE_READY = DRAIN + 7;
  // in-cluster merge, per softmax warpgroup and staging buffer: the k CTAs'
  // pieces of this CTA's columns have landed here (PEER_FULL, transaction
  // bytes) / every CTA has merged what this CTA sent it (PEER_EMPTY)
  const int PEER_FULL = DRAIN + 8, PEER_EMPTY = DRAIN + 8 + 2 * NWG;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      ptx::mbar_init(BAR(RING_FULL + i), 1);
      ptx::mbar_init(BAR(RING_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(Q_FULL + i), 1);
      ptx::mbar_init(BAR(Q_EMPTY + i), 1);
      ptx::mbar_init(BAR(S_FULL + i), 1);
      ptx::mbar_init(BAR(S_EMPTY + i), 4 * NWG);  // one arrival per softmax warp
      ptx::mbar_init(BAR(P_FULL + i), 4 * NWG);
      ptx::mbar_init(BAR(P_EMPTY + i), 1);
    }
    ptx::mbar_init(BAR(DRAIN), 1);
    ptx::mbar_init(BAR(DRAIN + 1), 1);
    ptx::mbar_init(BAR(PLAN_READY), 1);
    ptx::mbar_init(BAR(PRE_READY), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(OUT_FULL + i), NWG);  // each warpgroup's staging done
      ptx::mbar_init(BAR(OUT_EMPTY + i), 1);
    }
    if (cluster_merge) {
      for (int i = 0; i < 2 * NWG; ++i) {
        ptx::mbar_init(BAR(PEER_FULL + i), 1u);  // the local expect-tx arrival; the bytes come from st.async
        // one arrival per warp of the warpgroup in every CTA of the cluster
        ptx::mbar_init(BAR(PEER_EMPTY + i), 4u * static_cast<uint32_t>(p.cluster_k));
      }
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
    ptx::prefetch_tensormap(&p.tm_v);
  }
#ifdef GQA_TRACE
  __shared__ unsigned int trace_warps_done;  // warps that reached the teardown barrier
  if (threadIdx.x == 0) trace_warps_done = 0;
#endif
  // every warp reaches the CTA barriers converged (one arrival per warp)
  __syncwarp();
  __syncthreads();  // barriers initialised
  // The other CTAs of the cluster arrive on this CTA's barriers: all of them
  // must be initialised first.  Every thread arrives on the cluster's
  // hardware barrier here, after straight-line code (the cluster's CTAs are
  // scheduled together); a thread waits on it only before its first remote
  // arrival, or at teardown, by when the others have long arrived.
  if (cluster_merge) ptx::cluster_arrive();
  bool cluster_waited = !cluster_merge;

  // This CTA's work items, 32 candidates at a time (one per lane), written to
  // the shared list by the 32 lanes of one warp.  Owned items form a
  // contiguous run of candidates (pairs from the first one at or after this
  // CTA's first unit; split items c, c + C, ...).
  // Clamped lengths (flagging raw lengths outside [0, S_max]) and, for the
  // balanced plan, the exclusive prefix sums of their pairs' units, staged by
  // the 32 lanes of one warp.
  auto stage_lengths = [&](int lane) {
    if (lens_in_smem) {
      for (int i = lane; i < B; i += 32) {
        const int raw = p.seqlens[i];
        const int L = clamp_len(raw, plan.max_seqlen);
        if (raw != L) detail::set_error(p.err_word, kErrBadSeqlen, nullptr);
        s_len[i] = L;
      }
      __syncwarp();
      if (plan.mode == PLAN_BALANCED) {
        int run = 0;
        for (int base = 0; base < B; base += 32) {
          const int i = base + lane;
          const int nb = i < B ? pair_units(num_blocks(s_len[i]), plan.item_units) : 0;
          int incl = nb;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          if (i < B) s_pre[i] = run + incl - nb;
          run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_pre[B] = run;
      }
    }
    __threadfence_block();
    __syncwarp();
  };

  auto build_list = [&](int lane) {
    WorkIter base_it;
    base_it.init_warp(plan, lens_in_smem ? s_len : p.seqlens, s_len, s_pre, blockIdx.x, lane);
    const bool balanced = plan.mode == PLAN_BALANCED;
    long long p0 = 0, total = 0;
    if (balanced) {
      p0 = static_cast<long long>(base_it.bal.b) * plan.kv_heads + base_it.bal.h;
      total = static_cast<long long>(B) * plan.kv_heads;
    } else {
      total = static_cast<long long>(B) * plan.kv_heads * plan.num_splits;
    }
    int count = 0;
    for (int chunk = 0;; chunk += 32) {
      WorkItem w;
      bool owned = false;
      if (balanced) {
        const long long pr = p0 + chunk + lane;
        if (pr < total && base_it.bal.b < B) {
          BalancedIter bi = base_it.bal;
          bi.b = static_cast<int>(pr / plan.kv_heads);
          bi.h = static_cast<int>(pr - static_cast<long long>(bi.b) * plan.kv_heads);
          // next() returns the first owned pair at or after this one: this
          // candidate is owned iff it returns the candidate itself
          owned = bi.next(w) && (static_cast<long long>(w.b) * plan.kv_heads + w.h == pr);
        }
      } else {
        const long long wi = blockIdx.x + static_cast<long long>(chunk + lane) * plan.num_ctas;
        if (wi < total) {
          SplitIter si = base_it.s;
          si.w = wi;
          owned = si.next(w);
        }
      }
      const unsigned mask = __ballot_sync(0xffffffffu, owned);
      const int run = (~mask == 0u) ? 32 : __ffs(~mask) - 1;  // leading owned candidates
      if (owned && lane < run && count + lane < kMaxListItems) list_items[count + lane] = w;
      count += run;
      if (run < 32) break;
    }
    if (lane == 0) list_hdr[0] = count <= kMaxListItems ? count : -1;
    __threadfence_block();
  };

  uint32_t tmem_base = 0;
  WorkIter prod_it;  // the producer's own walk over the plan (warp 0)
  if (warp == 0) {
    // Warm L2 with the lengths while the previous kernel finishes: a prefetch
    // returns no data, so it cannot observe a value that kernel still writes.
    if (lens_in_smem && lane * 32 < B) ptx::prefetch_l2(p.seqlens + lane * 32);
    // Inputs may be produced by the previous kernel in the stream.
    ptx::griddep_wait();
    if (lane == 0) GQA_TRACE_EVENT(TR_START, 0);
    if (plan.mode == PLAN_BALANCED) {
      stage_lengths(lane);
      if (lane == 0) GQA_TRACE_EVENT(TR_LENS, 0);
      if (lane == 0) ptx::mbar_arrive(BAR(PRE_READY));  // lengths and prefix sums staged
      prod_it.init_warp(plan, lens_in_smem ? s_len : p.seqlens, s_len, s_pre, blockIdx.x, lane);
    } else {
      // split items: each reads its raw length (clamped the same way)
      prod_it.init_warp(plan, p.seqlens, s_len, s_pre, blockIdx.x, lane);
    }
    if (lane == 0) GQA_TRACE_EVENT(TR_ITER, 0);
  } else {
    if (NPAD == 16 && threadIdx.x == kSoftmaxThread0) {
      // This CTA's first tiles are prefetched into L2 before the grid
      // dependency (while the previous launch finishes) and while the
      // producer builds the plan, guessed as if every sequence had max_seqlen
      // positions (a wrong guess costs a few tiles of bandwidth).  A prefetch
      // returns no data, so it cannot observe a value the previous launch
      // still writes.  Measured on GB300: 0.2-1.3 us per call faster for the
      // stream-bound 16-column kernels; the softmax-bound 32-column kernels
      // gain nothing from earlier first tiles and lost 0.2 us to the extra TMA
      // work.
      const int nblk = num_blocks(plan.max_seqlen);
      const int H = plan.kv_heads;
      const long long pairs = static_cast<long long>(B) * H;
      long long pair = -1;
      int blk = 0;
      if (plan.mode == PLAN_BALANCED) {
        const long long vl = pair_units(nblk, plan.item_units);
        const long long U = pairs * vl;
        const long long C = U < plan.num_ctas ? U : plan.num_ctas;
        if (U > 0 && blockIdx.x < C) {
          const long long lo = muldiv(blockIdx.x, U, C);
          pair = div_nonneg(lo, vl);
          const long long off = lo - pair * vl - plan.item_units;
          blk = off > 0 ? static_cast<int>(off) : 0;
        }
      } else if (blockIdx.x < pairs * plan.num_splits) {
        const int S = plan.num_splits;
        pair = div_nonneg(blockIdx.x, S);
        const int s = static_cast<int>(blockIdx.x - pair * S);
        int splits = (nblk + plan.min_blocks - 1) / plan.min_blocks;
        splits = splits < 1 ? 1 : (splits > S ? S : splits);
        blk = s < splits ? static_cast<int>(muldiv(s, nblk, splits)) : nblk;
      }
      if (pair >= 0 && pair < pairs && blk < nblk) {
        const int b = static_cast<int>(div_nonneg(pair, H));
        const int h = static_cast<int>(pair - static_cast<long long>(b) * H);
#pragma unroll
        for (int kc = 0; kc < KCH; ++kc) {
          ptx::tma_prefetch_l2_4d(&p.tm_q, kc * 64, h * p.G, 0, b);
          ptx::tma_prefetch_l2_4d(&p.tm_k, kc * 64, h, blk * kBlockN, b);
          ptx::tma_prefetch_l2_4d(&p.tm_v, kc * 64, h, blk * kBlockN, b);
          if (blk + 1 < nblk) {
            ptx::tma_prefetch_l2_4d(&p.tm_k, kc * 64, h, (blk + 1) * kBlockN, b);
            ptx::tma_prefetch_l2_4d(&p.tm_v, kc * 64, h, (blk + 1) * kBlockN, b);
          }
          if (blk + 2 < nblk) {
            ptx::tma_prefetch_l2_4d(&p.tm_v, kc * 64, h, (blk + 2) * kBlockN, b);
            ptx::tma_prefetch_l2_4d(&p.tm_k, kc * 64, h, (blk + 2) * kBlockN, b);
          }
          if (blk + 3 < nblk) ptx::tma_prefetch_l2_4d(&p.tm_k, kc * 64, h, (blk + 3) * kBlockN, b);
        }
      }
    }
    if (warp == 1) {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish();
    }
    // Padding rows of Q (beyond nq*G) and both P buffers start at zero; TMA
    // never writes them.
    const int nv = p.nq * p.G;
    const int tid = threadIdx.x - 32;
    for (int i = tid; i < static_cast<int>(NB) * KCH * NPAD; i += kThreads - 32) {
      const int row = i % NPAD;
      if (row < nv) continue;
      uint4* dst = reinterpret_cast<uint4*>(qbuf + (i / NPAD) * NPAD * 128 + row * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    }
    uint4* pz = reinterpret_cast<uint4*>(pbuf);
    for (int i = tid; i < 2 * Cfg::kPBytes / 16; i += kThreads - 32) pz[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    // Outputs and workspace may still be read by the previous kernel.
    ptx::griddep_wait();
    if (warp == 2) {
      bool staged = true;
      if (plan.mode == PLAN_BALANCED) staged = ptx::mbar_wait_bounded(BAR(PRE_READY), 0, abort_flag, p.timeout_ns);
      else stage_lengths(lane);
      if (staged) {
        build_list(lane);
      } else {
        detail::set_error(p.err_word, kErrTimeout, abort_flag);
        if (lane == 0) list_hdr[0] = 0;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(BAR(PLAN_READY));
    }
    if (!ptx::mbar_wait_bounded(BAR(PLAN_READY), 0, abort_flag, p.timeout_ns))
      detail::set_error(p.err_word, kErrTimeout, abort_flag);
    ptx::tc_fence_before();
    ptx::named_barrier_sync(2, kThreads - 32);
    ptx::tc_fence_after();
    tmem_base = *tmem_slot;
    if (threadIdx.x == 32) GQA_TRACE_EVENT(TR_SETUP, 0);
  }
  // Uniform for warps 1..6: written (on a failed plan wait) before barrier 2.
  const bool plan_ok = (warp == 0) || (*abort_flag == 0);
  const int32_t* lens_raw = lens_in_smem ? s_len : p.seqlens;

  // Who issues an item's output copies.  Issuing a bulk copy can wait behind
  // the SM's queued TMA loads for hundreds of cycles.  With several softmax
  // warpgroups (32 columns) the softmax is the bottleneck, and the value-MMA
  // thread (idle while the softmax finishes an item) issues them once every
  // warpgroup has staged its columns.  With one warpgroup (16 columns) the KV
  // stream is the bottleneck and the first softmax thread issues them itself:
  // measured on GB300, that build's softmax loop runs faster.
  constexpr bool kPvStores = (NWG > 1);

  // Writes item wi's rows from staging buffer ob with bulk copies: nq copies
  // of G contiguous rows (the G query heads of one token) for O, the same for
  // the LSEs and, for the first piece of a balanced-plan pair, its piece
  // count.
  auto store_item = [&](const WorkItem& wi, int ob) {
    const int rows_total = plan.batch * p.nq * p.Hq;
    const long long pair_idx = static_cast<long long>(wi.b) * plan.kv_heads + wi.h;
    const bool with_o = wi.blk_begin < wi.blk_end;  // an empty split publishes only lse = -inf
    const bool final_out = wi.slot < 0;
    const uint32_t esz = (final_out && p.out_dtype != kOutF32) ? 2u : 4u;
    const uint32_t row_bytes = static_cast<uint32_t>(p.G) * HEAD_DIM * esz;
    const float* lse_st = lse_of(ob);
    for (int t = 0; t < p.nq; ++t) {
      const long long row0 = (static_cast<long long>(wi.b) * p.nq + t) * p.Hq + static_cast<long long>(wi.h) * p.G;
      if (final_out || with_o) {
        uint8_t* dst = final_out
            ? static_cast<uint8_t*>(p.out) + row0 * HEAD_DIM * esz
            : reinterpret_cast<uint8_t*>(p.o_part + (static_cast<long long>(wi.slot) * rows_total + row0) * HEAD_DIM);
        if (detail::write_ok(p.err_word, final_out ? p.out : static_cast<void*>(p.o_part),
                             final_out ? p.out_bytes : p.o_part_bytes, dst, row_bytes))
          ptx::bulk_store(dst, ptx::smem_u32(obuf_of(ob) + static_cast<uint32_t>(t) * row_bytes), row_bytes);
      }
      float* lse_dst = final_out ? (p.lse != nullptr ? p.lse + row0 : nullptr)
                                 : p.lse_part + static_cast<long long>(wi.slot) * rows_total + row0;
      if (lse_dst != nullptr &&
          detail::write_ok(p.err_word, final_out ? p.lse : p.lse_part, final_out ? p.lse_bytes : p.lse_part_bytes,
                           lse_dst, static_cast<unsigned long long>(p.G) * 4u)) {
        if (p.lse_bulk) {
          ptx::bulk_store(lse_dst, ptx::smem_u32(lse_st + t * p.G), static_cast<uint32_t>(p.G) * 4u);
        } else {
          for (int g2 = 0; g2 < p.G; ++g2) lse_dst[g2] = lse_st[t * p.G + g2];
        }
      }
    }
    if (wi.first_piece && p.n_pieces != nullptr &&
        detail::write_ok(p.err_word, p.n_pieces, p.n_pieces_bytes, p.n_pieces + pair_idx * 4, 16u)) {
      np_of(ob)[0] = wi.n_pieces;
      ptx::fence_proxy_async_smem();
      ptx::bulk_store(p.n_pieces + pair_idx * 4, ptx::smem_u32(np_of(ob)), 16u);
    }
    ptx::bulk_commit();
  };

  // =============================================================== producer
  if (!plan_ok) {
    // the plan never arrived: nothing was issued, go straight to teardown
  } else if (warp == 0) {
    if (lane == 0) {
      GQA_TRACE_EVENT(TR_PROD_T0, 0);
      const uint64_t policy = ptx::l2_policy_evict_first();
      uint32_t tk = 0, tv = 0;  // K / V tiles issued into their rings
      int kq = 0;       // non-empty items
      bool have_prev = false, ok = true;
      int pb = 0, ph = 0, pblk = 0;
      // tile `half` of block blk: d elements [half * kTileDim, (half + 1) * kTileDim)
      auto load_tile = [&](bool is_v, int b, int h, int blk, int half) -> bool {
        const uint32_t n = is_v ? tv : tk;
        const uint32_t stage = is_v ? NSK + n % NSV : n % NSK;
        const uint32_t phase = (n / (is_v ? NSV : NSK)) & 1u;
        if (!is_v) GQA_TRACE_EVENT(TR_PROD_WAIT, tk);
        // the first pass over a ring needs no wait: a fresh barrier's
        // preceding phase counts as complete
        if (n >= (is_v ? NSV : NSK) &&
            !ptx::mbar_wait_bounded(BAR(RING_EMPTY + stage), phase ^ 1u, abort_flag, p.timeout_ns))
          return false;
        ptx::mbar_arrive_expect_tx(BAR(RING_FULL + stage), Cfg::kSlotBytes);
        detail::check_coord(p.err_word, b >= 0 && b < plan.batch && h >= 0 && h < plan.kv_heads && blk >= 0 &&
                                            blk * kBlockN < plan.max_seqlen && half >= 0 && half < TPB);
        uint8_t* dst = ring + stage * Cfg::kSlotBytes;
        const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
#pragma unroll
        for (int kc = 0; kc < TCH; ++kc)
          ptx::tma_load_4d_hint(ptx::smem_u32(dst + kc * 16384), map, BAR(RING_FULL + stage),
                                (half * TCH + kc) * 64, h, blk * kBlockN, b, policy);
        if (is_v) {
          GQA_TRACE_EVENT(TR_PROD_V, tv);
          ++tv;
        } else {
          GQA_TRACE_EVENT(TR_PROD_K, tk);
          ++tk;
        }
        return true;
      };
      WorkItem it;
      while (ok && prod_it.next(it)) {
        if (it.blk_begin >= it.blk_end) continue;
        GQA_TRACE_EVENT(TR_PROD_PLAN, static_cast<uint32_t>(kq));
        const int qb = static_cast<int>(static_cast<uint32_t>(kq) % NB);
        if (kq >= static_cast<int>(NB) &&
            !ptx::mbar_wait_bounded(BAR(Q_EMPTY + qb), ((static_cast<uint32_t>(kq) / NB) & 1u) ^ 1u, abort_flag,
                                    p.timeout_ns)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(BAR(Q_FULL + qb), KCH * p.nq * p.G * 128);
        detail::check_coord(p.err_word, it.b >= 0 && it.b < plan.batch && it.h >= 0 && (it.h + 1) * p.G <= p.Hq);
#pragma unroll
        for (int kc = 0; kc < KCH; ++kc)
          ptx::tma_load_4d(ptx::smem_u32(qbuf + qb * Cfg::kQBytes + kc * NPAD * 128), &p.tm_q,
                           BAR(Q_FULL + qb), kc * 64, it.h * p.G, 0, it.b);
        GQA_TRACE_EVENT(TR_PROD_Q, static_cast<uint32_t>(kq));
        ++kq;
        for (int blk = it.blk_begin; blk < it.blk_end && ok; ++blk) {
          for (int hf = 0; hf < TPB && ok; ++hf) ok = load_tile(false, it.b, it.h, blk, hf);
          for (int hf = 0; hf < TPB && ok && have_prev; ++hf) ok = load_tile(true, pb, ph, pblk, hf);
          pb = it.b; ph = it.h; pblk = blk; have_prev = true;
        }
      }
      for (int hf = 0; hf < TPB && ok && have_prev; ++hf) ok = load_tile(true, pb, ph, pblk, hf);
      if (!ok) {
        detail::set_error(p.err_word, kErrTimeout, abort_flag);
        // let the copies already issued land before the CTA exits
        for (uint32_t u = tk > NSK ? tk - NSK : 0u; u < tk; ++u)
          ptx::mbar_wait_bounded(BAR(RING_FULL + u % NSK), (u / NSK) & 1u, nullptr, p.timeout_ns);
        for (uint32_t u = tv > NSV ? tv - NSV : 0u; u < tv; ++u)
          ptx::mbar_wait_bounded(BAR(RING_FULL + NSK + u % NSV), (u / NSV) & 1u, nullptr, p.timeout_ns);
        for (int k = (kq > static_cast<int>(NB) ? kq - static_cast<int>(NB) : 0); k < kq; ++k)
          ptx::mbar_wait_bounded(BAR(Q_FULL + static_cast<int>(static_cast<uint32_t>(k) % NB)),
                                 (static_cast<uint32_t>(k) / NB) & 1u, nullptr, p.timeout_ns);
      }
    }
    __syncwarp();
  }
  // ======================================================= MMA issuers
  // Two single-thread issuers: warp 1 the score MMAs (QK), warp 2 the value
  // MMAs (PV).  One issuing thread alone spends ~60 cycles per tcgen05.mma
  // at these shapes; splitting the two kinds lets their issue overlap.  Each
  // consumes its own ring in order (K of block g is K-ring tile g, V of block
  // g is V-ring tile g; the producer issues K0 K1 V0 K2 V1 ...) and releases
  // the stages with its own commits.
  else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      const bool is_qk = (warp == 1);
      const uint64_t ring_desc = ptx::smem_desc_sw128(ptx::smem_u32(ring), 16, 1024);
      const uint64_t q_desc = ptx::smem_desc_sw128(ptx::smem_u32(qbuf), 16, 1024);
      const uint64_t v_desc =
          ptx::smem_desc_sw128(ptx::smem_u32(ring), Cfg::kTileDim == 128 ? 16384 : 8192, 1024);
      const uint64_t p_desc = ptx::smem_desc_sw128(ptx::smem_u32(pbuf), 16, 1024);
      constexpr uint32_t kSlot16 = Cfg::kSlotBytes >> 4;  // descriptor units (16 B)
      bool ok = true;
      uint32_t g = 0;  // blocks of this CTA
      int kq = 0;      // non-empty items
      ItemSource iter;
      iter.init(list_hdr, list_items, plan, lens_raw, s_len, s_pre);
      WorkItem it;
      if (is_qk) {
        constexpr uint32_t idesc_qk = ptx::idesc_f16_f32(128, NPAD, 0, 0, !IN_F16);
        while (ok && iter.next(it)) {
          if (it.blk_begin >= it.blk_end) continue;
          const int qb = static_cast<int>(static_cast<uint32_t>(kq) % NB);
          if (!ptx::mbar_wait_bounded(BAR(Q_FULL + qb), (static_cast<uint32_t>(kq) / NB) & 1u, abort_flag,
                                      p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint64_t qd = q_desc + static_cast<uint64_t>(qb * (Cfg::kQBytes >> 4));
          for (int blk = it.blk_begin; blk < it.blk_end; ++blk, ++g) {
            const uint32_t sl = g & 1u;
            ok = g < 2 || ptx::mbar_wait_bounded(BAR(S_EMPTY + sl), ((g >> 1) & 1u) ^ 1u, abort_flag, p.timeout_ns);
            if (!ok) break;
            const uint32_t d_tmem = tmem_base + (sl ? kSCol1 : kSCol0);
            // S^T = K Q^T over d, one ring tile (at most 128 elements of d) at a time
#pragma unroll
            for (int hf = 0; hf < TPB; ++hf) {
              const uint32_t u = g * TPB + static_cast<uint32_t>(hf);  // K-ring tile
              const uint32_t stage = u % NSK;
              ok = ptx::mbar_wait_bounded(BAR(RING_FULL + stage), (u / NSK) & 1u, abort_flag, p.timeout_ns);
              if (!ok) break;
              if (hf == 0) GQA_TRACE_EVENT(TR_MMA_K, g);
              ptx::tc_fence_after();
              const uint64_t kd = ring_desc + static_cast<uint64_t>(stage * kSlot16);
#pragma unroll
              for (int kk = 0; kk < Cfg::kTileDim / 16; ++kk) {
                const int k = hf * (Cfg::kTileDim / 16) + kk;  // 16-element step of d
                const uint32_t off_a = static_cast<uint32_t>((kk >> 2) * (16384 >> 4) + (kk & 3) * 2);
                const uint32_t off_b = static_cast<uint32_t>((k >> 2) * (NPAD * 128 >> 4) + (k & 3) * 2);
                ptx::mma_f16_ss(d_tmem, kd + off_a, qd + off_b, idesc_qk, k > 0 ? 1u : 0u);
              }
              if (hf == TPB - 1) ptx::mma_commit(BAR(S_FULL + sl));
              ptx::mma_commit(BAR(RING_EMPTY + stage));
            }
            if (!ok) break;
            if (blk == it.blk_end - 1) ptx::mma_commit(BAR(Q_EMPTY + qb));
            GQA_TRACE_EVENT(TR_MMA_QK, g);
          }
          if (!ok) break;
          ++kq;
        }
      } else {
        constexpr uint32_t idesc_pv = ptx::idesc_f16_f32(128, Cfg::kPvN, 1, 0, !IN_F16);
        uint32_t k = 0;  // items
        while (ok && iter.next(it)) {
          for (int blk = it.blk_begin; blk < it.blk_end; ++blk, ++g) {
            const uint32_t sl = g & 1u;
            if (!ptx::mbar_wait_bounded(BAR(P_FULL + sl), (g >> 1) & 1u, abort_flag, p.timeout_ns)) {
              ok = false;
              break;
            }
            GQA_TRACE_EVENT(TR_MMA_P, g);
            const uint64_t pd = p_desc + static_cast<uint64_t>(sl * (Cfg::kPBytes >> 4));
            const bool first = (blk == it.blk_begin);
            // O^T += V^T P^T, one ring tile (d-half) at a time into its own
            // accumulator (head_dim 256: columns kOCol and kOCol + NPAD)
#pragma unroll
            for (int hf = 0; hf < TPB; ++hf) {
              const uint32_t u = g * TPB + static_cast<uint32_t>(hf);  // V-ring tile
              const uint32_t stage = NSK + u % NSV;
              if (!ptx::mbar_wait_bounded(BAR(RING_FULL + stage), (u / NSV) & 1u, abort_flag, p.timeout_ns)) {
                ok = false;
                break;
              }
              if (hf == 0) GQA_TRACE_EVENT(TR_MMA_V, g);
              ptx::tc_fence_after();
              const uint64_t vd = v_desc + static_cast<uint64_t>(stage * kSlot16);
              const uint32_t o_tmem = tmem_base + kOCol + static_cast<uint32_t>(hf * NPAD);
              if constexpr (Cfg::kTileDim == 128) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t off_b = static_cast<uint32_t>((kk >> 2) * (NPAD * 128 >> 4) + (kk & 3) * 2);
                  ptx::mma_f16_ss(o_tmem, vd + static_cast<uint32_t>(kk * (2048 >> 4)), pd + off_b, idesc_pv,
                                   (kk > 0 || !first) ? 1u : 0u);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  ptx::mma_f16_ss(o_tmem, vd + static_cast<uint32_t>(kk * (2048 >> 4)),
                                   pd + static_cast<uint32_t>(kk * 2), idesc_pv, (kk > 0 || !first) ? 1u : 0u);
                }
              }
              if (hf == TPB - 1) ptx::mma_commit(BAR(P_EMPTY + sl));
              ptx::mma_commit(BAR(RING_EMPTY + stage));
            }
            if (!ok) break;
            GQA_TRACE_EVENT(TR_MMA_PV, g);
          }
          if (!ok) break;
          if (kPvStores && !cluster_merge) {
            // The softmax warpgroup hands over this item's staged rows before
            // it sends the next item's first P, so nothing is delayed by
            // waiting here.  With two buffers, once this item's copies are
            // issued the previous item's copies have read theirs and it can be
            // reused; with one, this item's copies must have read it.
            const int ob = static_cast<int>(k % NB);
            if (!ptx::mbar_wait_bounded(BAR(OUT_FULL + ob), (k / NB) & 1u, abort_flag, p.timeout_ns)) {
              ok = false;
              break;
            }
            store_item(it, ob);
            if constexpr (NB == 1) {
              ptx::bulk_wait_read_all();
              ptx::mbar_arrive(BAR(OUT_EMPTY));
            } else if (k >= 1) {
              ptx::bulk_wait_read_all_but_last();
              ptx::mbar_arrive(BAR(OUT_EMPTY + (ob ^ 1)));
            }
          }
          ++k;
        }
        ptx::bulk_wait_all();  // this CTA's outputs are in global memory
        GQA_TRACE_EVENT(TR_SM_E1, 0);
        ptx::griddep_launch_dependents();
      }
      if (!ok) detail::set_error(p.err_word, kErrTimeout, abort_flag);
      // every MMA this thread issued has completed before TMEM is released
      const uint32_t drain = BAR(DRAIN + (is_qk ? 0 : 1));
      ptx::mma_commit(drain);
      ptx::mbar_wait_bounded(drain, 0, nullptr, p.timeout_ns);
    }
    __syncwarp();
  }
  // ===================================================== softmax warpgroup
  else {
    const int tq = warp & 3;          // TMEM lane quarter of this warp
    const int r = tq * 32 + lane;     // TMEM lane = KV row of S^T = row of O^T
    const uint32_t lane_addr = static_cast<uint32_t>(tq * 32) << 16;
    const int nv = p.nq * p.G;        // valid columns
    const int wg = NWG == 1 ? 0 : (warp - 3) >> 2;  // this softmax warpgroup
    const int c0 = wg * NC;                         // its first column
    const int sm0 = kSoftmaxThread0 + 128 * wg;     // its first thread
    const uint32_t xbar = 1u + 2u * static_cast<uint32_t>(wg);  // its named barrier
    const int cq = c0 + 2 * (lane & 3);             // this lane's two score columns
    // This lane's row of the transposed P store: column c0 + lane % 8,
    // positions tq*32 + 8 (lane / 8) .. + 7 (one 16-byte chunk of the
    // 64-position atom tq / 2, 128-byte swizzled).
    const uint32_t p_addr0 = [&] {
      const int n = c0 + (lane & 7);
      const int chunk = (tq & 1) * 4 + (lane >> 3);
      return ptx::smem_u32(pbuf) + static_cast<uint32_t>((tq >> 1) * (NPAD * 128) + n * 128 + ((chunk ^ (n & 7)) << 4));
    }();
    uint32_t* xflags = xflags_of(wg);
    float* xvals = xvals_of(wg);
    bool local_abort = false;
    uint32_t xc = 0;                  // exchange counter
    GQA_TRACE_STAMPS(ep_ts, kTraceEpStamps);

    // Exchange: every warp posts flags (lane 0) and, optionally, per-column
    // values (after a quad reduction lane q < 4 posts columns 2q and
    // 2q + 1); after the barrier all four warps see the same data.  Returns
    // the OR of the flags.
    auto exchange = [&](uint32_t flags, bool with_vals, float va, float vb) -> uint32_t {
      const uint32_t buf = xc & 1u;
      ++xc;
      if (lane == 0) xflags[buf * 4 + tq] = flags;
      if (with_vals && lane < 4)
        *reinterpret_cast<float2*>(xvals + (buf * 4 + tq) * NC + 2 * lane) = make_float2(va, vb);
      ptx::named_barrier_sync(xbar, 128);
      return xflags[buf * 4 + 0] | xflags[buf * 4 + 1] | xflags[buf * 4 + 2] | xflags[buf * 4 + 3];
    };
    // Per-column combination of the four warps' values of the last exchange,
    // read as 16-byte vectors.
    auto xcombine = [&](float (&outv)[NC], bool is_max) {
      const float4* base = reinterpret_cast<const float4*>(xvals + ((xc - 1) & 1u) * 4 * NC);
#pragma unroll
      for (int c4 = 0; c4 < NC / 4; ++c4) {
        const float4 a = base[0 * (NC / 4) + c4], b4 = base[1 * (NC / 4) + c4];
        const float4 c = base[2 * (NC / 4) + c4], d4 = base[3 * (NC / 4) + c4];
        if (is_max) {
          outv[4 * c4 + 0] = fmaxf(fmaxf(a.x, b4.x), fmaxf(c.x, d4.x));
          outv[4 * c4 + 1] = fmaxf(fmaxf(a.y, b4.y), fmaxf(c.y, d4.y));
          outv[4 * c4 + 2] = fmaxf(fmaxf(a.z, b4.z), fmaxf(c.z, d4.z));
          outv[4 * c4 + 3] = fmaxf(fmaxf(a.w, b4.w), fmaxf(c.w, d4.w));
        } else {
          outv[4 * c4 + 0] = (a.x + b4.x) + (c.x + d4.x);
          outv[4 * c4 + 1] = (a.y + b4.y) + (c.y + d4.y);
          outv[4 * c4 + 2] = (a.z + b4.z) + (c.z + d4.z);
          outv[4 * c4 + 3] = (a.w + b4.w) + (c.w + d4.w);
        }
      }
    };

    // Staging buffer of the next item: free once the copies of the item two
    // before it have read it.  Thread 0 of the warpgroup waits; the result
    // joins the next exchange's flags.
    uint32_t k_out = 0;  // items staged
    auto wait_staging = [&]() -> bool {
      if (threadIdx.x != sm0) return true;
      if constexpr (cluster_merge) {
        // every CTA has merged what this one sent into its buffer NB items before
        if (k_out < NB) return true;
        return ptx::mbar_wait_cluster_bounded(BAR(PEER_EMPTY + 2 * wg + static_cast<int>(k_out % NB)),
                                              ((k_out / NB) & 1u) ^ 1u, abort_flag, p.timeout_ns);
      }
      if constexpr (!kPvStores) {
        ptx::bulk_wait_read_all();
        return true;
      } else {
        if (k_out < NB) return true;
        return ptx::mbar_wait_bounded(BAR(OUT_EMPTY + (k_out % NB)), ((k_out / NB) & 1u) ^ 1u, abort_flag,
                                      p.timeout_ns);
      }
    };
    // In-cluster merge (CLUSTER; "Building a Faster GQA Decode Kernel for
    // Blackwell SM100", section "Reducing inside a thread block cluster",
    // with a fixed-order sum in place of the page's reduce-add into a zeroed
    // output).  CTA j of a cluster of k owns output columns [j d/k, (j+1) d/k)
    // of the pair.  Each CTA sends the normalised fp32 rows of its piece, and
    // their LSEs, straight into the owners' shared memory (send_piece: st.async
    // completing on the owner's PEER_FULL barrier), laid out [piece][column]
    // [row] with the LSEs [piece][row].  The owner then merges locally --
    // M = max_s lse_s, w_s = exp(lse_s - M), O = sum_s w_s O_s / sum_s w_s
    // in piece order s = 0..k-1, empty pieces (lse = -inf) skipped -- writes
    // its columns out (CTA 0 also the LSEs) and tells every sender, per warp,
    // that its buffer is free again (PEER_EMPTY).  A wait that runs out sets
    // the error word; the merge then carries on (its outputs are invalid) so
    // that every warp still reaches the warpgroup's barriers.
    auto send_piece = [&](const float* vals, int dr, bool with_lse, float lse_val) {
      // vals: this thread's NC values of O row dr (columns c0 .. c0 + NC)
      const uint32_t kc = static_cast<uint32_t>(p.cluster_k);
      const uint32_t crank = ptx::cluster_ctarank();
      const int ldk = kLogD - (__ffs(static_cast<int>(kc)) - 1);  // k is a power of two
      const int dk = 1 << ldk;
      const int ob = static_cast<int>(k_out % NB);
      const uint32_t full_bar = BAR(PEER_FULL + 2 * wg + ob);
      const uint32_t j = static_cast<uint32_t>(dr >> ldk);
      const int c = dr & (dk - 1);
      const uint32_t dst = ptx::map_shared_rank(
          ptx::smem_u32(obuf_of(ob)) + static_cast<uint32_t>(((static_cast<int>(crank) * dk + c) * NPAD + c0) * 4), j);
      const uint32_t rbar = ptx::map_shared_rank(full_bar, j);
#pragma unroll
      for (int q = 0; q < NC / 4; ++q)
        ptx::st_async_v4(dst + 16u * q, make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]),
                         rbar);
      if (with_lse) {  // this thread holds column dr's LSE (dr in [c0, c0 + NC)): to every CTA
        const uint32_t l_loc = ptx::smem_u32(lse_of(ob) + static_cast<int>(crank) * NPAD + dr);
        for (uint32_t s2 = 0; s2 < kc; ++s2)
          ptx::st_async_f32(ptx::map_shared_rank(l_loc, s2), lse_val, ptx::map_shared_rank(full_bar, s2));
      }
    };

    auto cluster_merge_item = [&](const WorkItem& wi, bool last_item) {
      const uint32_t kc = static_cast<uint32_t>(p.cluster_k);
      const uint32_t crank = ptx::cluster_ctarank();
      const int ob = static_cast<int>(k_out % NB);
      const uint32_t full_bar = BAR(PEER_FULL + 2 * wg + ob);
      const uint32_t empty_bar = BAR(PEER_EMPTY + 2 * wg + ob);
      const int ldk = kLogD - (__ffs(static_cast<int>(kc)) - 1);  // k is a power of two
      const int dk = 1 << ldk;  // output columns of this CTA
      // bytes every CTA sends this warpgroup: its rows of these columns and their LSEs
      if (threadIdx.x == sm0)
        ptx::mbar_arrive_expect_tx(full_bar, kc * static_cast<uint32_t>(dk * NC * 4 + NC * 4));
      if (!ptx::mbar_wait_cluster_bounded(full_bar, (k_out / NB) & 1u, abort_flag, p.timeout_ns))
        detail::set_error(p.err_word, kErrTimeout, abort_flag);
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_FULL - TR_EP_L);
      if (!last_item && threadIdx.x == sm0) ptx::bulk_wait_read_all();  // earlier copies have read fin
      if (!last_item) ptx::named_barrier_sync(xbar, 128);                 // ... before fin is rewritten

      constexpr float kLog2e = 1.4426950408889634f;
      const int ncv = dk >> 2;  // 4-column groups per row
      const int lncv = ldk - 2;
      const bool out16 = p.out_dtype != kOutF32;
      const float* recv = reinterpret_cast<const float*>(obuf_of(ob));  // [piece][column][row]
      const float* recv_lse = lse_of(ob);                                // [piece][row]
      uint8_t* fin_w = fin_buf + wg * (NC * HEAD_DIM * 2);
      float* fin_lse = reinterpret_cast<float*>(fin_buf + NPAD * HEAD_DIM * 2);
      // One (row, 4-column group) per thread and pass: NC rows x d / (4k)
      // groups, at most HEAD_DIM of them (k >= 2).  All passes are merged
      // into registers first; the received pieces are then released to
      // their senders (PEER_EMPTY) before any output is written, so that the
      // release at cluster scope does not wait for this warp's global stores.
      constexpr int kPasses = (Cfg::kNC * HEAD_DIM / 8 + 127) / 128;
      float4 res[kPasses];
      float res_lse[kPasses];
#pragma unroll
      for (int ps = 0; ps < kPasses; ++ps) {
        res[ps] = make_float4(0.f, 0.f, 0.f, 0.f);
        res_lse[ps] = -INFINITY;
        const int tw = static_cast<int>(threadIdx.x) - sm0 + 128 * ps;
        const int n = c0 + (tw >> lncv), cg = tw & (ncv - 1);
        if (tw >= NC * ncv || n >= nv) continue;
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterK; ++s2)
          if (s2 < static_cast<int>(kc)) M = fmaxf(M, recv_lse[s2 * NPAD + n]);
        if (M != -INFINITY) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          float W = 0.f;
#pragma unroll
          for (int s2 = 0; s2 < kMaxClusterK; ++s2) {
            if (s2 < static_cast<int>(kc)) {
              const float l2 = recv_lse[s2 * NPAD + n];
              const float w = l2 == -INFINITY ? 0.f : ptx::ex2_approx((l2 - M) * kLog2e);
              W += w;
              if (w != 0.f) {
                const float* o2 = recv + (s2 * dk + cg * 4) * NPAD + n;
                acc.x += w * o2[0]; acc.y += w * o2[NPAD]; acc.z += w * o2[2 * NPAD]; acc.w += w * o2[3 * NPAD];
              }
            }
          }
          const float inv = 1.0f / W;
          acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
          res[ps] = acc;
          res_lse[ps] = M + 0.69314718055994531f * __log2f(W);
        }
      }
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, kTraceEpComputed);
      __syncwarp();  // this warp's reads of the received pieces are done
      // After the last item nothing is sent again: instead of these
      // arrivals, the cluster barrier at the end keeps every CTA resident
      // until all have merged.
      if (!last_item && lane == 0)
        for (uint32_t s2 = 0; s2 < kc; ++s2) ptx::mbar_arrive_cluster(ptx::map_shared_rank(empty_bar, s2));
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_MERGED - TR_EP_L);
#pragma unroll
      for (int ps = 0; ps < kPasses; ++ps) {
        const int tw = static_cast<int>(threadIdx.x) - sm0 + 128 * ps;
        const int n = c0 + (tw >> lncv), cg = tw & (ncv - 1);
        if (tw >= NC * ncv || n >= nv) continue;
        const float4 acc = res[ps];
        const int col = static_cast<int>(crank) * dk + cg * 4;
        const int t = n / p.G;
        const long long grow =
            (static_cast<long long>(wi.b) * p.nq + t) * p.Hq + static_cast<long long>(wi.h) * p.G + (n - t * p.G);
        uint2 packed = make_uint2(0u, 0u);
        if (out16) {
          if constexpr (IN_F16) {
            __half2 a = __floats2half2_rn(acc.x, acc.y), b2 = __floats2half2_rn(acc.z, acc.w);
            packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b2));
          } else {
            __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b2 = __floats2bfloat162_rn(acc.z, acc.w);
            packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b2));
          }
        }
        if (last_item) {
          // Nothing of this CTA is still streaming in: plain stores, straight
          // from registers (16- or 8-byte aligned: col is a multiple of 4).
          if (out16) {
            uint16_t* dst = static_cast<uint16_t*>(p.out) + grow * HEAD_DIM + col;
            if (detail::write_ok(p.err_word, p.out, p.out_bytes, dst, 8u)) *reinterpret_cast<uint2*>(dst) = packed;
          } else {
            float* dst = static_cast<float*>(p.out) + grow * HEAD_DIM + col;
            if (detail::write_ok(p.err_word, p.out, p.out_bytes, dst, 16u)) *reinterpret_cast<float4*>(dst) = acc;
          }
          if (crank == 0 && cg == 0 && p.lse != nullptr &&
              detail::write_ok(p.err_word, p.lse, p.lse_bytes, p.lse + grow, 4u))
            p.lse[grow] = res_lse[ps];
        } else {
          const int e = (n - c0) * dk + cg * 4;  // element of this warpgroup's merged rows
          if (out16) *reinterpret_cast<uint2*>(fin_w + e * 2) = packed;
          else *reinterpret_cast<float4*>(fin_w + e * 4) = acc;
          if (crank == 0 && cg == 0) fin_lse[n] = res_lse[ps];
        }
      }
      if (!last_item) {
        // Later items still stream K/V tiles into this SM, and plain stores
        // would queue behind them: the merged rows leave by bulk copies.
        ptx::fence_proxy_async_smem();       // the merged rows are read by bulk copies
        ptx::named_barrier_sync(xbar, 128);  // every warp's rows are in fin
        if (threadIdx.x == sm0) {
          const uint32_t esz = out16 ? 2u : 4u;
          const uint32_t slice = static_cast<uint32_t>(dk) * esz;
          const int n_end = c0 + NC < nv ? c0 + NC : nv;
          for (int n2 = c0; n2 < n_end; ++n2) {
            const int t = n2 / p.G, g2 = n2 - t * p.G;
            const long long grow =
                (static_cast<long long>(wi.b) * p.nq + t) * p.Hq + static_cast<long long>(wi.h) * p.G + g2;
            uint8_t* dst = static_cast<uint8_t*>(p.out) + (grow * HEAD_DIM + static_cast<long long>(crank) * dk) * esz;
            if (detail::write_ok(p.err_word, p.out, p.out_bytes, dst, slice))
              ptx::bulk_store(dst, ptx::smem_u32(fin_w + (n2 - c0) * slice), slice);
          }
          if (crank == 0 && p.lse != nullptr) {
            // runs of rows of one query token are contiguous in lse
            for (int n2 = c0; n2 < n_end;) {
              const int t = n2 / p.G;
              const int run_end = (t + 1) * p.G < n_end ? (t + 1) * p.G : n_end;
              const long long grow = (static_cast<long long>(wi.b) * p.nq + t) * p.Hq +
                                     static_cast<long long>(wi.h) * p.G + (n2 - t * p.G);
              if (!detail::write_ok(p.err_word, p.lse, p.lse_bytes, p.lse + grow,
                                    static_cast<unsigned long long>(run_end - n2) * 4u)) {
                // outside lse: skipped (debug builds)
              } else if (p.lse_bulk) {
                ptx::bulk_store(p.lse + grow, ptx::smem_u32(fin_lse + n2), static_cast<uint32_t>(run_end - n2) * 4u);
              } else {
                for (int i = n2; i < run_end; ++i) p.lse[grow + (i - n2)] = fin_lse[i];
              }
              n2 = run_end;
            }
          }
          ptx::bulk_commit();
        }
      }
      ++k_out;
    };

    // Makes the staged rows visible to the async proxy and writes them out
    // (or hands them to the value-MMA thread, or merges them in the cluster).
    // Returns false on a timeout.
    auto hand_over = [&](const WorkItem& wi, bool last_item) -> bool {
      if constexpr (cluster_merge) {
        cluster_merge_item(wi, last_item);
        return true;
      }
      ptx::fence_proxy_async_smem();
      ptx::named_barrier_sync(xbar, 128);
      if (threadIdx.x == sm0) {
        if constexpr (kPvStores) ptx::mbar_arrive(BAR(OUT_FULL + (k_out % NB)));
        else store_item(wi, static_cast<int>(k_out % NB));
      }
      ++k_out;
      return true;
    };

    ItemSource iter;
    iter.init(list_hdr, list_items, plan, lens_raw, s_len, s_pre);
    WorkItem it;
    uint32_t g = 0;
    bool aborted = false;
    while (!aborted && iter.next(it)) {
      if (it.blk_begin >= it.blk_end) {
        // empty item: final output O = 0, lse = -inf; partial lse = -inf
        const bool st_ok = wait_staging();
        if (exchange(st_ok ? 0u : 2u, false, 0.f, 0.f) & 2u) { aborted = true; break; }
        if constexpr (cluster_merge) {
          if (!cluster_waited) {  // every CTA's barriers are initialised
            ptx::cluster_wait();
            cluster_waited = true;
          }
          float zeros[NC];
#pragma unroll
          for (int n = 0; n < NC; ++n) zeros[n] = 0.f;
          for (int dr = r; dr < HEAD_DIM; dr += 128) send_piece(zeros, dr, dr >= c0 && dr < c0 + NC, -INFINITY);
          if (!hand_over(it, !iter.has_next())) { aborted = true; break; }
          continue;
        }
        uint8_t* ob = obuf_of(static_cast<int>(k_out % NB));
        for (int dr = r; dr < HEAD_DIM; dr += 128) {  // rows r (and r + 128 for head_dim 256)
          for (int n = c0; n < c0 + NC && n < nv; ++n) {
            if (it.slot < 0 && p.out_dtype != kOutF32)
              reinterpret_cast<__nv_bfloat16*>(ob)[n * HEAD_DIM + dr] = __float2bfloat16_rn(0.f);  // +0: all-zero bits
            else
              reinterpret_cast<float*>(ob)[n * HEAD_DIM + dr] = 0.f;
          }
        }
        if (r >= c0 && r < c0 + NC && r < nv) lse_of(static_cast<int>(k_out % NB))[r] = -INFINITY;
        if (!hand_over(it, !iter.has_next())) { aborted = true; break; }
        continue;
      }
      const int L = it.L;
      // This thread's columns cq, cq + 1 (cq = c0 + 2 (lane % 4)): per-lane
      // denominators and -max as the addend of the scaled scores (max:
      // scaled, log2 units; kNoMax while the max is -inf: any visible score
      // then votes).  The warpgroup's -max of all its columns, the same in
      // every thread, rescales O.
      float l2[2] = {0.f, 0.f}, nms2[2] = {kNoMax, kNoMax};
      float nms8[NC];
#pragma unroll
      for (int n = 0; n < NC; ++n) nms8[n] = kNoMax;

      for (int blk = it.blk_begin; blk < it.blk_end; ++blk, ++g) {
        const bool first = (blk == it.blk_begin);
        const uint32_t sl = g & 1u;
        // ---- scores: x[2 j + i] = S^T(position pj = tq*32 + 8 j + lane/4, column cq + i)
        float x[8];
        if (!local_abort)
          local_abort = !ptx::mbar_wait_bounded(BAR(S_FULL + sl), (g >> 1) & 1u, abort_flag, p.timeout_ns);
        local_abort = __any_sync(0xffffffffu, local_abort);
        if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_S, g);
        ptx::tc_fence_after();
        if (!local_abort) {
          const uint32_t s_addr = tmem_base + lane_addr + (sl ? kSCol1 : kSCol0) + c0;
          float lo[4], hi[4];
          ptx::tmem_ld_16x256b_x1(s_addr, lo);                  // positions 0..15 of the quarter
          ptx::tmem_ld_16x256b_x1(s_addr + (16u << 16), hi);    // positions 16..31
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) { x[i] = lo[i]; x[4 + i] = hi[i]; }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k] = -INFINITY;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && !local_abort) ptx::mbar_arrive(BAR(S_EMPTY + sl));  // S slot free for QK(g+2)
        if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_LD, g);

        // ---- mask: position pos is visible to column n when pos < L and,
        // with the causal mask, n / G >= pos - (L - nq)  (bottom-right).
        // Blocks whose rows are all visible to every column skip it; their
        // padding columns (n >= nq*G, zero query rows) stay unmasked, which
        // only feeds O columns that are never written out.
        const bool interior = (blk + 1) * kBlockN <= L - (p.causal ? p.nq - 1 : 0);
        if (!interior) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pos = blk * kBlockN + tq * 32 + 8 * j + (lane >> 2);
            int n_min = 0;
            if (p.causal) {
              const int ahead = pos - (L - p.nq);
              n_min = ahead > 0 ? ahead * p.G : 0;
            }
            const bool row_valid = pos < L;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const bool vis = row_valid && cq + i >= n_min && cq + i < nv;
              x[2 * j + i] = vis ? x[2 * j + i] : -INFINITY;
            }
          }
        }
        // t = scaled score - running max, in log2 units: one FFMA per score
        // feeds both the rescale vote and the exponent
        float t[8];
        bool need = false;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          t[k] = fmaf(x[k], p.scale_log2, nms2[k & 1]);
          need |= t[k] > kRescaleThreshold;
        }
        // An item's first block always takes the max below (m is -inf; with
        // every score masked it leaves m = -inf and l = 0, as skipping it
        // would), so it needs no vote; the max exchange carries the abort flag.
        // The vote is one named barrier that ORs the warpgroup's predicates;
        // an abort joins it, and the max exchange below then carries it.
        uint32_t fl = 1u;
        if (!first) fl = ptx::named_barrier_or(xbar, 128, need || local_abort) ? 1u : 0u;
        if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_X, g);

        // ---- correction (only when some column's max moved past the threshold)
        if (fl & 1u) {
          float ma = fmaxf(fmaxf(x[0], x[2]), fmaxf(x[4], x[6]));
          float mb = fmaxf(fmaxf(x[1], x[3]), fmaxf(x[5], x[7]));
          detail::quad_reduce<true>(ma, mb);
          if (!first && !local_abort) {
            // O may be rescaled only after PV(g-1) has landed
            local_abort = !ptx::mbar_wait_bounded(BAR(P_EMPTY + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u,
                                                  abort_flag, p.timeout_ns);
          }
          local_abort = __any_sync(0xffffffffu, local_abort);
          const uint32_t f2 = exchange(local_abort ? 2u : 0u, true, ma, mb);
          if (f2 & 2u) { aborted = true; break; }
          // New maxima: M_n = max(m_n, scale * max of the block's column n).
          // With 16 columns this lane's two columns go first (their
          // exponentials wait on them) and the warpgroup's eight after, and an
          // item's first block, with no O to rescale and no denominator yet,
          // only records the maxima.  With 32 columns the eight go first and
          // every block takes the same path (measured faster on GB300: the
          // 608-thread kernel is at its register limit, and small changes move
          // its spills).
          float alpha[NC];
          auto own_columns = [&]() {
            const float* xv = xvals + ((xc - 1) & 1u) * 4 * NC + (cq - c0);
            const float2 w0 = *reinterpret_cast<const float2*>(xv);
            const float2 w1 = *reinterpret_cast<const float2*>(xv + NC);
            const float2 w2 = *reinterpret_cast<const float2*>(xv + 2 * NC);
            const float2 w3 = *reinterpret_cast<const float2*>(xv + 3 * NC);
            const float bm[2] = {fmaxf(fmaxf(w0.x, w1.x), fmaxf(w2.x, w3.x)),
                                 fmaxf(fmaxf(w0.y, w1.y), fmaxf(w2.y, w3.y))};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float mo = nms2[i] == kNoMax ? -INFINITY : -nms2[i];
              const float mn = fmaxf(mo, bm[i] * p.scale_log2);
              const float ms = mn == -INFINITY ? 0.f : mn;
              if (!first) l2[i] *= ptx::ex2_approx(mo - ms);
              nms2[i] = mn == -INFINITY ? kNoMax : -mn;
            }
          };
          auto all_columns = [&]() {
            float bmax[NC];
            xcombine(bmax, true);  // of the unscaled scores: the scale is positive
#pragma unroll
            for (int n = 0; n < NC; ++n) {
              const float mo = nms8[n] == kNoMax ? -INFINITY : -nms8[n];
              const float mn = fmaxf(mo, bmax[n] * p.scale_log2);
              const float ms = mn == -INFINITY ? 0.f : mn;
              alpha[n] = (NPAD == 16 && first) ? 0.f : ptx::ex2_approx(mo - ms);
              nms8[n] = mn == -INFINITY ? kNoMax : -mn;
            }
          };
          if constexpr (NPAD == 16) {
            own_columns();
            all_columns();
          } else {
            all_columns();
            // this lane's two columns: entries 2 (lane % 4) and + 1
            const int q = lane & 3;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              nms2[i] = q == 0 ? nms8[i] : q == 1 ? nms8[2 + i] : q == 2 ? nms8[4 + i] : nms8[6 + i];
              l2[i] *= q == 0 ? alpha[i] : q == 1 ? alpha[2 + i] : q == 2 ? alpha[4 + i] : alpha[6 + i];
            }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) t[k] = fmaf(x[k], p.scale_log2, nms2[k & 1]);
          if (!first) {
            // this warpgroup's O columns: c0 + [0, NC), and for head_dim 64
            // the same columns of the second stacked half at +NPAD
            ptx::tc_fence_after();
#pragma unroll
            for (int h2 = 0; h2 < Cfg::kOWidth / NPAD; ++h2) {
              const uint32_t col = kOCol + static_cast<uint32_t>(h2 * NPAD + c0);
              float o8[NC];
              ptx::tmem_ld_32x32b<NC>(tmem_base + lane_addr + col, o8);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < NC; ++i) o8[i] *= alpha[i];
              ptx::tmem_st_32x32b<NC>(tmem_base + lane_addr + col, o8);
            }
            ptx::tmem_wait_st();
          }
        }

        // ---- probabilities; the denominators are accumulated per lane
        float pr[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pr[k] = ptx::ex2_approx(t[k]);
          l2[k & 1] += pr[k];
        }
        // P buffer sl is free once PV(g-2) has completed
        if (!local_abort && g >= 2)
          local_abort = !ptx::mbar_wait_bounded(BAR(P_EMPTY + sl), ((g >> 1) & 1u) ^ 1u, abort_flag, p.timeout_ns);
        local_abort = __any_sync(0xffffffffu, local_abort);
        if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_PE, g);
        if (!local_abort) {
          // P^T as the K-major B operand (row n, positions contiguous, 128-byte
          // swizzle): matrix j of the transposed store holds positions
          // tq*32 + 8 j .. + 7 of columns c0 .. c0 + 7; this lane's register
          // j packs its columns cq, cq + 1 at position 8 j + lane / 4.
          uint32_t pw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if constexpr (IN_F16) {
              const __half2 h = __floats2half2_rn(pr[2 * j], pr[2 * j + 1]);
              pw[j] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
              const __nv_bfloat162 h = __floats2bfloat162_rn(pr[2 * j], pr[2 * j + 1]);
              pw[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
          }
          ptx::stmatrix_x4_trans(p_addr0 + sl * static_cast<uint32_t>(Cfg::kPBytes), pw[0], pw[1], pw[2], pw[3]);
          // Tail block: V rows past the sequence end hold whatever the cache
          // holds there; zero them so that 0 * garbage cannot poison O.
          const int tail_rows = L - blk * kBlockN;
          const int cap_rows = plan.max_seqlen - blk * kBlockN;
          if (wg == 0 && tail_rows < kBlockN && cap_rows > tail_rows) {
            // Wait for V(g)'s tiles to land.  A parity wait is sound once the
            // previous tile of the same stage (NSV tiles earlier) has landed:
            // PV(g-2) is done, which covers it when a ring stage pair holds
            // two blocks; with two tiles per block (head_dim 256) the ring
            // holds one block and PV(g-1) must be done as well.
            if constexpr (TPB > 1) {
              if (!local_abort && g >= 1)
                local_abort = !ptx::mbar_wait_bounded(BAR(P_EMPTY + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u,
                                                      abort_flag, p.timeout_ns);
            }
#pragma unroll
            for (int hf = 0; hf < TPB; ++hf) {
              const uint32_t u = g * TPB + static_cast<uint32_t>(hf);
              const uint32_t stage = NSK + u % NSV;
              if (!local_abort)
                local_abort = !ptx::mbar_wait_bounded(BAR(RING_FULL + stage), (u / NSV) & 1u, abort_flag,
                                                      p.timeout_ns);
              local_abort = __any_sync(0xffffffffu, local_abort);
              if (!local_abort && r >= tail_rows && r < cap_rows) {
#pragma unroll
                for (int kc = 0; kc < TCH; ++kc) {
                  uint4* row = reinterpret_cast<uint4*>(ring + stage * Cfg::kSlotBytes + kc * 16384 + r * 128);
#pragma unroll
                  for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
                }
              }
            }
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && !local_abort) ptx::mbar_arrive(BAR(P_FULL + sl));
        if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_PF, g);
      }
      if (aborted) break;

      // ---------------------------------------------------------- epilogue
      // The denominators are final once the last P is out: reduce and
      // exchange them while the item's last value MMA still runs, and wait
      // for it only before reading O.
      const uint32_t gl = g - 1;
      if (threadIdx.x == kSoftmaxThread0) GQA_TRACE_EVENT(TR_SM_E0, gl);
      float la = l2[0], lb = l2[1];
      detail::quad_reduce<false>(la, lb);
      const bool st_ok = wait_staging();  // staging buffer free after f3
      const uint32_t f3 = exchange((local_abort || !st_ok) ? 2u : 0u, true, la, lb);
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_L - TR_EP_L);
      if (f3 & 2u) { aborted = true; break; }
      float lt[NC];
      xcombine(lt, false);
      if (!local_abort && !ptx::mbar_wait_bounded(BAR(P_EMPTY + (gl & 1u)), (gl >> 1) & 1u, abort_flag,
                                                  p.timeout_ns)) {
        // recorded; the warps still meet at the barriers below (outputs invalid)
        local_abort = true;
        detail::set_error(p.err_word, kErrTimeout, abort_flag);
      }
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_PV - TR_EP_L);

      ptx::tc_fence_after();
      // 2 for head_dim 64 (stacked position halves, added below) and 256
      // (d-halves: rows r and r + 128 of O)
      constexpr int kHalves = Cfg::kOWidth / NPAD;
      float o[kHalves * NC];
#pragma unroll
      for (int h2 = 0; h2 < kHalves; ++h2) {
#pragma unroll
        for (int c = 0; c < NC; c += CW) {
          float o16[CW];
          ptx::tmem_ld_32x32b<CW>(tmem_base + lane_addr + kOCol + static_cast<uint32_t>(h2 * NPAD + c0 + c), o16);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < CW; ++i) o[h2 * NC + c + i] = o16[i];
        }
      }
      ptx::tc_fence_before();
      int d_row = r;
      bool writer = true;
      if constexpr (HEAD_DIM == 64) {
        // lanes 64..127 hold the second half-block's contribution in columns [N, 2N)
        // (one warpgroup: both P buffers are idle here; two: own scratch)
        float* xo = NWG == 1 ? reinterpret_cast<float*>(pbuf) : xo_buf;
        // [n][row] layout: the 32 lanes of a warp touch 32 consecutive words
        if (r >= 64) {
#pragma unroll
          for (int n = 0; n < NC; ++n) xo[(c0 + n) * 64 + (r - 64)] = o[NC + n];
        }
        ptx::named_barrier_sync(xbar, 128);
        if (r < 64) {
#pragma unroll
          for (int n = 0; n < NC; ++n) o[n] += xo[(c0 + n) * 64 + r];
        }
        ptx::named_barrier_sync(xbar, 128);  // xo is read before P is rewritten
        writer = r < 64;
      }
      constexpr int kRowsOut = HEAD_DIM == 256 ? 2 : 1;  // O rows of this thread: r (+ 128)
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_O - TR_EP_L);
      if constexpr (cluster_merge) {
        // the piece's rows go to the CTAs owning their columns
        if (!cluster_waited) {  // every CTA's barriers are initialised
          ptx::cluster_wait();
          cluster_waited = true;
        }
        if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_CW - TR_EP_L);
        if (writer) {
          float inv[NC];
#pragma unroll
          for (int n = 0; n < NC; ++n) inv[n] = lt[n] > 0.f ? ptx::rcp_approx(lt[n]) : 0.f;
          float lse_d = -INFINITY;  // the LSE of column d_row, when this thread holds it
#pragma unroll
          for (int n = 0; n < NC; ++n)
            if (c0 + n == d_row && lt[n] > 0.f) lse_d = 0.69314718055994531f * (__log2f(lt[n]) - nms8[n]);
#pragma unroll
          for (int h2 = 0; h2 < kRowsOut; ++h2) {
            float vals[NC];
#pragma unroll
            for (int n = 0; n < NC; ++n) vals[n] = o[h2 * NC + n] * inv[n];
            send_piece(vals, d_row + 128 * h2, h2 == 0 && d_row >= c0 && d_row < c0 + NC, lse_d);
          }
        }
      } else
      // Outputs go to shared memory in their global layout (row n = t*G + g
      // of this pair, d contiguous); the output warp writes them out.
      if (writer) {
        // fp32 for partials and fp32 outputs, else 16-bit outputs of the
        // input type
        const bool out16 = it.slot < 0 && p.out_dtype != kOutF32;
        uint8_t* obuf = obuf_of(static_cast<int>(k_out % NB));
#pragma unroll
        for (int n = 0; n < NC; ++n) {
          const float inv = lt[n] > 0.f ? ptx::rcp_approx(lt[n]) : 0.f;
          const int ng = c0 + n;
          if (ng < nv) {
#pragma unroll
            for (int h2 = 0; h2 < kRowsOut; ++h2) {
              const float val = o[h2 * NC + n] * inv;
              const int dr = d_row + 128 * h2;
              if (out16) {
                if constexpr (IN_F16)
                  reinterpret_cast<__half*>(obuf)[ng * HEAD_DIM + dr] = __float2half_rn(val);
                else
                  reinterpret_cast<__nv_bfloat16*>(obuf)[ng * HEAD_DIM + dr] = __float2bfloat16_rn(val);
              } else {
                reinterpret_cast<float*>(obuf)[ng * HEAD_DIM + dr] = val;
              }
            }
          }
        }
        if (d_row >= c0 && d_row < c0 + NC && d_row < nv) {
          float lt_n = 0.f, m_n = 0.f;
#pragma unroll
          for (int n = 0; n < NC; ++n)
            if (c0 + n == d_row) { lt_n = lt[n]; m_n = -nms8[n]; }
          lse_of(static_cast<int>(k_out % NB))[d_row] =
              lt_n > 0.f ? 0.69314718055994531f * (m_n + __log2f(lt_n)) : -INFINITY;
        }
      }
      if (threadIdx.x == kSoftmaxThread0 + 32) GQA_TRACE_STAMP(ep_ts, TR_EP_SENT - TR_EP_L);
      if (!hand_over(it, !iter.has_next())) { aborted = true; break; }
    }
    if constexpr (!kPvStores) {
      if (threadIdx.x == kSoftmaxThread0) ptx::bulk_wait_all();  // this CTA's outputs are in global memory
    }
    if (cluster_merge && threadIdx.x == sm0) {
      // Every CTA this one sent pieces to has merged them (so the stores have
      // landed) once it arrives on PEER_EMPTY: wait before exiting (bounded)
      // for every item but the last, whose merge the cluster barrier at the
      // end covers.
      for (uint32_t i = k_out >= NB ? k_out - NB : 0u; i + 1 < k_out; ++i)
        ptx::mbar_wait_cluster_bounded(BAR(PEER_EMPTY + 2 * wg + static_cast<int>(i % NB)), (i / NB) & 1u,
                                       abort_flag, p.timeout_ns);
      ptx::bulk_wait_all();  // this warpgroup's merged outputs are in global memory
    }
    if (aborted || local_abort) detail::set_error(p.err_word, kErrTimeout, abort_flag);
    if (threadIdx.x == kSoftmaxThread0 + 32) {
      GQA_TRACE_STAMP(ep_ts, TR_EP_EXIT - TR_EP_L);
      GQA_TRACE_FLUSH(ep_ts, kTraceEpStamps, TR_EP_L);
    }
    ptx::griddep_launch_dependents();
  }

  // ---------------------------------------------------------------- teardown
  if (!cluster_waited) ptx::cluster_wait();
  if (cluster_merge) {
    // No CTA leaves while another may still send into it or merge what it
    // sent: every thread of the cluster has finished its role here.
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait();
  }
#ifdef GQA_TRACE
  if (lane == 0) atomicAdd(&trace_warps_done, 1u);
#endif
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();  // every role is done with TMEM and shared memory
  if (threadIdx.x == 0) {
    GQA_TRACE_EVENT(TR_END, 0);
    GQA_TRACE_VALUE(TR_END, 1, trace_warps_done);
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace gqa
