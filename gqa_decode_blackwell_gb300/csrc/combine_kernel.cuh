// Log-sum-exp merge of split-KV partials ("Building a Faster GQA Decode Kernel
// for Blackwell SM100", sections "Combining the KV splits", "Starting combine
// early with PDL" and "Removing the max reset").
//
// Partials are normalised (O_s, lse_s) in fp32.  For one output row:
//   M = max_s lse_s;  w_s = exp(lse_s - M);  O = sum_s w_s O_s / sum_s w_s;
//   lse = M + ln(sum_s w_s).
// A split with lse_s = -inf is empty and its partial is ignored; a row whose
// splits are all empty gets O = 0 and lse = -inf.  The splits are summed in a fixed order,
// so the output is bit-identical from run to run, and the maximum is taken here
// from the staged lse values (no global running-max buffer, nothing to reset).
//
// One warp per row; each lane owns 8 (head_dim 256), 4 (128) or 2 (64)
// consecutive output elements, read as 32-, 16- or 8-byte vectors per split.
// Up to 64 splits the LSEs stay in two registers per lane; more splits (a
// long sequence cut over many CTAs) take a two-pass loop over groups of 32.
//
// Four warps per CTA at <= 48 registers a thread (6 K registers) fit beside a
// resident decode CTA (11 warps at 160 registers, or 19 at 96), so the merge's
// CTAs are placed while the decode kernel still runs.  The merge releases the
// next launch in the stream at once: that launch's own grid-dependency wait
// still covers every output written here.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace gqa {

constexpr int kCombineThreads = 128;

struct CombineParams {
  const float* o_part;      // [num_splits, rows, d]
  const float* lse_part;    // [num_splits, rows]
  const int32_t* n_pieces;  // optional [B * Hkv][4]: valid slots per pair in [0] (balanced plan)
  void* out;                // [rows, d] bf16, fp16 or fp32
  float* lse;               // [rows] or null
  long long rows;
  int num_splits;           // slots per row (all of them are merged when n_pieces is null)
  int out_dtype;            // 0 bf16, 1 fp32, 2 fp16 (gqa_dtype_t)
  int nq, Hq, G, kv_heads;  // row -> pair mapping for n_pieces
};

namespace detail {

template <int VEC>
__device__ __forceinline__ void load_vec(const float* src, float (&v)[VEC]) {
  if constexpr (VEC == 8) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
    const float4 y = __ldg(reinterpret_cast<const float4*>(src) + 1);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else if constexpr (VEC == 4) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = __ldg(reinterpret_cast<const float2*>(src));
    v[0] = x.x; v[1] = x.y;
  }
}

}  // namespace detail

template <int HEAD_DIM>
__global__ void __launch_bounds__(kCombineThreads, 10)
gqa_combine_kernel(const CombineParams p) {
  constexpr int VEC = HEAD_DIM / 32;  // elements per lane
  constexpr float kLog2e = 1.4426950408889634f;
  // The next launch may start its set-up now; it waits for this grid to
  // complete before it reads or writes anything this grid touches.
  ptx::griddep_launch_dependents();
  // Partials come from the preceding decode launch.
  ptx::griddep_wait();

  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (row >= p.rows) return;

  // split s of this row is partial row first + s * stride
  const long long first = row, stride = p.rows;
  int n = p.num_splits;
  const int32_t* rec = nullptr;
  if (p.n_pieces != nullptr) {
    // rows < 2^31 with piece counts (at most 512 sequences): 32-bit
    // divisions, not the emulated 64-bit ones
    const uint32_t r32 = static_cast<uint32_t>(row);
    const uint32_t bt = r32 / static_cast<uint32_t>(p.Hq);  // b * nq + t
    const uint32_t hq = r32 - bt * static_cast<uint32_t>(p.Hq);
    const uint32_t b = bt / static_cast<uint32_t>(p.nq);
    rec = p.n_pieces + (static_cast<long long>(b) * p.kv_heads + hq / static_cast<uint32_t>(p.G)) * 4;  // one 16-byte record per pair
  }
  constexpr int kSpec = 4;
  float l0, l1, spec[kSpec][VEC];
  auto lse_at = [&](int s) -> float { return p.lse_part[first + s * stride]; };
  auto o_at = [&](int s) -> const float* { return p.o_part + (first + s * stride) * HEAD_DIM + lane * VEC; };
  auto load_fast = [&](int slots) {
    // Up to 64 slots: the LSEs of every slot and the first kSpec partial
    // rows, all issued before the first use.  Slots past the valid count
    // are masked out, never used.
    l0 = lane < slots ? lse_at(lane) : -INFINITY;
    l1 = lane + 32 < slots ? lse_at(lane + 32) : -INFINITY;
#pragma unroll
    for (int s = 0; s < kSpec; ++s) {
      if (s < slots) {
        detail::load_vec<VEC>(o_at(s), spec[s]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) spec[s][i] = 0.f;
      }
    }
  };
  {
    // the addresses do not depend on the piece count, so the loads go out
    // together with it
    const int slots = p.num_splits;
    const int n_raw = rec != nullptr ? *rec : slots;
    const bool loaded = slots <= 64;
    if (loaded) load_fast(slots);
    if (rec != nullptr) {
      n = n_raw < slots ? n_raw : slots;
      if (n <= 1) return;  // written directly by the decode kernel
    }
    if (!loaded && n <= 64) load_fast(n);
  }

  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  float lse_out = -INFINITY;

  if (n <= 64) {
    if (lane >= n) l0 = -INFINITY;
    if (lane + 32 >= n) l1 = -INFINITY;
    float M = fmaxf(l0, l1);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      const float w0 = l0 == -INFINITY ? 0.f : ptx::ex2_approx((l0 - M) * kLog2e);
      const float w1 = l1 == -INFINITY ? 0.f : ptx::ex2_approx((l1 - M) * kLog2e);
      float W = w0 + w1;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
#pragma unroll
      for (int s = 0; s < kSpec; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w0, s);
        if (s < n && ws != 0.f) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[i] += ws * spec[s][i];
        }
      }
      // the rest kBatch at a time: a batch's loads go out together, then
      // its partials are added in split order
      constexpr int kBatch = 16 / VEC;
      for (int s = kSpec; s < n; s += kBatch) {
        float v[kBatch][VEC], wb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int sj = s + j;
          const float ws = __shfl_sync(0xffffffffu, sj < 32 ? w0 : w1, sj & 31);
          wb[j] = sj < n ? ws : 0.f;
          if (wb[j] != 0.f) {  // an empty split (or a weight that underflows) is not read
            detail::load_vec<VEC>(o_at(sj), v[j]);
          } else {
#pragma unroll
            for (int i = 0; i < VEC; ++i) v[j][i] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          if (wb[j] != 0.f) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += wb[j] * v[j][i];
          }
        }
      }
      const float inv = 1.0f / W;
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[i] *= inv;
      lse_out = M + 0.69314718055994531f * __log2f(W);
    }
  } else {
    // many splits: the maximum first, then weights and sums, 32 at a time
    float M = -INFINITY;
    for (int s0 = 0; s0 < n; s0 += 32)
      if (s0 + lane < n) M = fmaxf(M, lse_at(s0 + lane));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      float W = 0.f;
      for (int s0 = 0; s0 < n; s0 += 32) {
        const float l = s0 + lane < n ? lse_at(s0 + lane) : -INFINITY;
        const float w = l == -INFINITY ? 0.f : ptx::ex2_approx((l - M) * kLog2e);
        W += w;
        const int cnt = n - s0 < 32 ? n - s0 : 32;
        for (int j = 0; j < cnt; ++j) {
          const float ws = __shfl_sync(0xffffffffu, w, j);
          if (ws == 0.f) continue;
          float v[VEC];
          detail::load_vec<VEC>(o_at(s0 + j), v);
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[i] += ws * v[i];
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
      const float inv = 1.0f / W;
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[i] *= inv;
      lse_out = M + 0.69314718055994531f * __log2f(W);
    }
  }

  if (p.out_dtype == 1) {  // fp32
    float* dst = static_cast<float*>(p.out) + row * HEAD_DIM + lane * VEC;
    if constexpr (VEC == 8) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else if constexpr (VEC == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
    }
  } else {
    // two 16-bit values per 32-bit word, bf16 or fp16
    uint32_t w[VEC / 2];
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
      if (p.out_dtype == 2) {
        __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    uint16_t* dst = static_cast<uint16_t*>(p.out) + row * HEAD_DIM + lane * VEC;
    if constexpr (VEC == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (VEC == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint32_t*>(dst) = w[0];
  }
  if (lane == 0 && p.lse != nullptr) p.lse[row] = lse_out;
}

}  // namespace gqa
