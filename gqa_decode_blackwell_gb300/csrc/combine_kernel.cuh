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
// One warp per row; each lane owns 4 (head_dim 128) or 2 (head_dim 64)
// consecutive output elements, read as one 16- or 8-byte vector per split.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace gqa {

constexpr int kCombineThreads = 256;
constexpr int kMaxSplits = 64;

struct CombineParams {
  const float* o_part;      // [num_slots, rows, d]
  const float* lse_part;    // [num_slots, rows]
  const int32_t* n_pieces;  // optional [B * Hkv][4]: valid slots per pair in [0] (balanced plan)
  void* out;                // [rows, d] bf16 or fp32
  float* lse;               // [rows] or null
  long long rows;
  int num_splits;           // slots to merge when n_pieces is null
  int out_fp32;
  int nq, Hq, G, kv_heads;  // row -> pair mapping for n_pieces
};

template <int HEAD_DIM>
__global__ void __launch_bounds__(kCombineThreads)
gqa_combine_kernel(const CombineParams p) {
  constexpr int VEC = HEAD_DIM / 32;  // elements per lane
  // Partials come from the preceding decode launch.
  ptx::griddep_wait();

  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (row >= p.rows) return;

  // Every load below is independent of the others, so they are all issued
  // before the first use: the piece count, the LSEs of every allocated slot
  // and the first kSpec partial rows.  Slots beyond the valid count are
  // allocated memory whose values are masked out, never used.
  constexpr int kSpec = 4;
  const int slots = p.num_splits;  // allocated slots
  int n = slots;
  const int* np_ptr = nullptr;
  if (p.n_pieces != nullptr) {
    const long long bt = row / p.Hq;            // b * nq + t
    const int hq = static_cast<int>(row % p.Hq);
    const long long b = bt / p.nq;
    np_ptr = p.n_pieces + (b * p.kv_heads + hq / p.G) * 4;  // one 16-byte record per pair
  }
  const int n_raw = np_ptr != nullptr ? *np_ptr : slots;
  float l0 = lane < slots ? p.lse_part[static_cast<long long>(lane) * p.rows + row] : -INFINITY;
  float l1 = lane + 32 < slots ? p.lse_part[static_cast<long long>(lane + 32) * p.rows + row] : -INFINITY;
  float spec[kSpec][VEC];
#pragma unroll
  for (int s = 0; s < kSpec; ++s) {
    if (s < slots) {
      const float* src = p.o_part + (static_cast<long long>(s) * p.rows + row) * HEAD_DIM + lane * VEC;
      if constexpr (VEC == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        spec[s][0] = v.x; spec[s][1] = v.y; spec[s][2] = v.z; spec[s][3] = v.w;
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src));
        spec[s][0] = v.x; spec[s][1] = v.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) spec[s][i] = 0.f;
    }
  }
  if (np_ptr != nullptr) {
    n = n_raw < slots ? n_raw : slots;
    if (n <= 1) return;                          // written directly by the decode kernel
  }
  if (lane >= n) l0 = -INFINITY;
  if (lane + 32 >= n) l1 = -INFINITY;
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  float lse_out = -INFINITY;

  if (M != -INFINITY) {
    constexpr float kLog2e = 1.4426950408889634f;
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
    for (int s = kSpec; s < n; ++s) {
      const float ws = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
      if (ws == 0.f) continue;  // empty split (or a weight that underflows): not used
      const float* src = p.o_part + (static_cast<long long>(s) * p.rows + row) * HEAD_DIM + lane * VEC;
      if constexpr (VEC == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] += ws * v.x; acc[1] += ws * v.y; acc[2] += ws * v.z; acc[3] += ws * v.w;
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] += ws * v.x; acc[1] += ws * v.y;
      }
    }
    const float inv = 1.0f / W;
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] *= inv;
    lse_out = M + 0.69314718055994531f * __log2f(W);
  }

  if (p.out_fp32) {
    float* dst = static_cast<float*>(p.out) + row * HEAD_DIM + lane * VEC;
    if constexpr (VEC == 4) *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + row * HEAD_DIM + lane * VEC;
    if constexpr (VEC == 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
      __nv_bfloat162 c = __floats2bfloat162_rn(acc[2], acc[3]);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&c);
      *reinterpret_cast<uint2*>(dst) = u;
    } else {
      *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0], acc[1]);
    }
  }
  if (lane == 0 && p.lse != nullptr) p.lse[row] = lse_out;
  ptx::griddep_launch_dependents();
}

}  // namespace gqa
