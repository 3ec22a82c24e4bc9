// Split-KV work planning, shared by the decode kernel, the combine kernel and
// the host-side plan introspection entry point.
//
// A "unit" is one 128-position KV block of one (batch, KV head) pair.  The
// decode grid is persistent: CTA c walks a deterministic list of work items,
// each a contiguous block range [blk_begin, blk_end) of one pair, writing
// either the final output (the item is the whole pair) or a partial
// (O_s, lse_s) into workspace slot `slot`.  Splitting the KV length so that a
// small batch fills the GPU, and merging the partials by log-sum-exp, follows
// "Building a Faster GQA Decode Kernel for Blackwell SM100", section
// "Combining the KV splits".  The two partitions below are this library's
// own (the page leaves its split heuristic unstated).
//
//  * PLAN_SPLITS: sequence b is cut into splits_b = clamp(ceil(nblk_b /
//    min_blocks), 1, S) contiguous block ranges; split s covers blocks
//    [s*nblk_b/splits_b, (s+1)*nblk_b/splits_b).  Items (b, h, s) are dealt
//    round-robin to the CTAs.  Splits s >= splits_b are empty items that only
//    publish lse = -inf.
//  * PLAN_BALANCED: the U units of all pairs, ordered (b, h, block), are cut
//    into C' = min(C, U) equal contiguous ranges, one per CTA (CTA c < C'
//    owns units [floor(cU/C'), floor((c+1)U/C')), at least one each; CTAs
//    c >= C' own nothing).  Each non-empty pair also counts X = item_units
//    units before its blocks, which hold no work: a work item costs a fixed
//    time (Q load, pipeline fill, epilogue) worth a few blocks, so a CTA
//    whose range takes in the start of a pair -- and with it one more item --
//    gets X fewer blocks.  Because no range is empty, the CTAs touching a
//    pair's blocks are consecutive.  A pair whose blocks fall inside one CTA
//    is written as final output; a pair cut by CTA boundaries gets one
//    partial per CTA touching its blocks, in slot (c - first such CTA), and
//    the CTA holding its first block publishes the piece count for the
//    combine.
//    Pairs of empty sequences belong to the CTA whose range contains their
//    (zero-length) start; trailing ones to CTA C' - 1.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define GQA_HD __host__ __device__ __forceinline__
#else
#define GQA_HD inline
#endif

namespace gqa {

constexpr int kBlockN = 128;  // KV positions per block (the MMA M dimension)

enum PlanMode : int { PLAN_SPLITS = 0, PLAN_BALANCED = 1 };

struct PlanParams {
  int mode;           // PlanMode
  int batch;          // B
  int kv_heads;       // Hkv
  int max_seqlen;     // S_max: lengths are clamped to [0, S_max]
  int num_splits;     // PLAN_SPLITS: S
  int min_blocks;     // PLAN_SPLITS: minimum blocks per split
  int force_partial;  // PLAN_SPLITS: write partials even when S == 1
  int num_ctas;       // C: CTAs of the persistent grid
  int item_units;     // PLAN_BALANCED: X, the units a pair's item costs before its blocks
};

struct WorkItem {
  int b, h;
  int L;            // clamped sequence length
  int blk_begin;    // first KV block (inclusive)
  int blk_end;      // last KV block (exclusive); begin == end: empty item
  int slot;         // partial slot, or -1 for final output
  int first_piece;  // publishes the pair's piece count (PLAN_BALANCED)
  int n_pieces;     // pieces of this pair (PLAN_BALANCED) / splits of this sequence
};

GQA_HD int clamp_len(int L, int s_max) { return L < 0 ? 0 : (L > s_max ? s_max : L); }
GQA_HD int num_blocks(int L) { return (L + kBlockN - 1) / kBlockN; }
// Units of one pair in the balanced plan: its blocks plus X item units (none when empty).
GQA_HD int pair_units(int nblk, int X) { return nblk > 0 ? nblk + X : 0; }

// floor(a * b / c) for a, b >= 0 and c > 0.  GPUs emulate 64-bit division in
// software, so the common case where everything fits in 32 bits takes the
// 32-bit path.
GQA_HD long long muldiv(long long a, long long b, long long c) {
  const unsigned long long ab = static_cast<unsigned long long>(a) * static_cast<unsigned long long>(b);
  if (ab <= 0xffffffffull && c <= 0xffffffffll)
    return static_cast<long long>(static_cast<uint32_t>(ab) / static_cast<uint32_t>(c));
  return static_cast<long long>(ab / static_cast<unsigned long long>(c));
}

// floor(a / c) for a >= 0, c > 0, with the same 32-bit fast path.
GQA_HD long long div_nonneg(long long a, long long c) { return muldiv(a, 1, c); }

// CTA owning unit u under the balanced partition of U units over C CTAs:
// the largest c with floor(c*U/C) <= u.
GQA_HD int balanced_cta_of(long long u, long long U, int C) {
  return static_cast<int>(div_nonneg((u + 1) * static_cast<long long>(C) - 1, U));
}

// Round-robin over split items.  `lens` holds raw lengths (clamped here).
struct SplitIter {
  PlanParams pp;
  const int32_t* lens;
  long long w, total;
  int cta;

  GQA_HD void init(const PlanParams& p, const int32_t* l, int c) {
    pp = p; lens = l; cta = c; w = c;
    total = static_cast<long long>(p.batch) * p.kv_heads * p.num_splits;
  }
  GQA_HD bool next(WorkItem& it) {
    if (w >= total) return false;
    const int S = pp.num_splits;
    const long long pair = div_nonneg(w, S);
    const int s = static_cast<int>(w - pair * S);
    const long long bb = div_nonneg(pair, pp.kv_heads);
    it.h = static_cast<int>(pair - bb * pp.kv_heads);
    it.b = static_cast<int>(bb);
    it.L = clamp_len(lens[it.b], pp.max_seqlen);
    const int nblk = num_blocks(it.L);
    int splits = (nblk + pp.min_blocks - 1) / pp.min_blocks;
    splits = splits < 1 ? 1 : (splits > S ? S : splits);
    if (s < splits) {
      it.blk_begin = static_cast<int>(muldiv(s, nblk, splits));
      it.blk_end = static_cast<int>(muldiv(s + 1, nblk, splits));
    } else {
      it.blk_begin = it.blk_end = 0;
    }
    it.slot = (S == 1 && !pp.force_partial) ? -1 : s;
    it.first_piece = (s == 0);
    it.n_pieces = splits;
    w += pp.num_ctas;
    return true;
  }
};

// Contiguous equal ranges of units.  `lens` are clamped lengths and `pre`
// (B + 1 entries) the exclusive prefix sums of the units of one pair of each
// sequence: its blocks + X when it is non-empty, 0 when it is empty.
struct BalancedIter {
  const int32_t* lens;
  const int32_t* pre;
  long long U, lo, hi;
  int B, H, X;
  int b, h, cta, C;  // C: effective CTA count min(num_ctas, U), at least 1

  GQA_HD void init(const PlanParams& p, const int32_t* l, const int32_t* prefix, int c) {
    lens = l; pre = prefix; cta = c;
    B = p.batch; H = p.kv_heads; X = p.item_units;
    U = static_cast<long long>(H) * pre[B];
    C = U <= 0 ? 1 : (U < p.num_ctas ? static_cast<int>(U) : p.num_ctas);
    if (c >= C) {  // this CTA owns nothing
      b = B; h = 0; lo = hi = U;
      return;
    }
    lo = muldiv(c, U, C);
    hi = muldiv(c + 1, U, C);
    // first pair: the smallest b that reaches lo (the predicate is monotone in b)
    int a = 0, z = B;
    while (a < z) {
      const int mid = (a + z) / 2;
      if (reaches(mid)) z = mid; else a = mid + 1;
    }
    b = a;
    set_first_head();
  }
#ifdef __CUDACC__
  // The same result as init(), computed by the 32 lanes of a warp together:
  // lo and hi in two lanes at once, and the first pair by a ballot over 32
  // sequences at a time instead of a serial binary search.  Every lane must
  // call it; every lane ends with the same state.
  __device__ __forceinline__ void init_warp(const PlanParams& p, const int32_t* l, const int32_t* prefix, int c,
                                            int lane) {
    lens = l; pre = prefix; cta = c;
    B = p.batch; H = p.kv_heads; X = p.item_units;
    U = static_cast<long long>(H) * pre[B];
    C = U <= 0 ? 1 : (U < p.num_ctas ? static_cast<int>(U) : p.num_ctas);
    if (c >= C) {
      b = B; h = 0; lo = hi = U;
      return;
    }
    const long long v = muldiv(c + (lane & 1), U, C);
    lo = __shfl_sync(0xffffffffu, v, 0);
    hi = __shfl_sync(0xffffffffu, v, 1);
    b = B;
    for (int base = 0; base < B; base += 32) {
      const unsigned m = __ballot_sync(0xffffffffu, base + lane < B && reaches(base + lane));
      if (m != 0u) {
        b = base + __ffs(m) - 1;
        break;
      }
    }
    set_first_head();
  }
#endif
  // Sequence b holds a unit at or after lo, or starts at or after lo.
  GQA_HD bool reaches(int bb) const {
    return static_cast<long long>(H) * pre[bb + 1] > lo || static_cast<long long>(H) * pre[bb] >= lo;
  }
  // First head of the first pair: the head whose units contain lo.
  GQA_HD void set_first_head() {
    h = 0;
    if (b < B) {
      const long long start = static_cast<long long>(H) * pre[b];
      const int nblk = pre[b + 1] - pre[b];
      if (start < lo && nblk > 0) h = static_cast<int>(div_nonneg(lo - start, nblk));
    }
  }
  GQA_HD void advance() {
    if (++h == H) { h = 0; ++b; }
  }
  GQA_HD bool next(WorkItem& it) {
    while (b < B) {
      const int vl = pre[b + 1] - pre[b];  // units of each pair of sequence b
      const long long v_first = static_cast<long long>(H) * pre[b] + static_cast<long long>(h) * vl;
      if (vl == 0) {
        const bool owned = (v_first >= lo && v_first < hi) || (v_first == U && cta == C - 1);
        if (!owned) {
          if (v_first >= hi) return false;
          advance();
          continue;
        }
        it.b = b; it.h = h; it.L = lens[b];
        it.blk_begin = it.blk_end = 0;
        it.slot = -1; it.first_piece = 1; it.n_pieces = 1;
        advance();
        return true;
      }
      if (v_first >= hi) return false;
      // the pair's blocks: units [u_first, u_end), after its X item units
      const long long u_first = v_first + X;
      const long long u_end = v_first + vl;
      const long long pl = u_first > lo ? u_first : lo;
      const long long ph = u_end < hi ? u_end : hi;
      if (pl >= ph) { advance(); continue; }
      const int c_first = balanced_cta_of(u_first, U, C);
      const int c_last = balanced_cta_of(u_end - 1, U, C);
      it.b = b; it.h = h; it.L = lens[b];
      it.blk_begin = static_cast<int>(pl - u_first);
      it.blk_end = static_cast<int>(ph - u_first);
      it.n_pieces = c_last - c_first + 1;
      it.slot = it.n_pieces == 1 ? -1 : cta - c_first;
      it.first_piece = (pl == u_first);
      advance();
      return true;
    }
    return false;
  }
};

// Either iterator behind one interface (the mode is uniform per launch).
struct WorkIter {
  SplitIter s;
  BalancedIter bal;
  int mode;
  GQA_HD void init(const PlanParams& p, const int32_t* raw_lens, const int32_t* clamped_lens,
                   const int32_t* prefix, int cta) {
    mode = p.mode;
    if (mode == PLAN_BALANCED) bal.init(p, clamped_lens, prefix, cta);
    else s.init(p, raw_lens, cta);
  }
#ifdef __CUDACC__
  // Warp-cooperative init (all 32 lanes), same result as init().
  __device__ __forceinline__ void init_warp(const PlanParams& p, const int32_t* raw_lens,
                                            const int32_t* clamped_lens, const int32_t* prefix, int cta, int lane) {
    mode = p.mode;
    if (mode == PLAN_BALANCED) bal.init_warp(p, clamped_lens, prefix, cta, lane);
    else s.init(p, raw_lens, cta);
  }
#endif
  GQA_HD bool next(WorkItem& it) { return mode == PLAN_BALANCED ? bal.next(it) : s.next(it); }
};

}  // namespace gqa
