/*
 * gqa_decode.h -- C ABI of the GB300 (sm_103a) grouped-query attention decode
 * library.
 *
 * Operation.  For every batch entry b, new query token t < nq and query head
 * hq, with KV head h = hq / G (G = Hq / Hkv: consecutive query heads share a
 * KV head, "Flash Attention 4 - warp-role choreography and the edges",
 * section "Edge 2 - GQA"):
 *
 *     O[b,t,hq,:] = sum_j softmax_j(scale * q[b,t,hq,:] . K[b,j,h,:]) V[b,j,h,:]
 *     lse[b,t,hq] = ln sum_j exp(scale * q[b,t,hq,:] . K[b,j,h,:])
 *
 * ("Optimization diaries: S/P ping-pong for FlashAttention-4 decode", section
 * "Recap on the FA4 forward pass"), over the visible keys j: 0 <= j < L_b
 * (L_b = seqlens[b], which counts the nq new positions), and with the causal
 * flag also j <= L_b - nq + t (the new tokens are the last nq positions; a
 * query never sees a later key: same page as the GQA section, "Edge 1 -
 * causal masking").  A row with no visible key yields O = 0, lse = -inf
 * ("Building a Faster GQA Decode Kernel for Blackwell SM100", section
 * "Removing the max reset").  The KV length is split so that a small batch
 * fills the GPU, each split yields a partial (O_s, lse_s) in fp32, and a
 * second kernel merges them by log-sum-exp (same page, section "Combining the
 * KV splits").
 *
 * Conventions shared by every call:
 *   - Pointers are device pointers unless stated otherwise; the caller owns
 *     all memory.  The library never allocates, frees or memsets device
 *     memory (gqa_decode_attn_static_workspace uses a static array).  Calls
 *     are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and contain no host synchronisation.  gqa_decode_attn and
 *     gqa_decode_attn_split are captured in CUDA graphs and replayed in this
 *     library's tests and benchmark, after one call outside capture (the
 *     first call on a device sets kernel attributes); do the same.
 *   - Tensors are dense, row-major, in the layouts stated per argument.
 *   - Arguments are checked before anything is launched; an invalid call
 *     returns an error status and launches nothing.
 *   - The library computes on the current CUDA device; pointers must belong
 *     to it.
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or flag */
  GQA_ERR_UNSUPPORTED = 2,  /* valid but not implemented: head_dim, group size */
  GQA_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
  GQA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute) */
  GQA_ERR_TIMEOUT = 5,      /* a kernel wait ran out (see gqa_decode_get_error) */
  GQA_ERR_BAD_SEQLEN = 6,   /* a sequence length was < 0 or > max_seqlen */
  GQA_ERR_BOUNDS = 7        /* library built with -DGQA_DEBUG: a kernel caught (and skipped) a write
                               outside its buffer, or recorded a TMA tile origin outside its tensor */
} gqa_status_t;

typedef enum { GQA_DTYPE_BF16 = 0, GQA_DTYPE_FP32 = 1, GQA_DTYPE_FP16 = 2 } gqa_dtype_t;

/* How the split partials of a sequence are merged ("Building a Faster GQA
 * Decode Kernel for Blackwell SM100", sections "Combining the KV splits" and
 * "Reducing inside a thread block cluster"):
 *   GQA_REDUCE_COMBINE  the decode kernel writes fp32 partials to the
 *                       workspace and a second kernel merges them;
 *   GQA_REDUCE_CLUSTER  the k splits of one (batch, KV head) pair run as one
 *                       thread-block cluster and merge their partials in the
 *                       cluster's distributed shared memory, in a fixed split
 *                       order, each CTA writing d/k columns of the output: no
 *                       workspace, no second launch, nothing to zero, results
 *                       bit-identical from run to run.  Needs k = num_splits
 *                       a power of two <= 8 (num_splits = 0: the largest
 *                       power of two <= min(8, #SMs / pairs, blocks));
 *                       otherwise GQA_ERR_UNSUPPORTED;
 *   GQA_REDUCE_AUTO     the page's selection (at most four splits, or eight
 *                       with at most 64 CTAs) narrowed by measurement on
 *                       GB300: with num_splits = 0, the in-cluster merge when
 *                       the automatic plan would give every pair k >= 2 whole
 *                       CTAs of at most 32 blocks each (short sequences), the
 *                       k * pairs CTAs are at least 64 and each streams at
 *                       most 3 blocks more than one of that plan's; with an
 *                       explicit count, for 2 splits on
 *                       at least 128 CTAs; otherwise the combine kernel. */
typedef enum { GQA_REDUCE_AUTO = 0, GQA_REDUCE_COMBINE = 1, GQA_REDUCE_CLUSTER = 2 } gqa_reduction_t;

/* Problem description.  Q is [batch, q_tokens, q_heads, head_dim]; the K
 * and V caches are [batch, max_seqlen, kv_heads, head_dim]; all three are
 * in_dtype (bf16 or fp16).  Scores, softmax and accumulation are fp32; P
 * enters the value MMA in in_dtype. */
typedef struct {
  int batch;       /* B >= 0 */
  int q_tokens;    /* nq >= 1 new query tokens per sequence */
  int q_heads;     /* Hq, a multiple of kv_heads */
  int kv_heads;    /* Hkv >= 1 */
  int head_dim;    /* d: 64, 128 or 256 */
  int max_seqlen;  /* S_max >= 1: cache capacity along positions */
  float scale;     /* softmax scale; 0 selects 1/sqrt(head_dim) */
  int causal;      /* nonzero: causal mask among the nq new tokens */
  int out_dtype;   /* gqa_dtype_t of `out`: FP32, or in_dtype (a 16-bit
                      output of the other 16-bit type is GQA_ERR_UNSUPPORTED) */
  int in_dtype;    /* gqa_dtype_t of q, k_cache, v_cache: BF16 or FP16 */
  int reduction;   /* gqa_reduction_t: how split partials are merged (0 = auto) */
} gqa_desc_t;

/* Limits: q_tokens * (q_heads / kv_heads) <= 32 query rows per KV head, and
 * num_splits <= GQA_MAX_SPLITS. */
#define GQA_MAX_QROWS 32
#define GQA_MAX_SPLITS 64

/*
 * Bytes of device workspace gqa_decode_attn needs for this problem and split
 * request (the fp32 split partials, their LSEs and a per-(batch, KV head)
 * piece count; "Building a Faster GQA Decode Kernel for Blackwell SM100",
 * section "Combining the KV splits").  num_splits: 0 = automatic, 1..64 =
 * exactly that many contiguous 128-position-aligned splits per sequence.
 * Returns 0 when no workspace is needed (a single split), and also for an
 * invalid description.  Depends on the current device (its SM count).  The
 * in-cluster merge needs none.
 */
size_t gqa_decode_workspace_size(const gqa_desc_t* desc, int num_splits);

/*
 * Full decode: split-KV attention kernel, then (when the work was split) the
 * log-sum-exp combine kernel, chained with programmatic dependent launch
 * ("Building a Faster GQA Decode Kernel for Blackwell SM100", section
 * "Starting combine early with PDL").
 *   q          in_dtype [B, nq, Hq, d], 16-byte aligned
 *   k_cache    in_dtype [B, S_max, Hkv, d], 16-byte aligned
 *   v_cache    in_dtype [B, S_max, Hkv, d], 16-byte aligned
 *   seqlens    int32 [B] device array; L_b in [0, S_max] (values outside are
 *              clamped and flagged as GQA_ERR_BAD_SEQLEN by
 *              gqa_decode_get_error).  Positions in [L_b, S_max) may hold any
 *              values, they are never used.
 *   out        [B, nq, Hq, d] of desc->out_dtype, 16-byte aligned; written
 *              in full
 *   lse        fp32 [B, nq, Hq] natural-log LSE of the scaled scores, or NULL
 *   num_splits 0 = automatic (balanced contiguous ranges over all
 *              sequences), 1..64 = min(num_splits, ceil(L_b / 128)) splits
 *              of sequence b, as in gqa_decode_splitkv
 *   workspace  device buffer of >= gqa_decode_workspace_size() bytes,
 *              256-byte aligned (may be NULL when that size is 0); its
 *              contents need no initialisation
 */
gqa_status_t gqa_decode_attn(const gqa_desc_t* desc, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* out, float* lse,
                             int num_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gqa_decode_attn without a caller-provided workspace, for callers that
 * cannot allocate device memory where they call decode: plugins that must
 * stay inside a host framework's own memory arena, serving runtimes that fix
 * their memory footprint at start-up and forbid allocation afterwards, and
 * latency-critical paths that cannot afford cudaMalloc's implicit
 * device-wide synchronisation.  (The pages describe no such entry point; it
 * is this library's addition.)
 *
 * The split partials go to a workspace owned by the library: a static array
 * of GQA_STATIC_WORKSPACE_BYTES in device global memory, which every GPU that
 * loads the library holds until the process exits.  Arguments and results are
 * those of gqa_decode_attn.  A problem whose workspace
 * (gqa_decode_workspace_size) exceeds GQA_STATIC_WORKSPACE_BYTES is rejected
 * with GQA_ERR_WORKSPACE before anything is launched.  The call allocates and
 * frees nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept for the life of the
 * process: resetting a device (cudaDeviceReset) while this library is loaded
 * is not supported.  Every call on a device shares the one array, which
 * keeps the last call's contents, and nothing in it needs clearing: the
 * merge may load slots this call did not write (the partials of empty
 * splits), but their weight is exactly zero (lse = -inf, or a piece count
 * that excludes them), so they never affect the result.  Calls whose kernels
 * overlap on the GPU -- on different streams, or different host threads --
 * race on the array: order them on one stream.
 */
#define GQA_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)
gqa_status_t gqa_decode_attn_static_workspace(const gqa_desc_t* desc, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              const int32_t* seqlens, void* out, float* lse,
                                              int num_splits, void* stream);

/*
 * The two halves of gqa_decode_attn, for callers that want to run other work
 * between them or time them apart.  gqa_decode_attn_split runs the
 * split-KV decode kernel of gqa_decode_attn (same plan, same arguments):
 * rows whose KV range was not split are final in out / lse, split rows leave
 * their partials in the workspace.  gqa_decode_attn_merge then runs the
 * combine kernel of gqa_decode_attn over that workspace (no-op when nothing
 * was split).  The pair, on one stream, equals one gqa_decode_attn call; the
 * workspace must not be reused in between.
 */
gqa_status_t gqa_decode_attn_split(const gqa_desc_t* desc, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* seqlens, void* out,
                                   float* lse, int num_splits, void* workspace,
                                   size_t workspace_bytes, void* stream);
gqa_status_t gqa_decode_attn_merge(const gqa_desc_t* desc, void* out, float* lse, int num_splits,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The split step alone: for each sequence b the KV blocks are cut into
 * splits_b = min(num_splits, ceil(L_b / 128)) (at least 1) contiguous ranges;
 * split s covers blocks [s*nblk/splits_b, (s+1)*nblk/splits_b) with
 * nblk = ceil(L_b / 128).  Writes the normalised partial output and its LSE
 * of every split:
 *   o_part    fp32 [num_splits, B, nq, Hq, d], 16-byte aligned
 *   lse_part  fp32 [num_splits, B, nq, Hq], 16-byte aligned (its rows leave
 *             by bulk async copies; any other address is GQA_ERR_INVALID_ARG
 *             before launch); lse_part = -inf marks an empty split
 *             (s >= splits_b, or no visible key), whose o_part entries are
 *             left unwritten (gqa_decode_combine ignores them)
 * num_splits: 1..64.  gqa_decode_combine merges the result.
 */
gqa_status_t gqa_decode_splitkv(const gqa_desc_t* desc, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* seqlens, int num_splits,
                                float* o_part, float* lse_part, void* stream);

/*
 * Log-sum-exp merge of split partials ("Building a Faster GQA Decode Kernel
 * for Blackwell SM100", section "Combining the KV splits"): per row,
 * M = max_s lse_s, w_s = exp(lse_s - M), O = sum_s w_s O_s / sum_s w_s,
 * lse = M + ln sum_s w_s, summing splits in index order (bit-reproducible).
 * Splits with lse_s = -inf are skipped (their o_part values are ignored and
 * may be anything, NaN included); a row with no valid split gets O = 0,
 * lse = -inf.
 *   o_part    fp32 [num_splits, rows, head_dim], 16-byte aligned
 *   lse_part  fp32 [num_splits, rows]
 *   out       [rows, head_dim] of out_dtype, 16-byte aligned
 *   lse       fp32 [rows] or NULL
 * num_splits: 1..64; head_dim: 64, 128 or 256; rows >= 0.
 */
gqa_status_t gqa_decode_combine(const float* o_part, const float* lse_part, int num_splits,
                                int64_t rows, int head_dim, void* out, int out_dtype, float* lse,
                                void* stream);

/*
 * Reads (and, if `clear` is nonzero, resets) the device error word the
 * kernels set on the current device: GQA_ERR_TIMEOUT if a bounded wait ran
 * out (the kernel then returned early and its outputs are invalid),
 * GQA_ERR_BOUNDS (debug builds only) if a bounds check fired,
 * GQA_ERR_BAD_SEQLEN if a length was clamped, GQA_OK otherwise.  Synchronises
 * with the device (call it after the work of interest has finished).
 * After GQA_ERR_TIMEOUT from a decode kernel, treat the CUDA context as
 * suspect: the kernel's own clean-up waits are bounded too, so asynchronous
 * copies or MMAs it had issued may still have been in flight when it
 * returned.  Rebuild the context before relying on it again.
 */
gqa_status_t gqa_decode_get_error(int clear);

/* Static description of a status code. */
const char* gqa_status_string(gqa_status_t status);

/*
 * Host-side view of the work decomposition the decode kernel will use, for
 * inspection and testing.  seqlens_host: int32 [B] in host memory; sm_count:
 * SMs to plan for (0 = those of the current device; needs no GPU otherwise).  Fills
 * *num_ctas with the grid size, *plan_mode with 0 (fixed splits per sequence),
 * 2 (fixed splits merged inside thread-block clusters of num_splits CTAs,
 * CTA q*k + j taking piece j of the pairs of cluster q)
 * or 1 (balanced contiguous ranges; each non-empty (b, h) pair counts its
 * 128-position blocks plus X units for the item's fixed cost: X = 0 with a
 * grid of k CTAs per pair when k >= 2 fit on the SMs and S_max spans at most
 * 32 k blocks, else every SM and X = 1 for nq * G <= 16, 3 above) and *num_slots
 * with the partial slots per row (0 when no combine runs).  If `items` is not NULL, writes up to
 * max_items records of 8 int32 each -- cta, b, h, blk_begin, blk_end, slot
 * (-1 = final output), first_piece, n_pieces -- in the order each CTA
 * processes them, and returns the total count in *num_items.
 */
gqa_status_t gqa_decode_plan(const gqa_desc_t* desc, const int32_t* seqlens_host, int num_splits,
                             int sm_count, int* num_ctas, int* plan_mode, int* num_slots,
                             int32_t* items, int64_t max_items, int64_t* num_items);

/*
 * Failure-detection self-test: launches one CTA that waits, with the same
 * bounded wait the decode kernel uses, on a barrier nothing will ever
 * complete, for at most timeout_us microseconds.  Afterwards
 * gqa_decode_get_error() reports GQA_ERR_TIMEOUT and the context is intact.
 */
gqa_status_t gqa_decode_selftest_timeout(unsigned int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
