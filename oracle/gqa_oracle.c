/*
 * gqa_oracle.c -- plain fp64 CPU oracle for grouped-query attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py load this library.  It shares no
 * code, header, table or helper with the CUDA library it checks, and the
 * product path never calls it.
 *
 * What it computes, and where the definition comes from:
 *
 *  - Attention forward, S = Q K^T / sqrt(d), P = softmax(S) row-wise,
 *    O = P V ("Optimization diaries: S/P ping-pong for FlashAttention-4
 *    decode", section "Recap on the FA4 forward pass").  Computed exactly,
 *    two-pass: the max over visible scores first, then the sums.  No online
 *    update, no exp2, no splitting: the definition written out.
 *  - Several query heads share one KV head; query head hq reads KV head
 *    floor(hq / G) with G = Hq / Hkv ("Flash Attention 4 - warp-role
 *    choreography and the edges", section "Edge 2 - GQA").
 *  - Causal masking: a query never attends to a key in its future (same
 *    page, section "Edge 1 - causal masking").  Alignment is bottom-right:
 *    the nq new tokens are the last nq of the L_b cached positions, so
 *    token t sees positions j <= L_b - nq + t.
 *  - The log-sum-exp of a row, lse = M + ln(sum_j exp(s_j - M)), natural
 *    log, scores including the 1/sqrt(d) scale.
 *  - A row with no visible key has O = 0 and lse = -inf ("Building a Faster
 *    GQA Decode Kernel for Blackwell SM100", section "Removing the max
 *    reset": an entirely empty sequence produces zero output).
 *  - Split partials and their merge (same page, section "Combining the KV
 *    splits"): a split restricted to key positions [begin, end) yields a
 *    normalised (O_s, lse_s); the merge takes M = max_s lse_s, skips empty
 *    splits, weights w_s = exp(lse_s - M) and returns
 *    O = sum_s w_s O_s / sum_s w_s, lse = M + ln(sum_s w_s).
 *
 * Inputs are the exact bf16 or fp16 values (raw 16-bit patterns), widened to
 * double: bf16 is the upper half of an IEEE binary32; fp16 is IEEE binary16
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits; exponent 0
 * holds zero and the subnormals fraction * 2^-24, exponent 31 inf and NaN).
 *
 * Compile with -DORACLE_MUTANT=<n> to plant one deliberate mistake; the test
 * suite builds each mutant and checks that some pin rejects it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
  int batch;      /* B */
  int q_tokens;   /* nq */
  int q_heads;    /* Hq */
  int kv_heads;   /* Hkv */
  int head_dim;   /* d */
  int max_seqlen; /* S_max: cache capacity along positions */
  double scale;   /* score scale, normally 1/sqrt(d) */
  int causal;     /* bottom-right causal mask among the nq new tokens */
  int in_fp16;    /* inputs are fp16 bit patterns (else bf16) */
} gqa_oracle_shape;

static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double fp16_to_double(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 0x1f, frac = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)frac, -24); /* zero and subnormals */
  } else if (e == 31) {
    mag = frac == 0 ? INFINITY : NAN;
  } else {
#if ORACLE_MUTANT == 14 /* mistake: exponent bias 14 instead of 15 */
    mag = ldexp(1.0 + frac / 1024.0, e - 14);
#else
    mag = ldexp(1.0 + frac / 1024.0, e - 15);
#endif
  }
  return sign ? -mag : mag;
}

/* One input element, widened to double. */
static inline double elem_to_double(int in_fp16, uint16_t bits) {
  return in_fp16 ? fp16_to_double(bits) : bf16_to_double(bits);
}

double gqa_oracle_elem(int in_fp16, uint16_t bits) { return elem_to_double(in_fp16, bits); }

typedef struct {
  const gqa_oracle_shape* sh;
  const uint16_t *q, *k, *v;
  const int32_t* seqlens;
  const int32_t *pos_begin, *pos_end;
  double *out, *lse;
  long row_begin, row_end; /* rows are (b, t, hq) flattened */
  int status;
} oracle_job;

/* Index of element (b, j, h, x) in a cache laid out [B, S_max, Hkv, d]. */
static size_t cache_index(const gqa_oracle_shape* sh, int b, int j, int h, int x) {
#if ORACLE_MUTANT == 11 /* mistake: cache read as [B, Hkv, S_max, d] */
  return (((size_t)b * sh->kv_heads + h) * sh->max_seqlen + j) * sh->head_dim + x;
#else
  return (((size_t)b * sh->max_seqlen + j) * sh->kv_heads + h) * sh->head_dim + x;
#endif
}

static void* oracle_rows(void* arg) {
  oracle_job* job = (oracle_job*)arg;
  const gqa_oracle_shape* sh = job->sh;
  const int nq = sh->q_tokens, Hq = sh->q_heads, Hkv = sh->kv_heads, d = sh->head_dim;
  const int G = Hq / Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)(sh->max_seqlen > 0 ? sh->max_seqlen : 1));
  double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
  double* acc = (double*)malloc(sizeof(double) * (size_t)d);
  if (!s || !qrow || !acc) {
    job->status = -1;
    free(s); free(qrow); free(acc);
    return NULL;
  }
  for (long row = job->row_begin; row < job->row_end; ++row) {
    const int hq = (int)(row % Hq);
    const int t = (int)((row / Hq) % nq);
    const int b = (int)(row / ((long)Hq * nq));
#if ORACLE_MUTANT == 2 /* mistake: head map modulo instead of division */
    const int h = hq % Hkv;
#else
    const int h = hq / G;
#endif
    int L = job->seqlens[b];
    if (L < 0) L = 0;
    if (L > sh->max_seqlen) L = sh->max_seqlen;
    /* visible key positions: [lo, hi) */
    int lo = 0, hi = L;
#if ORACLE_MUTANT == 8 /* mistake: one key past the end */
    hi = L + 1 <= sh->max_seqlen ? L + 1 : L;
#endif
    if (sh->causal) {
#if ORACLE_MUTANT == 3 /* mistake: top-left causal alignment */
      int lim = t + 1;
#elif ORACLE_MUTANT == 13 /* mistake: a token does not see its own position */
      int lim = L - nq + t;
#else
      int lim = L - nq + t + 1;
#endif
      if (lim < hi) hi = lim;
    }
    if (job->pos_begin && job->pos_begin[b] > lo) lo = job->pos_begin[b];
    if (job->pos_end && job->pos_end[b] < hi) hi = job->pos_end[b];
    double* o = job->out + (size_t)row * d;
    if (hi <= lo) {
      for (int x = 0; x < d; ++x) o[x] = 0.0;
      job->lse[row] = -INFINITY;
      continue;
    }
    const uint16_t* qp = job->q + (size_t)row * d; /* q is [B, nq, Hq, d] */
    for (int x = 0; x < d; ++x) qrow[x] = elem_to_double(sh->in_fp16, qp[x]);
    /* pass 1: scores and their max */
    double M = -INFINITY;
    for (int j = lo; j < hi; ++j) {
      double dot = 0.0;
      for (int x = 0; x < d; ++x) dot += qrow[x] * elem_to_double(sh->in_fp16, job->k[cache_index(sh, b, j, h, x)]);
#if ORACLE_MUTANT == 1 /* mistake: scale dropped */
      s[j] = dot;
#else
      s[j] = sh->scale * dot;
#endif
      if (s[j] > M) M = s[j];
    }
    /* pass 2: Z = sum exp(s - M), acc = sum exp(s - M) V_j */
    double Z = 0.0;
    for (int x = 0; x < d; ++x) acc[x] = 0.0;
    for (int j = lo; j < hi; ++j) {
#if ORACLE_MUTANT == 5 /* mistake: max not subtracted */
      const double w = exp(s[j]);
#else
      const double w = exp(s[j] - M);
#endif
      Z += w;
#if ORACLE_MUTANT == 6 /* mistake: values read from the key cache */
      const uint16_t* vsrc = job->k;
#else
      const uint16_t* vsrc = job->v;
#endif
      for (int x = 0; x < d; ++x) acc[x] += w * elem_to_double(sh->in_fp16, vsrc[cache_index(sh, b, j, h, x)]);
    }
#if ORACLE_MUTANT == 7 /* mistake: no normalisation */
    for (int x = 0; x < d; ++x) o[x] = acc[x];
#else
    for (int x = 0; x < d; ++x) o[x] = acc[x] / Z;
#endif
#if ORACLE_MUTANT == 4 /* mistake: max term dropped from the log-sum-exp */
    job->lse[row] = log(Z);
#elif ORACLE_MUTANT == 5
    job->lse[row] = log(Z);
#else
    job->lse[row] = M + log(Z);
#endif
  }
  free(s); free(qrow); free(acc);
  return NULL;
}

/*
 * Attention of every (b, t, hq) row over its visible keys, optionally
 * restricted to key positions [pos_begin[b], pos_end[b]) (NULL = no bound).
 * q: bf16 or fp16 bits [B, nq, Hq, d]; k, v: the same type, [B, S_max, Hkv, d];
 * seqlens: [B] (L_b includes the nq new positions).
 * out: [B, nq, Hq, d] doubles; lse: [B, nq, Hq] doubles (natural log).
 * Returns 0, or -1 on a bad shape / allocation failure.
 */
int gqa_oracle_decode(const gqa_oracle_shape* sh, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const int32_t* seqlens, const int32_t* pos_begin,
                      const int32_t* pos_end, double* out, double* lse, int nthreads) {
  if (!sh || sh->batch < 0 || sh->q_tokens <= 0 || sh->q_heads <= 0 || sh->kv_heads <= 0 ||
      sh->head_dim <= 0 || sh->max_seqlen < 0 || sh->q_heads % sh->kv_heads != 0)
    return -1;
  const long rows = (long)sh->batch * sh->q_tokens * sh->q_heads;
  if (rows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > rows) nthreads = (int)rows;
  oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs); free(tids);
    return -1;
  }
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].sh = sh;
    jobs[i].q = q; jobs[i].k = k; jobs[i].v = v;
    jobs[i].seqlens = seqlens;
    jobs[i].pos_begin = pos_begin; jobs[i].pos_end = pos_end;
    jobs[i].out = out; jobs[i].lse = lse;
    jobs[i].row_begin = rows * i / nthreads;
    jobs[i].row_end = rows * (i + 1) / nthreads;
  }
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tids[i], NULL, oracle_rows, &jobs[i]) != 0) break;
    started = i;
  }
  oracle_rows(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
  /* rows of threads that failed to start are computed here */
  for (int i = started + 1; i < nthreads; ++i) oracle_rows(&jobs[i]);
  int status = 0;
  for (int i = 0; i < nthreads; ++i) status |= jobs[i].status;
  free(jobs); free(tids);
  return status;
}

/*
 * Merge of S split partials per row.  o_part: [S, rows, d]; lse_part:
 * [S, rows] (a split with lse = -inf is empty and is skipped).
 * out: [rows, d]; lse: [rows].  A row whose splits are all empty gives
 * O = 0 and lse = -inf.
 */
int gqa_oracle_combine(int num_splits, long rows, int head_dim, const double* o_part,
                       const double* lse_part, double* out, double* lse) {
  if (num_splits <= 0 || rows < 0 || head_dim <= 0) return -1;
  for (long r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int s = 0; s < num_splits; ++s) {
      const double l = lse_part[(size_t)s * rows + r];
      if (l > M) M = l;
    }
    double* o = out + (size_t)r * head_dim;
#if ORACLE_MUTANT != 10 /* mutant 10 drops the all-empty special case */
    if (M == -INFINITY) {
      for (int x = 0; x < head_dim; ++x) o[x] = 0.0;
      lse[r] = -INFINITY;
      continue;
    }
#endif
    double W = 0.0;
    for (int x = 0; x < head_dim; ++x) o[x] = 0.0;
    for (int s = 0; s < num_splits; ++s) {
      const double l = lse_part[(size_t)s * rows + r];
      if (l == -INFINITY && M != -INFINITY) continue; /* empty split */
#if ORACLE_MUTANT == 9 /* mistake: weight exponent with the wrong sign */
      const double w = exp(M - l);
#else
      const double w = exp(l - M);
#endif
      W += w;
      const double* os = o_part + ((size_t)s * rows + r) * head_dim;
      for (int x = 0; x < head_dim; ++x) o[x] += w * os[x];
    }
    for (int x = 0; x < head_dim; ++x) o[x] /= W;
#if ORACLE_MUTANT == 12 /* mistake: max term dropped from the merged lse */
    lse[r] = log(W);
#else
    lse[r] = M + log(W);
#endif
  }
  return 0;
}
