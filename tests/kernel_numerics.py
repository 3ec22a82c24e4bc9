"""A model of the decode kernel's floating-point arithmetic, in numpy.

Test infrastructure.  It explains the parity tests' regression bounds by
repeating on the CPU the rounding steps that the kernel takes and the fp64
oracle does not:

- scores in fp32 from exact products of the 16-bit inputs;
- scores scaled into log2 units by one fused multiply-add with a running max.
  The max is refreshed only when some score of the warpgroup's 8 columns
  exceeds it by more than the rescale threshold (8; "Flash Attention 4 -
  warp-role choreography and the edges", section "The correction").  Every
  column of that warpgroup then takes its new max;
- p = 2^t in fp32, summed in fp32 for the denominator but rounded to the
  input type (bf16 or fp16) for the value product;
- each split piece normalised in fp32, its LSE in natural-log units;
- the pieces merged with fp32 weights 2^((lse_s - M) log2 e) in split order,
  and the output rounded to its 16-bit type when it has one.

The model shares nothing with the kernels and is not the oracle: parity is
always checked against the oracle.  A column n of a (batch, KV head) pair is
query token n // G, head n % G of the group, as in the kernel.
"""
import numpy as np

LOG2E = np.float32(1.4426950408889634)
LN2 = 0.6931471805599453
BLOCK = 128
COLS_PER_WARPGROUP = 8


def to_bf16(x):
    """fp32 -> bf16 (round to nearest, ties to even), returned as fp32.
    NaN does not occur here."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def to_fp16(x):
    """fp32 -> fp16 (round to nearest, ties to even), returned as fp32."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


ROUND = {"bf16": to_bf16, "fp16": to_fp16, None: lambda x: np.asarray(x, dtype=np.float32)}


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def piece(qc, k, v, lo, hi, L, nq, G, scale, causal, threshold, p_type="bf16"):
    """One split piece, keys [lo, hi), of one (batch, KV head) pair.
    qc: [C, d] query columns (C = nq G), k, v: [positions, d].
    Returns the normalised O [C, d] and the LSE [C] (natural log), fp32."""
    C, d = qc.shape
    sl2 = f32(np.float32(scale) * LOG2E)
    m = np.full(C, -np.inf, np.float32)  # running max, scaled, log2 units
    l = np.zeros(C, np.float32)
    O = np.zeros((C, d), np.float32)
    tok = np.arange(C) // G
    for b0 in range(lo, hi, BLOCK):
        b1 = min(b0 + BLOCK, hi)
        pos = np.arange(b0, b1)
        s = f32(k[b0:b1].astype(np.float64) @ qc.T.astype(np.float64))  # [n, C]
        vis = pos[:, None] < L
        if causal:
            vis = vis & (pos[:, None] <= L - nq + tok[None, :])
        s = np.where(vis, s, np.float32(-np.inf))
        first = b0 == lo
        # -max as the addend; 2^100 while the max is -inf, so any visible score votes
        nms = np.where(np.isneginf(m), np.float32(2.0 ** 100), -m).astype(np.float32)
        t = f32(s.astype(np.float64) * sl2 + nms)
        bm = s.max(axis=0) * sl2
        for w0 in range(0, C, COLS_PER_WARPGROUP):
            cols = slice(w0, w0 + COLS_PER_WARPGROUP)
            if not (first or bool((t[:, cols] > threshold).any())):
                continue
            mo = m[cols]
            mn = np.maximum(mo, bm[cols]).astype(np.float32)
            ms = np.where(np.isneginf(mn), np.float32(0), mn)
            alpha = np.zeros_like(mo) if first else f32(np.exp2(mo.astype(np.float64) - ms))
            O[cols] = f32(O[cols] * alpha[:, None])
            l[cols] = f32(l[cols] * alpha)
            m[cols] = mn
        ms = np.where(np.isneginf(m), np.float32(0), m)
        t = f32(s.astype(np.float64) * sl2 - ms)
        p = f32(np.exp2(t.astype(np.float64)))
        l = f32(l + p.sum(axis=0, dtype=np.float32))
        pv = ROUND[p_type](p)
        O = f32(O.astype(np.float64) + pv.T.astype(np.float64) @ v[b0:b1].astype(np.float64))
    with np.errstate(divide="ignore", invalid="ignore"):
        Oo = np.where(l[:, None] > 0, f32(O / l[:, None]), np.float32(0))
        lse = np.where(l > 0, f32(LN2 * (m.astype(np.float64) + np.log2(l.astype(np.float64)))),
                       np.float32(-np.inf))
    return Oo, lse


def decode(q, k_cache, v_cache, seqlens, ranges, *, scale, causal=False, threshold=8.0, p_type="bf16",
           out_type="bf16"):
    """q [B, nq, Hq, d], caches [B, S_max, Hkv, d] (float arrays holding the
    16-bit inputs' values), seqlens [B]; ranges(b) -> the (lo, hi) key ranges
    of sequence b's split pieces.  p_type / out_type: the type P is rounded to
    for the value product and the output type ("bf16", "fp16"; None: fp32,
    no rounding).  Returns O [B, nq, Hq, d] and lse [B, nq, Hq] as the
    kernel's arithmetic produces them (float64 arrays)."""
    B, nq, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, nq, Hq, d))
    lse = np.full((B, nq, Hq), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        for h in range(Hkv):
            qc = q[b, :, h * G:(h + 1) * G].reshape(nq * G, d).astype(np.float32)
            Os, Ls = [], []
            for lo, hi in ranges(b):
                o_, l_ = piece(qc, k_cache[b, :, h], v_cache[b, :, h], lo, hi, L, nq, G, scale, causal,
                               threshold, p_type)
                Os.append(o_)
                Ls.append(l_)
            if not Os:
                continue
            Ls = np.array(Ls, np.float32)
            M = Ls.max(axis=0)
            Ms = np.where(np.isneginf(M), np.float32(0), M)
            w = np.where(np.isneginf(Ls), np.float32(0), f32(np.exp2(f32((Ls - Ms) * LOG2E))))
            acc = np.zeros_like(Os[0])
            for s, o_ in enumerate(Os):
                acc = f32(acc + w[s][:, None] * o_)
            W = w.sum(axis=0, dtype=np.float32)
            with np.errstate(divide="ignore", invalid="ignore"):
                O = np.where(W[:, None] > 0, f32(acc * f32(np.float32(1) / W)[:, None]), np.float32(0))
                lrow = np.where(W > 0, M + LN2 * np.log2(W), -np.inf)
            O = ROUND[out_type](O)
            out[b, :, h * G:(h + 1) * G] = O.reshape(nq, G, d)
            lse[b, :, h * G:(h + 1) * G] = lrow.reshape(nq, G)
    return out, lse
