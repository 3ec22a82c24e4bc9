"""The regression bounds of the GPU parity tests, derived on the CPU.

tests/kernel_numerics.py repeats the decode kernel's rounding steps.  These
tests check three things:
- the model itself is right: without its two departures from exact
  arithmetic (P rounded to bf16, a stale running max) it agrees with the
  fp64 oracle to fp32 round-off, causal masking and split merging included;
- the short-row bound REG_ABS is set by the stale max: a peaked row's worst
  error falls when the max is kept current and stays under the bound
  either way;
- the workloads' rows stay well under REG_LONG and REG_LSE.
Split pieces follow the documented partition (oracle.split_ranges) with the
piece counts that the automatic plan takes for these shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_decode_blackwell_gb300 import workloads
from tests import kernel_numerics as km
from tests.tolerances import REG_ABS, REG_LONG, REG_LSE

SHORT = workloads.shrink(workloads.CONFIGS["llama8b"], batch=2, seqlen=700)  # scale 0.3: peaked rows


def _run(cfg, splits, *, scale=0.0, threshold=8.0, p_type="bf16", out_type="bf16", dtype=torch.bfloat16):
    return _compare(workloads.make_inputs(cfg, dtype=dtype), splits, scale=scale, causal=cfg.causal,
                    threshold=threshold, p_type=p_type, out_type=out_type)


def _compare(inp, splits, *, scale=0.0, causal=False, threshold=8.0, p_type="bf16", out_type="bf16"):
    """Max error of the model against the oracle: |dO| (beyond one ulp of
    the output type for 16-bit outputs) and |dlse|, with `splits` pieces per
    sequence."""
    sc = scale if scale else 1.0 / float(inp.q.shape[-1]) ** 0.5
    ref_o, ref_l = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, scale=sc, causal=causal)
    begin, end = oracle.split_ranges(inp.seqlens.tolist(), splits)

    def ranges(b):
        return [(int(begin[s, b]), int(end[s, b])) for s in range(splits)]

    o, l = km.decode(inp.q.float().numpy(), inp.k_cache.float().numpy(), inp.v_cache.float().numpy(),
                     inp.seqlens.numpy(), ranges, scale=sc, causal=causal, threshold=threshold,
                     p_type=p_type, out_type=out_type)
    fin = ~np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ~fin)
    diff = np.abs(o - ref_o)
    if out_type is not None:  # beyond one ulp of the reference, as the GPU tests measure it
        mant, tiny = (7, 2.0 ** -126) if out_type == "bf16" else (10, 2.0 ** -14)
        ax = np.maximum(np.abs(ref_o), tiny)
        diff = diff - np.exp2(np.floor(np.log2(ax)) - mant)
    return float(diff.max()), float(np.abs(l[fin] - ref_l[fin]).max())


def test_bf16_rounding_is_round_to_nearest_even():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4096).astype(np.float32) * 300,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e-39, 65504.0, -2.5e-3])])
    # 1 + 2^-8 and 1 + 3 * 2^-8 sit halfway between bf16 neighbours: ties to even
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(km.to_bf16(x), want)


@pytest.mark.parametrize("name,splits", [("tiny", 1), ("spec", 2), ("short", 4), ("spec-edge", 5)])
def test_model_without_its_roundings_matches_the_oracle(name, splits):
    cfg = {"short": SHORT,
           "spec-edge": workloads.shrink(workloads.CONFIGS["spec"], batch=5, seqlen=1000)}.get(
        name, workloads.CONFIGS.get(name))
    err_o, err_l = _run(cfg, splits, scale=0.3 if name == "short" else 0.0, threshold=0.0, p_type=None,
                        out_type=None)
    assert err_o < 1e-5 and err_l < 1e-5  # fp32 round-off; the modelled roundings cost 1e-4 to 5e-3


def test_stale_max_sets_the_short_row_bound():
    """Peaked rows (scale 0.3, 700 keys, four pieces per pair, as the
    automatic plan takes them): the error with the threshold-8 max is several
    times the error with a current max, and both stay under REG_ABS."""
    stale, lse_err = _run(SHORT, 4, scale=0.3, out_type=None)
    current, _ = _run(SHORT, 4, scale=0.3, out_type=None, threshold=0.0)
    stale16, _ = _run(SHORT, 4, scale=0.3)
    assert 2e-3 < stale < REG_ABS
    assert current < stale / 2
    assert stale16 < REG_ABS and lse_err < REG_LSE


@pytest.mark.parametrize("name,splits", [("llama8b", 2), ("spec", 2), ("llama70b", 8)])
def test_workload_rows_sit_well_under_the_long_bound(name, splits):
    err_o, err_l = _run(workloads.CONFIGS[name], splits)
    assert err_o < REG_LONG / 2 and err_l < REG_LSE / 4


@pytest.mark.parametrize("which,splits", [(0, 8), (1, 3)])
def test_head_dim_256_rows(which, splits):
    """The head_dim 256 parity cases, held to the long-row bound on the GPU.
    The trace shape (32768 keys) sits far below it.  The ragged batch's
    largest error is in its 129-key sequence, a short row whose two pieces
    each take their max exactly: plain bf16 rounding of p, 7.8e-4, with
    only a 1.3x margin to the bound, so the model pins that margin here."""
    err_o, err_l = _compare(workloads.head_dim_256_inputs(which), splits, out_type=None)
    assert err_o < (REG_LONG / 4 if which == 0 else REG_LONG) and err_l < REG_LSE / 4


@pytest.mark.parametrize("name", ["llama8b", "spec"])
def test_fp16_inputs_round_p_three_bits_finer(name):
    """fp16 inputs: P enters the value product in fp16 (10 mantissa bits
    against bf16's 7), so the same shapes drawn in fp16 err several times
    less, far under the long-row bound."""
    cfg = workloads.CONFIGS[name]
    e16, l16 = _run(cfg, 2, p_type="fp16", out_type=None, dtype=torch.float16)
    e_bf, _ = _run(cfg, 2, p_type="bf16", out_type=None)
    assert e16 < e_bf / 4 and e16 < REG_LONG / 10 and l16 < REG_LSE / 4
