"""Each planted mistake in the oracle must be rejected by at least one pin.

The mutants are compiled from ``oracle/gqa_oracle.c`` with
``-DORACLE_MUTANT=<n>`` (a dropped scale, a wrong head map, a wrong causal
alignment or an off-by-one, a dropped max term, no max subtraction, values
read from the key cache, no normalisation, one key past the end, a sign error
or a missing max in the merge, a missing empty-row case, a transposed cache
layout, a wrong fp16 exponent bias).  CPU only.
"""
import math
import warnings

import numpy as np
import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    1: "score scale dropped",
    2: "head map hq % Hkv",
    3: "top-left causal alignment",
    4: "max term dropped from lse",
    5: "max not subtracted",
    6: "values read from the key cache",
    7: "no normalisation",
    8: "one key past the end",
    9: "merge weight sign",
    10: "merge of an all-empty row",
    11: "cache read as [B, Hkv, S, d]",
    12: "max term dropped from merged lse",
    13: "causal limit off by one",
    14: "fp16 exponent bias 14",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_some_pin_rejects_mutant(mutant, tmp_path):
    path = oracle.build(str(tmp_path / f"libgqa_oracle_m{mutant}.so"), mutant=mutant)
    orc = oracle.Oracle(path)
    rejected_by = None
    with warnings.catch_warnings(), np.errstate(all="ignore"):
        warnings.simplefilter("ignore")
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError, OverflowError):
                rejected_by = pin.__name__
                break
    assert rejected_by is not None, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


# ------------------------------------------------- the split partition
def _ranges(seqlens, num_splits, block, boundary, splits_of, clamp_end=True):
    sl = np.asarray(seqlens, dtype=np.int64)
    begin = np.zeros((num_splits, sl.shape[0]), dtype=np.int32)
    end = np.zeros_like(begin)
    for b, L in enumerate(sl):
        L = max(int(L), 0)
        nblk = -(-L // block)
        sp = splits_of(nblk)
        for s in range(min(sp, num_splits)):
            b0, b1 = boundary(s, nblk, sp), boundary(s + 1, nblk, sp)
            begin[s, b] = b0 * block
            end[s, b] = min(b1 * block, L) if clamp_end else b1 * block
    return begin, end


def _mut_ceil(seqlens, S, block=128, min_blocks=1):
    return _ranges(seqlens, S, block, lambda s, n, k: -(-s * n // k),
                   lambda n: min(max(-(-n // min_blocks), 1), S))


def _mut_no_min_blocks(seqlens, S, block=128, min_blocks=1):
    return _ranges(seqlens, S, block, lambda s, n, k: s * n // k, lambda n: min(max(n, 1), S))


def _mut_end_unclamped(seqlens, S, block=128, min_blocks=1):
    return _ranges(seqlens, S, block, lambda s, n, k: s * n // k,
                   lambda n: min(max(-(-n // min_blocks), 1), S), clamp_end=False)


def _mut_not_capped_by_blocks(seqlens, S, block=128, min_blocks=1):
    return _ranges(seqlens, S, block, lambda s, n, k: s * n // k, lambda n: S)


def _mut_floor_min_blocks(seqlens, S, block=128, min_blocks=1):
    return _ranges(seqlens, S, block, lambda s, n, k: s * n // k, lambda n: min(max(n // min_blocks, 1), S))


SPLIT_MUTANTS = {
    "ceil boundaries": _mut_ceil,
    "min_blocks ignored": _mut_no_min_blocks,
    "last range not clamped to L": _mut_end_unclamped,
    "split count not capped by the block count": _mut_not_capped_by_blocks,
    "floor(nblk / min_blocks) splits": _mut_floor_min_blocks,
}


def test_split_ranges_pin_accepts_the_oracle():
    oracle_pins.pin_split_ranges(None)


@pytest.mark.parametrize("name", sorted(SPLIT_MUTANTS))
def test_split_ranges_pin_rejects_mutant(name):
    with pytest.raises(AssertionError):
        oracle_pins.pin_split_ranges(None, split_ranges=SPLIT_MUTANTS[name])
