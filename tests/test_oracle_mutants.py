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
