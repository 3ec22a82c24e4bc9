"""bench.py's reference arm (the fp64 CPU oracle timed on the host cores):
the JSON line it prints and its behaviour on ranks other than 0 (CPU only)."""
import contextlib
import io
import json
import os

import pytest

import bench
import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _run(argv, env=None):
    buf = io.StringIO()
    old = {k: os.environ.get(k) for k in (env or {})}
    os.environ.update(env or {})
    try:
        with contextlib.redirect_stdout(buf):
            rc = bench.main(argv)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return rc, buf.getvalue()


def test_reference_line_has_the_contract_keys():
    rc, out = _run(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    assert rc == 0
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC
    assert j["unit"] == "GB/s" and j["higher_is_better"] is True and j["value"] > 0
    assert j["steps"] == 2 and j["warmup"] == 1 and j["n_gpus"] == 1
    assert j["config"]["workload"] == "tiny"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_prints_nothing_on_other_ranks():
    rc, out = _run(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"],
                   env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert rc == 0 and out.strip() == ""
