"""The ncu summaries under profiles/ are tied to the decode kernel's code by a
digest that ignores comments and layout: the committed summaries match the
committed sources, a comment edit keeps the digest, a code edit changes it,
and bench.py reads a summary's DRAM bytes and tensor-pipe utilisation only
while they match."""
import glob
import os

import pytest

import bench


def test_committed_summaries_match_the_kernel_sources():
    """Every summary carries the current digest and a positive byte count.
    A kernel edit that is not yet profiled is reported as a skip (bench.py
    then prints traffic: null), not as a failure of the CPU suite."""
    digest = bench.kernel_source_digest()
    paths = sorted(glob.glob(os.path.join(bench.PROFILES, "decode_kernel_*.md")))
    assert paths
    for path in paths:
        workload = os.path.basename(path)[len("decode_kernel_"):-len(".md")]
        traffic, source = bench.ncu_traffic(workload)
        if traffic is None and "changed" in source:
            pytest.skip(f"kernel code {digest} differs from the ncu summaries: re-capture them")
        assert traffic is not None and traffic > 0, (path, source, digest)
        tensor = bench.ncu_tensor_pct(workload)  # reported beside the DRAM figure
        assert tensor is not None and 0 < tensor < 100, (path, tensor)


def test_code_only_ignores_comments_and_layout():
    a = 'int f(int x) {  // first\n  return x + 1; /* two */ }\nconst char* s = "//kept /*kept*/";\n'
    b = 'int f(int x) { return x + 1; }\n// another comment\nconst char* s = "//kept /*kept*/";'
    assert bench._code_only(a) == bench._code_only(b)
    assert "//kept /*kept*/" in bench._code_only(a)
    c = a.replace("x + 1", "x + 2")
    assert bench._code_only(c) != bench._code_only(a)
    assert bench._code_only("char q = '\"'; int y; // \" not a string") == "char q = '\"'; int y;"


def test_summary_ignored_once_the_code_changes(tmp_path, monkeypatch):
    src = tmp_path / "gqa_decode_blackwell_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        with open(os.path.join(bench.ROOT, "gqa_decode_blackwell_gb300", "csrc", name)) as f:
            (src / name).write_text(f.read())
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILES", str(prof))
    (prof / "decode_kernel_ragged.md").write_text(
        f"- kernel_source_sha256: `{bench.kernel_source_digest()}`\n- dram_bytes_per_launch: `930257664`\n")
    assert bench.ncu_traffic("ragged")[0] == 930257664.0
    assert bench.ncu_tensor_pct("ragged") is None  # no such field: reported as null
    with open(prof / "decode_kernel_ragged.md", "a") as f:
        f.write("- tensor_pipe_active_pct: `3.1` (a remark after the value)\n")
    assert bench.ncu_tensor_pct("ragged") == 3.1
    k = src / "decode_kernel.cuh"
    k.write_text(k.read_text() + "\n// a comment\n")
    assert bench.ncu_traffic("ragged")[0] is not None
    k.write_text(k.read_text() + "\nstatic_assert(true, \"\");\n")
    traffic, why = bench.ncu_traffic("ragged")
    assert traffic is None and "changed" in why
    assert bench.ncu_tensor_pct("ragged") is None
