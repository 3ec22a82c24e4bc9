"""The C-ABI library loads, exports what the header declares, and rejects
invalid arguments before touching the GPU (CPU only)."""
import ctypes

import pytest

import gqa_decode_blackwell_gb300 as g
from gqa_decode_blackwell_gb300 import build as gbuild


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return g.lib()


def test_exports_every_header_function(L):
    names = g.header_functions()
    assert {"gqa_decode_attn", "gqa_decode_combine", "gqa_decode_splitkv", "gqa_decode_workspace_size",
            "gqa_decode_get_error", "gqa_status_string", "gqa_decode_plan",
            "gqa_decode_selftest_timeout"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(8):
        assert g.gqa_status_string(code) not in ("", "unknown status")
    assert g.gqa_status_string(99) == "unknown status"


def _desc(**kw):
    base = dict(batch=2, q_tokens=1, q_heads=8, kv_heads=2, head_dim=128, max_seqlen=256, scale=0.0, causal=0,
                out_dtype=0)
    base.update(kw)
    return g.gqa_desc_t(**base)


ALIGNED = 1 << 20   # fake, 16-byte aligned non-null "device" addresses: never dereferenced
MISALIGNED = ALIGNED + 2


def _attn(L, desc, q=ALIGNED, k=ALIGNED, v=ALIGNED, sl=ALIGNED, out=ALIGNED, lse=None, splits=0, ws=None, wsb=0):
    return L.gqa_decode_attn(ctypes.byref(desc), q, k, v, sl, out, lse, splits, ws, wsb, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(head_dim=96), g.GQA_ERR_UNSUPPORTED),
    (dict(head_dim=512), g.GQA_ERR_UNSUPPORTED),
    (dict(head_dim=192), g.GQA_ERR_UNSUPPORTED),
    (dict(q_heads=6, kv_heads=4), g.GQA_ERR_INVALID_ARG),
    (dict(q_tokens=0), g.GQA_ERR_INVALID_ARG),
    (dict(batch=-1), g.GQA_ERR_INVALID_ARG),
    (dict(max_seqlen=0), g.GQA_ERR_INVALID_ARG),
    (dict(out_dtype=7), g.GQA_ERR_INVALID_ARG),
    (dict(scale=-1.0), g.GQA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), g.GQA_ERR_INVALID_ARG),
    (dict(q_heads=64, kv_heads=1), g.GQA_ERR_UNSUPPORTED),   # 64 query rows per KV head
    (dict(q_tokens=8, q_heads=16, kv_heads=2), g.GQA_ERR_UNSUPPORTED),
])
def test_bad_descriptions(L, kw, expect):
    assert _attn(L, _desc(**kw)) == expect


def test_null_and_misaligned_pointers(L):
    d = _desc()
    assert L.gqa_decode_attn(None, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, 0, None, 0, None) \
        == g.GQA_ERR_INVALID_ARG
    for kw in (dict(q=None), dict(k=None), dict(v=None), dict(sl=None), dict(out=None),
               dict(q=MISALIGNED), dict(k=MISALIGNED), dict(v=MISALIGNED), dict(out=MISALIGNED),
               dict(sl=ALIGNED + 1), dict(lse=ALIGNED + 2)):
        assert _attn(L, d, **kw) == g.GQA_ERR_INVALID_ARG, kw


def test_bad_split_counts(L):
    d = _desc()
    assert _attn(L, d, splits=-1) == g.GQA_ERR_INVALID_ARG
    assert _attn(L, d, splits=65) == g.GQA_ERR_INVALID_ARG
    rc = L.gqa_decode_splitkv(ctypes.byref(d), ALIGNED, ALIGNED, ALIGNED, ALIGNED, 0, ALIGNED, ALIGNED, None)
    assert rc == g.GQA_ERR_INVALID_ARG
    rc = L.gqa_decode_splitkv(ctypes.byref(d), ALIGNED, ALIGNED, ALIGNED, ALIGNED, 2, MISALIGNED, ALIGNED, None)
    assert rc == g.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("G", [4, 8, 3])
def test_splitkv_rejects_lse_part_off_16_bytes(L, G):
    """The kernel writes lse_part rows with bulk async copies (16-byte
    aligned addresses only), so a 4- or 8-byte aligned lse_part is refused
    before anything is launched -- for every group size, including those
    whose rows would be 16-byte multiples."""
    d = _desc(q_heads=2 * G, kv_heads=2)
    for off in (4, 8, 12):
        rc = L.gqa_decode_splitkv(ctypes.byref(d), ALIGNED, ALIGNED, ALIGNED, ALIGNED, 2, ALIGNED, ALIGNED + off,
                                  None)
        assert rc == g.GQA_ERR_INVALID_ARG, off


def test_empty_batch_is_a_no_op(L):
    assert _attn(L, _desc(batch=0)) == g.GQA_OK


def test_combine_argument_checks(L):
    C = L.gqa_decode_combine
    assert C(ALIGNED, ALIGNED, 0, 4, 128, ALIGNED, 0, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(ALIGNED, ALIGNED, 65, 4, 128, ALIGNED, 0, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(ALIGNED, ALIGNED, 2, -1, 128, ALIGNED, 0, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(ALIGNED, ALIGNED, 2, 4, 80, ALIGNED, 0, None, None) == g.GQA_ERR_UNSUPPORTED
    assert C(ALIGNED, ALIGNED, 2, 4, 128, ALIGNED, 3, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(MISALIGNED, ALIGNED, 2, 4, 128, ALIGNED, 0, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(None, ALIGNED, 2, 4, 128, ALIGNED, 0, None, None) == g.GQA_ERR_INVALID_ARG
    assert C(ALIGNED, ALIGNED, 2, 0, 128, ALIGNED, 0, None, None) == g.GQA_OK


def test_selftest_argument_checks(L):
    assert L.gqa_decode_selftest_timeout(0, None) == g.GQA_ERR_INVALID_ARG
    assert L.gqa_decode_selftest_timeout(11_000_000, None) == g.GQA_ERR_INVALID_ARG


def test_workspace_size_of_invalid_description_is_zero(L):
    assert L.gqa_decode_workspace_size(ctypes.byref(_desc(head_dim=96)), 0) == 0
    assert L.gqa_decode_workspace_size(None, 0) == 0


def test_header_is_plain_c_and_links(L, tmp_path):
    """A C99 translation unit that includes the header and calls every
    declared function compiles warning-free and links against the library."""
    import os
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    calls = {
        "gqa_decode_workspace_size": "(void)gqa_decode_workspace_size(&d, 0);",
        "gqa_decode_attn": "(void)gqa_decode_attn(&d, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);",
        "gqa_decode_attn_static_workspace": "(void)gqa_decode_attn_static_workspace(&d, 0, 0, 0, 0, 0, 0, 0, 0);",
        "gqa_decode_attn_split": "(void)gqa_decode_attn_split(&d, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);",
        "gqa_decode_attn_merge": "(void)gqa_decode_attn_merge(&d, 0, 0, 0, 0, 0, 0);",
        "gqa_decode_splitkv": "(void)gqa_decode_splitkv(&d, 0, 0, 0, 0, 1, 0, 0, 0);",
        "gqa_decode_combine": "(void)gqa_decode_combine(0, 0, 1, 0, 64, 0, GQA_DTYPE_FP32, 0, 0);",
        "gqa_decode_get_error": "(void)gqa_decode_get_error(0);",
        "gqa_status_string": "(void)gqa_status_string(GQA_OK);",
        "gqa_decode_plan": "(void)gqa_decode_plan(&d, 0, 0, 1, &n, &m, &s, 0, 0, &ni);",
        "gqa_decode_selftest_timeout": "(void)gqa_decode_selftest_timeout(0u, 0);",
    }
    assert set(calls) == set(g.header_functions())
    src = tmp_path / "use.c"
    src.write_text('#include "gqa_decode.h"\n'
                   "int main(void) {\n"
                   "  gqa_desc_t d = {0};\n  int n = 0, m = 0, s = 0;\n  int64_t ni = 0;\n"
                   + "".join(f"  {c}\n" for c in calls.values()) +
                   "  (void)n; (void)m; (void)s; (void)ni;\n  return 0;\n}\n")
    lib = gbuild.LIB
    exe = tmp_path / "use"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(gbuild.ROOT, "include"), str(src), lib, "-o", str(exe)], check=True)
