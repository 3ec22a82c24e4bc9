"""Seeded synthetic inputs: deterministic, of the documented shapes (CPU)."""
import torch

from gqa_decode_blackwell_gb300 import workloads


def test_configs_have_documented_shapes():
    c = workloads.CONFIGS
    assert (c["tiny"].batch, c["tiny"].q_heads, c["tiny"].kv_heads, c["tiny"].head_dim, c["tiny"].seqlen) == \
        (1, 8, 1, 64, 512)
    assert c["tiny"].num_splits == (1, 4) and c["tiny"].out_dtype == "fp32"
    assert (c["llama8b"].batch, c["llama8b"].group, c["llama8b"].head_dim, c["llama8b"].seqlen) == (8, 4, 128, 4096)
    assert (c["llama70b"].batch, c["llama70b"].group, c["llama70b"].seqlen) == (16, 8, 8192)
    assert c["llama70b"].num_splits == (8,)
    assert (c["spec"].q_tokens, c["spec"].causal, c["spec"].group, c["spec"].head_dim) == (4, True, 8, 64)
    assert c["ragged"].ragged == (1024, 131072) and c["ragged"].key_offset_std == 0.5


def test_generator_is_deterministic_and_bf16():
    cfg = workloads.shrink(workloads.CONFIGS["spec"], batch=3, seqlen=300)
    a = workloads.make_inputs(cfg)
    b = workloads.make_inputs(cfg)
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache), (a.seqlens, b.seqlens)):
        assert torch.equal(x, y)
    assert a.q.dtype == a.k_cache.dtype == torch.bfloat16
    assert a.q.shape == (3, 4, 16, 64) and a.k_cache.shape == (3, 300, 2, 64)
    assert a.seqlens.dtype == torch.int32 and a.seqlens.tolist() == [300] * 3


def test_ragged_lengths_and_key_offset():
    cfg = workloads.shrink(workloads.CONFIGS["ragged"], ragged=(10, 200), seqlen=200)
    a = workloads.make_inputs(cfg)
    L = a.seqlens.tolist()
    assert all(10 <= x <= 200 for x in L) and a.k_cache.shape[1] == max(L)
    off = a.extras["key_offset"]
    assert off.shape == (cfg.kv_heads,)
    # the per-head offset moves the mean of that head's keys
    means = a.k_cache.float().mean(dim=(0, 1, 3))
    assert torch.allclose(means, off, atol=0.05)
