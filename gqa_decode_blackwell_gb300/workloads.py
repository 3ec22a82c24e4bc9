"""Seeded synthetic decode workloads: shapes and input generators only.

This module holds no attention arithmetic.  Both the CUDA path's tests and
the CPU oracle draw their inputs from here, so that the two sides see the
same bf16 values.

Recipe (every config): a CPU ``torch.Generator`` seeded with the config's
seed; draw order lengths (ragged config only), then q, then k one batch
entry at a time, then v one batch entry at a time, then the per-KV-head key
offsets (ragged config only).  Every tensor is drawn as fp32 ``randn`` and
rounded to bf16 (round-to-nearest-even, torch's ``.to``).  The cache
capacity S_max is the longest sequence, so positions past a shorter
sequence's length hold random (finite) values that the kernel must mask.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    q_tokens: int
    q_heads: int
    kv_heads: int
    head_dim: int
    seqlen: int                       # KV length of every sequence (includes the new tokens)
    seed: int
    causal: bool = False
    out_dtype: str = "bf16"           # "bf16" or "fp32"
    num_splits: Tuple[int, ...] = (0,)  # 0 = automatic split selection
    ragged: Optional[Tuple[int, int]] = None  # inclusive [lo, hi] for uniform lengths
    key_offset_std: float = 0.0       # std of a per-KV-head constant added to every key element
    description: str = ""

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads


# The five synthetic decode shapes.  Lengths include the new query tokens.
CONFIGS = {
    "tiny": DecodeConfig(
        "tiny", batch=1, q_tokens=1, q_heads=8, kv_heads=1, head_dim=64, seqlen=512, seed=1,
        out_dtype="fp32", num_splits=(1, 4),
        description="tiny GQA decode: B1, 8 query heads on 1 KV head, d64, L512, fp32 out"),
    "llama8b": DecodeConfig(
        "llama8b", batch=8, q_tokens=1, q_heads=32, kv_heads=8, head_dim=128, seqlen=4096, seed=2,
        description="Llama-3.1-8B-shaped decode: B8, 32/8 heads, d128, L4096, bf16 out"),
    "llama70b": DecodeConfig(
        "llama70b", batch=16, q_tokens=1, q_heads=64, kv_heads=8, head_dim=128, seqlen=8192, seed=3,
        num_splits=(8,),
        description="70B-shaped decode: B16, 64/8 heads, d128, L8192, 8 KV splits"),
    "spec": DecodeConfig(
        "spec", batch=32, q_tokens=4, q_heads=16, kv_heads=2, head_dim=64, seqlen=2048, seed=4,
        causal=True,
        description="speculative decode: B32, 4 new causal tokens, 16/2 heads, d64, L2048"),
    "ragged": DecodeConfig(
        "ragged", batch=4, q_tokens=1, q_heads=64, kv_heads=8, head_dim=128, seqlen=131072, seed=5,
        ragged=(1024, 131072), key_offset_std=0.5,
        description="long-context ragged decode: B4, 64/8 heads, d128, L~U[1024,131072], key offset"),
}

CONFIG_ORDER = ("tiny", "llama8b", "llama70b", "spec", "ragged")


@dataclass
class DecodeInputs:
    config: DecodeConfig
    q: torch.Tensor          # bf16 [B, nq, Hq, d]
    k_cache: torch.Tensor    # bf16 [B, S_max, Hkv, d]
    v_cache: torch.Tensor    # bf16 [B, S_max, Hkv, d]
    seqlens: torch.Tensor    # int32 [B]
    scale: float
    extras: dict = field(default_factory=dict)

    @property
    def max_seqlen(self) -> int:
        return int(self.k_cache.shape[1])

    def kv_bytes(self) -> int:
        """Bytes of K and V a decode must read: 4*d bytes per position per KV head
        (2-byte elements, bf16 or fp16)."""
        c = self.config
        return int(self.seqlens.clamp(min=0).sum().item()) * c.kv_heads * c.head_dim * 2 * 2

    def to(self, device) -> "DecodeInputs":
        return DecodeInputs(self.config, self.q.to(device), self.k_cache.to(device), self.v_cache.to(device),
                            self.seqlens.to(device), self.scale, dict(self.extras))


def seqlens_for(cfg: DecodeConfig, gen: torch.Generator) -> torch.Tensor:
    if cfg.ragged is not None:
        lo, hi = cfg.ragged
        return torch.randint(lo, hi + 1, (cfg.batch,), generator=gen, dtype=torch.int64).to(torch.int32)
    return torch.full((cfg.batch,), cfg.seqlen, dtype=torch.int32)


def make_inputs(cfg: DecodeConfig, seed: Optional[int] = None, capacity: Optional[int] = None,
                dtype: torch.dtype = torch.bfloat16) -> DecodeInputs:
    """Seeded CPU inputs for a config (see the module docstring for the recipe);
    dtype: the element type q, k and v are rounded to (bf16 or fp16)."""
    if dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"inputs are bf16 or fp16, not {dtype}")
    gen = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    seqlens = seqlens_for(cfg, gen)
    s_max = int(seqlens.max().item()) if cfg.batch > 0 else 0
    if capacity is not None:
        s_max = max(s_max, int(capacity))
    B, nq, Hq, Hkv, d = cfg.batch, cfg.q_tokens, cfg.q_heads, cfg.kv_heads, cfg.head_dim
    q = torch.randn(B, nq, Hq, d, generator=gen).to(dtype)
    k32 = [torch.randn(s_max, Hkv, d, generator=gen) for _ in range(B)]
    v = torch.stack([torch.randn(s_max, Hkv, d, generator=gen).to(dtype) for _ in range(B)]) \
        if B > 0 else torch.empty(0, s_max, Hkv, d, dtype=dtype)
    extras = {}
    if cfg.key_offset_std > 0:
        off = torch.randn(Hkv, generator=gen) * cfg.key_offset_std
        extras["key_offset"] = off
        k32 = [kb + off.view(1, Hkv, 1) for kb in k32]
    k = torch.stack([kb.to(dtype) for kb in k32]) if B > 0 else torch.empty_like(v)
    return DecodeInputs(cfg, q, k, v, seqlens, 1.0 / float(d) ** 0.5, extras)


def shrink(cfg: DecodeConfig, **changes) -> DecodeConfig:
    """A smaller variant of a config (same structure) for fast parity tests."""
    return replace(cfg, **changes)


def head_dim_256_inputs(which: int) -> DecodeInputs:
    """head_dim 256 test inputs, seeded randn rounded to bf16 (seed 600 +
    which; draw order q, k, v), scale 1/16.  which = 0: the split-reduction
    trace shape of "Building a Faster GQA Decode Kernel for Blackwell SM100"
    (one sequence of 32768 positions, 32 query heads on one KV head); which =
    1: a 16-column batch of lengths 9001, 3000 and 129."""
    gen = torch.Generator().manual_seed(600 + which)
    if which == 0:
        B, nq, Hq, Hkv, lens = 1, 1, 32, 1, [32768]
    else:
        B, nq, Hq, Hkv, lens = 3, 1, 16, 2, [9001, 3000, 129]
    s_max = max(lens)
    q = torch.randn(B, nq, Hq, 256, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, s_max, Hkv, 256, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, s_max, Hkv, 256, generator=gen).to(torch.bfloat16)
    return DecodeInputs(None, q, k, v, torch.tensor(lens, dtype=torch.int32), 1 / 16)
