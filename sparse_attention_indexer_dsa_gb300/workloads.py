"""Seeded synthetic inputs for the DSA lightning-indexer workloads.

This module only draws random inputs (numpy PCG64); it holds none of the
method's arithmetic and is the one module both the oracle-side tests and the
CUDA-side callers (tests, bench, smoke) share.  The shapes, value
distributions and document-length mix follow the workloads the indexer pages
describe (Megatron-LM PR #8403 "Test": seq 2048, top-k 256, 32 indexer heads;
PR #5992 "Key changes": MXFP8, THD packed sequences; PR #7522 "Changes":
KPool) and the five configurations this library is measured on.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


@dataclass
class Workload:
    name: str
    doc_lens: list            # document lengths (THD packing order)
    n_heads: int
    head_dim: int
    index_topk: int
    prec: str                 # "bf16", "mxfp8" or "fp8" (one scale per vector)
    values: str               # "int" | "normal" | "outlier"
    layernorm: bool = False
    rope_dim: int = 0
    rope_base: float = 10000.0
    rope_fp32: bool = True
    w_std: float = 0.125
    kpool: int = 1
    seed: int = 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.doc_lens))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.doc_lens)]).astype(np.int32)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.doc_lens))

    def causal_pairs(self) -> int:
        """Visible (query, key) pairs: sum over documents of L(L+1)/2 (pool
        mode: visible complete pools)."""
        if self.kpool > 1:
            P = self.kpool
            return int(sum(sum((p + 1) // P for p in range(L)) for L in self.doc_lens))
        return int(sum(L * (L + 1) // 2 for L in self.doc_lens))

    def flops(self) -> float:
        """Algorithmic tensor flops: 2*H*D per visible pair."""
        return 2.0 * self.n_heads * self.head_dim * self.causal_pairs()


def thd_lengths(rng: np.random.Generator, n_docs: int, lo: int, hi: int, total: int) -> list:
    """Lengths drawn uniform in [lo, hi], rescaled to sum to `total` (floored,
    remainder added to the last document)."""
    raw = rng.integers(lo, hi + 1, size=n_docs).astype(np.float64)
    lens = np.floor(raw * total / raw.sum()).astype(np.int64)
    lens[-1] += total - lens.sum()
    return [int(x) for x in lens]


def config(name: str) -> Workload:
    """The named workload (tiny, c2, c3, thd, kpool, target)."""
    if name == "tiny":
        return Workload("tiny", [256], 4, 64, 32, "bf16", "int", seed=1001)
    if name == "c2":
        return Workload("c2", [2048], 32, 128, 256, "bf16", "normal", layernorm=True,
                        rope_dim=64, rope_fp32=True, w_std=1 / np.sqrt(32), seed=1002)
    if name == "c3":
        return Workload("c3", [8192, 8192], 64, 128, 2048, "mxfp8", "normal", layernorm=True,
                        rope_dim=64, rope_fp32=True, w_std=0.125, seed=1003)
    if name == "thd":
        rng = np.random.default_rng(1004)
        lens = thd_lengths(rng, 8, 512, 8192, 32768)
        return Workload("thd", lens, 64, 128, 2048, "mxfp8", "outlier", w_std=0.125, seed=1004)
    if name == "kpool":
        return Workload("kpool", [16384], 64, 128, 2048, "bf16", "normal", w_std=0.125,
                        kpool=4, seed=1005)
    if name == "target":
        return Workload("target", [32768], 64, 128, 2048, "mxfp8", "normal", layernorm=True,
                        rope_dim=64, rope_fp32=True, w_std=0.125, seed=1006)
    raise KeyError(name)


def _truncate_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def make_inputs(wl: Workload, seed: Optional[int] = None) -> dict:
    """Raw inputs of a workload as numpy arrays: q [T,H,D] f32, k [T,D] f32,
    w [T,H] f32, cu_seqlens, and when used ln_gamma/ln_beta [D] f32,
    gate_bits [T] (bf16 bit patterns) and slot_bias [P] f32."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    out = {"cu_seqlens": wl.cu_seqlens}
    if wl.values == "int":
        out["q"] = rng.integers(-3, 4, size=(T, H, D)).astype(np.float32)
        out["k"] = rng.integers(-3, 4, size=(T, D)).astype(np.float32)
        out["w"] = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    else:
        out["q"] = rng.standard_normal((T, H, D), dtype=np.float32)
        out["k"] = rng.standard_normal((T, D), dtype=np.float32)
        if wl.values == "outlier":
            out["q"] *= np.where(rng.random((T, H, D)) < 0.01, 20.0, 1.0).astype(np.float32)
            out["k"] *= np.where(rng.random((T, D)) < 0.01, 20.0, 1.0).astype(np.float32)
        out["w"] = (rng.standard_normal((T, H), dtype=np.float32) * np.float32(wl.w_std)).astype(np.float32)
    if wl.layernorm:
        out["ln_gamma"] = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
        out["ln_beta"] = (0.1 * rng.standard_normal(D)).astype(np.float32)
    if wl.kpool > 1:
        out["gate_bits"] = _truncate_to_bf16_bits(rng.standard_normal(T, dtype=np.float32))
        out["slot_bias"] = (0.5 * rng.standard_normal(wl.kpool)).astype(np.float32)
    return out


def random_bf16_bits(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """BF16 bit patterns of N(0, std^2) draws (FP32 draw, low 16 bits dropped)."""
    return _truncate_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def random_e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniformly drawn finite OCP E4M3 byte codes (0x7F and 0xFF excluded)."""
    c = rng.integers(0, 254, size=shape)
    c = np.where(c >= 0x7F, c + 1, c)          # skip 0x7F
    return c.astype(np.uint8)


def random_ue8m0(rng: np.random.Generator, shape, lo: int = 120, hi: int = 134) -> np.ndarray:
    """UE8M0 scale bytes drawn uniform in [lo, hi]."""
    return rng.integers(lo, hi + 1, size=shape).astype(np.uint8)
