"""GB300 (sm_103a) DSA lightning-indexer: Python binding of libdsa_idx.so.

Thin layer over the C ABI (include/dsa_idx.h): it allocates outputs with
PyTorch, passes raw device pointers and the current CUDA stream, and turns
status codes into exceptions.  Every step of the computation runs in the
library's CUDA kernels; nothing here computes on the CPU and there is no
fallback path when the library or a GPU is missing.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _abi
from ._abi import (DSA_FLAG_COMPRESSED_KEYS, DSA_FLAG_DETERMINISTIC, DSA_FLAG_KPOOL_TAIL,  # noqa: F401
                   DSA_FLAG_SORT_BY_SCORE,
                   DSA_PREC_BF16, DSA_PREC_FP8, DSA_PREC_MXFP8)

__all__ = [
    "DsaError", "preprocess", "quantize_mxfp8", "quantize_fp8_rows", "kpool_compress", "score_topk", "score_topk_kv", "workspace",
    "read_status", "debug_mma_tile", "output_width",
]


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _abi.load()
        name = lib.dsa_idx_status_string(code).decode()
        msg = lib.dsa_idx_last_error().decode()
        super().__init__(f"{where}: {name}: {msg}")
        self.code = code


def _check(code: int, where: str) -> None:
    if code != 0:
        raise DsaError(code, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _prec(p) -> int:
    if isinstance(p, int):
        return p
    return {"bf16": DSA_PREC_BF16, "mxfp8": DSA_PREC_MXFP8, "fp8": DSA_PREC_FP8}[p]


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _abi.DSA_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return _abi.DSA_DTYPE_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _rule(r) -> int:
    return {"nosat": _abi.DSA_MX_SCALE_NOSAT, "floor": _abi.DSA_MX_SCALE_FLOOR}[r] if isinstance(r, str) else r


def output_width(index_topk: int, kpool_size: int = 1, tail: bool = True) -> int:
    return _abi.load().dsa_idx_output_width(index_topk, kpool_size, DSA_FLAG_KPOOL_TAIL if tail else 0)


def workspace(total_tokens: int, num_seqs: int, max_seqlen: int, n_heads: int, head_dim: int,
              index_topk: int, kpool_size: int = 1, prec="bf16", device=None) -> torch.Tensor:
    """Device workspace (uint8, 256-byte aligned) for score_topk."""
    n = _abi.load().dsa_idx_workspace_size(total_tokens, num_seqs, max_seqlen, n_heads, head_dim,
                                           index_topk, kpool_size, _prec(prec))
    if n == 0:
        raise ValueError("invalid workspace sizes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def preprocess(q: torch.Tensor, k: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
               ln_gamma: Optional[torch.Tensor] = None, ln_beta: Optional[torch.Tensor] = None,
               ln_eps: float = 1e-6, rope_dim: int = 64, rope_base: float = 10000.0,
               rope_interleaved: bool = False, rope_fp32: bool = True, out_prec="bf16",
               scale_rule="nosat", out=None):
    """Key LayerNorm -> RoPE -> quantise (dsa_idx_preprocess).

    q [T, H, D], k [T, D] (fp32 or bf16).  Returns (q_op [T*H, D], q_scale or
    None, k_op [T, D], k_scale or None); bf16 for BF16, uint8 E4M3 codes and
    [rows, D/32] UE8M0 bytes for MXFP8."""
    T, H, D = q.shape
    prec = _prec(out_prec)
    if out is None:
        if prec == DSA_PREC_BF16:
            q_op = torch.empty((T * H, D), dtype=torch.bfloat16, device=q.device)
            k_op = torch.empty((T, D), dtype=torch.bfloat16, device=q.device)
            q_sc = k_sc = None
        else:
            q_op = torch.empty((T * H, D), dtype=torch.uint8, device=q.device)
            k_op = torch.empty((T, D), dtype=torch.uint8, device=q.device)
            ns = 1 if prec == DSA_PREC_FP8 else D // 32   # scales per row
            q_sc = torch.empty((T * H, ns), dtype=torch.uint8, device=q.device)
            k_sc = torch.empty((T, ns), dtype=torch.uint8, device=q.device)
    else:
        q_op, q_sc, k_op, k_sc = out
    lib = _abi.load()
    code = lib.dsa_idx_preprocess(
        _ptr(q), _ptr(k), _dtype(q), _ptr(ln_gamma), _ptr(ln_beta), ln_eps, _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, T, max_seqlen, H, D, rope_dim, rope_base, int(rope_interleaved),
        int(rope_fp32), prec, _rule(scale_rule), _ptr(q_op), _ptr(q_sc), _ptr(k_op), _ptr(k_sc),
        _stream())
    _check(code, "dsa_idx_preprocess")
    return q_op, q_sc, k_op, k_sc


def quantize_mxfp8(x: torch.Tensor, scale_rule="nosat") -> Tuple[torch.Tensor, torch.Tensor]:
    """BF16/FP32 [rows, cols] -> (E4M3 codes uint8 [rows, cols], UE8M0 uint8 [rows, cols/32])."""
    x2 = x.reshape(-1, x.shape[-1])
    rows, cols = x2.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    code = _abi.load().dsa_idx_quantize_mxfp8(_ptr(x2), _dtype(x2), rows, cols, _rule(scale_rule),
                                              _ptr(codes), _ptr(scales), _stream())
    _check(code, "dsa_idx_quantize_mxfp8")
    return codes, scales


def quantize_fp8_rows(x: torch.Tensor, scale_rule="nosat") -> Tuple[torch.Tensor, torch.Tensor]:
    """BF16/FP32 [rows, 128] -> (E4M3 codes uint8 [rows, 128], UE8M0 uint8 [rows]): one scale per row."""
    x2 = x.reshape(-1, x.shape[-1])
    rows, cols = x2.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows,), dtype=torch.uint8, device=x.device)
    code = _abi.load().dsa_idx_quantize_fp8_rows(_ptr(x2), _dtype(x2), rows, cols, _rule(scale_rule),
                                                 _ptr(codes), _ptr(scales), _stream())
    _check(code, "dsa_idx_quantize_fp8_rows")
    return codes, scales


def kpool_compress(k: torch.Tensor, gate_bits: torch.Tensor, slot_bias: torch.Tensor,
                   cu_seqlens: torch.Tensor, pool_size: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """Pooled keys (bf16 [T // P, D]) and cu_pools (int32 [B+1])."""
    T, D = k.shape
    kp = torch.empty((T // pool_size, D), dtype=torch.bfloat16, device=k.device)
    cu_pools = torch.empty(cu_seqlens.numel(), dtype=torch.int32, device=k.device)
    code = _abi.load().dsa_idx_kpool_compress(
        _ptr(k), _dtype(k), _ptr(gate_bits), _ptr(slot_bias), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
        T, D, pool_size, _ptr(kp), _ptr(cu_pools), _stream())
    _check(code, "dsa_idx_kpool_compress")
    return kp, cu_pools


def _order_flag(order: str, return_scores: bool = True) -> int:
    if order not in ("index", "score"):
        raise ValueError(f"order must be 'index' or 'score', not {order!r}")
    if order == "score" and not return_scores:
        raise ValueError("order='score' ranks rows by their scores: return_scores must be True")
    return DSA_FLAG_SORT_BY_SCORE if order == "score" else 0


def score_topk(q_op: torch.Tensor, q_scale: Optional[torch.Tensor], k_op: torch.Tensor,
               k_scale: Optional[torch.Tensor], w: torch.Tensor, cu_seqlens: torch.Tensor,
               max_seqlen: int, n_heads: int, index_topk: int, prec="bf16", sm_scale: float = 1.0,
               kpool_size: int = 1, cu_pools: Optional[torch.Tensor] = None, tail: bool = True,
               return_scores: bool = True, ws: Optional[torch.Tensor] = None, out=None,
               compressed: bool = False, order: str = "index"):
    """Fused score + top-k (dsa_idx_score_topk).

    q_op [T*H, D] (bf16 or E4M3 codes), k_op [rows, D], w [T, H] fp32/bf16.
    kpool_size > 1: KPool pools of that size, or with compressed=True the
    compression ratio of caller-provided compressed keys (cu_pools = their
    per-document prefix; indices are reported per compressed key).
    order "index": each row in ascending index order; "score": score
    descending, index ascending (KPool tail tokens stay last).
    Returns (idx int32 [T, W], scores fp32 [T, W] or None, lens int32 [T])."""
    T = w.shape[0]
    D = q_op.shape[-1]
    B = cu_seqlens.numel() - 1
    if compressed:
        flags = DSA_FLAG_DETERMINISTIC | DSA_FLAG_COMPRESSED_KEYS
    else:
        flags = DSA_FLAG_DETERMINISTIC | (DSA_FLAG_KPOOL_TAIL if (kpool_size > 1 and tail) else 0)
    flags |= _order_flag(order, return_scores)
    W = _abi.load().dsa_idx_output_width(index_topk, kpool_size, flags)
    if out is None:
        idx = torch.empty((T, W), dtype=torch.int32, device=q_op.device)
        sc = torch.empty((T, W), dtype=torch.float32, device=q_op.device) if return_scores else None
        lens = torch.empty((T,), dtype=torch.int32, device=q_op.device)
    else:
        idx, sc, lens = out
    if ws is None:
        ws = workspace(T, B, max_seqlen, n_heads, D, index_topk, kpool_size, prec, q_op.device)
    code = _abi.load().dsa_idx_score_topk(
        _ptr(q_op), _ptr(q_scale), _ptr(k_op), _ptr(k_scale), _ptr(w), _dtype(w), sm_scale,
        _ptr(cu_seqlens), B, T, max_seqlen, n_heads, D, index_topk, _prec(prec), flags, kpool_size,
        _ptr(cu_pools), _ptr(idx), _ptr(sc), _ptr(lens), _ptr(ws), ws.numel(), _stream())
    _check(code, "dsa_idx_score_topk")
    return idx, sc, lens


def score_topk_kv(q_op: torch.Tensor, q_scale: Optional[torch.Tensor], k_op: torch.Tensor,
                  k_scale: Optional[torch.Tensor], w: torch.Tensor, cu_seqlens_q: torch.Tensor,
                  cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, n_heads: int,
                  index_topk: int, prec="bf16", sm_scale: float = 1.0, return_scores: bool = True,
                  ws: Optional[torch.Tensor] = None, out=None, order: str = "index"):
    """Fused score + top-k with more keys than queries per document
    (dsa_idx_score_topk_kv): document d's queries are its last T_d tokens.

    q_op [Tq*H, D], k_op [Tk, D], w [Tq, H].  order as in score_topk.
    Returns (idx int32 [Tq, k], scores fp32 [Tq, k] or None, lens int32
    [Tq]); indices are local to the document's keys."""
    Tq, Tk = w.shape[0], k_op.shape[0]
    D = q_op.shape[-1]
    B = cu_seqlens_q.numel() - 1
    if out is None:
        idx = torch.empty((Tq, index_topk), dtype=torch.int32, device=q_op.device)
        sc = torch.empty((Tq, index_topk), dtype=torch.float32, device=q_op.device) if return_scores else None
        lens = torch.empty((Tq,), dtype=torch.int32, device=q_op.device)
    else:
        idx, sc, lens = out
    if ws is None:
        ws = workspace(max(Tq, Tk), B, max(max_seqlen_q, max_seqlen_k), n_heads, D, index_topk, 1, prec,
                       q_op.device)
    code = _abi.load().dsa_idx_score_topk_kv(
        _ptr(q_op), _ptr(q_scale), _ptr(k_op), _ptr(k_scale), _ptr(w), _dtype(w), sm_scale,
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Tq, Tk, max_seqlen_q, max_seqlen_k, n_heads, D,
        index_topk, _prec(prec), DSA_FLAG_DETERMINISTIC | _order_flag(order, return_scores), _ptr(idx), _ptr(sc),
        _ptr(lens), _ptr(ws), ws.numel(), _stream())
    _check(code, "dsa_idx_score_topk_kv")
    return idx, sc, lens


def read_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream and return the device status word."""
    out = ctypes.c_int(0)
    _check(_abi.load().dsa_idx_read_status(_ptr(ws), _stream(), ctypes.byref(out)), "dsa_idx_read_status")
    return out.value


def debug_mma_tile(q_op, q_scale, q_row0: int, k_op, k_scale, k_row0: int, n_cols: int, prec="bf16"):
    """Raw fp32 accumulator [128, n_cols] of one tcgen05 tile (diagnostic)."""
    D = q_op.shape[-1]
    out = torch.empty((128, n_cols), dtype=torch.float32, device=q_op.device)
    ws = torch.empty(256, dtype=torch.uint8, device=q_op.device)
    code = _abi.load().dsa_idx_debug_mma_tile(
        _ptr(q_op), _ptr(q_scale), q_op.shape[0], q_row0, _ptr(k_op), _ptr(k_scale), k_op.shape[0],
        k_row0, D, n_cols, _prec(prec), _ptr(out), _ptr(ws), ws.numel(), _stream())
    _check(code, "dsa_idx_debug_mma_tile")
    return out, ws
