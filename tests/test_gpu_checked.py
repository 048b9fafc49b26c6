"""The checked build (libdsa_idx_checked.so, -DDSA_CHECKED): the stand-in for
a memory checker.  On clean inputs it must give the product library's results
bit for bit, write nothing outside its output buffers (guard rows around every
output hold a canary pattern that must survive), and report DSA_OK; on inputs
with a NaN or Inf (BF16 operands, FP32 head weights, an E4M3 NaN code, a UE8M0
NaN scale) or inconsistent cu_seqlens it must report DSA_ERR_INVALID_ARG in
the status word and leave the outputs untouched.  Nothing here faults: every
bad input is built on the host and caught by the library's own checks."""
import ctypes

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import _abi, build_lib
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host

pytestmark = pytest.mark.gpu

GUARD = 3                      # guard rows before and after every output
CANARY = 0x5A5A5A5A


@pytest.fixture(scope="module")
def chk():
    lib = ctypes.CDLL(build_lib.build_checked())
    for name, (res, args) in _abi.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    assert lib.dsa_idx_version() % 2 == 1
    return lib


def _guarded(rows, width, dtype):
    buf = torch.full(((rows + 2 * GUARD) * width,), CANARY, dtype=torch.int32, device="cuda")
    return buf, buf.view(dtype)[GUARD * width:(GUARD + rows) * width]


def _guards_intact(buf, rows, width):
    h = host(buf)
    return (h[:GUARD * width] == CANARY).all() and (h[(GUARD + rows) * width:] == CANARY).all()


def _call(lib, ops, w, cu, lens, H, k, prec, flags=_abi.DSA_FLAG_DETERMINISTIC, pool=1, cu_pools=None):
    """The checked library's dsa_idx_score_topk with guarded outputs; returns
    (status, idx, scores, lens, guards intact)."""
    q_op, q_sc, k_op, k_sc = ops
    T, D = sum(lens), q_op.shape[-1]
    Wd = lib.dsa_idx_output_width(k, pool, flags)
    bi, idx = _guarded(T, Wd, torch.int32)
    bs, sc = _guarded(T, Wd, torch.float32)
    bl, ln = _guarded(T, 1, torch.int32)
    ws = torch.empty(lib.dsa_idx_workspace_size(T, len(lens), max(lens), H, D, k, pool, prec), dtype=torch.uint8,
                     device="cuda")
    ptr = lambda t: None if t is None else t.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    code = lib.dsa_idx_score_topk(ptr(q_op), ptr(q_sc), ptr(k_op), ptr(k_sc), ptr(w),
                                  _abi.DSA_DTYPE_F32 if w.dtype == torch.float32 else _abi.DSA_DTYPE_BF16, 0.5,
                                  ptr(cu), len(lens), T, max(lens), H, D, k, prec, flags, pool, ptr(cu_pools),
                                  ptr(idx), ptr(sc), ptr(ln), ptr(ws), ws.numel(), st)
    assert code == _abi.DSA_OK, lib.dsa_idx_last_error()
    status = ctypes.c_int(-1)
    assert lib.dsa_idx_read_status(ptr(ws), st, ctypes.byref(status)) == _abi.DSA_OK
    ok = _guards_intact(bi, T, Wd) and _guards_intact(bs, T, Wd) and _guards_intact(bl, T, 1)
    return status.value, host(idx).reshape(T, Wd), host(sc).reshape(T, Wd), host(ln), ok


def _operands(prec, T, H, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T * H, D))
    k = rng.standard_normal((T, D))
    if prec == "bf16":
        qb, kb = O.float_to_bf16_bits(O.round_bf16(q)), O.float_to_bf16_bits(O.round_bf16(k))
        return [bf16_dev(qb), None, bf16_dev(kb), None], _abi.DSA_PREC_BF16
    if prec == "fp8":
        qc, qs, _ = O.quantize_fp8_rows(q)
        kc, ks, _ = O.quantize_fp8_rows(k)
        return [dev(qc), dev(qs), dev(kc), dev(ks)], _abi.DSA_PREC_FP8
    qc, qs, _ = O.quantize_mxfp8(q)
    kc, ks, _ = O.quantize_mxfp8(k)
    return [dev(qc), dev(qs), dev(kc), dev(ks)], _abi.DSA_PREC_MXFP8


@pytest.mark.parametrize("prec", ["bf16", "mxfp8", "fp8"])
@pytest.mark.parametrize("order", ["index", "score"])
def test_checked_build_matches_and_stays_in_bounds(chk, prec, order):
    lens, H, D, k = [300, 5, 700], 64, 128, 64
    T = sum(lens)
    ops, p = _operands(prec, T, H, D, seed=11)
    w = dev((np.random.default_rng(12).standard_normal((T, H)) * 0.2).astype(np.float32))
    cu = dev(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    flags = _abi.DSA_FLAG_DETERMINISTIC | (_abi.DSA_FLAG_SORT_BY_SCORE if order == "score" else 0)
    st, gi, gs, gl, ok = _call(chk, ops, w, cu, lens, H, k, p, flags)
    assert st == _abi.DSA_OK and ok
    ri, rs, rl = dsa.score_topk(*ops, w, cu, max(lens), H, k, prec, sm_scale=0.5, order=order)
    np.testing.assert_array_equal(gi, host(ri))
    np.testing.assert_array_equal(gs, host(rs))
    np.testing.assert_array_equal(gl, host(rl))


def test_checked_build_kpool_with_tail(chk):
    lens, H, D, k, P = [900, 37, 3], 64, 128, 256, 4
    T = sum(lens)
    rng = np.random.default_rng(13)
    qb = W.random_bf16_bits(rng, (T * H, D))
    pb = W.random_bf16_bits(rng, (T // P, D))
    w = dev((rng.standard_normal((T, H)) * 0.125).astype(np.float32))
    cu = dev(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    cp = dev(np.concatenate([[0], np.cumsum([L // P for L in lens])]).astype(np.int32))
    ops = [bf16_dev(qb), None, bf16_dev(pb), None]
    flags = _abi.DSA_FLAG_DETERMINISTIC | _abi.DSA_FLAG_KPOOL_TAIL
    st, gi, gs, gl, ok = _call(chk, ops, w, cu, lens, H, k, _abi.DSA_PREC_BF16, flags, pool=P, cu_pools=cp)
    assert st == _abi.DSA_OK and ok
    ri, rs, rl = dsa.score_topk(*ops, w, cu, max(lens), H, k, "bf16", sm_scale=0.5, kpool_size=P, cu_pools=cp,
                                tail=True)
    np.testing.assert_array_equal(gi, host(ri))
    np.testing.assert_array_equal(gl, host(rl))


@pytest.mark.parametrize("where", ["bf16-q-nan", "bf16-k-inf", "w-inf", "w-nan", "e4m3-nan", "ue8m0-nan"])
def test_checked_build_reports_non_finite_inputs(chk, where):
    lens, H, D, k = [260, 40], 16, 128, 32
    T = sum(lens)
    prec = "bf16" if where.startswith("bf16") or where.startswith("w") else "mxfp8"
    ops, p = _operands(prec, T, H, D, seed=14)
    w = dev((np.random.default_rng(15).standard_normal((T, H)) * 0.2).astype(np.float32))
    if where == "bf16-q-nan":
        ops[0].view(torch.int16)[7 * H + 3, 17] = 0x7FC0
    elif where == "bf16-k-inf":
        ops[2].view(torch.int16)[123, 64] = 0x7F80
    elif where == "w-inf":
        w[5, 2] = float("inf")
    elif where == "w-nan":
        w[T - 1, H - 1] = float("nan")
    elif where == "e4m3-nan":
        ops[2][200, 5] = 0x7F
    else:
        ops[1][9, 2] = 0xFF
    cu = dev(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    st, gi, gs, gl, ok = _call(chk, ops, w, cu, lens, H, k, p)
    assert st == _abi.DSA_ERR_INVALID_ARG, st
    assert ok
    assert (gl == CANARY).all() and (gi == CANARY).all()   # nothing written


def test_checked_build_reports_inconsistent_cu_seqlens(chk):
    lens, H, D, k = [200, 100], 16, 128, 16
    T = sum(lens)
    ops, p = _operands("bf16", T, H, D, seed=16)
    w = dev(np.ones((T, H), np.float32))
    cu = dev(np.array([0, 250, 300], np.int32))        # a document longer than max_seqlen (200)
    st, gi, gs, gl, ok = _call(chk, ops, w, cu, lens, H, k, p)
    assert st == _abi.DSA_ERR_INVALID_ARG and ok
