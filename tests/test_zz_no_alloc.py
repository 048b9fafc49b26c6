"""dsa_idx_score_topk_noalloc: the fused score + top-k for callers that cannot
supply device scratch memory (for example code that must not allocate once it
is running, or integrations that only receive input and output tensors).  Its
scratch is a fixed device array inside the library, so the tests check that
two calls in a row, through the C ABI, reproduce the workspace entry point
exactly (plain keys, rows in ranking order, KPool pools with the tail), that
the status word of a call whose bounded device wait ran out can be read back
through dsa_idx_score_topk_noalloc_status (and the next call runs clean), and
that sizes beyond the array are refused up front."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import _abi
from sparse_attention_indexer_dsa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(lib, ops, w, cu, lens, H, D, k, prec, out, flags=_abi.DSA_FLAG_DETERMINISTIC, pool=1, cu_pools=None):
    q_op, q_sc, k_op, k_sc = ops
    idx, sc, ln = out
    ptr = lambda t: None if t is None else t.data_ptr()
    code = lib.dsa_idx_score_topk_noalloc(
        ptr(q_op), ptr(q_sc), ptr(k_op), ptr(k_sc), ptr(w), _abi.DSA_DTYPE_F32, 0.5, ptr(cu), len(lens),
        sum(lens), max(lens), H, D, k, prec, flags, pool, ptr(cu_pools), ptr(idx), ptr(sc),
        ptr(ln), torch.cuda.current_stream().cuda_stream)
    return code


def _status(lib):
    st = ctypes.c_int(-1)
    assert lib.dsa_idx_score_topk_noalloc_status(torch.cuda.current_stream().cuda_stream,
                                                 ctypes.byref(st)) == _abi.DSA_OK
    return st.value


def _inputs(prec, lens, H, D, seed=123):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    q = torch.from_numpy(rng.standard_normal((T, H, D), dtype=np.float32)).cuda()
    kk = torch.from_numpy(rng.standard_normal((T, D), dtype=np.float32)).cuda()
    w = torch.from_numpy((rng.standard_normal((T, H)) * 0.2).astype(np.float32)).cuda()
    ops = dsa.preprocess(q, kk, cu, max(lens), rope_dim=64, out_prec=prec)
    return cu, kk, w, ops


def _twice(lib, ops, w, cu, lens, H, D, k, p, W_, ref, **kw):
    T = sum(lens)
    for _ in range(2):
        out = (torch.full((T, W_), 7, dtype=torch.int32, device="cuda"),
               torch.full((T, W_), 7.0, dtype=torch.float32, device="cuda"),
               torch.full((T,), 7, dtype=torch.int32, device="cuda"))
        assert _noalloc(lib, ops, w, cu, lens, H, D, k, p, out, **kw) == _abi.DSA_OK, lib.dsa_idx_last_error()
        torch.cuda.synchronize()
        assert _status(lib) == _abi.DSA_OK
        for a, b in zip(out, ref):
            assert torch.equal(a, b)


@pytest.mark.parametrize("prec", ["bf16", "mxfp8", "fp8"])
@pytest.mark.parametrize("order", ["index", "score"])
def test_noalloc_matches_workspace_entry_point_twice(prec, order):
    lib = _abi.load()
    lens, H, D, k = [700, 1, 260], 64, 128, 96
    cu, _, w, ops = _inputs(prec, lens, H, D)
    p = {"bf16": dsa.DSA_PREC_BF16, "mxfp8": dsa.DSA_PREC_MXFP8, "fp8": dsa.DSA_PREC_FP8}[prec]
    ref = dsa.score_topk(*ops, w, cu, max(lens), H, k, prec, sm_scale=0.5, order=order)
    flags = _abi.DSA_FLAG_DETERMINISTIC | (_abi.DSA_FLAG_SORT_BY_SCORE if order == "score" else 0)
    _twice(lib, ops, w, cu, lens, H, D, k, p, k, ref, flags=flags)


def test_noalloc_kpool_with_tail_matches_twice():
    """KPool pools of 4 with the tail: the pooled keys come from
    dsa_idx_kpool_compress; the scratch holds the same work list."""
    lib = _abi.load()
    lens, H, D, k, P = [900, 37, 3], 64, 128, 256, 4
    cu, kk, w, ops = _inputs("bf16", lens, H, D, seed=321)
    rng = np.random.default_rng(322)
    gate = torch.from_numpy(W.random_bf16_bits(rng, (sum(lens),)).view(np.int16)).cuda()
    bias = torch.from_numpy((0.5 * rng.standard_normal(P)).astype(np.float32)).cuda()
    kp, cp = dsa.kpool_compress(kk, gate, bias, cu, P)
    ops = (ops[0], None, kp, None)
    ref = dsa.score_topk(*ops, w, cu, max(lens), H, k, "bf16", sm_scale=0.5, kpool_size=P, cu_pools=cp, tail=True)
    flags = _abi.DSA_FLAG_DETERMINISTIC | _abi.DSA_FLAG_KPOOL_TAIL
    _twice(lib, ops, w, cu, lens, H, D, k, dsa.DSA_PREC_BF16, k + P - 1, ref, flags=flags, pool=P, cu_pools=cp)


def test_noalloc_timeout_status_is_readable_and_next_call_is_clean():
    """A bounded device wait that runs out (the producer withholds its first
    key stage through the library's test hook, 50 ms limit) is reported by
    dsa_idx_score_topk_noalloc_status; the next call runs clean."""
    lib = _abi.load()
    lens, H, D, k = [700], 64, 128, 32
    cu, _, w, ops = _inputs("bf16", lens, H, D, seed=5)
    T = sum(lens)
    out = (torch.empty((T, k), dtype=torch.int32, device="cuda"), torch.empty((T, k), dtype=torch.float32, device="cuda"),
           torch.empty((T,), dtype=torch.int32, device="cuda"))
    try:
        lib.dsa_idx_test_set_timeout_ns(50_000_000)
        lib.dsa_idx_test_set_fault_inject(1)
        assert _noalloc(lib, ops, w, cu, lens, H, D, k, dsa.DSA_PREC_BF16, out) == _abi.DSA_OK
        assert _status(lib) == _abi.DSA_ERR_TIMEOUT
    finally:
        lib.dsa_idx_test_set_fault_inject(0)
        lib.dsa_idx_test_set_timeout_ns(2_000_000_000)
    ref = dsa.score_topk(*ops, w, cu, max(lens), H, k, "bf16", sm_scale=0.5)
    _twice(lib, ops, w, cu, lens, H, D, k, dsa.DSA_PREC_BF16, k, ref)


def test_noalloc_refuses_sizes_beyond_its_array():
    lib = _abi.load()
    T = 1 << 20                        # needs ~8 MiB of scratch, above the 4 MiB array
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    P = z.data_ptr()
    code = lib.dsa_idx_score_topk_noalloc(P, None, P, None, P, 0, 1.0, P, 1, T, T, 64, 128, 16, 0, 1, 1,
                                          None, P, None, None, None)
    assert code == _abi.DSA_ERR_WORKSPACE
    assert b"fixed" in lib.dsa_idx_last_error()
