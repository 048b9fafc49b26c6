"""dsa_idx_score_topk_noalloc: the fused score + top-k for callers that cannot
supply device scratch memory (for example code that must not allocate once it
is running, or integrations that only receive input and output tensors).  Its
scratch is a fixed device array inside the library, so the test checks that
two calls in a row, through the C ABI, reproduce the workspace entry point
exactly, and that sizes beyond the array are refused up front."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import _abi
from sparse_attention_indexer_dsa_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(lib, ops, w, cu, lens, H, D, k, prec, out):
    q_op, q_sc, k_op, k_sc = ops
    idx, sc, ln = out
    ptr = lambda t: None if t is None else t.data_ptr()
    code = lib.dsa_idx_score_topk_noalloc(
        ptr(q_op), ptr(q_sc), ptr(k_op), ptr(k_sc), ptr(w), _abi.DSA_DTYPE_F32, 0.5, ptr(cu), len(lens),
        sum(lens), max(lens), H, D, k, prec, _abi.DSA_FLAG_DETERMINISTIC, 1, None, ptr(idx), ptr(sc),
        ptr(ln), torch.cuda.current_stream().cuda_stream)
    return code


@pytest.mark.parametrize("prec", ["bf16", "mxfp8"])
def test_noalloc_matches_workspace_entry_point_twice(prec):
    lib = _abi.load()
    rng = np.random.default_rng(123)
    lens, H, D, k = [700, 1, 260], 64, 128, 96
    T = sum(lens)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    q = torch.from_numpy(rng.standard_normal((T, H, D), dtype=np.float32)).cuda()
    kk = torch.from_numpy(rng.standard_normal((T, D), dtype=np.float32)).cuda()
    w = torch.from_numpy((rng.standard_normal((T, H)) * 0.2).astype(np.float32)).cuda()
    ops = dsa.preprocess(q, kk, cu, max(lens), rope_dim=64, out_prec=prec)
    p = dsa.DSA_PREC_BF16 if prec == "bf16" else dsa.DSA_PREC_MXFP8
    ref_idx, ref_sc, ref_ln = dsa.score_topk(*ops, w, cu, max(lens), H, k, prec, sm_scale=0.5)
    for _ in range(2):
        out = (torch.full((T, k), 7, dtype=torch.int32, device="cuda"),
               torch.full((T, k), 7.0, dtype=torch.float32, device="cuda"),
               torch.full((T,), 7, dtype=torch.int32, device="cuda"))
        assert _noalloc(lib, ops, w, cu, lens, H, D, k, p, out) == _abi.DSA_OK, lib.dsa_idx_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out[0], ref_idx)
        assert torch.equal(out[1], ref_sc)
        assert torch.equal(out[2], ref_ln)


def test_noalloc_refuses_sizes_beyond_its_array():
    lib = _abi.load()
    T = 1 << 20                        # needs ~8 MiB of scratch, above the 4 MiB array
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    P = z.data_ptr()
    code = lib.dsa_idx_score_topk_noalloc(P, None, P, None, P, 0, 1.0, P, 1, T, T, 64, 128, 16, 0, 1, 1,
                                          None, P, None, None, None)
    assert code == _abi.DSA_ERR_WORKSPACE
    assert b"fixed" in lib.dsa_idx_last_error()
