"""index_topk above 2048, up to the supported 4096 (4096 pools in KPool mode),
against the oracle: integer inputs bit-exact (indices, scores, lengths, ties to
the lower index), random operands within the stated tolerances, and rows in
ranking order, including KPool rows of more than 2048 pools, which are ranked
pool by pool (each pool's tokens stay together and ascending)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host
from tests.parity import REL_BF16, REL_MXFP8, compare_topk

pytestmark = pytest.mark.gpu


def _to_bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact for small integers


def _operands(q, k, prec):
    T, H, D = q.shape
    if prec == "bf16":
        return bf16_dev(_to_bf16(q.reshape(T * H, D))), None, bf16_dev(_to_bf16(k)), None
    quant = O.quantize_mxfp8 if prec == "mxfp8" else O.quantize_fp8_rows
    qc, qs, _ = quant(q.reshape(T * H, D))
    kc, ks, _ = quant(k)
    return dev(qc), dev(qs), dev(kc), dev(ks)


def _rows(lens, extra=()):
    cu = np.concatenate([[0], np.cumsum(lens)])
    rows = []
    for d in range(len(lens)):
        a, b = int(cu[d]), int(cu[d + 1])
        rows += list(range(a, min(b, a + 6))) + list(range(max(a, b - 12), b))
    rows += list(extra)
    return np.unique(np.asarray(rows, dtype=np.int64))


@pytest.mark.parametrize("prec,H,k,lens", [
    ("mxfp8", 64, 4096, [6000, 300]),
    ("bf16", 64, 4096, [5200]),
    ("fp8", 64, 3000, [4500, 17]),
    ("mxfp8", 32, 4096, [4600]),
    ("bf16", 16, 2049, [2500, 2049, 2048]),
])
def test_large_topk_integer_exact(prec, H, k, lens):
    """Integer scores full of ties: bit-exact, rows shorter than k select every
    visible key, rows longer than k keep exactly k, ties to the lower index."""
    rng = np.random.default_rng(600 + H + k)
    T, D = sum(lens), 128
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (T, D)).astype(np.float64)
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx, sc, ln = dsa.score_topk(*_operands(q, kk, prec), dev(w), dev(cu), max(lens), H, k, prec)
    torch.cuda.synchronize()
    rows = _rows(lens, extra=np.linspace(0, T - 1, 24).astype(int))
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k, rows=rows)
    gi, gs, gl = host(idx)[rows], host(sc)[rows], host(ln)[rows]
    np.testing.assert_array_equal(gl, ref["len"])
    np.testing.assert_array_equal(gi, ref["idx"])
    np.testing.assert_array_equal(gs, ref["score"].astype(np.float32))


@pytest.mark.parametrize("prec,k", [("mxfp8", 3000), ("mxfp8", 4096), ("bf16", 4096), ("fp8", 4096)])
def test_large_topk_random(prec, k):
    """N(0,1) operands at the target's shape (64 heads, D 128), rows of up to
    9000 keys: scores within the stated tolerance of the oracle's, swaps only
    at the selection boundary."""
    rng = np.random.default_rng(700 + k)
    lens, H, D = [9000, 2000], 64, 128
    T = sum(lens)
    q = rng.standard_normal((T, H, D))
    kk = rng.standard_normal((T, D))
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    if prec == "bf16":
        qb, kb = _to_bf16(q.reshape(T * H, D)), _to_bf16(kk)
        ops = (bf16_dev(qb), None, bf16_dev(kb), None)
        qd, kd = O.bf16_bits_to_float(qb), O.bf16_bits_to_float(kb)
    else:
        quant = O.quantize_mxfp8 if prec == "mxfp8" else O.quantize_fp8_rows
        qc, qs, qd = quant(q.reshape(T * H, D))
        kc, ks, kd = quant(kk)
        ops = (dev(qc), dev(qs), dev(kc), dev(ks))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx, sc, ln = dsa.score_topk(*ops, dev(w), dev(cu), max(lens), H, k, prec, sm_scale=0.5)
    torch.cuda.synchronize()
    rows = _rows(lens, extra=[4095, 4096, 4097, 6000])
    ref = O.indexer_topk(qd.reshape(T, H, D), kd, w.astype(np.float64), cu, k, sm_scale=0.5, rows=rows,
                         with_scale=True)
    compare_topk(host(idx), host(sc), host(ln), ref, REL_BF16 if prec == "bf16" else REL_MXFP8, rows=rows)


def test_large_topk_score_order_integer_exact():
    """Ranking order (score desc, index asc) of rows of up to 4096 entries."""
    rng = np.random.default_rng(801)
    lens, H, D, k = [5000, 40], 64, 128, 4096
    T = sum(lens)
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (T, D)).astype(np.float64)
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    g = dsa.score_topk(*_operands(q, kk, "mxfp8"), dev(w), dev(cu), max(lens), H, k, "mxfp8", order="score")
    torch.cuda.synchronize()
    rows = _rows(lens, extra=np.linspace(0, T - 1, 16).astype(int))
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k, rows=rows, order="score")
    gi, gs, gl = (host(t)[rows] for t in g)
    np.testing.assert_array_equal(gl, ref["len"])
    np.testing.assert_array_equal(gi, ref["idx"])
    np.testing.assert_array_equal(gs, ref["score"].astype(np.float32))


@pytest.mark.parametrize("order", ["index", "score"])
def test_kpool_more_than_2048_pools_integer_exact(order):
    """KPool with index_topk = 16384 tokens (4096 pools of 4) and the tail: in
    ranking order the pools are ranked by score (ties to the lower pool), each
    pool's four tokens together and ascending, the unscored tail last."""
    rng = np.random.default_rng(802)
    lens, H, D, P, k = [18000, 37], 64, 128, 4, 16384
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cp = np.concatenate([[0], np.cumsum([L // P for L in lens])]).astype(np.int32)
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    pk = rng.integers(-3, 4, (T // P, D)).astype(np.float64)      # pooled keys given directly
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    g = dsa.score_topk(bf16_dev(_to_bf16(q.reshape(T * H, D))), None, bf16_dev(_to_bf16(pk)), None, dev(w),
                       dev(cu), max(lens), H, k, "bf16", kpool_size=P, cu_pools=dev(cp), tail=True, order=order)
    torch.cuda.synchronize()
    rows = _rows(lens, extra=[16383, 16384, 16385, 16386, 17000])
    ref = O.kpool_topk(q, pk, w.astype(np.float64), cu, cp, k, P, True, rows=rows, order=order)
    gi, gs, gl = (host(t)[rows] for t in g)
    np.testing.assert_array_equal(gl, ref["len"])
    np.testing.assert_array_equal(gi, ref["idx"])
    np.testing.assert_array_equal(gs, ref["score"].astype(np.float32))


def test_index_topk_above_4096_refused():
    t = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError, match="UNSUPPORTED"):
        dsa.score_topk(t, None, t, None, torch.zeros(1, 64, device="cuda"), dev(np.array([0, 1], np.int32)), 1,
                       64, 4097, "bf16")
