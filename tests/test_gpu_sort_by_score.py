"""Rows in ranking order (DSA_FLAG_SORT_BY_SCORE): score descending, index
ascending, the order of the repeated-varlen-ends regression rows in PR #8403's
review ("Preservation and acceptance").  Integer inputs make every score
exact, so the GPU rows must equal the oracle's order="score" rows bit for bit;
on float inputs the ranking-order row must be the index-order row reordered by
the GPU's own scores."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from tests.gpu_util import bf16_dev, dev, host

pytestmark = pytest.mark.gpu


def _to_bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact for small integers


def _ints(rng, lens, H, D, qmax=3, wmax=2):
    T = sum(lens)
    q = rng.integers(-qmax, qmax + 1, (T, H, D)).astype(np.float64)
    k = rng.integers(-qmax, qmax + 1, (T, D)).astype(np.float64)
    w = rng.integers(-wmax, wmax + 1, (T, H)).astype(np.float32)
    return q, k, w


def _operands(q, k, prec):
    T, H, D = q.shape
    if prec == "bf16":
        return bf16_dev(_to_bf16(q.reshape(T * H, D))), None, bf16_dev(_to_bf16(k)), None
    if prec == "mxfp8":
        qc, qs, _ = O.quantize_mxfp8(q.reshape(T * H, D))
        kc, ks, _ = O.quantize_mxfp8(k)
        return dev(qc), dev(qs), dev(kc), dev(ks)
    qc, qs, _ = O.quantize_fp8_rows(q.reshape(T * H, D))
    kc, ks, _ = O.quantize_fp8_rows(k)
    return dev(qc), dev(qs), dev(kc), dev(ks)


def _check_exact(g, ref, rows=None):
    gi, gs, gl = (host(t) for t in g)
    if rows is not None:
        gi, gs, gl = gi[rows], gs[rows], gl[rows]
    np.testing.assert_array_equal(gl, ref["len"])
    np.testing.assert_array_equal(gi, ref["idx"])
    np.testing.assert_array_equal(gs, ref["score"].astype(np.float32))


@pytest.mark.parametrize("prec,H,k,lens", [
    ("bf16", 64, 40, [300, 77, 1]),
    ("bf16", 16, 300, [700, 129]),
    ("mxfp8", 64, 2048, [2600]),
    ("mxfp8", 32, 1, [130, 5]),
    ("fp8", 64, 1000, [1500, 260]),
    ("bf16", 4, 7, [260, 3, 0, 2]),
])
def test_score_order_integer_exact(prec, H, k, lens):
    rng = np.random.default_rng(500 + H + k)
    q, kk, w = _ints(rng, lens, H, 128)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    g = dsa.score_topk(*_operands(q, kk, prec), dev(w), dev(cu), max(lens), H, k, prec, order="score")
    torch.cuda.synchronize()
    T = sum(lens)
    rows = np.unique(np.concatenate([np.arange(0, min(T, 40)), np.arange(max(0, T - 40), T),
                                     np.linspace(0, T - 1, 40).astype(int)])) if T > 0 else np.arange(0)
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k, rows=rows, order="score")
    _check_exact(g, ref, rows)


def test_score_order_random_is_the_index_row_ranked():
    """Float operands (MXFP8, 64 heads, top-2048): the ranking-order row holds
    the same entries as the index-order row, ordered by the scores the GPU
    reports, ties to the lower index."""
    rng = np.random.default_rng(77)
    lens, H, D, k = [3000, 400], 64, 128, 2048
    T = sum(lens)
    qc, qs, _ = O.quantize_mxfp8(rng.standard_normal((T * H, D)))
    kc, ks, _ = O.quantize_mxfp8(rng.standard_normal((T, D)))
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    cu = dev(np.array([0, lens[0], T], np.int32))
    ops = (dev(qc), dev(qs), dev(kc), dev(ks), dev(w), cu, max(lens), H, k, "mxfp8")
    ia, sa, la = (host(t) for t in dsa.score_topk(*ops))
    ib, sb, lb = (host(t) for t in dsa.score_topk(*ops, order="score"))
    np.testing.assert_array_equal(la, lb)
    for t in range(T):
        n = int(la[t])
        perm = np.lexsort((ia[t, :n], -sa[t, :n].astype(np.float64)))
        np.testing.assert_array_equal(ib[t, :n], ia[t, :n][perm], err_msg=f"row {t}")
        np.testing.assert_array_equal(sb[t, :n], sa[t, :n][perm], err_msg=f"row {t}")
        assert (ib[t, n:] == -1).all() and np.isneginf(sb[t, n:]).all()


@pytest.mark.parametrize("P,tail", [(4, True), (2, False)])
def test_score_order_kpool_integer_exact(P, tail):
    """Pool mode: pools ranked by score (pool index ascending among ties),
    each pool's tokens ascending, then the query's tail tokens."""
    rng = np.random.default_rng(600 + P)
    lens, H, D, k = [1000, 37, 3], 64, 128, 256
    T = sum(lens)
    q, _, w = _ints(rng, lens, H, D)
    npool = [L // P for L in lens]
    kbar = rng.integers(-3, 4, (sum(npool), D)).astype(np.float64)
    kroom = np.zeros((T // P, D))                  # the key operand has room for T / P rows
    kroom[:len(kbar)] = kbar
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cp = np.concatenate([[0], np.cumsum(npool)]).astype(np.int32)
    g = dsa.score_topk(bf16_dev(_to_bf16(q.reshape(T * H, D))), None, bf16_dev(_to_bf16(kroom)), None, dev(w),
                       dev(cu), max(lens), H, k, "bf16", kpool_size=P, cu_pools=dev(cp), tail=tail, order="score")
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(0, 30), np.arange(990, T)])
    ref = O.kpool_topk(q, kbar, w.astype(np.float64), cu, cp, k, P, tail, rows=rows, order="score")
    _check_exact(g, ref, rows)


def test_score_order_compressed_keys_integer_exact():
    rng = np.random.default_rng(611)
    lens, H, D, k, ratio = [900, 250], 32, 128, 64, 4
    T = sum(lens)
    q, _, w = _ints(rng, lens, H, D)
    ncomp = [L // ratio for L in lens]
    kc = rng.integers(-3, 4, (sum(ncomp), D)).astype(np.float64)
    kroom = np.zeros((T // ratio, D))              # the key operand has room for T / ratio rows
    kroom[:len(kc)] = kc
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cc = np.concatenate([[0], np.cumsum(ncomp)]).astype(np.int32)
    g = dsa.score_topk(bf16_dev(_to_bf16(q.reshape(T * H, D))), None, bf16_dev(_to_bf16(kroom)), None, dev(w),
                       dev(cu), max(lens), H, k, "bf16", kpool_size=ratio, cu_pools=dev(cc), compressed=True,
                       order="score")
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(0, 20), np.arange(880, 920), np.arange(T - 20, T)])
    ref = O.compressed_topk(q, kc, w.astype(np.float64), cu, cc, k, ratio, rows=rows, order="score")
    _check_exact(g, ref, rows)


def test_score_order_key_offsets_integer_exact():
    """Queries that are the last tokens of longer key sequences."""
    rng = np.random.default_rng(622)
    lq, lk, H, D, k = [100, 7], [900, 7], 64, 128, 300
    Tq, Tk = sum(lq), sum(lk)
    q = rng.integers(-3, 4, (Tq, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (Tk, D)).astype(np.float64)
    w = rng.integers(-2, 3, (Tq, H)).astype(np.float32)
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    g = dsa.score_topk_kv(bf16_dev(_to_bf16(q.reshape(Tq * H, D))), None, bf16_dev(_to_bf16(kk)), None, dev(w),
                          dev(cq), dev(ck), max(lq), max(lk), H, k, "bf16", order="score")
    torch.cuda.synchronize()
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cq, k, order="score", cu_seqlens_k=ck)
    _check_exact(g, ref)


@pytest.mark.parametrize("outlier", [1.0, 20.0, 2.0 ** 20])
@pytest.mark.parametrize("k", [700, 2048, 3000])
def test_score_order_spread_and_crowded_rows(outlier, k):
    """Float operands with 1 % of the keys scaled by `outlier`: at 1 and 20 the
    rows' scores spread over the buckets of the ranking pass (its bucket rank),
    at 2^20 the other scores crowd into one bucket and the rows take the radix
    fallback.  Either way the ranking-order row must be the index-order row
    ordered by the GPU's own scores, ties to the lower index."""
    rng = np.random.default_rng(int(outlier) % 1000 + k)
    lens, H, D = [k + 900, 300], 32, 128
    T = sum(lens)
    kv = rng.standard_normal((T, D))
    kv[rng.random(T) < 0.01] *= outlier
    qc, qs, _ = O.quantize_mxfp8(rng.standard_normal((T * H, D)))
    kc, ks, _ = O.quantize_mxfp8(kv)
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    cu = dev(np.array([0, lens[0], T], np.int32))
    ops = (dev(qc), dev(qs), dev(kc), dev(ks), dev(w), cu, max(lens), H, k, "mxfp8")
    ia, sa, la = (host(t) for t in dsa.score_topk(*ops))
    ib, sb, lb = (host(t) for t in dsa.score_topk(*ops, order="score"))
    np.testing.assert_array_equal(la, lb)
    for t in range(T):
        n = int(la[t])
        perm = np.lexsort((ia[t, :n], -sa[t, :n].astype(np.float64)))
        np.testing.assert_array_equal(ib[t, :n], ia[t, :n][perm], err_msg=f"row {t}")
        np.testing.assert_array_equal(sb[t, :n], sa[t, :n][perm], err_msg=f"row {t}")
        assert (ib[t, n:] == -1).all() and np.isneginf(sb[t, n:]).all()
