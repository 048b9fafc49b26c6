"""Fused score + top-k (C ABI dsa_idx_score_topk) against the oracle.

Operands are generated directly in the scoring precision (BF16 bit patterns,
or E4M3 codes with UE8M0 scales) so both sides score identical values; the
end-to-end cases add preprocessing on each side."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import _abi
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host
from tests.parity import REL_BF16, REL_MXFP8, compare_topk

pytestmark = pytest.mark.gpu


def _run(q_op, q_sc, k_op, k_sc, w, lens, H, k, prec, sm_scale=1.0, pool=1, cu_pools=None, tail=True):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx, sc, ln = dsa.score_topk(q_op, q_sc, k_op, k_sc, w, dev(cu), max(lens), H, k, prec,
                                 sm_scale=sm_scale, kpool_size=pool, cu_pools=cu_pools, tail=tail)
    torch.cuda.synchronize()
    return host(idx), host(sc), host(ln), cu


def _bf16_case(rng, lens, H, D, wstd=0.3):
    T = sum(lens)
    qb = W.random_bf16_bits(rng, (T * H, D))
    kb = W.random_bf16_bits(rng, (T, D))
    w = (rng.standard_normal((T, H)) * wstd).astype(np.float32)
    return qb, kb, w


def test_tiny_integer_exact_all_rows():
    """Integer q, k in [-3,3], w in [-2,2]: every score is exact, so indices,
    scores and lengths must match the oracle bit for bit (ties to the lower
    index, many zero scores)."""
    wl = W.config("tiny")
    x = W.make_inputs(wl)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    qb = (x["q"].reshape(T * H, D).view(np.uint32) >> 16).astype(np.uint16)   # exact in BF16
    kb = (x["k"].view(np.uint32) >> 16).astype(np.uint16)
    g_idx, g_sc, g_ln, cu = _run(bf16_dev(qb), None, bf16_dev(kb), None, dev(x["w"]), wl.doc_lens, H,
                                 wl.index_topk, "bf16")
    ref = O.indexer_topk(x["q"].astype(np.float64), x["k"].astype(np.float64), x["w"].astype(np.float64),
                         cu, wl.index_topk)
    np.testing.assert_array_equal(g_ln, ref["len"])
    np.testing.assert_array_equal(g_idx, ref["idx"])
    np.testing.assert_array_equal(g_sc, ref["score"].astype(np.float32))


@pytest.mark.parametrize("H", [16, 64])
def test_integer_exact_mxfp8(H):
    """Integer inputs are exact in MXFP8 too (block scale 2^-7 or 2^-8), so
    the block-scaled path must also be bit-exact."""
    rng = np.random.default_rng(21 + H)
    lens = [300, 77]
    T, D, k = sum(lens), 128, 40
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (T, D)).astype(np.float64)
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    qc, qs, qd = O.quantize_mxfp8(q.reshape(T * H, D))
    kc, ks, kd = O.quantize_mxfp8(kk)
    assert np.array_equal(qd, q.reshape(T * H, D)) and np.array_equal(kd, kk)
    g_idx, g_sc, g_ln, cu = _run(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens, H, k, "mxfp8")
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k)
    np.testing.assert_array_equal(g_ln, ref["len"])
    np.testing.assert_array_equal(g_idx, ref["idx"])
    np.testing.assert_array_equal(g_sc, ref["score"].astype(np.float32))


@pytest.mark.parametrize("prec,k", [("bf16", 300), ("mxfp8", 300), ("mxfp8", 2048), ("bf16", 2048)])
def test_integer_exact_long_documents(prec, k):
    """Documents long enough that the candidate buffers hold thousands of
    entries when a query's final selection runs (the sample-bracketed exact
    select), with integer scores full of ties: still bit-exact, lowest index
    first among equal scores.  The oracle checks a spread of rows."""
    rng = np.random.default_rng(71 + k + (prec == "mxfp8"))
    lens, H, D = [2600, 1500], 64, 128
    T = sum(lens)
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (T, D)).astype(np.float64)
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    if prec == "mxfp8":
        qc, qs, _ = O.quantize_mxfp8(q.reshape(T * H, D))
        kc, ks, _ = O.quantize_mxfp8(kk)
        args = (dev(qc), dev(qs), dev(kc), dev(ks))
    else:
        to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact for small ints
        args = (bf16_dev(to_bf16(q.reshape(T * H, D))), None, bf16_dev(to_bf16(kk)), None)
    g_idx, g_sc, g_ln, cu = _run(*args, dev(w), lens, H, k, prec)
    rows = np.concatenate([np.arange(0, 8), np.arange(1000, 1008), np.arange(2580, 2600), np.arange(2600, 2610),
                           np.arange(T - 24, T)])
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k, rows=rows)
    np.testing.assert_array_equal(g_ln[rows], ref["len"])
    np.testing.assert_array_equal(g_idx[rows], ref["idx"])
    np.testing.assert_array_equal(g_sc[rows], ref["score"].astype(np.float32))


def test_mxfp8_long_document_random():
    """One 3000-token document at the target's shape (64 heads, top-2048):
    every late query ends with a full candidate buffer."""
    rng = np.random.default_rng(81)
    lens, H, D, k = [3000], 64, 128, 2048
    T = sum(lens)
    qc, qs, qd = O.quantize_mxfp8(rng.standard_normal((T * H, D)))
    kc, ks, kd = O.quantize_mxfp8(rng.standard_normal((T, D)))
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    g_idx, g_sc, g_ln, cu = _run(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens, H, k, "mxfp8")
    rows = np.concatenate([np.arange(2040, 2056), np.arange(T - 40, T)])
    ref = O.indexer_topk(qd.reshape(T, H, D), kd, w.astype(np.float64), cu, k, rows=rows, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_MXFP8, rows=rows)


BF16_CASES = [
    # lens, H, D, k
    ([700], 64, 128, 64),
    ([1, 5, 130, 257, 129, 128], 32, 128, 16),
    ([1000, 33], 16, 128, 300),
    ([517], 8, 64, 100),
    ([260, 3], 4, 64, 7),
    ([384], 64, 128, 1),
    ([200], 64, 128, 2048),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=[str(i) for i in range(len(BF16_CASES))])
def test_bf16_random_operands(case):
    lens, H, D, k = case
    rng = np.random.default_rng(31 + len(lens) + H + k)
    qb, kb, w = _bf16_case(rng, lens, H, D)
    g_idx, g_sc, g_ln, cu = _run(bf16_dev(qb), None, bf16_dev(kb), None, dev(w), lens, H, k, "bf16", sm_scale=0.7)
    T = sum(lens)
    ref = O.indexer_topk(O.bf16_bits_to_float(qb).reshape(T, H, D), O.bf16_bits_to_float(kb),
                         w.astype(np.float64), cu, k, sm_scale=0.7, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_BF16)


def test_bf16_weights_in_bf16():
    rng = np.random.default_rng(41)
    lens, H, D, k = [333], 32, 128, 50
    qb, kb, _ = _bf16_case(rng, lens, H, D)
    wb = W.random_bf16_bits(rng, (sum(lens), H), 0.3)
    g_idx, g_sc, g_ln, cu = _run(bf16_dev(qb), None, bf16_dev(kb), None, bf16_dev(wb), lens, H, k, "bf16")
    T = sum(lens)
    ref = O.indexer_topk(O.bf16_bits_to_float(qb).reshape(T, H, D), O.bf16_bits_to_float(kb),
                         O.bf16_bits_to_float(wb), cu, k, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_BF16)


MX_CASES = [
    ([600, 130], 64, 256),
    ([1, 2, 3, 250, 513], 32, 64),
    ([400], 16, 2048),
    ([389], 4, 33),
]


@pytest.mark.parametrize("case", MX_CASES, ids=[str(i) for i in range(len(MX_CASES))])
def test_mxfp8_random_operands(case):
    lens, H, k = case
    D = 128
    T = sum(lens)
    rng = np.random.default_rng(51 + H + k)
    # MXFP8 data as the quantiser would produce it from N(0,1) values
    qc, qs, qd = O.quantize_mxfp8(rng.standard_normal((T * H, D)))
    kc, ks, kd = O.quantize_mxfp8(rng.standard_normal((T, D)) * np.where(rng.random((T, D)) < 0.01, 20, 1))
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    g_idx, g_sc, g_ln, cu = _run(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens, H, k, "mxfp8")
    ref = O.indexer_topk(qd.reshape(T, H, D), kd, w.astype(np.float64), cu, k, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_MXFP8)


def test_pool_mode_bf16():
    """KPool selection: score complete pools, keep index_topk / P of them,
    expand to tokens, append the incomplete tail (PR #7522 "Changes")."""
    rng = np.random.default_rng(61)
    lens, H, D, k, P = [1100, 37, 2], 64, 128, 256, 4
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    cp = np.concatenate([[0], np.cumsum([L // P for L in lens])]).astype(np.int32)
    qb = W.random_bf16_bits(rng, (T * H, D))
    pb = W.random_bf16_bits(rng, (T // P, D))        # pooled keys given directly
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    for tail in (True, False):
        g_idx, g_sc, g_ln, _ = _run(bf16_dev(qb), None, bf16_dev(pb), None, dev(w), lens, H, k, "bf16",
                                    pool=P, cu_pools=dev(cp), tail=tail)
        ref = O.kpool_topk(O.bf16_bits_to_float(qb).reshape(T, H, D), O.bf16_bits_to_float(pb), w.astype(np.float64),
                           cu, cp, k, P, tail, with_scale=True)
        compare_topk(g_idx, g_sc, g_ln, ref, REL_BF16, pool=P, tail=tail)


def test_end_to_end_c2_like():
    """LayerNorm + RoPE (FP32) -> BF16 scoring, the 2048-token / 32-head /
    top-256 configuration, all rows."""
    wl = W.config("c2")
    x = W.make_inputs(wl)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    cu_d = dev(wl.cu_seqlens)
    q_op, q_sc, k_op, k_sc = dsa.preprocess(dev(x["q"]), dev(x["k"]), cu_d, wl.max_seqlen, dev(x["ln_gamma"]),
                                            dev(x["ln_beta"]), 1e-6, 64, 10000.0, False, True, "bf16")
    idx, sc, ln = dsa.score_topk(q_op, q_sc, k_op, k_sc, dev(x["w"]), cu_d, wl.max_seqlen, H, wl.index_topk, "bf16")
    qf, kf = O.preprocess(x["q"], x["k"], wl.cu_seqlens, x["ln_gamma"], x["ln_beta"], 1e-6, 64, 10000.0, False, True)
    rows = np.arange(0, T, 3)
    ref = O.indexer_topk(O.round_bf16(qf), O.round_bf16(kf), x["w"].astype(np.float64), wl.cu_seqlens,
                         wl.index_topk, rows=rows, with_scale=True)
    # the preprocessing chains differ by FP32 rounding (float64 on the oracle
    # side); the stated tolerance, relative to M, applies as it is
    compare_topk(host(idx), host(sc), host(ln), ref, REL_BF16, rows=rows, n_heads=H)


def test_deterministic_replay():
    """Three replays, one of them with a concurrent stream busy, give
    byte-identical outputs (PR #8403 review finding 3: bit-exact replay)."""
    rng = np.random.default_rng(71)
    lens, H, D, k = [1500, 700], 64, 128, 512
    qc, qs, _ = O.quantize_mxfp8(rng.standard_normal((sum(lens) * H, D)))
    kc, ks, _ = O.quantize_mxfp8(rng.standard_normal((sum(lens), D)))
    w = (rng.standard_normal((sum(lens), H)) * 0.125).astype(np.float32)
    args = (dev(qc), dev(qs), dev(kc), dev(ks), dev(w))
    outs = []
    side = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device="cuda")
    for rep in range(3):
        if rep == 1:
            with torch.cuda.stream(side):
                for _ in range(4):
                    big = big @ big
                    big = big / big.norm()
        outs.append(_run(*args, lens, H, k, "mxfp8")[:3])
    torch.cuda.synchronize()
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert a.tobytes() == b.tobytes()


def test_empty_and_degenerate_documents():
    rng = np.random.default_rng(81)
    lens = [0, 1, 0, 129, 0]
    H, D, k = 16, 128, 8
    T = sum(lens)
    qb, kb, w = _bf16_case(rng, lens, H, D)
    g_idx, g_sc, g_ln, cu = _run(bf16_dev(qb), None, bf16_dev(kb), None, dev(w), lens, H, k, "bf16")
    ref = O.indexer_topk(O.bf16_bits_to_float(qb).reshape(T, H, D), O.bf16_bits_to_float(kb),
                         w.astype(np.float64), cu, k, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_BF16)


def test_invalid_cu_seqlens_sets_status():
    """cu_seqlens that do not end at total_tokens are caught on the device:
    the status word says INVALID_ARG and nothing is launched past the check."""
    H, D, k = 16, 128, 8
    qb = np.zeros((64 * H, D), np.uint16)
    kb = np.zeros((64, D), np.uint16)
    w = np.zeros((64, H), np.float32)
    cu = dev(np.array([0, 30, 70], np.int32))         # ends at 70, total_tokens is 64
    ws = dsa.workspace(64, 2, 40, H, D, k)
    idx, sc, ln = dsa.score_topk(bf16_dev(qb), None, bf16_dev(kb), None, dev(w), cu, 40, H, k, "bf16", ws=ws)
    assert dsa.read_status(ws) == 1


def test_host_argument_errors():
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError, match="UNSUPPORTED"):
        dsa.score_topk(t.view(1, 16), None, t.view(1, 16), None, torch.zeros(1, 3, device="cuda"),
                       dev(np.array([0, 1], np.int32)), 1, 3, 1, "bf16")


# ---------------------------------------------------------------- global causal offsets

def _run_kv(q_op, q_sc, k_op, k_sc, w, lens_q, lens_k, H, k, prec, sm_scale=1.0):
    cuq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cuk = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    idx, sc, ln = dsa.score_topk_kv(q_op, q_sc, k_op, k_sc, w, dev(cuq), dev(cuk), max(max(lens_q), 1),
                                    max(lens_k), H, k, prec, sm_scale=sm_scale)
    torch.cuda.synchronize()
    return host(idx), host(sc), host(ln), cuq, cuk


KV_CASES = [
    # lens_q, lens_k, H, k, prec
    ([64, 300, 1, 0], [700, 300, 130, 5], 64, 256, "bf16"),
    ([64, 300, 1, 0], [700, 300, 130, 5], 64, 256, "mxfp8"),
    ([40, 200], [2500, 900], 64, 2048, "mxfp8"),
    ([3, 129, 17], [3, 400, 1000], 16, 100, "bf16"),
]


@pytest.mark.parametrize("case", KV_CASES, ids=[str(i) for i in range(len(KV_CASES))])
def test_kv_offsets_random(case):
    """Queries that are the last T_d tokens of S_d keys ([P1] review finding
    2, global causal offsets), BF16 and MXFP8, including T_d = S_d, T_d = 1
    and T_d = 0."""
    lens_q, lens_k, H, k, prec = case
    D = 128
    Tq, Tk = sum(lens_q), sum(lens_k)
    rng = np.random.default_rng(101 + H + k)
    w = (rng.standard_normal((Tq, H)) * 0.2).astype(np.float32)
    if prec == "bf16":
        qb = W.random_bf16_bits(rng, (Tq * H, D))
        kb = W.random_bf16_bits(rng, (Tk, D))
        args = (bf16_dev(qb), None, bf16_dev(kb), None)
        qd, kd, rel = O.bf16_bits_to_float(qb), O.bf16_bits_to_float(kb), REL_BF16
    else:
        qc, qs, qd = O.quantize_mxfp8(rng.standard_normal((Tq * H, D)))
        kc, ks, kd = O.quantize_mxfp8(rng.standard_normal((Tk, D)))
        args = (dev(qc), dev(qs), dev(kc), dev(ks))
        rel = REL_MXFP8
    g_idx, g_sc, g_ln, cuq, cuk = _run_kv(*args, dev(w), lens_q, lens_k, H, k, prec, sm_scale=0.5)
    ref = O.indexer_topk(qd.reshape(Tq, H, D), kd, w.astype(np.float64), cuq, k, sm_scale=0.5, with_scale=True,
                         cu_seqlens_k=cuk)
    compare_topk(g_idx, g_sc, g_ln, ref, rel)


def test_kv_offsets_integer_exact():
    """Integer scores (ties everywhere) with offsets: bit-exact."""
    rng = np.random.default_rng(111)
    lens_q, lens_k, H, D, k = [50, 7, 260], [1800, 7, 300], 64, 128, 512
    Tq, Tk = sum(lens_q), sum(lens_k)
    q = rng.integers(-3, 4, (Tq, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (Tk, D)).astype(np.float64)
    w = rng.integers(-2, 3, (Tq, H)).astype(np.float32)
    qc, qs, _ = O.quantize_mxfp8(q.reshape(Tq * H, D))
    kc, ks, _ = O.quantize_mxfp8(kk)
    g_idx, g_sc, g_ln, cuq, cuk = _run_kv(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens_q, lens_k, H, k, "mxfp8")
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cuq, k, cu_seqlens_k=cuk)
    np.testing.assert_array_equal(g_ln, ref["len"])
    np.testing.assert_array_equal(g_idx, ref["idx"])
    np.testing.assert_array_equal(g_sc, ref["score"].astype(np.float32))


def test_kv_more_queries_than_keys_sets_status():
    """T_d > S_d is caught on the device: DSA_ERR_INVALID_ARG in the status word."""
    H, D, k = 16, 128, 8
    lens_q, lens_k = [10, 5], [10, 4]
    Tq, Tk = sum(lens_q), sum(lens_k)
    qb = torch.zeros((Tq * H, D), dtype=torch.bfloat16, device="cuda")
    kb = torch.zeros((Tk, D), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((Tq, H), dtype=torch.float32, device="cuda")
    cuq = dev(np.array([0, 10, 15], np.int32))
    cuk = dev(np.array([0, 10, 14], np.int32))
    ws = dsa.workspace(max(Tq, Tk), 2, 10, H, D, k, 1, "bf16", qb.device)
    dsa.score_topk_kv(qb, None, kb, None, w, cuq, cuk, 10, 10, H, k, "bf16", ws=ws)
    assert dsa.read_status(ws) == _abi.DSA_ERR_INVALID_ARG


# ---------------------------------------------------------------- compressed keys (ratio > 1)

COMP_CASES = [
    # lens, ratio, H, k, prec
    ([1500, 37, 400], 4, 64, 256, "bf16"),
    ([1500, 37, 400], 4, 64, 256, "mxfp8"),
    ([4000, 900], 2, 64, 2048, "mxfp8"),
    ([2000, 3, 700], 16, 32, 50, "bf16"),
]


@pytest.mark.parametrize("case", COMP_CASES, ids=[str(i) for i in range(len(COMP_CASES))])
def test_compressed_keys_random(case):
    """Caller-provided compressed keys ([P2], the indexer's ratio): key c of a
    document covers its tokens c*ratio .. c*ratio + ratio - 1 and is visible
    once complete; indices are per compressed key."""
    lens, ratio, H, k, prec = case
    D = 128
    T = sum(lens)
    ncomp = [L // ratio for L in lens]
    cc = np.concatenate([[0], np.cumsum(ncomp)]).astype(np.int32)
    rng = np.random.default_rng(121 + ratio + k)
    w = (rng.standard_normal((T, H)) * 0.2).astype(np.float32)
    rows_k = max(T // ratio, 1)     # the documented room: total_tokens / ratio rows
    if prec == "bf16":
        qb = W.random_bf16_bits(rng, (T * H, D))
        kb = W.random_bf16_bits(rng, (rows_k, D))
        args = (bf16_dev(qb), None, bf16_dev(kb), None)
        qd, kd, rel = O.bf16_bits_to_float(qb), O.bf16_bits_to_float(kb), REL_BF16
    else:
        qc, qs, qd = O.quantize_mxfp8(rng.standard_normal((T * H, D)))
        kc, ks, kd = O.quantize_mxfp8(rng.standard_normal((rows_k, D)))
        args = (dev(qc), dev(qs), dev(kc), dev(ks))
        rel = REL_MXFP8
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx, sc, ln = dsa.score_topk(*args, dev(w), dev(cu), max(lens), H, k, prec, sm_scale=0.5, kpool_size=ratio,
                                 cu_pools=dev(cc), compressed=True)
    torch.cuda.synchronize()
    ref = O.compressed_topk(qd.reshape(T, H, D), kd, w.astype(np.float64), cu, cc, k, ratio, sm_scale=0.5,
                            with_scale=True)
    compare_topk(host(idx), host(sc), host(ln), ref, rel)


def test_compressed_keys_too_few_rows_sets_status():
    """A document with fewer compressed keys than complete groups is caught on
    the device (DSA_ERR_INVALID_ARG in the status word)."""
    H, D, k, ratio = 16, 128, 8, 4
    lens = [40, 12]
    T = sum(lens)
    qb = torch.zeros((T * H, D), dtype=torch.bfloat16, device="cuda")
    kb = torch.zeros((T // ratio, D), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((T, H), dtype=torch.float32, device="cuda")
    cu = dev(np.array([0, 40, 52], np.int32))
    cc = dev(np.array([0, 9, 12], np.int32))     # document 0 has 10 complete groups
    ws = dsa.workspace(T, 2, 40, H, D, k, ratio, "bf16", qb.device)
    dsa.score_topk(qb, None, kb, None, w, cu, 40, H, k, "bf16", kpool_size=ratio, cu_pools=cc, compressed=True,
                   ws=ws)
    assert dsa.read_status(ws) == _abi.DSA_ERR_INVALID_ARG


# ---------------------------------------------------------------- FP8 with per-vector scales

FP8_CASES = [
    ([600, 130], 64, 256),
    ([1, 2, 3, 250, 513], 32, 64),
    ([2500], 64, 2048),
    ([389], 16, 33),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[str(i) for i in range(len(FP8_CASES))])
def test_fp8_rows_random_operands(case):
    """FP8 scoring with one UE8M0 scale per q row and per key (kind::f8f6f4,
    scales folded into the head weights and the key's score): both sides
    score identical dequantised operands, so FP32 accumulation is the only
    difference."""
    lens, H, k = case
    D = 128
    T = sum(lens)
    rng = np.random.default_rng(131 + H + k)
    q = rng.standard_normal((T * H, D)) * np.exp2(rng.integers(-4, 5, (T * H, 1)))
    kk = rng.standard_normal((T, D)) * np.where(rng.random((T, D)) < 0.01, 20, 1)
    qc, qs, qd = O.quantize_fp8_rows(q)
    kc, ks, kd = O.quantize_fp8_rows(kk)
    w = (rng.standard_normal((T, H)) * 0.125).astype(np.float32)
    g_idx, g_sc, g_ln, cu = _run(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens, H, k, "fp8", sm_scale=0.25)
    ref = O.indexer_topk(qd.reshape(T, H, D), kd, w.astype(np.float64), cu, k, sm_scale=0.25, with_scale=True)
    compare_topk(g_idx, g_sc, g_ln, ref, REL_BF16)


def test_fp8_rows_integer_exact():
    """Integers in [-3, 3] are exact in per-vector FP8 (row scale 2^-7), so the
    indices and scores must be bit-exact, ties to the lower index."""
    rng = np.random.default_rng(141)
    lens, H, D, k = [900, 77], 64, 128, 300
    T = sum(lens)
    q = rng.integers(-3, 4, (T, H, D)).astype(np.float64)
    kk = rng.integers(-3, 4, (T, D)).astype(np.float64)
    w = rng.integers(-2, 3, (T, H)).astype(np.float32)
    qc, qs, qd = O.quantize_fp8_rows(q.reshape(T * H, D))
    kc, ks, kd = O.quantize_fp8_rows(kk)
    assert np.array_equal(qd, q.reshape(T * H, D)) and np.array_equal(kd, kk)
    g_idx, g_sc, g_ln, cu = _run(dev(qc), dev(qs), dev(kc), dev(ks), dev(w), lens, H, k, "fp8")
    rows = np.concatenate([np.arange(0, 40), np.arange(860, 940), np.arange(T - 20, T)])
    ref = O.indexer_topk(q, kk, w.astype(np.float64), cu, k, rows=rows)
    np.testing.assert_array_equal(g_ln[rows], ref["len"])
    np.testing.assert_array_equal(g_idx[rows], ref["idx"])
    np.testing.assert_array_equal(g_sc[rows], ref["score"].astype(np.float32))


def test_fp8_rows_end_to_end_with_preprocess():
    """Key LayerNorm + RoPE + per-vector FP8 on both sides, then scoring."""
    wl = W.Workload("c2-fp8", [1500, 300], 32, 128, 256, "fp8", "normal", layernorm=True, rope_dim=64,
                    rope_fp32=True, w_std=1 / np.sqrt(32), seed=1008)
    x = W.make_inputs(wl)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    cu = wl.cu_seqlens
    ops = dsa.preprocess(dev(x["q"]), dev(x["k"]), dev(cu), wl.max_seqlen, dev(x["ln_gamma"]), dev(x["ln_beta"]),
                         1e-6, 64, 10000.0, False, True, "fp8")
    idx, sc, ln = dsa.score_topk(*ops, dev(x["w"]), dev(cu), wl.max_seqlen, H, wl.index_topk, "fp8")
    torch.cuda.synchronize()
    qf, kf = O.preprocess(x["q"], x["k"], cu, x["ln_gamma"], x["ln_beta"], 1e-6, 64, 10000.0, False, True)
    _, _, qd = O.quantize_fp8_rows(qf.reshape(T * H, D))
    _, _, kd = O.quantize_fp8_rows(kf)
    rows = np.concatenate([np.arange(0, 30), np.arange(1400, 1530), np.arange(T - 30, T)])
    ref = O.indexer_topk(qd.reshape(T, H, D), kd, x["w"].astype(np.float64), cu, wl.index_topk, rows=rows,
                         with_scale=True)
    # the two carriers differ by FP32 rounding, which can move an element by one E4M3 step
    compare_topk(host(idx), host(sc), host(ln), ref, REL_MXFP8, rows=rows)
