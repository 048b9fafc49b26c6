"""Parity at the full sizes of the measured configurations, in the launch
configuration bench.py times.

* End to end: the seeded inputs resident on the device, dsa_idx_preprocess
  (key LayerNorm, RoPE, quantisation; KPool: pool compression) and the fused
  score + top-k over every query; sampled rows (the first two and last two
  queries of every document and a seeded spread) are checked against the
  oracle, which computes them one by one from the same seeded inputs.
* Identical operands: the oracle quantises the seeded inputs itself (MXFP8,
  per-vector FP8 or BF16; KPool: its own pooled keys), the GPU scores exactly
  those bytes, and the sampled rows must agree at the stated tolerances with
  no widening: this isolates the fused scoring kernel at full size.
* MXFP8 against BF16 scoring on the same inputs (the precision comparison the
  indexer pages make): the per-row top-k overlap of the two GPU selections
  must follow the oracle's overlap on the sampled rows.

Each test prints its parity statistics (pytest -s shows them)."""
import json

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host
from tests.parity import REL_BF16, REL_MXFP8, compare_topk, topk_overlap

pytestmark = pytest.mark.gpu

CASES = [("c3", "mxfp8"), ("c3", "bf16"), ("thd", "mxfp8"), ("kpool", "bf16"), ("target", "mxfp8"),
         ("target", "bf16"), ("target", "fp8")]


def rel_for(prec):
    return REL_BF16 if prec == "bf16" else REL_MXFP8


def report(name, stats):
    print(json.dumps({"parity": name, **stats}))


def sample_rows(wl, n_spread=24, seed=0):
    cu = wl.cu_seqlens
    rows = []
    for d in range(len(wl.doc_lens)):
        a, b = int(cu[d]), int(cu[d + 1])
        rows += [r for r in (a, a + 1, b - 2, b - 1) if a <= r < b]
    rows += np.random.default_rng(seed).choice(wl.total_tokens, n_spread, replace=False).tolist()
    return np.unique(np.asarray(rows, dtype=np.int64))


def oracle_rows(wl, x, prec, rows):
    """The oracle's preprocessing and selection for the sampled query rows
    (a query's RoPE and quantisation depend on its own row only; the keys are
    processed whole)."""
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    cu = wl.cu_seqlens
    pos = O.positions_in_document(cu)
    kk = np.asarray(x["k"], np.float64)
    if wl.layernorm:
        kk = O.key_layernorm(kk, x["ln_gamma"], x["ln_beta"], 1e-6)
    kf = O.round_fp32(O.apply_rope(kk, pos, wl.rope_dim, wl.rope_base))
    qf = O.round_fp32(O.apply_rope(np.asarray(x["q"][rows], np.float64), pos[rows][:, None], wl.rope_dim,
                                   wl.rope_base))
    qq = np.zeros((T, H, D))
    w = x["w"].astype(np.float64)
    if wl.kpool > 1:
        kbar, cpools = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], cu, wl.kpool)
        qq[rows] = O.round_bf16(qf)
        return O.kpool_topk(qq, O.round_bf16(kbar), w, cu, cpools, wl.index_topk, wl.kpool, True, rows=rows,
                            with_scale=True)
    qq[rows] = O.scoring_operand(qf.reshape(-1, D), prec)[0].reshape(len(rows), H, D)
    return O.indexer_topk(qq, O.scoring_operand(kf, prec)[0], w, cu, wl.index_topk, rows=rows, with_scale=True)


MAX_LEN = W.Workload("max-seqlen", [65536], 16, 128, 2048, "mxfp8", "normal", layernorm=True, rope_dim=64,
                     rope_fp32=True, w_std=0.25, seed=1009)


def gpu_end_to_end(wl, x, prec):
    T, H, D, K = wl.total_tokens, wl.n_heads, wl.head_dim, wl.index_topk
    cu = dev(wl.cu_seqlens)
    k = dev(x["k"])
    g = dev(x["ln_gamma"]) if wl.layernorm else None
    b = dev(x["ln_beta"]) if wl.layernorm else None
    qo, qs, ko, ks = dsa.preprocess(dev(x["q"]), k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base,
                                    False, True, prec)
    pool = {}
    if wl.kpool > 1:
        ko, cpools = dsa.kpool_compress(k, dev(x["gate_bits"].view(np.int16)), dev(x["slot_bias"]), cu, wl.kpool)
        ks = None
        pool = dict(kpool_size=wl.kpool, cu_pools=cpools, tail=True)
    ws = dsa.workspace(T, len(wl.doc_lens), wl.max_seqlen, H, D, K, wl.kpool, prec, qo.device)
    idx, sc, ln = dsa.score_topk(qo, qs, ko, ks, dev(x["w"]), cu, wl.max_seqlen, H, K, prec, ws=ws, **pool)
    assert dsa.read_status(ws) == 0
    out = host(idx), host(sc), host(ln)
    del qo, qs, ko, ks, idx, sc, ln
    torch.cuda.empty_cache()
    return out


def check_lengths(wl, gi, gl):
    """Every row: lengths and padding follow from the visibility rule alone."""
    K = wl.index_topk
    pos = O.positions_in_document(wl.cu_seqlens)
    if wl.kpool > 1:
        P = wl.kpool
        exp_len = np.minimum((pos + 1) // P, K // P) * P + (pos + 1) % P
    else:
        exp_len = np.minimum(pos + 1, K)
    np.testing.assert_array_equal(gl, exp_len)
    assert all((gi[t, gl[t]:] == -1).all() for t in range(0, wl.total_tokens, 97))


@pytest.mark.parametrize("name,prec", CASES + [("max-seqlen", "mxfp8")],
                         ids=[f"{n}-{p}" for n, p in CASES] + ["max-seqlen-mxfp8"])
def test_full_size_sampled_rows(name, prec):
    """End to end on the measured configurations, and one document of the
    longest supported length (65536 tokens: local indices up to 65535, 512 key
    tiles).  The two preprocessing chains round to FP32 independently (float64
    on the oracle side), which can move a rare scoring operand by one step of
    its format; the tolerance stays the stated one."""
    wl = MAX_LEN if name == "max-seqlen" else W.config(name)
    x = W.make_inputs(wl)
    gi, gs, gl = gpu_end_to_end(wl, x, prec)
    check_lengths(wl, gi, gl)
    rows = sample_rows(wl)
    ref = oracle_rows(wl, x, prec, rows)
    st = compare_topk(gi, gs, gl, ref, rel_for(prec), pool=wl.kpool, tail=True, rows=rows,
                      head_dim=wl.head_dim, n_heads=wl.n_heads)
    report(f"end-to-end {name} {prec}", st)


# ---------------------------------------------------------------- identical operands

def oracle_quantised(x2d, prec, chunk=1 << 19):
    """The oracle's scoring operand of every row of x2d, computed in chunks of
    rows: (payload for the device: E4M3 codes or BF16 bits, scale bytes or
    None)."""
    R, D = x2d.shape
    if prec == "bf16":
        bits = np.empty((R, D), np.uint16)
        for r0 in range(0, R, chunk):
            bits[r0:r0 + chunk] = O.float_to_bf16_bits(O.round_bf16(x2d[r0:r0 + chunk]))
        return bits, None
    codes = np.empty((R, D), np.uint8)
    scales = np.empty((R, D // 32) if prec == "mxfp8" else (R,), np.uint8)
    quant = O.quantize_mxfp8 if prec == "mxfp8" else O.quantize_fp8_rows
    for r0 in range(0, R, chunk):
        c, s, _ = quant(x2d[r0:r0 + chunk])
        codes[r0:r0 + chunk] = c
        scales[r0:r0 + chunk] = s
    return codes, scales


def dequantised(payload, scales, prec, rows_sel):
    if prec == "bf16":
        return O.bf16_bits_to_float(payload[rows_sel])
    if prec == "mxfp8":
        return O.dequantize_mxfp8(payload[rows_sel], scales[rows_sel])
    return O.dequantize_fp8_rows(payload[rows_sel], scales[rows_sel])


def to_device(payload, scales, prec):
    if prec == "bf16":
        return bf16_dev(payload), None
    return dev(payload), dev(scales)


IDENT_CASES = [("target", "mxfp8"), ("target", "bf16"), ("target", "fp8"), ("c3", "mxfp8"), ("thd", "mxfp8"),
               ("kpool", "bf16"), ("kpool", "mxfp8")]


@pytest.mark.parametrize("name,prec", IDENT_CASES, ids=[f"{n}-{p}" for n, p in IDENT_CASES])
def test_full_size_identical_operands(name, prec):
    """The fused kernel alone at full size: both sides score the oracle's own
    quantisation of the seeded inputs (no preprocessing), so the only
    difference left is the FP32 accumulation, and the stated tolerances apply
    as they are (2e-3 BF16, 1.5e-2 8-bit, relative to M)."""
    wl = W.config(name)
    x = W.make_inputs(wl)
    T, H, D, K = wl.total_tokens, wl.n_heads, wl.head_dim, wl.index_topk
    cu = wl.cu_seqlens
    rows = sample_rows(wl)
    q2 = x["q"].reshape(T * H, D)
    qp, qsc = oracle_quantised(q2, prec)
    q_rows = (rows[:, None] * H + np.arange(H)[None, :]).reshape(-1)
    qd = np.zeros((T, H, D))
    qd[rows] = dequantised(qp, qsc, prec, q_rows).reshape(len(rows), H, D)
    pool = {}
    if wl.kpool > 1:
        kbar, cpools = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], cu, wl.kpool)
        kp, ksc = oracle_quantised(O.round_bf16(kbar), prec)
        kd = dequantised(kp, ksc, prec, np.arange(kp.shape[0]))
        pool = dict(kpool_size=wl.kpool, cu_pools=dev(cpools.astype(np.int32)), tail=True)
    else:
        kp, ksc = oracle_quantised(x["k"], prec)
        kd = dequantised(kp, ksc, prec, np.arange(T))
    q_op, q_sc = to_device(qp, qsc, prec)
    k_op, k_sc = to_device(kp, ksc, prec)
    del qp, qsc
    ws = dsa.workspace(T, len(wl.doc_lens), wl.max_seqlen, H, D, K, wl.kpool, prec, q_op.device)
    idx, sc, ln = dsa.score_topk(q_op, q_sc, k_op, k_sc, dev(x["w"]), dev(cu), wl.max_seqlen, H, K, prec, ws=ws,
                                 **pool)
    assert dsa.read_status(ws) == 0
    gi, gs, gl = host(idx), host(sc), host(ln)
    del q_op, q_sc, k_op, k_sc, idx, sc, ln
    torch.cuda.empty_cache()
    check_lengths(wl, gi, gl)
    w = x["w"].astype(np.float64)
    if wl.kpool > 1:
        ref = O.kpool_topk(qd, kd, w, cu, cpools, K, wl.kpool, True, rows=rows, with_scale=True)
    else:
        ref = O.indexer_topk(qd, kd, w, cu, K, rows=rows, with_scale=True)
    st = compare_topk(gi, gs, gl, ref, rel_for(prec), pool=wl.kpool, tail=True, rows=rows, head_dim=D, n_heads=H)
    report(f"identical-operands {name} {prec}", st)


# ---------------------------------------------------------------- MXFP8 against BF16

@pytest.mark.parametrize("name", ["c3", "target"])
def test_mxfp8_against_bf16_overlap(name):
    """MXFP8 and BF16 scoring of the same preprocessed inputs select slightly
    different keys (the quantisation moves scores near the k-th).  The GPU's
    per-row overlap |S_mxfp8 & S_bf16| / k must follow the oracle's on the
    sampled rows (each GPU row may differ from its oracle row by 1 % swaps, so
    within 2 %), and over all rows stay above the floor the oracle's sampled
    rows show (c3: mean 0.99, worst 0.973; target: mean 0.978, worst 0.959 on
    24 seeded rows)."""
    wl = W.config(name)
    x = W.make_inputs(wl)
    gi_m, _, gl_m = gpu_end_to_end(wl, x, "mxfp8")
    gi_b, _, gl_b = gpu_end_to_end(wl, x, "bf16")
    ov_all = topk_overlap(gi_m, gl_m, gi_b, gl_b)
    rows = np.sort(np.random.default_rng(5).choice(wl.total_tokens, 24, replace=False))
    ref_m = oracle_rows(wl, x, "mxfp8", rows)
    ref_b = oracle_rows(wl, x, "bf16", rows)
    ov_ora = topk_overlap(ref_m["idx"], ref_m["len"], ref_b["idx"], ref_b["len"])
    ov_gpu = ov_all[rows]
    print(json.dumps({"overlap": name, "gpu_mean_all_rows": float(ov_all.mean()),
                      "gpu_min_all_rows": float(ov_all.min()), "gpu_sampled": ov_gpu.round(4).tolist(),
                      "oracle_sampled": ov_ora.round(4).tolist()}))
    assert np.all(np.abs(ov_gpu - ov_ora) <= 0.02 + 1e-12), (ov_gpu, ov_ora)
    floor_mean, floor_min = (0.98, 0.95) if name == "c3" else (0.97, 0.94)
    assert ov_all.mean() >= floor_mean and ov_all.min() >= floor_min, (ov_all.mean(), ov_all.min())
