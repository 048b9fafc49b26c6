"""KPool compression (PR #7522 "Changes") against the oracle, and the KPool
workload end to end (compress -> pool-mode score + top-k)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host
from tests.parity import REL_BF16, REL_MXFP8, compare_topk

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,D,lens,src", [(4, 128, [1000, 3, 57], "f32"), (2, 64, [9, 0, 31], "bf16"),
                                          (8, 128, [64, 71], "f32")])
def test_kpool_compress(P, D, lens, src):
    rng = np.random.default_rng(91 + P)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    k = rng.standard_normal((T, D)).astype(np.float32)
    gate = W.random_bf16_bits(rng, (T,))
    bias = (0.5 * rng.standard_normal(P)).astype(np.float32)
    if src == "bf16":
        kb = (k.view(np.uint32) >> 16).astype(np.uint16)
        kin, kv = bf16_dev(kb), O.bf16_bits_to_float(kb)
    else:
        kin, kv = dev(k), k.astype(np.float64)
    kp, cp = dsa.kpool_compress(kin, dev(gate.view(np.int16)), dev(bias), dev(cu), P)
    ref, rcp = O.kpool_compress(kv, O.bf16_bits_to_float(gate), bias, cu, P)
    np.testing.assert_array_equal(host(cp), rcp)
    n = int(rcp[-1])
    got = host(kp.float())[:n]
    # FP32 softmax/FMA vs float64, then one BF16 rounding: within one BF16 ulp
    _, e2 = np.frexp(np.abs(ref))
    ulp = np.ldexp(1.0, np.maximum(e2 - 1, -126) - 7)
    assert np.all(np.abs(got - ref) <= ulp * 1.001 + 1e-30)
    assert np.mean(got == O.round_bf16(ref)) > 0.99


def test_kpool_workload_end_to_end():
    """The 16384-token KPool configuration scaled down (same H, D, P, top-k),
    compress on the GPU, score pools in BF16, expand, append the tail."""
    wl = W.Workload("kpool-small", [3000, 700], 64, 128, 2048, "bf16", "normal", w_std=0.125, kpool=4, seed=1005)
    x = W.make_inputs(wl)
    T, H, D, P = wl.total_tokens, wl.n_heads, wl.head_dim, wl.kpool
    cu = dev(wl.cu_seqlens)
    kp, cp = dsa.kpool_compress(dev(x["k"]), dev(x["gate_bits"].view(np.int16)), dev(x["slot_bias"]), cu, P)
    qb = (x["q"].reshape(T * H, D).view(np.uint32) >> 16).astype(np.uint16)   # BF16 queries (truncated input)
    idx, sc, ln = dsa.score_topk(bf16_dev(qb), None, kp, None, dev(x["w"]), cu, wl.max_seqlen, H,
                                 wl.index_topk, "bf16", kpool_size=P, cu_pools=cp, tail=True)
    kbar, rcp = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], wl.cu_seqlens, P)
    rows = np.concatenate([np.arange(0, 64), np.arange(2900, 3010), np.arange(T - 40, T)])
    ref = O.kpool_topk(O.bf16_bits_to_float(qb).reshape(T, H, D), O.round_bf16(kbar), x["w"].astype(np.float64),
                       wl.cu_seqlens, rcp, wl.index_topk, P, True, rows=rows, with_scale=True)
    # pooled keys may differ by one BF16 ulp between the two sides (FP32 against
    # float64 softmax pooling); the stated tolerance, relative to M, absorbs it
    compare_topk(host(idx), host(sc), host(ln), ref, REL_BF16, pool=P, tail=True, rows=rows)


def test_kpool_mxfp8_scoring():
    """KPool with MXFP8 scoring: the pooled BF16 keys are quantised to MXFP8
    (dsa_idx_quantize_mxfp8) and scored against MXFP8 queries in pool mode.
    The oracle quantises its own pooled keys the same way; the two sides'
    pooled keys may differ by one BF16 ulp, which can move a key element by
    one E4M3 step: the stated tolerance, relative to M, absorbs it."""
    wl = W.Workload("kpool-mx", [2600, 700], 64, 128, 2048, "mxfp8", "normal", w_std=0.125, kpool=4, seed=1007)
    x = W.make_inputs(wl)
    T, H, D, P = wl.total_tokens, wl.n_heads, wl.head_dim, wl.kpool
    cu = dev(wl.cu_seqlens)
    kp, cp = dsa.kpool_compress(dev(x["k"]), dev(x["gate_bits"].view(np.int16)), dev(x["slot_bias"]), cu, P)
    kc, ks = dsa.quantize_mxfp8(kp)
    qc, qs = dsa.quantize_mxfp8(dev(x["q"].reshape(T * H, D)))
    idx, sc, ln = dsa.score_topk(qc, qs, kc, ks, dev(x["w"]), cu, wl.max_seqlen, H, wl.index_topk, "mxfp8",
                                 kpool_size=P, cu_pools=cp, tail=True)
    kbar, rcp = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], wl.cu_seqlens, P)
    _, _, kq = O.quantize_mxfp8(O.round_bf16(kbar))
    _, _, qq = O.quantize_mxfp8(x["q"].reshape(T * H, D).astype(np.float64))
    rows = np.concatenate([np.arange(0, 40), np.arange(2560, 2620), np.arange(T - 40, T)])
    ref = O.kpool_topk(qq.reshape(T, H, D), kq, x["w"].astype(np.float64), wl.cu_seqlens, rcp, wl.index_topk, P,
                       True, rows=rows, with_scale=True)
    compare_topk(host(idx), host(sc), host(ln), ref, REL_MXFP8, pool=P, tail=True, rows=rows)


def test_kpool_fp8_scoring():
    """KPool with per-vector FP8 scoring: the pooled BF16 keys get one UE8M0
    scale per pooled row (dsa_idx_quantize_fp8_rows), laid out per key tile
    for the block-scaled MMA like the MXFP8 key scales.  Same reasoning and
    tolerance as the MXFP8 case."""
    wl = W.Workload("kpool-f8", [2600, 700], 64, 128, 2048, "fp8", "normal", w_std=0.125, kpool=4, seed=1011)
    x = W.make_inputs(wl)
    T, H, D, P = wl.total_tokens, wl.n_heads, wl.head_dim, wl.kpool
    cu = dev(wl.cu_seqlens)
    kp, cp = dsa.kpool_compress(dev(x["k"]), dev(x["gate_bits"].view(np.int16)), dev(x["slot_bias"]), cu, P)
    kc, ks = dsa.quantize_fp8_rows(kp)
    qc, qs = dsa.quantize_fp8_rows(dev(x["q"].reshape(T * H, D)))
    idx, sc, ln = dsa.score_topk(qc, qs, kc, ks, dev(x["w"]), cu, wl.max_seqlen, H, wl.index_topk, "fp8",
                                 kpool_size=P, cu_pools=cp, tail=True)
    kbar, rcp = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], wl.cu_seqlens, P)
    _, _, kq = O.quantize_fp8_rows(O.round_bf16(kbar))
    _, _, qq = O.quantize_fp8_rows(x["q"].reshape(T * H, D).astype(np.float64))
    rows = np.concatenate([np.arange(0, 40), np.arange(2560, 2620), np.arange(T - 40, T)])
    ref = O.kpool_topk(qq.reshape(T, H, D), kq, x["w"].astype(np.float64), wl.cu_seqlens, rcp, wl.index_topk, P,
                       True, rows=rows, with_scale=True)
    compare_topk(host(idx), host(sc), host(ln), ref, REL_MXFP8, pool=P, tail=True, rows=rows)
