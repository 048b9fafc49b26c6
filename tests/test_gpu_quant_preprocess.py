"""Preprocessing and MXFP8 quantisation kernels against the oracle.

The stand-alone quantiser gets the same FP32/BF16 input as the oracle and
must match it bit for bit (codes and scale bytes).  The fused preprocess
computes LayerNorm/RoPE in FP32 where the oracle uses float64, so its output
must be a correct rounding of a value within a few FP32 ulps of the oracle's
exact carrier (checked as |gpu - carrier| <= half a format ulp + slack)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_indexer_dsa_gb300 as dsa
from sparse_attention_indexer_dsa_gb300 import workloads as W
from tests.gpu_util import bf16_dev, dev, host

pytestmark = pytest.mark.gpu


def _edge_rows(rng):
    x = rng.standard_normal((37, 128)).astype(np.float32)
    x[0] = 0.0                                            # zero blocks
    x[1, :32] = 448.0 * 2.0 ** -3                         # exact binade edge
    x[1, 32:64] = np.nextafter(np.float32(448.0 * 2.0 ** 5), np.float32(np.inf))
    x[2] *= 1e-38                                         # subnormal amax
    x[3] *= 1e30
    x[4, :32] = 1.9                                       # floor rule saturates
    x[5] = np.arange(128, dtype=np.float32) - 64.0        # integers
    grid = O.e4m3_decode(np.arange(0, 0x7E))
    x[6, :125] = (grid[1:] + grid[:-1]) / 2 * 2.0 ** -4   # RNE ties after scaling
    return x


@pytest.mark.parametrize("rule", ["nosat", "floor"])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_bit_exact(rule, src):
    rng = np.random.default_rng(11)
    x = _edge_rows(rng)
    x = np.concatenate([x, (rng.standard_normal((1000, 128)) * np.exp2(rng.integers(-30, 30, (1000, 1)))).astype(np.float32)])
    if src == "bf16":
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        xin = bf16_dev(bits)
        xv = O.bf16_bits_to_float(bits)
    else:
        xin = dev(x)
        xv = x.astype(np.float64)
    codes, scales = dsa.quantize_mxfp8(xin, rule)
    rc, rs, _ = O.quantize_mxfp8(xv, rule)
    np.testing.assert_array_equal(host(scales), rs)
    np.testing.assert_array_equal(host(codes), rc)


def test_quantize_64_cols_and_ragged_rows():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((333, 64)).astype(np.float32)
    codes, scales = dsa.quantize_mxfp8(dev(x))
    rc, rs, _ = O.quantize_mxfp8(x.astype(np.float64))
    np.testing.assert_array_equal(host(scales), rs)
    np.testing.assert_array_equal(host(codes), rc)


def _check_rounding(gpu_vals, carrier, mag, mant_bits, emin, slack=16 * 2.0 ** -24):
    """The GPU value must be a correct rounding (to the format) of a value
    within `slack * mag` of the oracle's exact carrier, where `mag` is the
    magnitude of the terms that formed the carrier (LayerNorm and the RoPE
    rotation cancel, so FP32 errors scale with their inputs, not the result)."""
    c = np.asarray(carrier, np.float64)
    _, e2 = np.frexp(np.abs(c) + slack * mag)
    ulp = np.ldexp(1.0, np.maximum(e2 - 1, emin) - mant_bits)
    bound = 0.5 * ulp * (1 + 1e-9) + slack * mag + 1e-30
    err = np.abs(np.asarray(gpu_vals, np.float64) - c)
    assert np.all(err <= bound), (err / bound).max()


def _rope_mag(a, rope_dim, inter):
    """|a_i| + |a_partner| on rotated dims, |a_i| elsewhere."""
    m = np.abs(np.asarray(a, np.float64)).copy()
    if rope_dim == 0:
        return m
    h = rope_dim // 2
    if inter:
        s = m[..., 0:rope_dim:2] + m[..., 1:rope_dim:2]
        m[..., 0:rope_dim:2] = s
        m[..., 1:rope_dim:2] = s
    else:
        s = m[..., :h] + m[..., h:rope_dim]
        m[..., :h] = s
        m[..., h:rope_dim] = s
    return m


CASES = [
    dict(lens=[64, 191, 5], H=16, D=128, ln=True, rope=64, inter=False, fp32=True),
    dict(lens=[300], H=64, D=128, ln=True, rope=64, inter=True, fp32=True),
    dict(lens=[130, 2], H=32, D=128, ln=False, rope=0, inter=False, fp32=True),
    dict(lens=[77, 100], H=8, D=128, ln=True, rope=128, inter=False, fp32=False),
    dict(lens=[40, 9], H=4, D=64, ln=True, rope=32, inter=False, fp32=True),
    dict(lens=[33], H=1, D=64, ln=False, rope=64, inter=True, fp32=False),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_preprocess_bf16_out(case, src):
    rng = np.random.default_rng(13)
    lens, H, D = case["lens"], case["H"], case["D"]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = (rng.standard_normal((T, D)) * 3 + 0.5).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32)
    if src == "bf16":
        qb, kb = (q.view(np.uint32) >> 16).astype(np.uint16), (k.view(np.uint32) >> 16).astype(np.uint16)
        qin, kin = bf16_dev(qb), bf16_dev(kb)
        qv, kv = O.bf16_bits_to_float(qb), O.bf16_bits_to_float(kb)
    else:
        qin, kin, qv, kv = dev(q), dev(k), q.astype(np.float64), k.astype(np.float64)
    gd, bd = (dev(g), dev(b)) if case["ln"] else (None, None)
    q_op, _, k_op, _ = dsa.preprocess(qin, kin, dev(cu), max(lens), gd, bd, 1e-6, case["rope"], 10000.0,
                                      case["inter"], case["fp32"], "bf16")
    # oracle carrier before the final BF16 rounding of the scoring boundary
    pos = O.positions_in_document(cu)
    kk = kv
    if case["ln"]:
        kk = O.key_layernorm(kk, g, b, 1e-6)
        if not case["fp32"]:
            kk = O.round_bf16(kk)
    kk = O.apply_rope(kk, pos, case["rope"], 10000.0, case["inter"])
    qq = O.apply_rope(qv, pos[:, None], case["rope"], 10000.0, case["inter"])
    gq = host(q_op.float()).reshape(T, H, D)
    gk = host(k_op.float())
    if case["ln"]:
        z = (kv - kv.mean(-1, keepdims=True)) / np.sqrt(kv.var(-1, keepdims=True) + 1e-6)
        k_terms = np.abs(z * g) + np.abs(b)
    else:
        k_terms = np.abs(kv)
    # the default path rounds the LayerNorm output to BF16 before RoPE: one BF16
    # ulp of slack when FP32 and float64 LayerNorm land on different sides
    k_slack = 2.0 ** -8 if (case["ln"] and not case["fp32"]) else 16 * 2.0 ** -24
    _check_rounding(gq, qq, _rope_mag(qv, case["rope"], case["inter"]), 7, -126)
    _check_rounding(gk, kk, _rope_mag(k_terms, case["rope"], case["inter"]), 7, -126, k_slack)
    # rope_fp32=0: the values are BF16 already and equal to the oracle almost everywhere
    if not case["fp32"]:
        qb_ora, kb_ora = O.preprocess(qv, kv, cu, g if case["ln"] else None, b if case["ln"] else None,
                                      1e-6, case["rope"], 10000.0, case["inter"], False)
        assert np.mean(gq == qb_ora) > 0.99 and np.mean(gk == kb_ora) > 0.97


@pytest.mark.parametrize("case", CASES[:4], ids=[str(i) for i in range(4)])
def test_preprocess_mxfp8_out(case):
    rng = np.random.default_rng(14)
    lens, H, D = case["lens"], case["H"], case["D"]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = rng.standard_normal((T, D)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32)
    gd, bd = (dev(g), dev(b)) if case["ln"] else (None, None)
    q_op, q_sc, k_op, k_sc = dsa.preprocess(dev(q), dev(k), dev(cu), max(lens), gd, bd, 1e-6, case["rope"],
                                            10000.0, case["inter"], case["fp32"], "mxfp8")
    qf, kf = O.preprocess(q, k, cu, g if case["ln"] else None, b if case["ln"] else None, 1e-6,
                          case["rope"], 10000.0, case["inter"], case["fp32"])
    _, rqs, rq = O.quantize_mxfp8(qf.reshape(T * H, D))
    _, rks, rk = O.quantize_mxfp8(kf)
    gq = O.dequantize_mxfp8(host(q_op), host(q_sc))
    gk = O.dequantize_mxfp8(host(k_op), host(k_sc))
    # scale bytes agree except where the block max sits on a binade edge
    assert np.mean(host(q_sc) == rqs) > 0.999 and np.mean(host(k_sc) == rks) > 0.99
    same = np.repeat(host(q_sc) == rqs, 32, axis=1)
    assert np.mean(gq[same] == rq[same]) > 0.999
    err = np.abs(gq - rq)
    assert np.all(err <= np.ldexp(1.0, host(q_sc).astype(int).repeat(32, axis=1) - 127 + 8 - 3) + 1e-30)
    errk = np.abs(gk - rk)
    assert np.all(errk <= np.ldexp(1.0, host(k_sc).astype(int).repeat(32, axis=1) - 127 + 8 - 3) + 1e-30)


@pytest.mark.parametrize("rule", ["nosat", "floor"])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_fp8_rows_bit_exact(rule, src):
    """Per-vector FP8 (one UE8M0 scale per 128-element row) against the
    oracle's quantize_fp8_rows on identical input, bit for bit."""
    rng = np.random.default_rng(15)
    x = _edge_rows(rng)
    x = np.concatenate([x, (rng.standard_normal((1000, 128)) * np.exp2(rng.integers(-30, 30, (1000, 1)))).astype(np.float32)])
    if src == "bf16":
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        xin = bf16_dev(bits)
        xv = O.bf16_bits_to_float(bits)
    else:
        xin = dev(x)
        xv = x.astype(np.float64)
    codes, scales = dsa.quantize_fp8_rows(xin, rule)
    rc, rs, _ = O.quantize_fp8_rows(xv, rule)
    np.testing.assert_array_equal(host(scales), rs)
    np.testing.assert_array_equal(host(codes), rc)


@pytest.mark.parametrize("case", CASES[:4], ids=[str(i) for i in range(4)])
def test_preprocess_fp8_out(case):
    """Fused preprocess with per-vector FP8 output: the GPU's FP32 carrier
    and the oracle's float64 one differ by FP32 rounding only, so scale bytes
    agree almost everywhere and every value is within one E4M3 step."""
    rng = np.random.default_rng(16)
    lens, H, D = case["lens"], case["H"], case["D"]
    if D != 128:
        pytest.skip("FP8 output needs head_dim 128")
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = rng.standard_normal((T, D)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32)
    gd, bd = (dev(g), dev(b)) if case["ln"] else (None, None)
    q_op, q_sc, k_op, k_sc = dsa.preprocess(dev(q), dev(k), dev(cu), max(lens), gd, bd, 1e-6, case["rope"],
                                            10000.0, case["inter"], case["fp32"], "fp8")
    qf, kf = O.preprocess(q, k, cu, g if case["ln"] else None, b if case["ln"] else None, 1e-6,
                          case["rope"], 10000.0, case["inter"], case["fp32"])
    _, rqs, rq = O.quantize_fp8_rows(qf.reshape(T * H, D))
    _, rks, rk = O.quantize_fp8_rows(kf)
    gqs, gks = host(q_sc).reshape(-1), host(k_sc).reshape(-1)
    gq = O.e4m3_decode(host(q_op)) * np.ldexp(1.0, gqs.astype(int) - 127)[:, None]
    gk = O.e4m3_decode(host(k_op)) * np.ldexp(1.0, gks.astype(int) - 127)[:, None]
    assert np.mean(gqs == rqs) > 0.999 and np.mean(gks == rks) > 0.99
    same = gqs == rqs
    assert np.mean(gq[same] == rq[same]) > 0.999
    # one E4M3 step in the top binade of the coarser of the two scales
    step = np.ldexp(1.0, np.maximum(gqs, rqs).astype(int) - 127 + 8 - 3)[:, None]
    assert np.all(np.abs(gq - rq) <= step + 1e-30)
    stepk = np.ldexp(1.0, np.maximum(gks, rks).astype(int) - 127 + 8 - 3)[:, None]
    assert np.all(np.abs(gk - rk) <= stepk + 1e-30)


@pytest.mark.parametrize("out_prec", ["mxfp8", "fp8", "bf16"])
def test_fused_quantiser_bit_exact_on_its_input(out_prec):
    """The fused preprocess with no key LayerNorm and no rotary dims on FP32
    input: its carrier is the input itself, so the quantiser inside the fused
    kernel must give the oracle's quantisation of that input bit for bit
    (codes and scale bytes; BF16: the RNE bit patterns), queries and keys,
    including the edge rows of the stand-alone quantiser test."""
    rng = np.random.default_rng(17)
    lens, H, D = [37, 5, 90], 8, 128
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    edge = _edge_rows(rng)
    q = (rng.standard_normal((T * H, D)) * np.exp2(rng.integers(-20, 20, (T * H, 1)))).astype(np.float32)
    q[:len(edge)] = edge
    k = (rng.standard_normal((T, D)) * np.exp2(rng.integers(-20, 20, (T, 1)))).astype(np.float32)
    k[:len(edge)] = edge[::-1]
    q_op, q_sc, k_op, k_sc = dsa.preprocess(dev(q.reshape(T, H, D)), dev(k), dev(cu), max(lens), None, None,
                                            1e-6, 0, 10000.0, False, True, out_prec)
    if out_prec == "bf16":
        np.testing.assert_array_equal(host(q_op.view(torch.int16)).view(np.uint16),
                                      O.float_to_bf16_bits(O.round_bf16(q.astype(np.float64))))
        np.testing.assert_array_equal(host(k_op.view(torch.int16)).view(np.uint16),
                                      O.float_to_bf16_bits(O.round_bf16(k.astype(np.float64))))
        return
    quant = O.quantize_mxfp8 if out_prec == "mxfp8" else O.quantize_fp8_rows
    rqc, rqs, _ = quant(q.astype(np.float64))
    rkc, rks, _ = quant(k.astype(np.float64))
    np.testing.assert_array_equal(host(q_sc).reshape(rqs.shape), rqs)
    np.testing.assert_array_equal(host(q_op), rqc)
    np.testing.assert_array_equal(host(k_sc).reshape(rks.shape), rks)
    np.testing.assert_array_equal(host(k_op), rkc)
