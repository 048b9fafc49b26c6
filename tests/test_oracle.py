"""Pins of the CPU oracle against things other than itself: library routines,
closed forms, brute force on tiny inputs, invariants and the worked examples
the pages print (tests/golden/).  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from sparse_attention_indexer_dsa_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- formats

def _fp32_samples(rng, n=20000):
    """FP32 values over many binades, plus exact BF16/E4M3 midpoints."""
    v = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    # midpoints between consecutive BF16 values (ties) and their neighbours
    base = (rng.standard_normal(2000).astype(np.float32).view(np.uint32) & 0xFFFF0000)
    mid = (base | 0x8000).view(np.float32)
    odd = ((base | 0x10000) | 0x8000).view(np.float32)
    return np.concatenate([v, mid, odd, np.array([0.0, -0.0, 1e-40, -3e-39], np.float32)])


def test_round_bf16_matches_torch_cast():
    x = _fp32_samples(np.random.default_rng(0))
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_round_fp32_matches_numpy_cast():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-130, 60, 20000))
    np.testing.assert_array_equal(O.round_fp32(x), x.astype(np.float32).astype(np.float64))


def test_round_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(2)
    x = rng.uniform(-448, 448, 20000) * np.exp2(rng.integers(-12, 1, 20000))
    grid = O.e4m3_decode(np.arange(0, 0x7F))
    mids = (grid[1:] + grid[:-1]) / 2                  # exact ties
    x = np.concatenate([x, mids, -mids, [448.0, -448.0, 0.0]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(O.round_e4m3_sat(x.astype(np.float32).astype(np.float64)), ref)


def test_round_e4m3_saturates():
    np.testing.assert_array_equal(O.round_e4m3_sat([500.0, -1e9, 464.0]), [448.0, -448.0, 448.0])


def test_e4m3_codes_match_torch_and_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    vals = O.e4m3_decode(codes)
    np.testing.assert_array_equal(vals, ref)
    np.testing.assert_array_equal(O.e4m3_encode(vals), codes)
    assert O.e4m3_decode([0x7E])[0] == 448.0 and O.e4m3_decode([0x01])[0] == 2.0 ** -9
    assert O.e4m3_decode([0x38])[0] == 1.0


def test_signed_zero_survives_rounding_and_quantisation():
    """-0 rounds to -0 in every format and quantises to the E4M3 code 0x80,
    as torch's casts do."""
    z = np.array([-0.0, 0.0])
    for r in (O.round_bf16(z), O.round_fp32(z), O.round_e4m3_sat(z)):
        assert np.signbit(r[0]) and not np.signbit(r[1])
    ref = torch.tensor([-0.0, 0.0]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    row = np.zeros((1, 32))
    row[0, 5] = -0.0
    row[0, 6] = 1.5
    np.testing.assert_array_equal(O.quantize_mxfp8(row)[0][0, 5:7], [ref[0], O.quantize_mxfp8(row)[0][0, 6]])
    assert O.quantize_fp8_rows(row)[0][0, 5] == ref[0] == 0x80
    assert O.e4m3_encode(O.round_e4m3_sat(z)).tolist() == ref.tolist()


def test_bf16_bits_round_trip():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 16, 5000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # finite only
    vals = O.bf16_bits_to_float(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(vals, ref)
    np.testing.assert_array_equal(O.float_to_bf16_bits(vals), bits)


# ----------------------------------------------------------------- MXFP8

def test_mx_exponent_definition():
    rng = np.random.default_rng(4)
    for a in np.concatenate([rng.uniform(0, 10, 500) * np.exp2(rng.integers(-60, 60, 500)),
                             [448.0, 448.0 * 2 ** -7, 448.0 * 2 ** 3 * (1 + 2 ** -40), 1e-45]]):
        e = O.mx_block_exponent(float(a))
        assert a <= 448.0 * 2.0 ** e
        assert e == -127 or a > 448.0 * 2.0 ** (e - 1)


def test_mx_exponent_exact_binade_edges():
    for e in range(-20, 20):
        assert O.mx_block_exponent(448.0 * 2.0 ** e) == e
        assert O.mx_block_exponent(np.nextafter(448.0 * 2.0 ** e, np.inf)) == e + 1
    assert O.mx_block_exponent(0.0) == -127
    assert O.mx_block_exponent(1e300) == 127
    # floor rule: e = floor(log2 amax) - 8
    assert O.mx_block_exponent(1.0, "floor") == -8
    assert O.mx_block_exponent(1.99, "floor") == -8


def test_mxfp8_payload_matches_torch_cast_of_scaled_block():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 128)) * np.exp2(rng.integers(-8, 8, (64, 1)))).astype(np.float32)
    codes, sb, deq = O.quantize_mxfp8(x.astype(np.float64))
    e = sb.astype(np.int64) - 127
    scaled = x.astype(np.float64).reshape(64, 4, 32) / np.exp2(e)[..., None]
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(codes.reshape(64, 4, 32), ref.view(torch.uint8).numpy())
    np.testing.assert_array_equal(O.dequantize_mxfp8(codes, sb), deq)
    assert np.abs(O.e4m3_decode(codes)).max() <= 448.0


def test_mxfp8_block_power_of_two_invariance():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 128))
    c0, s0, d0 = O.quantize_mxfp8(x)
    for m in (-5, 3, 17):
        c1, s1, d1 = O.quantize_mxfp8(x * 2.0 ** m)
        np.testing.assert_array_equal(c1, c0)
        np.testing.assert_array_equal(s1.astype(int), s0.astype(int) + m)
        np.testing.assert_array_equal(d1, d0 * 2.0 ** m)


def test_mxfp8_grid_values_round_trip_and_zero_block():
    rng = np.random.default_rng(7)
    codes = W.random_e4m3_codes(rng, (4, 128))
    codes[:, ::32] = 0x7E                                   # every block reaches 448
    x = O.e4m3_decode(codes) * 2.0 ** 5
    c, s, d = O.quantize_mxfp8(x)
    np.testing.assert_array_equal(d, x)
    np.testing.assert_array_equal(s, np.full((4, 4), 127 + 5, np.uint8))
    c, s, d = O.quantize_mxfp8(np.zeros((2, 64)))
    assert (s == 0).all() and (d == 0).all() and (c == 0).all()


def test_mxfp8_integer_inputs_are_exact():
    rng = np.random.default_rng(8)
    x = rng.integers(-3, 4, (32, 128)).astype(np.float64)
    _, _, d = O.quantize_mxfp8(x)
    np.testing.assert_array_equal(d, x)


def test_mxfp8_floor_rule_saturates_large_mantissas():
    x = np.zeros((1, 32))
    x[0, 0] = 1.9            # floor rule: e=-8, 1.9*256 = 486.4 > 448 -> saturates
    x[0, 1] = 0.5
    c, s, d = O.quantize_mxfp8(x, "floor")
    assert s[0, 0] == 127 - 8 and d[0, 0] == 448.0 * 2.0 ** -8
    c, s, d = O.quantize_mxfp8(x, "nosat")
    assert s[0, 0] == 127 - 7 and abs(d[0, 0] - 1.9) < 1.9 * 2 ** -4


# ----------------------------------------------------------------- preprocessing

def test_layernorm_matches_torch_layer_norm():
    rng = np.random.default_rng(9)
    k = rng.standard_normal((50, 128)) * 3 + 1
    g = 1 + 0.1 * rng.standard_normal(128)
    b = 0.1 * rng.standard_normal(128)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(k), (128,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-6).numpy()
    np.testing.assert_allclose(O.key_layernorm(k, g, b, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_layernorm_closed_form_moments():
    rng = np.random.default_rng(10)
    k = rng.standard_normal((20, 64)) * 0.01
    eps = 1e-4
    y = O.key_layernorm(k, np.ones(64), np.zeros(64), eps)
    var = k.var(axis=-1)
    np.testing.assert_allclose(y.mean(axis=-1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=-1), var / (var + eps), rtol=1e-10)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((7, 128))
    pos = rng.integers(0, 40000, 7)
    th = 10000.0 ** (-np.arange(32) * 2 / 64)
    for inter in (False, True):
        y = O.apply_rope(x, pos, 64, 10000.0, inter)
        if inter:
            z = (x[:, 0:64:2] + 1j * x[:, 1:64:2]) * np.exp(1j * pos[:, None] * th)
            np.testing.assert_allclose(y[:, 0:64:2], z.real, atol=1e-12)
            np.testing.assert_allclose(y[:, 1:64:2], z.imag, atol=1e-12)
        else:
            z = (x[:, :32] + 1j * x[:, 32:64]) * np.exp(1j * pos[:, None] * th)
            np.testing.assert_allclose(y[:, :32], z.real, atol=1e-12)
            np.testing.assert_allclose(y[:, 32:64], z.imag, atol=1e-12)
        np.testing.assert_array_equal(y[:, 64:], x[:, 64:])


def test_rope_unit_vector_position_one():
    x = np.zeros((1, 128))
    x[0, 0] = 1.0
    y = O.apply_rope(x, np.array([1]), 64, 10000.0)
    assert y[0, 0] == pytest.approx(math.cos(1.0)) and y[0, 32] == pytest.approx(math.sin(1.0))


def test_rope_invariants():
    rng = np.random.default_rng(12)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    y0 = O.apply_rope(q[None], np.array([0]), 64, 10000.0)
    np.testing.assert_array_equal(y0[0], q)
    y = O.apply_rope(q[None], np.array([1234]), 64, 10000.0)[0]
    np.testing.assert_allclose(y[:32] ** 2 + y[32:64] ** 2, q[:32] ** 2 + q[32:64] ** 2, rtol=1e-12)
    dots = []
    for m, n in [(10, 3), (1007, 1000), (30007, 30000)]:
        qm = O.apply_rope(q[None], np.array([m]), 64, 10000.0)[0]
        kn = O.apply_rope(k[None], np.array([n]), 64, 10000.0)[0]
        dots.append(qm @ kn)
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    np.testing.assert_array_equal(O.apply_rope(q[None], np.array([55]), 0, 10000.0)[0], q)


def test_positions_restart_per_document():
    np.testing.assert_array_equal(O.positions_in_document([0, 3, 3, 5]), [0, 1, 2, 0, 1])


def test_preprocess_rope_fp32_and_bf16_paths():
    rng = np.random.default_rng(13)
    T, H, D = 6, 2, 128
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = rng.standard_normal((T, D)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32)
    cu = np.array([0, 4, 6])
    pos = O.positions_in_document(cu)
    qf, kf = O.preprocess(q, k, cu, g, b, 1e-6, 64, 10000.0, False, rope_fp32=True)
    ln = O.key_layernorm(k, g, b, 1e-6)
    np.testing.assert_array_equal(kf, O.round_fp32(O.apply_rope(ln, pos, 64, 10000.0)))
    np.testing.assert_array_equal(qf, O.round_fp32(O.apply_rope(q, pos[:, None], 64, 10000.0)))
    qb, kb = O.preprocess(q, k, cu, g, b, 1e-6, 64, 10000.0, False, rope_fp32=False)
    np.testing.assert_array_equal(kb, O.round_bf16(O.apply_rope(O.round_bf16(ln), pos, 64, 10000.0)))
    assert not np.array_equal(kb, O.round_bf16(kf))   # the BF16 round trip changes values


# ----------------------------------------------------------------- scores

def _brute_scores(q_t, k_vis, w_t, sm):
    out = []
    for s in range(k_vis.shape[0]):
        tot = 0.0
        for j in range(q_t.shape[0]):
            dot = sum(float(q_t[j, d]) * float(k_vis[s, d]) for d in range(q_t.shape[1]))
            tot += float(w_t[j]) * max(dot, 0.0)
        out.append(sm * tot)
    return np.array(out)


def test_scores_brute_force():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((3, 5))
    k = rng.standard_normal((6, 5))
    w = rng.standard_normal(3)
    np.testing.assert_allclose(O.indexer_scores(q, k, w, 0.7), _brute_scores(q, k, w, 0.7), rtol=1e-12)
    A = O.error_scale(q, k, w, 0.7)
    bruteA = [0.7 * sum(abs(w[j]) * sum(abs(q[j, d] * k[s, d]) for d in range(5)) for j in range(3))
              for s in range(6)]
    np.testing.assert_allclose(A, bruteA, rtol=1e-12)
    assert (np.abs(O.indexer_scores(q, k, w, 0.7)) <= A + 1e-12).all()


def test_relu_magnitude_brute_force_and_bounds():
    """M[s] = |sm| sum_j |w_j| max(q_j . k_s, 0), against a plain triple loop;
    |I| <= M <= A on random rows, and M == |I| when every weight is positive."""
    rng = np.random.default_rng(15)
    q = rng.standard_normal((4, 6))
    k = rng.standard_normal((7, 6))
    w = rng.standard_normal(4)
    M = O.relu_magnitude(q, k, w, -0.6)
    brute = [0.6 * sum(abs(w[j]) * max(sum(q[j, d] * k[s, d] for d in range(6)), 0.0) for j in range(4))
             for s in range(7)]
    np.testing.assert_allclose(M, brute, rtol=1e-12)
    I = O.indexer_scores(q, k, w, -0.6)
    A = O.error_scale(q, k, w, -0.6)
    assert (np.abs(I) <= M + 1e-12).all() and (M <= A + 1e-12).all()
    wp = np.abs(w)
    np.testing.assert_allclose(O.relu_magnitude(q, k, wp, 0.6), O.indexer_scores(q, k, wp, 0.6), rtol=1e-12)
    res = O.indexer_topk(q[None].repeat(3, 0), k[:3], w[None].repeat(3, 0), [0, 3], 2, with_scale=True)
    np.testing.assert_allclose(res["all_mags"][2], O.relu_magnitude(q, k[:3], w), rtol=1e-12)


def test_mx_block_exponents_equal_the_scalar_search():
    """The array form of the block-exponent search gives the scalar search's
    exponent for every value: zero, subnormals, exact binade edges 448 * 2^e
    and their neighbours, the UE8M0 clamp at both ends, and random values."""
    rng = np.random.default_rng(16)
    edges = [0.0, 5e-324, 2.0 ** -140, 2.0 ** -127 * 448, 2.0 ** 127 * 448, 3.4e38, 1e300]
    for e in range(-130, 130, 7):
        b = 448.0 * 2.0 ** e
        edges += [b, np.nextafter(b, 0), np.nextafter(b, np.inf)]
    vals = np.concatenate([edges, np.abs(rng.standard_normal(2000)) * np.exp2(rng.integers(-140, 140, 2000))])
    for rule in ("nosat", "floor"):
        got = O.mx_block_exponents(vals, rule)
        want = [O.mx_block_exponent(float(v), rule) for v in vals]
        np.testing.assert_array_equal(got, want)


def test_fp8_rows_dequantisation_round_trip():
    rng = np.random.default_rng(17)
    x = rng.standard_normal((9, 128)) * np.exp2(rng.integers(-20, 20, (9, 1)))
    codes, sb, deq = O.quantize_fp8_rows(x)
    np.testing.assert_array_equal(O.dequantize_fp8_rows(codes, sb), deq)
    # one byte per row: a row scaled by 2^m dequantises to the scaled values
    c2, s2, d2 = O.quantize_fp8_rows(x * 8.0)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2.astype(int), sb.astype(int) + 3)
    np.testing.assert_array_equal(O.dequantize_fp8_rows(c2, s2), deq * 8.0)


def test_preprocess_bf16_path_query_closed_form():
    """Default (rope_fp32 = 0) chain, query side: a query whose rotary pair
    (0, 32) is the unit vector (1, 0) becomes (cos(p), sin(p)) at position p
    (theta_0 = 1), rounded once to BF16 (torch's cast of the float64 cosine
    and sine); the NoPE half comes out as its own BF16 rounding; position 0
    leaves the rotary dims unrotated."""
    T, H, D = 7, 1, 128
    q = np.zeros((T, H, D), np.float32)
    q[:, 0, 0] = 1.0
    q[:, 0, 64:] = np.linspace(-3.3, 3.7, 64, dtype=np.float32)
    k = np.ones((T, D), np.float32)
    cu = np.array([0, T])
    qb, _ = O.preprocess(q, k, cu, None, None, 1e-6, 64, 10000.0, False, rope_fp32=False)
    to_bf16 = lambda v: torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    for p in range(T):
        assert qb[p, 0, 0] == to_bf16(math.cos(p))
        assert qb[p, 0, 32] == to_bf16(math.sin(p))
        np.testing.assert_array_equal(qb[p, 0, 64:], to_bf16(q[p, 0, 64:].astype(np.float64)))
    assert qb[0, 0, 0] == 1.0 and qb[0, 0, 32] == 0.0


def test_golden_bf16_scoring_boundary():
    g = _golden("bf16_scoring_boundary.json")
    q = np.array([[g["q"]]])
    k = np.array([[g["k"]]])
    w = np.array([g["w"]])
    qb, _, _ = O.scoring_operand(O.round_fp32(q), "bf16")
    kb, _, _ = O.scoring_operand(O.round_fp32(k), "bf16")
    assert O.indexer_scores(qb, kb, w, g["sm_scale"])[0] == g["expected_bf16_score"]
    f = O.indexer_scores(O.round_fp32(q), O.round_fp32(k), w, g["sm_scale"])[0]
    assert abs(f - g["expected_fp32_score_approx"]) < g["fp32_abs_tol"]


def test_golden_repeated_varlen_ends_format():
    g = _golden("repeated_varlen_ends_format.json")
    T = sum(g["doc_lens"])
    q = np.array(g["q"]).reshape(T, 1, 1)
    k = np.array(g["k"]).reshape(T, 1)
    w = np.array(g["w"]).reshape(T, 1)
    cu = np.concatenate([[0], np.cumsum(g["doc_lens"])])
    r = O.indexer_topk(q, k, w, cu, g["index_topk"], rows=g["rows"], order="score")
    np.testing.assert_array_equal(r["idx"], g["expected_indices"])
    np.testing.assert_array_equal(r["len"], g["expected_lengths"])
    np.testing.assert_array_equal(r["score"], g["expected_scores"])


# ----------------------------------------------------------------- selection

def _dominates(sa, a, sb, b):
    return sa > sb or (sa == sb and a < b)


def test_select_topk_brute_force_dominance():
    rng = np.random.default_rng(15)
    for _ in range(200):
        n = int(rng.integers(1, 9))
        s = rng.integers(-2, 3, n).astype(np.float64)      # many ties
        s[rng.random(n) < 0.2] = -0.0
        kk = int(rng.integers(1, 10))
        ch = O.select_topk(s, kk)
        assert len(ch) == min(kk, n) and len(set(ch.tolist())) == len(ch)
        rest = [i for i in range(n) if i not in set(ch.tolist())]
        for a in ch:
            for b in rest:
                assert _dominates(s[a], a, s[b], b)
        # exhaustive: the chosen set is the unique set dominating its complement
        valid = [set(c) for c in itertools.combinations(range(n), min(kk, n))
                 if all(_dominates(s[a], a, s[b], b) for a in c for b in set(range(n)) - set(c))]
        assert valid == [set(ch.tolist())]


def test_selection_invariants_on_integer_workload():
    wl = W.config("tiny")
    x = W.make_inputs(wl)
    cu = wl.cu_seqlens
    rows = np.arange(0, wl.total_tokens, 7)
    r = O.indexer_topk(x["q"].astype(np.float64), x["k"].astype(np.float64), x["w"].astype(np.float64),
                       cu, wl.index_topk, rows=rows, with_scale=True)
    for i, t in enumerate(rows):
        n = min(wl.index_topk, t + 1)
        idx = r["idx"][i]
        assert r["len"][i] == n
        assert (idx[:n] >= 0).all() and (idx[:n] <= t).all() and (idx[n:] == -1).all()
        assert len(set(idx[:n].tolist())) == n
        assert (np.diff(idx[:n]) > 0).all()
    # permuting heads jointly in q and w leaves the selection unchanged (exact: integers)
    perm = np.random.default_rng(16).permutation(wl.n_heads)
    r2 = O.indexer_topk(x["q"][:, perm].astype(np.float64), x["k"].astype(np.float64),
                        x["w"][:, perm].astype(np.float64), cu, wl.index_topk, rows=rows)
    np.testing.assert_array_equal(r2["idx"], r["idx"])
    # scaling w by 2^m leaves the selection unchanged
    r3 = O.indexer_topk(x["q"].astype(np.float64), x["k"].astype(np.float64),
                        x["w"].astype(np.float64) * 8.0, cu, wl.index_topk, rows=rows)
    np.testing.assert_array_equal(r3["idx"], r["idx"])


def test_all_visible_selected_when_k_exceeds_row():
    rng = np.random.default_rng(17)
    q = rng.standard_normal((10, 2, 8))
    k = rng.standard_normal((10, 8))
    w = rng.standard_normal((10, 2))
    r = O.indexer_topk(q, k, w, [0, 10], 16)
    for t in range(10):
        np.testing.assert_array_equal(r["idx"][t, :t + 1], np.arange(t + 1))


def test_thd_documents_equal_separate_runs():
    rng = np.random.default_rng(18)
    lens = [5, 9, 3]
    T = sum(lens)
    q = rng.standard_normal((T, 2, 8))
    k = rng.standard_normal((T, 8))
    w = rng.standard_normal((T, 2))
    cu = np.concatenate([[0], np.cumsum(lens)])
    r = O.indexer_topk(q, k, w, cu, 4)
    for d, L in enumerate(lens):
        a = cu[d]
        rd = O.indexer_topk(q[a:a + L], k[a:a + L], w[a:a + L], [0, L], 4)
        np.testing.assert_array_equal(r["idx"][a:a + L], rd["idx"])
        np.testing.assert_array_equal(r["score"][a:a + L], rd["score"])


def test_global_offsets_equal_last_rows_of_full_run():
    """Queries that are the last T_d of S_d tokens ([P1] review finding 2,
    global causal offsets) score exactly like those rows of the full
    self-attention run over all S_d tokens."""
    rng = np.random.default_rng(19)
    lens_k, lens_q = [12, 7, 4, 9], [5, 7, 0, 1]
    S = sum(lens_k)
    q_full = rng.integers(-2, 3, (S, 3, 8)).astype(np.float64)   # integers: ties exercise the rule
    k = rng.integers(-2, 3, (S, 8)).astype(np.float64)
    w_full = rng.integers(-2, 3, (S, 3)).astype(np.float64)
    cuk = np.concatenate([[0], np.cumsum(lens_k)])
    cuq = np.concatenate([[0], np.cumsum(lens_q)])
    rows_full = np.concatenate([np.arange(cuk[d + 1] - lens_q[d], cuk[d + 1]) for d in range(4)]).astype(np.int64)
    full = O.indexer_topk(q_full, k, w_full, cuk, 6, rows=rows_full)
    off = O.indexer_topk(q_full[rows_full], k, w_full[rows_full], cuq, 6, cu_seqlens_k=cuk)
    np.testing.assert_array_equal(off["idx"], full["idx"])
    np.testing.assert_array_equal(off["score"], full["score"])
    np.testing.assert_array_equal(off["len"], full["len"])


def test_global_offsets_brute_force():
    """Explicit loops: query i of document d sees keys 0 .. S_d - T_d + i of
    that document; the best min(k, visible) by (score desc, index asc),
    listed in ascending index."""
    rng = np.random.default_rng(20)
    lens_k, lens_q = [6, 3], [2, 3]
    q = rng.standard_normal((5, 2, 4))
    k = rng.standard_normal((9, 4))
    w = rng.standard_normal((5, 2))
    cuk, cuq = [0, 6, 9], [0, 2, 5]
    r = O.indexer_topk(q, k, w, cuq, 3, cu_seqlens_k=cuk)
    row = 0
    for d in range(2):
        for i in range(lens_q[d]):
            p = lens_k[d] - lens_q[d] + i
            sc = _brute_scores(q[row], k[cuk[d]:cuk[d] + p + 1], w[row], 1.0)
            best = sorted(range(p + 1), key=lambda s_: (-sc[s_], s_))[:3]
            n = len(best)
            assert r["len"][row] == n
            np.testing.assert_array_equal(r["idx"][row][:n], sorted(best))
            np.testing.assert_allclose(r["score"][row][:n], sc[sorted(best)], rtol=1e-12)
            row += 1


# ----------------------------------------------------------------- FP8 with per-vector scales

def test_fp8_rows_of_32_equal_the_mx_block_rule():
    """A 32-element row is one MX block: the per-vector quantiser must agree
    with the (separately pinned) MXFP8 quantiser code for code."""
    x = np.random.default_rng(24).standard_normal((300, 32)) * np.exp(np.random.default_rng(25).uniform(-20, 20, (300, 1)))
    c1, s1, d1 = O.quantize_fp8_rows(x)
    c2, s2, d2 = O.quantize_mxfp8(x)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2[:, 0])
    np.testing.assert_array_equal(d1, d2)


def test_fp8_rows_power_of_two_invariance_and_range():
    rng = np.random.default_rng(26)
    x = rng.standard_normal((50, 128))
    c, sb, d = O.quantize_fp8_rows(x)
    c8, sb8, d8 = O.quantize_fp8_rows(x * 2.0 ** 9)
    np.testing.assert_array_equal(c8, c)
    np.testing.assert_array_equal(sb8.astype(int), sb.astype(int) + 9)
    amax = np.abs(x).max(axis=1)
    scale = np.ldexp(1.0, sb.astype(int) - 127)
    assert (amax <= 448 * scale).all() and (amax > 448 * scale / 2).all()   # the smallest such exponent
    assert np.abs(d - x).max(axis=1).max() <= (scale * 2.0 ** 5).max()        # within half an E4M3 step


def test_fp8_scale_folding_is_exact():
    """The per-vector scales are positive powers of two and ReLU is positively
    homogeneous, so scoring the dequantised operands equals scoring the raw
    payloads with w_j * s_q[j] and the result times s_k, exactly."""
    rng = np.random.default_rng(27)
    q = rng.standard_normal((4, 32)) * 3
    k = rng.standard_normal((9, 32))
    w = rng.standard_normal(4)
    qc, qs, qd = O.quantize_fp8_rows(q)
    kc, ks, kd = O.quantize_fp8_rows(k)
    direct = O.indexer_scores(qd, kd, w, 0.5)
    sq = np.ldexp(1.0, qs.astype(int) - 127)
    sk = np.ldexp(1.0, ks.astype(int) - 127)
    folded = O.indexer_scores(O.e4m3_decode(qc), O.e4m3_decode(kc), w * sq, 0.5) * sk
    np.testing.assert_array_equal(folded, direct)


# ----------------------------------------------------------------- compressed keys

def test_compressed_ratio_one_is_the_plain_indexer():
    rng = np.random.default_rng(21)
    lens = [9, 4]
    q = rng.standard_normal((13, 2, 8))
    k = rng.standard_normal((13, 8))
    w = rng.standard_normal((13, 2))
    cu = [0, 9, 13]
    a = O.compressed_topk(q, k, w, cu, cu, 5, 1)
    b = O.indexer_topk(q, k, w, cu, 5)
    for key in ("idx", "score", "len"):
        np.testing.assert_array_equal(a[key], b[key])


def test_compressed_selection_matches_kpool_pools():
    """Given pooled keys, the compressed selection of index_topk / P keys is
    exactly the set of pools KPool expands (its tokens / P, tail excluded)."""
    rng = np.random.default_rng(22)
    lens, P, kk = [23, 10], 4, 12
    T = sum(lens)
    q = rng.integers(-2, 3, (T, 2, 8)).astype(np.float64)
    k = rng.standard_normal((T, 8))
    w = rng.integers(-2, 3, (T, 2)).astype(np.float64)
    cu = np.array([0, 23, 33])
    kbar, cp = O.kpool_compress(k, rng.standard_normal(T), rng.standard_normal(P), cu, P)
    c = O.compressed_topk(q, kbar, w, cu, cp, kk // P, P)
    kp = O.kpool_topk(q, kbar, w, cu, cp, kk, P, always_select_tail=False)
    for r in range(T):
        n = c["len"][r]
        assert kp["len"][r] == n * P
        np.testing.assert_array_equal(kp["idx"][r][:n * P:P] // P, c["idx"][r][:n])
        np.testing.assert_array_equal(kp["score"][r][:n * P:P], c["score"][r][:n])


def test_compressed_visibility_brute_force():
    rng = np.random.default_rng(23)
    ratio, L = 3, 11
    q = rng.standard_normal((L, 2, 4))
    kc = rng.standard_normal((4, 4))     # ceil(11 / 3): the last one is never complete
    w = rng.standard_normal((L, 2))
    r = O.compressed_topk(q, kc, w, [0, L], [0, 4], 2, ratio)
    for t in range(L):
        nvis = sum(1 for c in range(4) if c * ratio + ratio - 1 <= t)
        sc = _brute_scores(q[t], kc[:nvis], w[t], 1.0)
        best = sorted(sorted(range(nvis), key=lambda s_: (-sc[s_], s_))[:2])
        assert r["len"][t] == len(best)
        np.testing.assert_array_equal(r["idx"][t][:len(best)], best)
        assert (r["idx"][t][len(best):] == -1).all()


# ----------------------------------------------------------------- KPool

def test_kpool_single_slot_reduces_to_plain_indexer():
    rng = np.random.default_rng(19)
    T, D = 12, 16
    k = rng.standard_normal((T, D))
    kbar, cp = O.kpool_compress(k, rng.standard_normal(T), np.zeros(1), [0, 7, 12], 1)
    np.testing.assert_array_equal(kbar, k)
    np.testing.assert_array_equal(cp, [0, 7, 12])
    q = rng.standard_normal((T, 2, D))
    w = rng.standard_normal((T, 2))
    a = O.kpool_topk(q, kbar, w, [0, 7, 12], cp, 3, 1)
    b = O.indexer_topk(q, k, w, [0, 7, 12], 3)
    np.testing.assert_array_equal(a["idx"], b["idx"])


def test_kpool_softmax_weights():
    rng = np.random.default_rng(20)
    k = rng.standard_normal((9, 8))
    kbar, cp = O.kpool_compress(k, np.zeros(9), np.zeros(4), [0, 9], 4)
    np.testing.assert_allclose(kbar, [k[0:4].mean(0), k[4:8].mean(0)], rtol=1e-12)
    assert list(cp) == [0, 2]
    from scipy.special import softmax
    g = rng.standard_normal(9)
    b = rng.standard_normal(4)
    kbar, _ = O.kpool_compress(k, g, b, [0, 9], 4)
    np.testing.assert_allclose(kbar[1], softmax(g[4:8] + b) @ k[4:8], rtol=1e-12)


def test_kpool_selection_tail_and_visibility():
    rng = np.random.default_rng(21)
    P, T, D = 4, 23, 8
    k = rng.standard_normal((T, D))
    q = rng.standard_normal((T, 2, D))
    w = np.abs(rng.standard_normal((T, 2)))
    cu = [0, 13, 23]
    kbar, cp = O.kpool_compress(k, rng.standard_normal(T), rng.standard_normal(P), cu, P)
    r = O.kpool_topk(q, kbar, w, cu, cp, 8, P, True)
    for t in range(T):
        d = 0 if t < 13 else 1
        p = t - cu[d]
        nvis = (p + 1) // P
        toks = r["idx"][t][: r["len"][t]]
        assert (toks <= p).all() and len(set(toks.tolist())) == len(toks)
        npool = min(2, nvis)
        tail = (p + 1) % P
        assert r["len"][t] == npool * P + tail
        np.testing.assert_array_equal(toks[npool * P:], np.arange(P * nvis, p + 1))
        assert np.isinf(r["score"][t][npool * P: npool * P + tail]).all()
        for c in range(npool):           # expansion: P consecutive tokens of one pool
            blk = toks[c * P:(c + 1) * P]
            assert blk[0] % P == 0 and (np.diff(blk) == 1).all()
    r2 = O.kpool_topk(q, kbar, w, cu, cp, 8, P, False)
    assert (r2["len"] % P == 0).all()


# ----------------------------------------------------------------- ranking order

def _ranked(idx, sc, n):
    """Entries [0, n) reordered by a plain sort on (score desc, index asc)."""
    order = sorted(range(n), key=lambda e: (-float(sc[e]), int(idx[e])))
    return idx[order], sc[order]


def test_score_order_ranks_the_index_order_rows():
    """order="score" holds the same entries as order="index", ranked by their
    own scores with ties to the lower index (integer scores: many ties)."""
    rng = np.random.default_rng(801)
    lens, H, D, k = [40, 1, 23], 4, 8, 9
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q = rng.integers(-2, 3, (T, H, D)).astype(np.float64)
    kk = rng.integers(-2, 3, (T, D)).astype(np.float64)
    w = rng.integers(-1, 2, (T, H)).astype(np.float64)
    a = O.indexer_topk(q, kk, w, cu, k)
    b = O.indexer_topk(q, kk, w, cu, k, order="score")
    np.testing.assert_array_equal(a["len"], b["len"])
    for r in range(T):
        n = int(a["len"][r])
        assert (np.diff(a["idx"][r, :n]) > 0).all()
        ri, rs = _ranked(a["idx"][r], a["score"][r], n)
        np.testing.assert_array_equal(b["idx"][r, :n], ri)
        np.testing.assert_array_equal(b["score"][r, :n], rs)
        assert (b["idx"][r, n:] == -1).all()
        if n:   # the first entry is the best visible key (brute force)
            s = O.indexer_scores(q[r], kk[cu[np.searchsorted(cu, r, side="right") - 1]:r + 1], w[r])
            assert b["score"][r, 0] == s.max() and b["idx"][r, 0] == int(np.flatnonzero(s == s.max())[0])


@pytest.mark.parametrize("P,tail", [(4, True), (2, False)])
def test_kpool_score_order_ranks_pools_and_keeps_the_tail_last(P, tail):
    rng = np.random.default_rng(802 + P)
    lens, H, D, k = [37, 6], 4, 8, 4 * P
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    npool = [L // P for L in lens]
    cp = np.concatenate([[0], np.cumsum(npool)])
    q = rng.integers(-2, 3, (T, H, D)).astype(np.float64)
    kb = rng.integers(-2, 3, (sum(npool), D)).astype(np.float64)
    w = rng.integers(-1, 2, (T, H)).astype(np.float64)
    a = O.kpool_topk(q, kb, w, cu, cp, k, P, tail)
    b = O.kpool_topk(q, kb, w, cu, cp, k, P, tail, order="score")
    np.testing.assert_array_equal(a["len"], b["len"])
    for r in range(T):
        n = int(a["len"][r])
        ntail = int(np.sum(np.isposinf(a["score"][r, :n])))
        npt = n - ntail
        # pools: groups of P consecutive tokens, ranked by (score desc, pool asc)
        pa = a["idx"][r, :npt].reshape(-1, P)[:, 0] // P
        sa = a["score"][r, :npt].reshape(-1, P)[:, 0]
        rp, _ = _ranked(pa, sa, len(pa))
        exp = (rp[:, None] * P + np.arange(P)[None, :]).reshape(-1)
        np.testing.assert_array_equal(b["idx"][r, :npt], exp)
        # the tail: unchanged, last
        np.testing.assert_array_equal(b["idx"][r, npt:n], a["idx"][r, npt:n])
        assert np.isposinf(b["score"][r, npt:n]).all()


def test_compressed_score_order_ranks_the_index_order_rows():
    rng = np.random.default_rng(803)
    lens, H, D, k, ratio = [50, 9], 4, 8, 5, 4
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    nc = [L // ratio for L in lens]
    cc = np.concatenate([[0], np.cumsum(nc)])
    q = rng.integers(-2, 3, (T, H, D)).astype(np.float64)
    kc = rng.integers(-2, 3, (sum(nc), D)).astype(np.float64)
    w = rng.integers(-1, 2, (T, H)).astype(np.float64)
    a = O.compressed_topk(q, kc, w, cu, cc, k, ratio)
    b = O.compressed_topk(q, kc, w, cu, cc, k, ratio, order="score")
    for r in range(T):
        n = int(a["len"][r])
        ri, rs = _ranked(a["idx"][r], a["score"][r], n)
        np.testing.assert_array_equal(b["idx"][r, :n], ri)
        np.testing.assert_array_equal(b["score"][r, :n], rs)
