"""Double-precision CPU oracle of the DSA lightning-indexer hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its reference arm) may import this
module.  It shares no code with the CUDA library and never calls it; the CUDA
path never calls it either.

It is written to be read against the pages it follows (public Megatron-LM pull
requests):

* [P1] PR #8403, "cuDNN DSA indexer precision options": "What does this PR do?"
  (``dsa_indexer_rope_fp32``, ``dsa_indexer_scoring_precision``), "Motivation"
  (the default path materialises BF16 between key LayerNorm and RoPE), review
  finding 1 (ReLU scoring), finding 2 (BF16 rounding of FP32 carriers at the
  scoring boundary, worked example q = k = 1.001 -> 1.0; output format of the
  repeated-varlen-ends regression), finding 3 (``_indexer_forward(q, k, w,
  ratio, sm_scale, precision)`` with q (1,128,32,128) against k (1,128,1,128):
  one key head shared by every query head).
* [P2] PR #5992, "[DeepSeek-V4] Add compact BF16 and MXFP8 DSA indexer
  support": "Key changes" (BF16 -> MXFP8 quantisation: E4M3 payload with UE8M0
  scales per 32 elements; THD cu_seqlens; deterministic Top-K tie breaking).
* [P3] PR #7522, "KPool (pooled-key) DSA indexer support": "Changes" (pooled
  keys with a BF16 per-token gate and an FP32 per-slot bias, pool selection
  expanded back to tokens, always_select_tail, restart at document
  boundaries, NoPE).

The score itself, I[t,s] = sm_scale * sum_j w[t,j] * ReLU(q[t,j] . k[s]), and
"top-k keys per causally visible query" are what those pages imply (finding 1's
ReLU assertion, finding 3's per-head weights and shared key head); the pages
never print the formula.  Where the pages are silent, the reading taken is
stated at the function it concerns.

Every floating-point step is done in float64.  Rounding to the narrow formats
(BF16, FP32, E4M3) is a single round-to-nearest-even from the float64 value,
written out below from the definition of a binary floating-point format.

Parity pins: every public function here is pinned by tests/test_oracle.py
against closed forms, library routines (torch's bfloat16 / float8_e4m3fn casts,
torch's layer_norm, complex multiplication, scipy's softmax), brute force on
tiny inputs and the worked examples the pages print (tests/golden/).  No
function is unpinned.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0          # largest finite OCP E4M3 value, 1.75 * 2^8
E4M3_MANT_BITS = 3
E4M3_EMIN = -6            # smallest normal exponent of E4M3
BF16_MANT_BITS = 7
FP32_MANT_BITS = 23
FP_EMIN_8BIT_EXP = -126   # smallest normal exponent of FP32 and BF16
UE8M0_BIAS = 127


def round_to_format(x, mant_bits: int, emin: int, max_finite: float = math.inf,
                    saturate: bool = False) -> np.ndarray:
    """Round float64 values to a binary format with `mant_bits` explicit
    mantissa bits and smallest normal exponent `emin`, to nearest, ties to
    even (subnormals kept).

    The spacing of the format around |x| is 2^(floor(log2|x|) - mant_bits) for
    normal numbers and 2^(emin - mant_bits) below 2^emin; x / spacing is
    rounded half-to-even (np.rint) and scaled back.  Both scalings are exact
    (powers of two); -0 stays -0.  Values beyond max_finite become +-inf, or
    +-max_finite when `saturate`.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    nz = ax > 0
    out = np.where(nz, 0.0, x)          # a zero rounds to itself, sign included
    _, e2 = np.frexp(ax[nz])            # ax = m * 2^e2, m in [0.5, 1)
    exp = np.maximum(e2 - 1, emin)      # floor(log2|x|), clamped to subnormal range
    spacing = np.ldexp(1.0, exp - mant_bits)
    out[nz] = np.rint(x[nz] / spacing) * spacing
    over = np.abs(out) > max_finite
    if np.any(over):
        out[over] = np.sign(out[over]) * (max_finite if saturate else math.inf)
    return out


def round_bf16(x) -> np.ndarray:
    """Round to BF16 (8 exponent bits, 7 mantissa bits), RNE.  [P1] finding 2:
    BF16 scoring rounds FP32 carriers to BF16."""
    return round_to_format(x, BF16_MANT_BITS, FP_EMIN_8BIT_EXP, 3.3895313892515355e38)


def round_fp32(x) -> np.ndarray:
    """Round to IEEE binary32, RNE (the FP32 carrier of [P1] rope_fp32)."""
    return round_to_format(x, FP32_MANT_BITS, FP_EMIN_8BIT_EXP, 3.4028234663852886e38)


def round_e4m3_sat(x) -> np.ndarray:
    """Round to OCP FP8 E4M3 (4 exponent bits, bias 7, 3 mantissa bits, no
    infinities, max 448), RNE, saturating to +-448."""
    return round_to_format(x, E4M3_MANT_BITS, E4M3_EMIN, E4M3_MAX, saturate=True)


def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3 byte codes: sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0; exponent 0 is subnormal (mant * 2^-9); 0x7F/0xFF NaN."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(values) -> np.ndarray:
    """Byte code of values that are exactly representable in E4M3 (inverse of
    e4m3_decode; -0 encodes as 0x80)."""
    v = np.asarray(values, dtype=np.float64)
    sign = np.signbit(v).astype(np.int64)
    a = np.abs(v)
    code = np.zeros(v.shape, dtype=np.int64)
    normal = a >= 2.0 ** E4M3_EMIN
    _, e2 = np.frexp(a[normal])
    ex = e2 - 1
    mant = a[normal] / np.ldexp(1.0, ex) * 8 - 8
    code[normal] = ((ex + 7) << 3) | mant.astype(np.int64)
    sub = ~normal
    code[sub] = (a[sub] / 2.0 ** -9).astype(np.int64)
    return ((sign << 7) | code).astype(np.uint8)


def bf16_bits_to_float(bits) -> np.ndarray:
    """Value of BF16 bit patterns (the upper half of an FP32 word)."""
    b = np.asarray(bits, dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def float_to_bf16_bits(values) -> np.ndarray:
    """Bit pattern of values already exactly representable in BF16."""
    f = np.asarray(values, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# MXFP8 quantisation ([P2] "Key changes": BF16 -> MXFP8, E4M3 payload with a
# UE8M0 scale per 32 elements)
# ---------------------------------------------------------------------------

MX_BLOCK = 32


def mx_block_exponent(amax: float, rule: str = "nosat") -> int:
    """UE8M0 exponent e (scale 2^e) of one 32-element block with largest
    magnitude `amax`.

    rule "nosat" (default; reading of the pages' BF16->MXFP8 conversion): the
    smallest integer e with amax <= 448 * 2^e, so the largest element maps to
    at most 448 and nothing saturates.  rule "floor": e = floor(log2 amax) - 8
    (8 = exponent of E4M3's largest binade), elements above 448*2^e saturate.
    e is clamped to the UE8M0 range [-127, 127]; amax = 0 gives -127.
    Found by a plain search with exact float64 comparisons.
    """
    if not amax > 0:
        return -UE8M0_BIAS
    _, e2 = math.frexp(amax)
    fl = e2 - 1                                  # floor(log2 amax)
    if rule == "floor":
        e = fl - 8
    else:
        e = fl - 10
        while amax > E4M3_MAX * 2.0 ** e:
            e += 1
    return int(min(max(e, -UE8M0_BIAS), UE8M0_BIAS))


def mx_block_exponents(amax, rule: str = "nosat") -> np.ndarray:
    """mx_block_exponent applied to every element of the array `amax`, the
    same search written over arrays: start below the answer (floor(log2 amax)
    - 10 for "nosat") and step e up while amax > 448 * 2^e, with exact float64
    comparisons; clamp to [-127, 127]; amax = 0 gives -127."""
    a = np.asarray(amax, dtype=np.float64)
    pos = a > 0
    _, e2 = np.frexp(np.where(pos, a, 1.0))
    fl = e2.astype(np.int64) - 1                 # floor(log2 amax)
    if rule == "floor":
        e = fl - 8
    else:
        e = fl - 10
        while True:
            up = pos & (a > E4M3_MAX * np.ldexp(1.0, e))
            if not up.any():
                break
            e = e + up
    e = np.where(pos, e, -UE8M0_BIAS)
    return np.clip(e, -UE8M0_BIAS, UE8M0_BIAS).astype(np.int64)


def quantize_mxfp8(x, rule: str = "nosat") -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise rows of x [..., D] (D a multiple of 32) to MXFP8.

    Per block of 32 consecutive elements along the last axis: e from
    mx_block_exponent(max |x|), payload = E4M3_RNE_sat(x / 2^e).
    Returns (codes uint8 [..., D], scale bytes uint8 [..., D/32] = e + 127,
    dequantised float64 values payload * 2^e).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % MX_BLOCK == 0
    xb = x.reshape(-1, D // MX_BLOCK, MX_BLOCK)
    amax = np.abs(xb).max(axis=-1)
    e = mx_block_exponents(amax, rule)
    scale = np.ldexp(1.0, e)[..., None]
    payload = round_e4m3_sat(xb / scale)
    deq = (payload * scale).reshape(x.shape)
    codes = e4m3_encode(payload).reshape(x.shape)
    sbytes = (e + UE8M0_BIAS).astype(np.uint8).reshape(x.shape[:-1] + (D // MX_BLOCK,))
    return codes, sbytes, deq


def quantize_fp8_rows(x, rule: str = "nosat") -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """FP8 with one UE8M0 scale per vector ([P1] "What does this PR do?": the
    SM90 path's FP8 scoring with per-vector UE8M0 scales).  Each row of x
    [..., D] gets the exponent mx_block_exponent(max |row|, rule), i.e. the
    MXFP8 block rule applied to the whole row, and payload =
    E4M3_RNE_sat(x / 2^e).  Returns (codes uint8 [..., D], scale bytes uint8
    [...] = e + 127, dequantised float64 values payload * 2^e).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    xr = x.reshape(-1, D)
    amax = np.abs(xr).max(axis=-1)
    e = mx_block_exponents(amax, rule)
    scale = np.ldexp(1.0, e)[:, None]
    payload = round_e4m3_sat(xr / scale)
    deq = (payload * scale).reshape(x.shape)
    codes = e4m3_encode(payload).reshape(x.shape)
    sbytes = (e + UE8M0_BIAS).astype(np.uint8).reshape(x.shape[:-1])
    return codes, sbytes, deq


def dequantize_mxfp8(codes, scale_bytes) -> np.ndarray:
    """float64 value of MXFP8 data: e4m3_decode(code) * 2^(scale_byte - 127)."""
    codes = np.asarray(codes)
    sb = np.asarray(scale_bytes, dtype=np.int64)
    D = codes.shape[-1]
    vals = e4m3_decode(codes).reshape(-1, D // MX_BLOCK, MX_BLOCK)
    scale = np.ldexp(1.0, sb.reshape(-1, D // MX_BLOCK) - UE8M0_BIAS)[..., None]
    return (vals * scale).reshape(codes.shape)


def dequantize_fp8_rows(codes, scale_bytes) -> np.ndarray:
    """float64 value of per-vector FP8 data: e4m3_decode(code) * 2^(byte - 127)
    with one scale byte per row."""
    codes = np.asarray(codes)
    sb = np.asarray(scale_bytes, dtype=np.int64)
    return e4m3_decode(codes) * np.ldexp(1.0, sb - UE8M0_BIAS)[..., None]


# ---------------------------------------------------------------------------
# Preprocessing: key LayerNorm -> RoPE ([P1] "What does this PR do?",
# "Motivation"; [P3] "Changes": NoPE = no rotary)
# ---------------------------------------------------------------------------

def key_layernorm(k, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm over the last axis: (k - mean) / sqrt(var + eps) * gamma + beta,
    biased variance, two passes (mean first, then the mean of squared
    deviations).  Applied to keys only ("key LayerNorm -> RoPE")."""
    k = np.asarray(k, dtype=np.float64)
    mu = k.mean(axis=-1, keepdims=True)
    var = ((k - mu) ** 2).mean(axis=-1, keepdims=True)
    return (k - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def rope_inv_freq(rope_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i / rope_dim), i = 0 .. rope_dim/2 - 1."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / rope_dim)


def apply_rope(x, pos, rope_dim: int, base: float, interleaved: bool = False) -> np.ndarray:
    """Rotary embedding of the first `rope_dim` dims of x [..., D] at integer
    positions pos (broadcast against x[..., 0]); the remaining dims pass
    through.  Pair i (rotate-half: dims i and i + rope_dim/2; interleaved:
    dims 2i and 2i+1) is rotated by angle pos * theta_i:
        (a, b) -> (a cos - b sin, b cos + a sin).
    rope_dim = 0 is the identity (NoPE)."""
    x = np.array(x, dtype=np.float64, copy=True)
    if rope_dim == 0:
        return x
    half = rope_dim // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(rope_dim, base)
    c, s = np.cos(ang), np.sin(ang)
    if interleaved:
        a = x[..., 0:rope_dim:2].copy()
        b = x[..., 1:rope_dim:2].copy()
        x[..., 0:rope_dim:2] = a * c - b * s
        x[..., 1:rope_dim:2] = b * c + a * s
    else:
        a = x[..., :half].copy()
        b = x[..., half:rope_dim].copy()
        x[..., :half] = a * c - b * s
        x[..., half:rope_dim] = b * c + a * s
    return x


def positions_in_document(cu_seqlens) -> np.ndarray:
    """Position of every packed token within its own document (restarting at
    0 at each cu_seqlens boundary)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for d in range(len(cu) - 1):
        pos[cu[d]:cu[d + 1]] = np.arange(cu[d + 1] - cu[d])
    return pos


def preprocess(q, k, cu_seqlens, gamma=None, beta=None, eps: float = 1e-6,
               rope_dim: int = 64, base: float = 10000.0, interleaved: bool = False,
               rope_fp32: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """Query/key preprocessing up to the scoring carrier.

    q [T, H, D], k [T, D] (values of the input dtype).  Keys: LayerNorm (when
    gamma is given), then RoPE; queries: RoPE only.  rope_fp32 (the [P1]
    option): the chain is kept in FP32 and the result is the FP32 carrier.
    Otherwise (the default path of [P1] "Motivation") BF16 is materialised
    after the LayerNorm and after RoPE.  Returned values are float64 holding
    the carrier's values (FP32- or BF16-representable).
    """
    pos = positions_in_document(cu_seqlens)
    kk = np.asarray(k, dtype=np.float64)
    if gamma is not None:
        kk = key_layernorm(kk, gamma, beta, eps)
        if not rope_fp32:
            kk = round_bf16(kk)
    kk = apply_rope(kk, pos, rope_dim, base, interleaved)
    qq = apply_rope(np.asarray(q, dtype=np.float64), pos[:, None], rope_dim, base, interleaved)
    rnd = round_fp32 if rope_fp32 else round_bf16
    return rnd(qq), rnd(kk)


def scoring_operand(carrier, prec: str, rule: str = "nosat"):
    """Scoring operand from a carrier: "bf16" -> RNE to BF16 ([P1] finding 2);
    "mxfp8" -> quantize_mxfp8 along the last axis; "fp8" -> quantize_fp8_rows
    (one scale per row).  Returns (values float64,
    codes or None, scale bytes or None)."""
    if prec == "bf16":
        return round_bf16(carrier), None, None
    if prec == "fp8":
        codes, sb, deq = quantize_fp8_rows(carrier, rule)
        return deq, codes, sb
    codes, sb, deq = quantize_mxfp8(carrier, rule)
    return deq, codes, sb


# ---------------------------------------------------------------------------
# Scores and selection ([P1] findings 1-3, [P2] deterministic tie break)
# ---------------------------------------------------------------------------

def indexer_scores(q_t, k_vis, w_t, sm_scale: float = 1.0) -> np.ndarray:
    """I[s] = sm_scale * sum_j w_t[j] * max(q_t[j] . k_vis[s], 0) for one query.
    q_t [H, D], k_vis [n, D] (the keys the query sees), w_t [H]."""
    acc = np.asarray(q_t, np.float64) @ np.asarray(k_vis, np.float64).T   # [H, n]
    return sm_scale * (np.asarray(w_t, np.float64) @ np.maximum(acc, 0.0))


def error_scale(q_t, k_vis, w_t, sm_scale: float = 1.0) -> np.ndarray:
    """A[s] = |sm_scale| * sum_j |w_t[j]| * sum_d |q_t[j,d] * k_vis[s,d]|: the
    magnitude every rounding error of I[s] is measured against."""
    acc = np.abs(np.asarray(q_t, np.float64)) @ np.abs(np.asarray(k_vis, np.float64)).T
    return abs(sm_scale) * (np.abs(np.asarray(w_t, np.float64)) @ acc)


def relu_magnitude(q_t, k_vis, w_t, sm_scale: float = 1.0) -> np.ndarray:
    """M[s] = |sm_scale| * sum_j |w_t[j]| * max(q_t[j] . k_vis[s], 0): the sum
    of the magnitudes of the terms the score adds up (|I[s]| <= M[s] <= A[s]).
    Relative score tolerances are measured against it."""
    acc = np.asarray(q_t, np.float64) @ np.asarray(k_vis, np.float64).T   # [H, n]
    return abs(sm_scale) * (np.abs(np.asarray(w_t, np.float64)) @ np.maximum(acc, 0.0))


def select_topk(scores, k: int) -> np.ndarray:
    """Indices of the min(k, n) best entries under the total order (score
    descending, index ascending); -0 and +0 are equal.  Returned in that
    order."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))
    return order[:min(k, n)]


def _finish_row(chosen, scores, width: int, order: str):
    chosen = np.asarray(chosen, dtype=np.int64)
    if order == "index":
        chosen = np.sort(chosen)
    idx = np.full(width, -1, dtype=np.int64)
    sc = np.full(width, -np.inf)
    idx[:len(chosen)] = chosen
    sc[:len(chosen)] = scores[chosen]
    return idx, sc, len(chosen)


def indexer_topk(q_op, k_op, w, cu_seqlens, index_topk: int, sm_scale: float = 1.0,
                 rows: Optional[Sequence[int]] = None, order: str = "index",
                 with_scale: bool = False, cu_seqlens_k=None):
    """Top-k per query over its causally visible keys.

    q_op [T, H, D], k_op [S, D]: scoring operands (already rounded /
    dequantised); w [T, H]; cu_seqlens [B+1] for the queries and, when
    given, cu_seqlens_k [B+1] for the keys (default: the same).  Document d
    has T_d queries and S_d >= T_d keys; its queries are its last T_d tokens,
    so query i of it sits at position p = S_d - T_d + i (the global causal
    offset of [P1] review finding 2) and sees local keys 0 .. p (diagonal
    included).  Selected indices are local to the document's keys; fewer than
    k visible keys -> -1 / -inf padding and len = p + 1.  order "index":
    ascending index (the library's default row order); "score": (score desc,
    index asc).  Returns dict(rows, idx [R, k], score [R, k], len [R], and
    when with_scale all_scores / all_scales / all_mags: lists of the full
    score, error-scale A and ReLU-magnitude M rows).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, dtype=np.int64)
    T = int(cu[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    doc_of = np.searchsorted(cu, rows, side="right") - 1
    R = len(rows)
    out_idx = np.full((R, index_topk), -1, dtype=np.int64)
    out_sc = np.full((R, index_topk), -np.inf)
    out_len = np.zeros(R, dtype=np.int64)
    all_scores, all_scales, all_mags = [], [], []
    for r, (t, d) in enumerate(zip(rows, doc_of)):
        a = cu[d]
        off = (cuk[d + 1] - cuk[d]) - (cu[d + 1] - cu[d])
        assert off >= 0, "a document has more queries than keys"
        p = off + t - a
        kv = k_op[cuk[d]:cuk[d] + p + 1]
        s = indexer_scores(q_op[t], kv, w[t], sm_scale)
        chosen = select_topk(s, index_topk)
        out_idx[r], out_sc[r], out_len[r] = _finish_row(chosen, s, index_topk, order)
        if with_scale:
            all_scores.append(s)
            all_scales.append(error_scale(q_op[t], kv, w[t], sm_scale))
            all_mags.append(relu_magnitude(q_op[t], kv, w[t], sm_scale))
        assert p + 1 == len(s)
    res = dict(rows=rows, idx=out_idx, score=out_sc, len=out_len)
    if with_scale:
        res["all_scores"] = all_scores
        res["all_scales"] = all_scales
        res["all_mags"] = all_mags
    return res


# ---------------------------------------------------------------------------
# KPool ([P3] "Changes")
# ---------------------------------------------------------------------------

def kpool_compress(k, gate, slot_bias, cu_seqlens, pool_size: int):
    """Pooled keys: in every document, complete group p of pool_size tokens
    (local tokens p*P .. p*P+P-1) becomes
        kbar_p = sum_i softmax_i(gate[p*P+i] + slot_bias[i]) * k[p*P+i],
    softmax over the P slots (max-subtracted exp / sum).  Pooling restarts at
    each document; an incomplete last group is not pooled (it only ever
    serves as a query's tail).  Returns (kbar float64 [total_pools, D],
    cu_pools int64 [B+1])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    P = pool_size
    k = np.asarray(k, np.float64)
    g = np.asarray(gate, np.float64)
    b = np.asarray(slot_bias, np.float64)
    pools, cu_pools = [], [0]
    for d in range(len(cu) - 1):
        a, L = cu[d], cu[d + 1] - cu[d]
        for p in range(L // P):
            toks = a + p * P + np.arange(P)
            logit = g[toks] + b
            e = np.exp(logit - logit.max())
            pools.append((e / e.sum()) @ k[toks])
        cu_pools.append(cu_pools[-1] + L // P)
    D = k.shape[1]
    kbar = np.array(pools, dtype=np.float64).reshape(-1, D)
    return kbar, np.array(cu_pools, dtype=np.int64)


def compressed_topk(q_op, kc_op, w, cu_seqlens, cu_comp, index_topk: int, ratio: int,
                    sm_scale: float = 1.0, rows: Optional[Sequence[int]] = None, order: str = "index",
                    with_scale: bool = False):
    """Top-k over compressed keys ([P2] "[DeepSeek-V4] Add compact BF16 and
    MXFP8 DSA indexer support": the indexer's `ratio`).  Compressed key c of
    a document stands for its tokens c*ratio .. c*ratio + ratio - 1 and,
    like a complete KPool pool, is visible to the query at local position p
    once complete: c < (p+1) // ratio.  Each query keeps the best
    min(index_topk, visible) compressed keys (score desc, index asc); indices
    are local to the document's compressed keys (no expansion to tokens);
    -1 / -inf padding; len = number kept.  kc_op [total compressed, D],
    cu_comp [B+1] its per-document prefix (at least floor(L/ratio) keys per
    document; extra keys are never visible).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = np.asarray(cu_comp, dtype=np.int64)
    T = int(cu[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    doc_of = np.searchsorted(cu, rows, side="right") - 1
    R = len(rows)
    out_idx = np.full((R, index_topk), -1, dtype=np.int64)
    out_sc = np.full((R, index_topk), -np.inf)
    out_len = np.zeros(R, dtype=np.int64)
    all_scores, all_scales, all_mags = [], [], []
    for r, (t, d) in enumerate(zip(rows, doc_of)):
        p = t - cu[d]
        nvis = (p + 1) // ratio
        kv = kc_op[cc[d]:cc[d] + nvis]
        s = indexer_scores(q_op[t], kv, w[t], sm_scale)
        chosen = select_topk(s, index_topk)
        out_idx[r], out_sc[r], out_len[r] = _finish_row(chosen, s, index_topk, order)
        if with_scale:
            all_scores.append(s)
            all_scales.append(error_scale(q_op[t], kv, w[t], sm_scale))
            all_mags.append(relu_magnitude(q_op[t], kv, w[t], sm_scale))
    res = dict(rows=rows, idx=out_idx, score=out_sc, len=out_len)
    if with_scale:
        res["all_scores"] = all_scores
        res["all_scales"] = all_scales
        res["all_mags"] = all_mags
    return res


def kpool_topk(q_op, kbar_op, w, cu_seqlens, cu_pools, index_topk: int, pool_size: int,
               always_select_tail: bool = True, sm_scale: float = 1.0,
               rows: Optional[Sequence[int]] = None, order: str = "index",
               with_scale: bool = False):
    """Pool selection expanded to tokens ([P3] "Changes").

    Query at local position p sees the complete pools c with c*P + P-1 <= p,
    i.e. c < (p+1) // P.  It keeps the best index_topk // P of them (score
    desc, pool index asc), expands each to its P tokens, and with
    always_select_tail appends its own incomplete pool, tokens
    P*((p+1)//P) .. p, when (p+1) % P != 0.  Row layout (width index_topk +
    P - 1): pool tokens (pools ascending, or by score), then tail tokens, then
    -1.  Scores: the pool's score for its tokens, +inf for tail tokens, -inf
    for padding.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cp = np.asarray(cu_pools, dtype=np.int64)
    P = pool_size
    kp = index_topk // P
    width = index_topk + (P - 1 if always_select_tail else 0)
    T = int(cu[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    doc_of = np.searchsorted(cu, rows, side="right") - 1
    R = len(rows)
    out_idx = np.full((R, width), -1, dtype=np.int64)
    out_sc = np.full((R, width), -np.inf)
    out_len = np.zeros(R, dtype=np.int64)
    all_scores, all_scales, all_mags = [], [], []
    for r, (t, d) in enumerate(zip(rows, doc_of)):
        p = t - cu[d]
        nvis = (p + 1) // P
        kv = kbar_op[cp[d]:cp[d] + nvis]
        s = indexer_scores(q_op[t], kv, w[t], sm_scale)
        chosen = select_topk(s, kp)
        if order == "index":
            chosen = np.sort(chosen)
        toks, scs = [], []
        for c in chosen:
            toks.extend(range(c * P, c * P + P))
            scs.extend([s[c]] * P)
        if always_select_tail and (p + 1) % P != 0:
            tail = list(range(P * nvis, p + 1))
            toks.extend(tail)
            scs.extend([np.inf] * len(tail))
        out_idx[r, :len(toks)] = toks
        out_sc[r, :len(toks)] = scs
        out_len[r] = len(toks)
        if with_scale:
            all_scores.append(s)
            all_scales.append(error_scale(q_op[t], kv, w[t], sm_scale))
            all_mags.append(relu_magnitude(q_op[t], kv, w[t], sm_scale))
    res = dict(rows=rows, idx=out_idx, score=out_sc, len=out_len)
    if with_scale:
        res["all_scores"] = all_scores
        res["all_scales"] = all_scales
        res["all_mags"] = all_mags
    return res
