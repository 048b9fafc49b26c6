"""GPU-vs-oracle comparison rules for the fused score + top-k.

Scores.  The score I = sm_scale * sum_j w_j * ReLU(q_j . k) adds up the terms
w_j * ReLU(acc_j); its rounding errors are measured against the sum of their
magnitudes, M = |sm_scale| * sum_j |w_j| * ReLU(q_j . k) (|I| <= M).  "Relative"
precision is read as relative to M.  On top of that comes a rigorous allowance
for the FP32 accumulation of the contraction itself: every acc_j = q_j . k sums
D products in FP32, so its error is at most D * 2^-23 * sum_d |q_jd k_d| (a
bound that also covers truncating accumulation), which, through the 1-Lipschitz
ReLU and the head weights, gives gamma_D * A with A = |sm_scale| * sum_j |w_j|
* sum_d |q_jd k_d| and gamma_D = D * 2^-23; the FP32 head sum adds H * 2^-23 * M.
A GPU score passes when

    |I_gpu - I_oracle| <= tol = (rel + H * 2^-23) * M + D * 2^-23 * A,

rel = 2e-3 for BF16 scoring and 1.5e-2 for the 8-bit formats (the oracle
applying the same E4M3/UE8M0 quantisation).

Index sets.  Equal, except a key the GPU took in place of an oracle key, when
each of the two lies within tol_i + tol_kth of the oracle's k-th score (a swap
at the selection boundary).  The number of swapped keys of a row is bounded
(default: 1 % of the row, at least one).  Integer-valued inputs: bit-exact.

compare_topk returns the statistics the parity reports print: rows checked,
rows with swaps, swapped keys (total and worst row), the largest score error
as a fraction of its tolerance and of M, and the mean fraction of a row's
visible keys that lie inside the swap band (how much room the rule leaves).
"""
from __future__ import annotations

import math

import numpy as np

REL_BF16 = 2e-3
REL_MXFP8 = 1.5e-2
U32 = 2.0 ** -23           # FP32 unit roundoff, doubled to cover truncation


def tolerance(rel, M, A, head_dim, n_heads):
    return (rel + n_heads * U32) * M + head_dim * U32 * A


def compare_topk(g_idx, g_sc, g_len, ref, rel: float, exact: bool = False, pool: int = 1,
                 tail: bool = True, rows=None, head_dim: int = 128, n_heads: int = 64,
                 swap_frac: float = 0.01):
    """Assert parity of GPU rows against an oracle result dict (with_scale=True
    unless exact).  Returns a dict of statistics."""
    rows = ref["rows"] if rows is None else rows
    st = dict(rows=0, rows_with_swaps=0, swaps=0, max_swaps_row=0, max_err_over_tol=0.0,
              max_err_over_M=0.0, band_frac=0.0, band_rows=0)
    for r, t in enumerate(rows):
        gi, gs, gl = g_idx[t], g_sc[t] if g_sc is not None else None, int(g_len[t])
        oi, osc, ol = ref["idx"][r], ref["score"][r], int(ref["len"][r])
        st["rows"] += 1
        assert gl == ol, f"row {t}: len {gl} != oracle {ol}"
        if exact:
            np.testing.assert_array_equal(gi, oi, err_msg=f"row {t} indices")
            if gs is not None:
                np.testing.assert_array_equal(gs, osc.astype(np.float32), err_msg=f"row {t} scores")
            continue
        assert (gi[gl:] == -1).all(), f"row {t}: padding"
        if gs is not None:
            assert np.all(np.isneginf(gs[gl:])), f"row {t}: padding scores"
        s_all = ref["all_scores"][r]
        tol = tolerance(rel, ref["all_mags"][r], ref["all_scales"][r], head_dim, n_heads)
        M = ref["all_mags"][r]
        if pool > 1:
            # pool tokens: P consecutive tokens per pool, pooled score; then the tail
            n_tail = int(np.sum(np.isposinf(osc[:ol])))
            n_pool_tok = ol - n_tail
            np.testing.assert_array_equal(gi[n_pool_tok:gl], oi[n_pool_tok:ol], err_msg=f"row {t} tail")
            if gs is not None:
                assert np.all(np.isposinf(gs[n_pool_tok:gl])), f"row {t} tail scores"
            gp = gi[:n_pool_tok].reshape(-1, pool)
            assert (gp[:, 0] % pool == 0).all() and (np.diff(gp, axis=1) == 1).all(), f"row {t} expansion"
            g_keys = gp[:, 0] // pool
            o_keys = oi[:n_pool_tok].reshape(-1, pool)[:, 0] // pool
            g_scores = gs[:n_pool_tok].reshape(-1, pool)[:, 0] if gs is not None else None
        else:
            g_keys, o_keys = gi[:gl], oi[:ol]
            g_scores = gs[:gl] if gs is not None else None
        assert len(set(g_keys.tolist())) == len(g_keys), f"row {t}: duplicate keys"
        assert (np.diff(g_keys) > 0).all(), f"row {t}: not ascending"
        if g_scores is not None and len(g_keys):
            err = np.abs(g_scores.astype(np.float64) - s_all[g_keys])
            bad = err > tol[g_keys] + 1e-300
            assert not bad.any(), (f"row {t}: score error {err[bad][:4]} above tolerance {tol[g_keys][bad][:4]} "
                                   f"(M {M[g_keys][bad][:4]}) at keys {g_keys[bad][:4]}")
            st["max_err_over_tol"] = max(st["max_err_over_tol"], float(np.max(err / (tol[g_keys] + 1e-300))))
            st["max_err_over_M"] = max(st["max_err_over_M"], float(np.max(err / (M[g_keys] + 1e-300))))
        if len(o_keys) < len(s_all) and len(o_keys):
            kth = int(o_keys[np.argmin(s_all[o_keys])])
            band = np.abs(s_all - s_all[kth]) <= tol + tol[kth]
            st["band_frac"] += float(np.mean(band))
            st["band_rows"] += 1
        gset, oset = set(g_keys.tolist()), set(o_keys.tolist())
        if gset != oset:
            kth = int(o_keys[np.argmin(s_all[o_keys])])
            for i in gset ^ oset:
                lim = tol[i] + tol[kth]
                assert abs(s_all[i] - s_all[kth]) <= lim, (
                    f"row {t}: key {i} (score {s_all[i]}) swapped with the boundary score "
                    f"{s_all[kth]} beyond tolerance {lim}")
            n_sw = len(gset - oset)
            allowed = max(1, math.ceil(swap_frac * len(o_keys)))
            assert n_sw <= allowed, f"row {t}: {n_sw} swapped keys, more than {allowed}"
            st["rows_with_swaps"] += 1
            st["swaps"] += n_sw
            st["max_swaps_row"] = max(st["max_swaps_row"], n_sw)
    st["band_frac"] = st["band_frac"] / st["band_rows"] if st["band_rows"] else 0.0
    return st


def topk_overlap(idx_a, len_a, idx_b, len_b, rows=None):
    """Per-row overlap |A & B| / max(|A|, |B|) of two top-k index sets (rows
    with nothing selected count as 1)."""
    T = idx_a.shape[0]
    rows = np.arange(T) if rows is None else rows
    out = np.ones(len(rows))
    for r, t in enumerate(rows):
        na, nb = int(len_a[t]), int(len_b[t])
        if max(na, nb) == 0:
            continue
        a = np.asarray(idx_a[t, :na])
        b = np.asarray(idx_b[t, :nb])
        out[r] = len(np.intersect1d(a, b, assume_unique=True)) / max(na, nb)
    return out
