"""GPU-vs-oracle comparison rules for the fused score + top-k.

Scores: every entry the GPU returns must be within rel * A of the oracle's
score of that same key, where A = |sm_scale| * sum_j |w_j| * sum_d |q_jd k_d|
is the magnitude the rounding errors of I scale with (the head-weighted ReLU
sum cancels, so |I| itself is no yardstick).  rel = 2e-3 for BF16 scoring and
1.5e-2 for MXFP8 (the oracle applies the same E4M3/UE8M0 quantisation).

Index sets: equal, except keys the GPU took instead of oracle keys when both
oracle scores are within rel * (A_i + A_kth) of the oracle's k-th score (a
swap at the selection boundary).  Integer-valued inputs: bit-exact.
"""
from __future__ import annotations

import numpy as np

REL_BF16 = 2e-3
REL_MXFP8 = 1.5e-2


def compare_topk(g_idx, g_sc, g_len, ref, rel: float, exact: bool = False, pool: int = 1,
                 tail: bool = True, rows=None):
    """Assert parity of GPU rows against an oracle result dict (with_scale=True).
    Returns the number of rows with tolerated boundary swaps."""
    rows = ref["rows"] if rows is None else rows
    swaps = 0
    for r, t in enumerate(rows):
        gi, gs, gl = g_idx[t], g_sc[t] if g_sc is not None else None, int(g_len[t])
        oi, osc, ol = ref["idx"][r], ref["score"][r], int(ref["len"][r])
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
        A = ref["all_scales"][r]
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
        if g_scores is not None:
            err = np.abs(g_scores.astype(np.float64) - s_all[g_keys])
            bad = err > rel * A[g_keys] + 1e-30
            assert not bad.any(), (f"row {t}: score error {err[bad][:4]} vs A {A[g_keys][bad][:4]} "
                                   f"at keys {g_keys[bad][:4]}")
        gset, oset = set(g_keys.tolist()), set(o_keys.tolist())
        if gset != oset:
            kth = int(o_keys[np.argmin(s_all[o_keys])]) if len(o_keys) else 0
            for i in gset ^ oset:
                tol = rel * (A[i] + A[kth]) + 1e-30
                assert abs(s_all[i] - s_all[kth]) <= tol, (
                    f"row {t}: key {i} (score {s_all[i]}) swapped with the boundary score "
                    f"{s_all[kth]} beyond tolerance {tol}")
            swaps += 1
    return swaps
