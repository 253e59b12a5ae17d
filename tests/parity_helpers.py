"""Comparison rules between the CUDA path and the float64 oracle.

Tolerances (the method's outputs are decisions plus a few probabilities):

* accepted lengths and emitted tokens: bit-exact for greedy and tree modes.
* sampling: a row must match the oracle exactly unless the oracle flags it
  (a uniform within FLAG_WINDOW = 1e-6 of an acceptance threshold p/q, or
  u*R within 1e-6*R of the CDF value at the chosen token or the one before
  it).  A flagged row may differ, but only to another outcome that the exact
  law reaches within the window: the oracle measures the GPU's claim
  (accepted length, drawn token) with ``oracle.sample_claim`` and its
  violation must stay below FLAG_WINDOW.  The tokens before the accepted
  length must still be the drafts and the ones after it -1.
* how many rows are flagged depends on the inputs only.  The oracle reports,
  per row, the chance ``flag_prob`` that fresh uniforms land in a window
  (the acceptance windows of the decided positions plus the CDF boundaries
  of the drawn distribution).  The count must stay within a Poisson bound of
  its expectation mu = sum(flag_prob): floor(mu + 4 sqrt(mu) + 1).  With
  V >= 50 a window of 1e-6 around each of V CDF boundaries already exceeds
  1e-4 of the uniform's range, so a fixed rate of 1e-4 flagged rows is below
  what the exact law itself produces; on the V=128256 Zipf workload mu is
  about 2.7% of rows.
* p(x_i), q(x_i): within 1e-5 relative of the oracle's float64 value (plus
  1e-37 absolute, below which float32 outputs lose relative precision).
* residual mass R: within 1e-5 relative or 1e-7 absolute, whichever is
  looser (fp32 p - q cancellation bounds R's absolute error near 1e-7), of
  the R of the row the GPU drew from.
"""
from __future__ import annotations

import numpy as np

import oracle

FLAG_WINDOW = oracle.FLAG_WINDOW
PQ_RTOL = 1e-5
PQ_ATOL = 1e-37
R_RTOL = 1e-5
R_ATOL = 1e-7


def flag_allowance(mu: float) -> int:
    """Largest flagged-row count accepted when mu flags are expected."""
    return int(np.floor(mu + 4.0 * np.sqrt(mu) + 1.0))


def flagged_rows(orc: dict, window: float = FLAG_WINDOW) -> np.ndarray:
    return (orc["acc_margin"] < window) | (orc["cdf_margin"] < window)


def _check_structure(n, tok, drafts, rows_idx):
    """Tokens before the accepted length are the drafts, the ones after it -1."""
    for i in rows_idx:
        k = drafts.shape[1]
        assert 0 <= n[i] <= k, f"row {i}: accepted length {n[i]} outside [0, {k}]"
        assert (tok[i, :n[i]] == drafts[i, :n[i]]).all(), f"row {i}: accepted tokens differ"
        assert (tok[i, n[i] + 1:] == -1).all(), f"row {i}: slots after the draw are not -1"


def compare_sample(gpu: dict, orc: dict, rows=None, allow_flags=None, case=None,
                   window=FLAG_WINDOW, pq_rtol=PQ_RTOL):
    """Assert sampling parity.  ``gpu`` holds numpy copies of the CUDA outputs
    (accepted_len, out_tokens, p, q, resid_mass); ``orc`` the oracle's result
    for the same rows (computed with the same flag ``window``); ``case`` the
    inputs (needed to validate rows that differ).  ``rows`` selects which GPU
    rows ``orc`` covers.  Returns a summary dict."""
    sel = slice(None) if rows is None else rows
    g_n = np.asarray(gpu["accepted_len"])[sel]
    g_tok = np.asarray(gpu["out_tokens"])[sel]
    g_p = np.asarray(gpu["p"], dtype=np.float64)[sel]
    g_q = np.asarray(gpu["q"], dtype=np.float64)[sel]
    g_R = np.asarray(gpu["resid_mass"], dtype=np.float64)[sel]
    n_rows = g_n.shape[0]
    flags = flagged_rows(orc, window)
    nflag = int(flags.sum())
    mu = float(np.sum(orc["flag_prob"]))
    if allow_flags is None:
        allow_flags = flag_allowance(mu)
    assert nflag <= allow_flags, f"{nflag} flagged rows of {n_rows} (expected {mu:.2f})"

    # p and q on every row and position
    for name, gv, ov in (("p", g_p, orc["p"]), ("q", g_q, orc["q"])):
        err = np.abs(gv - ov)
        lim = pq_rtol * np.abs(ov) + PQ_ATOL
        worst = np.unravel_index(np.argmax(err - lim), err.shape) if err.size else None
        assert (err <= lim).all(), f"{name} out of tolerance at {worst}: gpu {gv[worst]} " \
            f"oracle {ov[worst]}"

    differ = (g_n != orc["accepted_len"]) | (g_tok != orc["out_tokens"]).any(axis=1)
    bad_n = np.nonzero(~flags & (g_n != orc["accepted_len"]))[0]
    assert bad_n.size == 0, f"accepted_len differs on unflagged rows {bad_n[:10]}: " \
        f"gpu {g_n[bad_n[:10]]} oracle {orc['accepted_len'][bad_n[:10]]}"
    bad_t = np.nonzero(~flags & differ)[0]
    assert bad_t.size == 0, f"out_tokens differ on unflagged rows {bad_t[:10]}: " \
        f"gpu {g_tok[bad_t[:3]]} oracle {orc['out_tokens'][bad_t[:3]]}"

    # rows that differ (all flagged): the GPU's outcome must be one the exact
    # law reaches within the window, with that outcome's residual mass
    ref_R = np.asarray(orc["resid_mass"], dtype=np.float64).copy()
    idx = np.nonzero(differ)[0]
    max_violation = 0.0
    if idx.size:
        assert case is not None, "rows differ and no inputs were given to validate them"
        case_rows = np.arange(case.B)[sel][idx]
        drafts = np.asarray(case.tokens)[case_rows]
        _check_structure(g_n[idx], g_tok[idx], drafts, range(idx.size))
        viol, claim_R = oracle.sample_claim(
            case.target[case_rows], None if case.draft is None else case.draft[case_rows],
            drafts, case.u_accept[case_rows], case.u_sample[case_rows], case.temperature,
            g_n[idx], g_tok[idx, g_n[idx]], dtype=case.dtype)
        max_violation = float(viol.max())
        assert (viol < window).all(), \
            f"rows {idx[viol >= window]} hold outcomes outside the window: " \
            f"violations {viol[viol >= window]}"
        ref_R[idx] = claim_R
    errR = np.abs(g_R - ref_R)
    limR = np.maximum(max(R_RTOL, pq_rtol) * np.abs(ref_R), R_ATOL)
    badR = np.nonzero(errR > limR)[0]
    assert badR.size == 0, f"resid_mass out of tolerance rows {badR[:10]}: " \
        f"gpu {g_R[badR[:5]]} oracle {ref_R[badR[:5]]}"
    relp = np.abs(g_p - orc["p"]) / np.maximum(np.abs(orc["p"]), 1e-300)
    return dict(rows=n_rows, flagged=nflag, expected_flags=mu, flag_allowance=allow_flags,
                differing=int(idx.size), max_violation=max_violation,
                max_rel_p=float(relp.max()) if relp.size else 0.0,
                mean_accepted=float(g_n.mean()) if n_rows else 0.0)


def compare_exact(gpu: dict, orc: dict, keys, rows=None):
    sel = slice(None) if rows is None else rows
    for k in keys:
        g = np.asarray(gpu[k])[sel]
        o = np.asarray(orc[k])
        bad = np.nonzero((g != o).reshape(g.shape[0], -1).any(axis=1))[0]
        assert bad.size == 0, f"{k} differs at rows {bad[:10]}: gpu {g[bad[:3]]} " \
            f"oracle {o[bad[:3]]}"
