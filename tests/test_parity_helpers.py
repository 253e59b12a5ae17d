"""CPU checks of the parity rules themselves (oracle against perturbed copies of
its own results), so the GPU parity tests run well-exercised comparison code."""
import numpy as np
import pytest

from speculative_decoding_verification_56_gb300 import synth
import parity_helpers as ph


def _as_gpu(r):
    return dict(accepted_len=r["accepted_len"].copy(), out_tokens=r["out_tokens"].copy(),
                p=r["p"].astype(np.float32), q=r["q"].astype(np.float32),
                resid_mass=r["resid_mass"].astype(np.float32))


@pytest.fixture(scope="module")
def res(oracle_mod):
    c = synth.peaked(seed=3)
    r = oracle_mod.verify_sample(c.target, c.draft, c.tokens, c.u_accept, c.u_sample,
                                 c.temperature, dtype=c.dtype)
    return c, r, _as_gpu(r)


def test_identical_passes(res):
    c, r, gpu = res
    s = ph.compare_sample(gpu, r, case=c)
    assert s["rows"] == c.B and s["flagged"] == 0 and s["differing"] == 0


def test_token_mismatch_detected(res):
    c, r, gpu = res
    g = {k: v.copy() for k, v in gpu.items()}
    g["out_tokens"][2, g["accepted_len"][2]] += 1
    with pytest.raises(AssertionError, match="out_tokens"):
        ph.compare_sample(g, r, case=c)


def test_probability_drift_detected(res):
    c, r, gpu = res
    g = {k: v.copy() for k, v in gpu.items()}
    g["p"][1, 1] *= 1.0 + 5e-5
    with pytest.raises(AssertionError, match="p out of tolerance"):
        ph.compare_sample(g, r, case=c)


def test_flagged_row_must_hold_a_valid_outcome(res):
    # a flagged row may differ, but only to an outcome the exact law reaches
    # within the window; a token far from u*R is not one
    c, r, gpu = res
    r2 = {k: v.copy() for k, v in r.items()}
    r2["cdf_margin"][4] = 1e-9
    g = {k: v.copy() for k, v in gpu.items()}
    n4 = g["accepted_len"][4]
    g["out_tokens"][4, n4] = (g["out_tokens"][4, n4] + c.V // 2) % c.V
    with pytest.raises(AssertionError, match="outside the window"):
        ph.compare_sample(g, r2, allow_flags=1, case=c)
    with pytest.raises(AssertionError, match="no inputs"):
        ph.compare_sample(g, r2, allow_flags=1)


def test_flag_count_bound(res):
    c, r, gpu = res
    r2 = {k: v.copy() for k, v in r.items()}
    r2["cdf_margin"][:] = 1e-9          # every row flagged: far above the expectation
    with pytest.raises(AssertionError, match="flagged rows"):
        ph.compare_sample(gpu, r2, case=c)
    assert ph.flag_allowance(0.0) == 1 and ph.flag_allowance(4.0) == 13


def _boundary_case(oracle_mod):
    """A bonus draw whose u*R sits on a CDF boundary to float32 precision:
    the boundary is computed here from the softmax of the row (numpy,
    float64), independently of the oracle's inverse CDF."""
    V, B = 40, 3
    rng = np.random.default_rng(8)
    zt = rng.standard_normal((B, 1, V)).astype(np.float32)
    p = np.exp(zt[:, 0].astype(np.float64) - zt[:, 0].max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    C = np.cumsum(p, axis=1)
    j = np.array([10, 20, 30])
    us = np.array([np.float32(C[b, j[b]]) for b in range(B)], np.float32)
    c = synth.ChainInputs("boundary", B, 0, V, "f32", 1.0, zt, np.zeros((B, 0, V), np.float32),
                          np.zeros((B, 0), np.int32), np.zeros((B, 0), np.float32), us)
    return c, j


def test_claim_on_a_boundary_accepts_both_neighbours(oracle_mod):
    c, j = _boundary_case(oracle_mod)
    r = oracle_mod.verify_sample(c.target, c.draft, c.tokens, c.u_accept, c.u_sample, 1.0)
    assert (r["cdf_margin"] < 1e-7).all()
    zeros = np.zeros(c.B, np.int32)
    for cand in (j, j + 1):          # the tokens on either side of the boundary
        viol, R = oracle_mod.sample_claim(c.target, c.draft, c.tokens, c.u_accept, c.u_sample,
                                          1.0, zeros, cand)
        assert (viol < 1e-7).all() and (R == 0).all()
    far, _ = oracle_mod.sample_claim(c.target, c.draft, c.tokens, c.u_accept, c.u_sample, 1.0,
                                     zeros, j + 3)
    assert (far > 1e-3).all()
    # the comparison accepts the neighbour that is not the oracle's choice
    other = np.where(r["out_tokens"][:, 0] == j, j + 1, j)
    g = _as_gpu(r)
    g["out_tokens"][:, 0] = other
    s = ph.compare_sample(g, r, allow_flags=c.B, case=c)   # flagged on purpose
    assert s["differing"] == c.B and s["max_violation"] < 1e-7


def test_compare_exact_subset(oracle_mod):
    t = synth.tree(seed=1, B=3, N=20, V=300)
    r = oracle_mod.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth)
    big = {k: np.concatenate([v, v]) for k, v in r.items()}
    ph.compare_exact(big, r, ["accepted_len", "path_nodes", "out_tokens"], rows=slice(0, 3))
    big["path_nodes"][1, 0] = 7
    with pytest.raises(AssertionError):
        ph.compare_exact(big, r, ["path_nodes"], rows=slice(0, 3))
