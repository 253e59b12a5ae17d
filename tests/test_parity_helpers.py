"""CPU checks of the parity rules themselves (oracle against perturbed copies of
its own results), so the GPU parity tests run well-exercised comparison code."""
import numpy as np
import pytest

from speculative_decoding_verification_56_gb300 import synth
import parity_helpers as ph


@pytest.fixture(scope="module")
def res(oracle_mod):
    c = synth.peaked(seed=3)
    r = oracle_mod.verify_sample(c.target, c.draft, c.tokens, c.u_accept, c.u_sample,
                                 c.temperature, dtype=c.dtype)
    gpu = dict(accepted_len=r["accepted_len"].copy(), out_tokens=r["out_tokens"].copy(),
               p=r["p"].astype(np.float32), q=r["q"].astype(np.float32),
               resid_mass=r["resid_mass"].astype(np.float32))
    return c, r, gpu


def test_identical_passes(res):
    c, r, gpu = res
    s = ph.compare_sample(gpu, r)
    assert s["rows"] == c.B and s["flagged"] == 0


def test_token_mismatch_detected(res):
    _, r, gpu = res
    g = {k: v.copy() for k, v in gpu.items()}
    g["out_tokens"][2, 0] += 1
    with pytest.raises(AssertionError, match="out_tokens"):
        ph.compare_sample(g, r)


def test_probability_drift_detected(res):
    _, r, gpu = res
    g = {k: v.copy() for k, v in gpu.items()}
    g["p"][1, 1] *= 1.0 + 5e-5
    with pytest.raises(AssertionError, match="p out of tolerance"):
        ph.compare_sample(g, r)


def test_flagged_rows_are_excused_but_counted(res):
    _, r, gpu = res
    r2 = {k: v.copy() for k, v in r.items()}
    r2["cdf_margin"][4] = 1e-9
    g = {k: v.copy() for k, v in gpu.items()}
    g["out_tokens"][4, 0] += 1
    s = ph.compare_sample(g, r2, allow_flags=1)
    assert s["flagged"] == 1
    with pytest.raises(AssertionError, match="flagged"):
        ph.compare_sample(g, r2)


def test_compare_exact_subset(oracle_mod):
    t = synth.tree(seed=1, B=3, N=20, V=300)
    r = oracle_mod.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth)
    big = {k: np.concatenate([v, v]) for k, v in r.items()}
    ph.compare_exact(big, r, ["accepted_len", "path_nodes", "out_tokens"], rows=slice(0, 3))
    big["path_nodes"][1, 0] = 7
    with pytest.raises(AssertionError):
        ph.compare_exact(big, r, ["path_nodes"], rows=slice(0, 3))
