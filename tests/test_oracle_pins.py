"""Pins of the float64 oracle against facts that do not come from the oracle.

* the worked example printed on the "EAGLE math" page (golden fixture);
* exact enumeration of the first emitted token's law, obtained from the
  oracle's own decisions by bisection over float32 uniforms, against
  softmax(target/T) ("EAGLE-3 speculative decoding review", section "Does Using
  a Small Model's Answer Reduce Quality?": accepted mass min(p,q) plus the
  normalised residual recovers p);
* chi-square goodness of fit of emitted tokens against p at every reached
  position (review page, "Interpreting 'No Quality Loss' Precisely":
  sampling keeps the target distribution);
* the expected-tokens law E = (1 - alpha^(gamma+1)) / (1 - alpha) ("EAGLE
  math", "Vanilla speculative decoding") by Monte Carlo;
* greedy verification equals target-only argmax decoding (review page,
  greedy bullets);
* brute-force top-down search of tiny draft trees; the chain tree reduces to
  greedy verification; the star tree to "any child equal to the root argmax".
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

from speculative_decoding_verification_56_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

F32_ONE_BITS = int(np.float32(1.0).view(np.uint32))


def f32_from_bits(b):
    return float(np.uint32(b).view(np.float32))


def smallest_u_where(pred):
    """Smallest float32 u in [0, 1) with pred(u) True (pred monotone False->True);
    returns 1.0 when pred is False on all of [0, 1)."""
    lo, hi = 0, F32_ONE_BITS  # invariant: pred false below lo, answer in [lo, hi]
    if pred(0.0):
        return 0.0
    lo = 1
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(f32_from_bits(mid)):
            hi = mid
        else:
            lo = mid + 1
    return f32_from_bits(lo)  # == 1.0 when never true


# ---------------------------------------------------------------------------
# worked example printed on the page
# ---------------------------------------------------------------------------

def test_worked_example_expected_tokens_and_speedup(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "eagle_math_worked_example.json")))
    half = 0.5 * 10 ** (-g["printed_decimals"])
    for case in g["cases"]:
        e = oracle_mod.expected_tokens(case["alpha"], g["gamma"])
        s = oracle_mod.speedup_model(case["alpha"], g["gamma"], g["c"])
        assert abs(e - case["E"]) <= half + 1e-12, (case, e)
        assert abs(s - case["speedup"]) <= half + 1e-12, (case, s)


@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.7, 0.95, 1.0])
@pytest.mark.parametrize("gamma", [0, 1, 4, 7])
def test_expected_tokens_closed_form(oracle_mod, alpha, gamma):
    closed = gamma + 1.0 if alpha == 1.0 else (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert oracle_mod.expected_tokens(alpha, gamma) == pytest.approx(closed, rel=1e-13)


# ---------------------------------------------------------------------------
# exact enumeration of the emitted-token law
# ---------------------------------------------------------------------------

def _call(oracle_mod, zt, zd, T, toks, ua, us):
    B = 1
    k = zd.shape[0]
    return oracle_mod.verify_sample(zt.reshape(B, k + 1, -1), zd.reshape(B, k, -1),
                                    np.array(toks, np.int32).reshape(B, k),
                                    np.array(ua, np.float32).reshape(B, k),
                                    np.array([us], np.float32), T, dtype="f32")


def _emission_law_at(oracle_mod, zt, zd, T, pos):
    """Law of the token emitted at position ``pos`` given that the first ``pos``
    drafts were accepted, measured from the oracle's decisions."""
    k, V = zd.shape
    q = special.softmax(zd[pos].astype(np.float64) / T)
    base_tok = [0] * k
    base_ua = [0.0] * k            # u = 0 accepts every earlier position (p > 0)
    # P(accept | x) as the measure of the accepting uniforms
    p_acc = np.zeros(V)
    for x in range(V):
        toks = list(base_tok)
        toks[pos] = x

        def rejected(u, toks=toks):
            ua = list(base_ua)
            ua[pos] = u
            return _call(oracle_mod, zt, zd, T, toks, ua, 0.5)["accepted_len"][0] == pos
        p_acc[x] = smallest_u_where(rejected)
    # residual law: reject at pos with the draft whose p/q is smallest
    p = special.softmax(zt[pos].astype(np.float64) / T)
    xr = int(np.argmin(p / q))
    toks = list(base_tok)
    toks[pos] = xr
    ua = list(base_ua)
    ua[pos] = float(np.nextafter(np.float32(1.0), np.float32(0.0)))
    assert _call(oracle_mod, zt, zd, T, toks, ua, 0.5)["accepted_len"][0] == pos
    cdf = np.zeros(V)
    for j in range(V):
        cdf[j] = smallest_u_where(
            lambda u: _call(oracle_mod, zt, zd, T, toks, ua, u)["out_tokens"][0, pos] > j)
    p_res = np.diff(np.concatenate([[0.0], cdf]))
    emit = q * p_acc + (1.0 - np.dot(q, p_acc)) * p_res
    return emit, p


@pytest.mark.parametrize("seed,V,T", [(0, 5, 1.0), (1, 8, 0.7), (2, 16, 1.3), (3, 6, 0.5)])
def test_emission_law_equals_target_first_position(oracle_mod, seed, V, T):
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((2, V)) * 1.5).astype(np.float32)
    zd = (zt[:1] + rng.standard_normal((1, V))).astype(np.float32)
    emit, p = _emission_law_at(oracle_mod, zt, zd, T, 0)
    assert np.abs(emit - p).max() < 2e-6 * V, (emit, p)


@pytest.mark.parametrize("seed", [4, 5])
def test_emission_law_equals_target_later_position(oracle_mod, seed):
    """Position 1 must use target row 1 and draft row 1 (row alignment)."""
    V, T = 7, 0.9
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((3, V)) * 2.0).astype(np.float32)
    zd = (zt[:2] + rng.standard_normal((2, V)) * 0.8).astype(np.float32)
    emit, p = _emission_law_at(oracle_mod, zt, zd, T, 1)
    assert np.abs(emit - p).max() < 2e-6 * V
    # and it is not the law of any other row
    for other in (0, 2):
        po = special.softmax(zt[other].astype(np.float64) / T)
        assert np.abs(emit - po).max() > 1e-3


@pytest.mark.parametrize("k", [1, 3])
def test_bonus_token_law_is_last_target_row(oracle_mod, k):
    V, T = 9, 1.1
    rng = np.random.default_rng(10 + k)
    zt = (rng.standard_normal((k + 1, V)) * 2.0).astype(np.float32)
    zd = (zt[:k] + rng.standard_normal((k, V))).astype(np.float32)
    toks, ua = [0] * k, [0.0] * k
    assert _call(oracle_mod, zt, zd, T, toks, ua, 0.5)["accepted_len"][0] == k
    cdf = np.array([smallest_u_where(
        lambda u: _call(oracle_mod, zt, zd, T, toks, ua, u)["out_tokens"][0, k] > j)
        for j in range(V)])
    law = np.diff(np.concatenate([[0.0], cdf]))
    p = special.softmax(zt[k].astype(np.float64) / T)
    assert np.abs(law - p).max() < 2e-6 * V


# ---------------------------------------------------------------------------
# chi-square over many seeded trials
# ---------------------------------------------------------------------------

def _trials(B, zt_row, zd_row, rng):
    zt = np.broadcast_to(zt_row, (B,) + zt_row.shape).copy()
    zd = np.broadcast_to(zd_row, (B,) + zd_row.shape).copy()
    return zt, zd


def _chisq_pvalue(samples, probs):
    V = probs.size
    obs = np.bincount(samples, minlength=V).astype(np.float64)
    exp = probs * samples.size
    keep = exp > 5
    obs_k = np.append(obs[keep], obs[~keep].sum())
    exp_k = np.append(exp[keep], exp[~keep].sum())
    if exp_k[-1] == 0:
        obs_k, exp_k = obs_k[:-1], exp_k[:-1]
    return stats.chisquare(obs_k, exp_k).pvalue


@pytest.mark.parametrize("seed,T,dtype", [(0, 1.0, "f32"), (1, 0.8, "bf16")])
def test_chisquare_every_position(oracle_mod, seed, T, dtype):
    B, k, V = 200_000, 3, 8
    rng = np.random.default_rng(seed)
    zt_row = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    zd_row = (zt_row[:k] + rng.standard_normal((k, V)) * 0.9).astype(np.float32)
    if dtype == "bf16":
        zt_row = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(zt_row))
        zd_row = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(zd_row))
    zt, zd = _trials(B, zt_row, zd_row, rng)
    qs = [special.softmax(zd_row[i].astype(np.float64) / T) for i in range(k)]
    toks = np.stack([rng.choice(V, size=B, p=qs[i]) for i in range(k)], axis=1).astype(np.int32)
    ua = synth.uniforms_f32(rng, (B, k))
    us = synth.uniforms_f32(rng, (B,))
    if dtype == "bf16":
        zt_s, zd_s = synth.f32_to_bf16_bits(zt), synth.f32_to_bf16_bits(zd)
    else:
        zt_s, zd_s = zt, zd
    res = oracle_mod.verify_sample(zt_s, zd_s, toks, ua, us, T, dtype=dtype)
    n = res["accepted_len"]
    for j in range(k + 1):
        reached = n >= j
        emitted = res["out_tokens"][reached, j]
        p = special.softmax(zt_row[j].astype(np.float64) / T)
        pv = _chisq_pvalue(emitted, p)
        assert pv > 1e-3, (j, pv)
    # a wrong law is detected by the same statistic
    p_wrong = special.softmax(zd_row[0].astype(np.float64) / T)
    assert _chisq_pvalue(res["out_tokens"][:, 0], p_wrong) < 1e-6


def test_chisquare_k0_is_plain_sampling(oracle_mod):
    B, V, T = 100_000, 10, 1.0
    rng = np.random.default_rng(7)
    row = (rng.standard_normal((1, V)) * 2).astype(np.float32)
    zt = np.broadcast_to(row, (B, 1, V)).copy()
    res = oracle_mod.verify_sample(zt, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                                   np.zeros((B, 0), np.float32), synth.uniforms_f32(rng, (B,)), T)
    assert (res["accepted_len"] == 0).all()
    assert _chisq_pvalue(res["out_tokens"][:, 0], special.softmax(row[0].astype(np.float64))) > 1e-3


# ---------------------------------------------------------------------------
# expected tokens per pass
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("alpha_target", [0.7, 0.8, 0.9])
def test_expected_tokens_monte_carlo(oracle_mod, alpha_target):
    B, k = 200_000, 4
    a = 0.35
    b = a + (1.0 - alpha_target)           # |a - b| = 1 - alpha
    zt_row = np.array([0.0, np.log((1 - a) / a)], np.float32)
    zd_row = np.array([0.0, np.log((1 - b) / b)], np.float32)
    p = special.softmax(zt_row.astype(np.float64))
    q = special.softmax(zd_row.astype(np.float64))
    alpha = np.minimum(p, q).sum()          # exact per-row acceptance of these logits
    assert abs(alpha - alpha_target) < 1e-6
    rng = np.random.default_rng(int(alpha_target * 100))
    zt = np.broadcast_to(zt_row, (B, k + 1, 2)).copy()
    zd = np.broadcast_to(zd_row, (B, k, 2)).copy()
    toks = (rng.random((B, k)) >= q[0]).astype(np.int32)
    res = oracle_mod.verify_sample(zt, zd, toks, synth.uniforms_f32(rng, (B, k)),
                                   synth.uniforms_f32(rng, (B,)), 1.0)
    emitted = res["accepted_len"].astype(np.float64) + 1.0
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    se = emitted.std() / np.sqrt(B)
    assert abs(emitted.mean() - E) < 5 * se, (emitted.mean(), E, se)
    # per-position acceptance is alpha: P(n >= i) = alpha^i
    for i in range(1, k + 1):
        frac = (res["accepted_len"] >= i).mean()
        assert abs(frac - alpha ** i) < 5 * np.sqrt(alpha ** i * (1 - alpha ** i) / B)


# ---------------------------------------------------------------------------
# boundary cases of the acceptance rule
# ---------------------------------------------------------------------------

def test_identical_rows_accept_everything(oracle_mod):
    c = synth.make_chain_case(B=20, k=4, V=50, seed=3)
    ua = np.full((20, 4), np.nextafter(np.float32(1), np.float32(0)), np.float32)
    res = oracle_mod.verify_sample(c.target, c.target[:, :4], c.tokens, ua, c.u_sample, 1.0)
    assert (res["accepted_len"] == 4).all()
    assert (res["resid_mass"] == 0).all()
    assert np.allclose(res["p"], res["q"])


def test_zero_probability_cases(oracle_mod):
    V = 6
    zt = np.zeros((1, 3, V), np.float32)
    zd = np.zeros((1, 2, V), np.float32)
    zt[0, 0, 2] = -5000.0     # p(2) underflows to 0 at position 0
    zd[0, 1, 4] = -5000.0     # q(4) underflows to 0 at position 1
    # position 0: p = 0 rejects even with u = 0 (0 * q < 0 is false)
    r = oracle_mod.verify_sample(zt, zd, np.array([[2, 4]]), np.array([[0.0, 0.5]], np.float32),
                                 np.array([0.3], np.float32), 1.0)
    assert r["accepted_len"][0] == 0 and r["p"][0, 0] == 0.0
    assert r["out_tokens"][0, 0] != 2 and r["out_tokens"][0, 1] == -1
    # position 1: q = 0 accepts for any u (p > 0)
    r = oracle_mod.verify_sample(zt, zd, np.array([[0, 4]]),
                                 np.array([[0.0, np.nextafter(np.float32(1), np.float32(0))]],
                                          np.float32), np.array([0.3], np.float32), 1.0)
    assert r["accepted_len"][0] == 2 and r["q"][0, 1] == 0.0


def test_p_q_reported_for_every_row(oracle_mod):
    # uniform rows: p(x) = q(x) = 1/V exactly.  The draft favours token 1 at
    # position 0 (q > p there), so u just below 1 rejects position 0; the rows
    # after the rejection still report their p and q
    V, k = 8, 4
    zt = np.zeros((1, k + 1, V), np.float32)
    zd = np.zeros((1, k, V), np.float32)
    zd[0, 0, 1] = 3.0
    ua = np.full((1, k), np.nextafter(np.float32(1), np.float32(0)), np.float32)
    r = oracle_mod.verify_sample(zt, zd, np.array([[1, 2, 3, 4]]), ua, np.array([0.5], np.float32),
                                 1.0)
    assert r["accepted_len"][0] == 0
    assert r["p"][0, 0] == 1.0 / V and r["q"][0, 0] > 1.0 / V
    assert (r["p"][0, 1:] == 1.0 / V).all() and (r["q"][0, 1:] == 1.0 / V).all()


def test_residual_zero_falls_back_to_target_row(oracle_mod):
    V = 5
    zt = np.zeros((1, 2, V), np.float32)
    zt[0, 0] = [0.0, 1.0, -5000.0, 0.5, 0.2]
    zd = zt[:, :1].copy()                      # identical rows, token has p = q = 0
    us = np.array([0.8], np.float32)
    r = oracle_mod.verify_sample(zt, zd, np.array([[2]]), np.array([[0.0]], np.float32), us, 1.0)
    assert r["accepted_len"][0] == 0 and r["fallback"][0] == 1 and r["resid_mass"][0] == 0
    p = special.softmax(zt[0, 0].astype(np.float64))
    expect = int(np.searchsorted(np.cumsum(p), 0.8 * p.sum(), side="right"))
    assert r["out_tokens"][0, 0] == expect


def test_invalid_inputs_raise(oracle_mod):
    c = synth.make_chain_case(B=2, k=2, V=10, seed=1)
    bad = c.tokens.copy()
    bad[1, 1] = 10
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.verify_sample(c.target, c.draft, bad, c.u_accept, c.u_sample, 1.0)
    t = c.target.copy()
    t[0, 0, 3] = np.inf
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.verify_sample(t, c.draft, c.tokens, c.u_accept, c.u_sample, 1.0)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.verify_greedy(t, c.tokens)


# ---------------------------------------------------------------------------
# greedy == target-only argmax decoding
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k", [0, 1, 5])
def test_greedy_equals_argmax_decoding(oracle_mod, dtype, k):
    B, V = 300, 23
    rng = np.random.default_rng(k)
    # small integer logits: many ties, lowest index must win
    zt = rng.integers(-3, 4, size=(B, k + 1, V)).astype(np.float32)
    g = np.argmax(zt, axis=-1)                         # library argmax: first maximum
    toks = np.where(rng.random((B, k)) < 0.75, g[:, :k],
                    rng.integers(0, V, size=(B, k))).astype(np.int32)
    stored = synth.f32_to_bf16_bits(zt) if dtype == "bf16" else zt
    res = oracle_mod.verify_greedy(stored, toks, dtype=dtype)
    for b in range(B):
        n = 0
        while n < k and toks[b, n] == g[b, n]:
            n += 1
        assert res["accepted_len"][b] == n
        expect = list(g[b, :n + 1]) + [-1] * (k - n)
        assert list(res["out_tokens"][b]) == expect
    assert (res["argmax"] == g).all()


# ---------------------------------------------------------------------------
# draft trees: brute-force top-down search
# ---------------------------------------------------------------------------

def _tree_bruteforce(rows, tok, par):
    """Follow target greedy decoding down the tree from the root, exploring
    every child whose token equals the current row's argmax."""
    N = len(par)
    children = [[] for _ in range(N)]
    for v in range(1, N):
        children[par[v]].append(v)
    best = (0, 0)           # (depth, node)
    stack = [(0, 0)]
    while stack:
        v, d = stack.pop()
        if d > best[0] or (d == best[0] and v < best[1]):
            best = (d, v)
        g = int(np.argmax(rows[v]))
        for c in children[v]:
            if tok[c] == g:
                stack.append((c, d + 1))
    d, v = best
    path = [v]
    while path[-1] != 0:
        path.append(par[path[-1]])
    path = path[::-1]
    return d, path, [tok[x] for x in path[1:]] + [int(np.argmax(rows[v]))]


@pytest.mark.parametrize("seed", range(6))
def test_tree_bruteforce(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    B, V, max_depth = 40, 6, 5
    N = int(rng.integers(1, 13))
    zt = rng.integers(-2, 3, size=(B, N, V)).astype(np.float32)
    par = np.stack([synth.make_tree_parents(rng, N, max_depth, 3) for _ in range(B)])
    g = np.argmax(zt, axis=-1)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for v in range(1, N):
            if rng.random() < 0.7:
                tok[b, v] = g[b, par[b, v]]
    res = oracle_mod.verify_tree_greedy(zt, tok, par, max_depth, dtype="f32")
    W = max_depth + 1
    for b in range(B):
        d, path, toks = _tree_bruteforce(zt[b], tok[b], par[b])
        assert res["accepted_len"][b] == d
        assert list(res["path_nodes"][b]) == path + [-1] * (W - len(path))
        assert list(res["out_tokens"][b]) == toks + [-1] * (W - len(toks))


def test_chain_tree_reduces_to_greedy(oracle_mod):
    c = synth.make_chain_case(B=50, k=6, V=30, seed=9, greedy_force=0.8)
    k = c.k
    par = np.tile(np.arange(-1, k, dtype=np.int32), (c.B, 1))     # parent[v] = v - 1
    tok = np.concatenate([np.zeros((c.B, 1), np.int32), c.tokens], axis=1)
    tr = oracle_mod.verify_tree_greedy(c.target, tok, par, k, dtype="f32")
    gr = oracle_mod.verify_greedy(c.target, c.tokens, dtype="f32")
    assert (tr["accepted_len"] == gr["accepted_len"]).all()
    assert (tr["out_tokens"] == gr["out_tokens"]).all()


def test_star_tree(oracle_mod):
    B, N, V = 60, 9, 7
    rng = np.random.default_rng(2)
    zt = rng.standard_normal((B, N, V)).astype(np.float32)
    par = np.zeros((B, N), np.int32)
    par[:, 0] = -1
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    res = oracle_mod.verify_tree_greedy(zt, tok, par, 1, dtype="f32")
    g0 = np.argmax(zt[:, 0], axis=-1)
    for b in range(B):
        hits = [v for v in range(1, N) if tok[b, v] == g0[b]]
        if hits:
            v = hits[0]
            assert res["accepted_len"][b] == 1
            assert list(res["path_nodes"][b]) == [0, v]
            assert list(res["out_tokens"][b]) == [g0[b], int(np.argmax(zt[b, v]))]
        else:
            assert res["accepted_len"][b] == 0
            assert list(res["out_tokens"][b]) == [g0[b], -1]


def test_malformed_trees_raise(oracle_mod):
    zt = np.zeros((1, 4, 5), np.float32)
    tok = np.zeros((1, 4), np.int32)
    for par in ([-1, 0, 2, 1], [-1, 0, 1, 5], [0, 0, 1, 2], [-1, -1, 0, 1]):
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.verify_tree_greedy(zt, tok, np.array([par], np.int32), 5, dtype="f32")
    with pytest.raises(oracle_mod.OracleError):   # depth 3 > max_depth 2
        oracle_mod.verify_tree_greedy(zt, tok, np.array([[-1, 0, 1, 2]], np.int32), 2, dtype="f32")


# ---------------------------------------------------------------------------
# Tree attention mask (review page, "EAGLE-2: Does Every Context Need the Same
# Draft Tree?" and "Must the Feature Be Predicted Exactly?": each node sees
# the shared prefix, its parent and its ancestors, and no other branch)
# ---------------------------------------------------------------------------

def _mask_bool(mask, N):
    """uint32 words [..., W] -> bool [..., N]."""
    bits = np.unpackbits(mask.view(np.uint8), axis=-1, bitorder="little")
    return bits[..., :N].astype(bool)


def _closure(par):
    """Reflexive-transitive closure of the child->parent relation by
    Warshall's algorithm on the adjacency matrix: reach[v, u] iff u is v or
    an ancestor of v."""
    N = len(par)
    reach = np.eye(N, dtype=bool)
    for v in range(1, N):
        reach[v, par[v]] = True
    for m in range(N):
        reach |= reach[:, m:m + 1] & reach[m:m + 1, :]
    return reach


def test_tree_mask_chain_is_causal(oracle_mod):
    # a chain is ordinary decoding: the tree block is the lower-triangular mask
    for N in (1, 2, 31, 32, 33, 70):
        par = np.array([[-1] + list(range(N - 1))], dtype=np.int32)
        mask, depth, bad = oracle_mod.tree_mask(par)
        assert not bad
        assert np.array_equal(_mask_bool(mask[0], N), np.tri(N, dtype=bool))
        assert np.array_equal(depth[0], np.arange(N))


def test_tree_mask_star_sees_root_and_self(oracle_mod):
    N = 40
    par = np.array([[-1] + [0] * (N - 1)], dtype=np.int32)
    mask, depth, bad = oracle_mod.tree_mask(par)
    want = np.eye(N, dtype=bool)
    want[:, 0] = True
    assert not bad
    assert np.array_equal(_mask_bool(mask[0], N), want)
    assert np.array_equal(depth[0], [0] + [1] * (N - 1))


@pytest.mark.parametrize("seed", range(5))
def test_tree_mask_equals_closure(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    B, N = 3, [5, 33, 97][seed % 3]
    par = np.stack([synth.make_tree_parents(rng, N, max_depth=8, max_children=4)
                    for _ in range(B)]).astype(np.int32)
    mask, depth, bad = oracle_mod.tree_mask(par)
    assert not bad
    for b in range(B):
        reach = _closure(par[b])
        got = _mask_bool(mask[b], N)
        assert np.array_equal(got, reach)
        assert np.array_equal(depth[b], reach.sum(1) - 1)  # ancestors + self
        # siblings never see each other
        for u in range(1, N):
            for v in range(u + 1, N):
                if par[b, u] == par[b, v]:
                    assert not got[u, v] and not got[v, u]
        # no bit past N in the last word
        W = mask.shape[-1]
        if N % 32:
            assert not (mask[b, :, W - 1] >> np.uint32(N % 32)).any()


def test_tree_mask_malformed(oracle_mod):
    # node 2 points forward: its chain stops at itself; node 3 below it too
    par = np.array([[-1, 0, 3, 2, 1]], dtype=np.int32)
    mask, depth, bad = oracle_mod.tree_mask(par)
    got = _mask_bool(mask[0], 5)
    assert bad
    assert got[2].nonzero()[0].tolist() == [2] and depth[0, 2] == -1
    assert got[3].nonzero()[0].tolist() == [2, 3] and depth[0, 3] == -1
    assert got[4].nonzero()[0].tolist() == [0, 1, 4] and depth[0, 4] == 2


# ---------------------------------------------------------------------------
# KV commit of the accepted path (review page, "The Complete EAGLE-3
# Inference Process" step 5: keep only the accepted path's cache entries)
# ---------------------------------------------------------------------------

def _tagged_cache(planes, B, L, E, base, N):
    """Entries tagged by what they hold: prefix position t -> (p, b, t, 0);
    tree node v (at base + v - 1) -> (p, b, v, 1); unused tail -> (p, b, t, 2)."""
    c = np.zeros((planes, B, L, E), dtype=np.int32)
    for p in range(planes):
        for b in range(B):
            for t in range(L):
                v = t - base[b] + 1
                kind = 0 if t < base[b] else (1 if v < N else 2)
                tag = v if kind == 1 else t
                c[p, b, t, :] = [p, b, tag, kind] + [1000 * p + 10 * b + kind] * (E - 4)
    return c


def _appended(c, b, base, path, d):
    """The cache a plain decoder would hold after appending the accepted
    tokens one by one: prefix, then the entries of nodes v_1..v_d in order."""
    planes = c.shape[0]
    rows = []
    for p in range(planes):
        prefix = [c[p, b, t].copy() for t in range(base)]
        acc = [c[p, b, base + path[i] - 1].copy() for i in range(1, d + 1)]
        rows.append(np.array(prefix + acc))
    return rows


@pytest.mark.parametrize("seed", range(4))
def test_kv_commit_equals_appending_the_path(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    planes, B, N, E, W = 3, 4, 12, 6, 7
    base = rng.integers(1, 8, size=B).astype(np.int32)
    L = int(base.max()) + N + 3
    c = _tagged_cache(planes, B, L, E, base, N)
    par = np.stack([synth.make_tree_parents(rng, N, max_depth=W - 1) for _ in range(B)])
    path = np.full((B, W), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):                      # a random root-to-node path
        v = int(rng.integers(N))
        chain = [v]
        while chain[-1] != 0:
            chain.append(int(par[b, chain[-1]]))
        chain = chain[::-1]
        acc[b] = len(chain) - 1
        path[b, :len(chain)] = chain
    out, new_len, bad = oracle_mod.kv_commit(c, base, acc, path, N)
    assert not bad
    assert np.array_equal(new_len, base + acc)
    for b in range(B):
        want = _appended(c, b, base[b], path[b], acc[b])
        for p in range(planes):
            n = base[b] + acc[b]
            assert np.array_equal(out[p, b, :n], want[p])
            assert np.array_equal(out[p, b, n:], c[p, b, n:])   # untouched past the new end
            # the accepted entries are the path's nodes, in order
            assert out[p, b, base[b]:n, 2].tolist() == path[b, 1:acc[b] + 1].tolist()


def test_kv_commit_chain_and_empty_paths_change_nothing(oracle_mod):
    planes, B, N, E = 2, 3, 8, 4
    base = np.array([2, 5, 1], dtype=np.int32)
    L = 16
    c = _tagged_cache(planes, B, L, E, base, N)
    path = np.full((B, 6), -1, dtype=np.int32)
    path[:, 0] = 0
    path[0, 1:4] = [1, 2, 3]                 # a chain: nodes already in place
    acc = np.array([3, 0, 0], dtype=np.int32)
    out, new_len, bad = oracle_mod.kv_commit(c, base, acc, path, N)
    assert not bad and np.array_equal(out, c)
    assert new_len.tolist() == [5, 5, 1]


def test_kv_commit_overlapping_moves(oracle_mod):
    # path 0 -> 2 -> 3 -> 5: node 2 moves onto node 1's slot while node 3
    # moves onto node 2's old slot (a source of an earlier move)
    c = _tagged_cache(1, 1, 12, 4, np.array([2]), 8)
    path = np.array([[0, 2, 3, 5, -1]], dtype=np.int32)
    out, new_len, _ = oracle_mod.kv_commit(c, [2], [3], path, 8)
    assert out[0, 0, 2:5, 2].tolist() == [2, 3, 5]
    assert new_len.tolist() == [5]


def test_kv_commit_malformed_left_untouched(oracle_mod):
    c = _tagged_cache(2, 3, 10, 4, np.array([2, 2, 2]), 6)
    path = np.array([[1, 2, -1], [0, 6, -1], [0, 1, -1]], dtype=np.int32)
    out, new_len, bad = oracle_mod.kv_commit(c, [2, 2, 6], [1, 1, 1], path, 6)
    assert bad
    assert np.array_equal(out, c)            # bad root, node >= N, tree past L
    assert new_len.tolist() == [2, 2, 6]


# ---------------------------------------------------------------------------
# LM head fused with greedy verification ("EAGLE math", "Why feature drafting
# lands a higher acceptance rate": logits come from the target's LM head,
# z = W_LM h; review page greedy bullets)
# ---------------------------------------------------------------------------

def _bf16_normal(rng, shape, scale=1.0):
    return synth.f32_to_bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


def test_lm_head_matches_float64_matmul(oracle_mod):
    rng = np.random.default_rng(0)
    B, k, d, V = 3, 2, 48, 257
    H = _bf16_normal(rng, (B * (k + 1), d))
    W = _bf16_normal(rng, (V, d), 0.5)
    res = oracle_mod.lm_head_greedy(H, W, np.zeros((B, k), np.int32))
    z = synth.bf16_bits_to_f32(H).astype(np.float64) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
    assert np.array_equal(res["argmax"], z.argmax(1))
    top2 = np.sort(z, axis=1)[:, -2:]
    assert np.allclose(res["gap"], top2[:, 1] - top2[:, 0], rtol=1e-12, atol=1e-12)
    wa = synth.bf16_bits_to_f32(W).astype(np.float64)[res["argmax"]]
    assert np.allclose(res["mag"], np.abs(wa * synth.bf16_bits_to_f32(H)).sum(1), rtol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_lm_head_equals_unfused_greedy_on_exact_logits(oracle_mod, seed):
    # small integers: every logit is exact in float32, so verifying the
    # materialised logits must give the same acceptance as the fused form
    rng = np.random.default_rng(seed)
    B, k, d, V = 6, 4, 40, 300
    H = synth.f32_to_bf16_bits(rng.integers(-3, 4, (B * (k + 1), d)).astype(np.float32))
    W = synth.f32_to_bf16_bits(rng.integers(-3, 4, (V, d)).astype(np.float32))
    z = (synth.bf16_bits_to_f32(H).astype(np.float64) @
         synth.bf16_bits_to_f32(W).astype(np.float64).T).astype(np.float32)
    g = z.reshape(B, k + 1, V).argmax(-1)
    tokens = np.where(rng.random((B, k)) < 0.7, g[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    fused = oracle_mod.lm_head_greedy(H, W, tokens)
    plain = oracle_mod.verify_greedy(z.reshape(B, k + 1, V), tokens, dtype="f32")
    assert np.array_equal(fused["accepted_len"], plain["accepted_len"])
    assert np.array_equal(fused["out_tokens"], plain["out_tokens"])


def test_lm_head_ties_and_subset(oracle_mod):
    rng = np.random.default_rng(5)
    B, k, d, V = 4, 1, 16, 20
    H = _bf16_normal(rng, (B * (k + 1), d))
    W = _bf16_normal(rng, (V, d))
    W[7] = W[3]                                # identical vocabulary rows
    h = synth.bf16_bits_to_f32(H).astype(np.float64)
    W[3] = synth.f32_to_bf16_bits(np.float32(4.0) * np.sign(h[0]).astype(np.float32))
    W[7] = W[3]
    res = oracle_mod.lm_head_greedy(H, W, np.zeros((B, k), np.int32))
    assert res["argmax"][0] == 3 and res["gap"][0] == 0.0   # lowest index wins a tie
    sub = oracle_mod.lm_head_greedy(H, W, np.zeros((B, k), np.int32), seqs=[2])
    assert np.array_equal(sub["argmax"][4:6], res["argmax"][4:6])
    assert (sub["argmax"][:4] == -2).all()


# ---------------------------------------------------------------------------
# EAGLE-2 tree growth ("EAGLE math", "EAGLE-2: dynamic draft trees": expand
# the nodes with the highest cumulative draft probability, re-rank under a
# fixed node budget)
# ---------------------------------------------------------------------------

def _softmax64(z, T):
    z = np.asarray(z, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def test_tree_grow_one_layer_is_top_m_of_the_root_row(oracle_mod):
    rng = np.random.default_rng(0)
    B, K, V, T, M = 3, 12, 40, 0.9, 7
    z = (2 * rng.standard_normal((B, 1, K, V))).astype(np.float32)
    r = oracle_mod.tree_grow(z, T, M, dtype="f32")
    for b in range(B):
        q = _softmax64(z[b, 0, 0], T)
        top = np.argsort(-q, kind="stable")[:M]      # library sort, lowest index on ties
        assert r["tokens"][b, 1:].tolist() == sorted(top.tolist(), key=lambda x: -q[x])
        assert (r["parents"][b, 1:] == 0).all() and (r["depth"][b, 1:] == 1).all()
        assert np.allclose(r["values"][b, 1:], np.log(q[r["tokens"][b, 1:]]), atol=1e-12)


def test_tree_grow_two_layers_full_expansion(oracle_mod):
    # K = V: every token is expanded; the frontier is every child ranked by
    # value; the result is the M most probable paths of length <= 2
    rng = np.random.default_rng(1)
    V = K = 4
    T, M = 1.0, 9
    z = (1.5 * rng.standard_normal((1, 2, K, V))).astype(np.float32)
    r = oracle_mod.tree_grow(z, T, M, dtype="f32")
    q0 = _softmax64(z[0, 0, 0], T)
    rank = sorted(range(V), key=lambda x: (-q0[x], x))   # frontier slot of child x
    paths = [((x,), np.log(q0[x])) for x in range(V)]
    for slot, x in enumerate(rank):
        q1 = _softmax64(z[0, 1, slot], T)
        paths += [((x, y), np.log(q0[x]) + np.log(q1[y])) for y in range(V)]
    best = sorted(paths, key=lambda p: -p[1])[:M]
    got = set()
    for v in range(1, M + 1):
        chain = [r["tokens"][0, v]]
        p = r["parents"][0, v]
        while p != 0:
            chain.append(r["tokens"][0, p])
            p = r["parents"][0, p]
        got.add(tuple(chain[::-1]))
    assert got == {p[0] for p in best}


def test_tree_grow_k1_is_the_greedy_chain(oracle_mod):
    rng = np.random.default_rng(2)
    B, D, V = 2, 5, 30
    z = (2 * rng.standard_normal((B, D, 1, V))).astype(np.float32)
    r = oracle_mod.tree_grow(z, 1.0, D, dtype="f32")
    for b in range(B):
        assert r["tokens"][b, 1:].tolist() == [int(np.argmax(z[b, d, 0])) for d in range(D)]
        assert r["parents"][b, 1:].tolist() == list(range(D))


@pytest.mark.parametrize("seed", range(3))
def test_tree_grow_structure(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    B, D, K, V, M = 4, 4, 3, 50, 15
    z = (2 * rng.standard_normal((B, D, K, V))).astype(np.float32)
    r = oracle_mod.tree_grow(z, 0.8, M, dtype="f32")
    for b in range(B):
        par, dep, val = r["parents"][b], r["depth"][b], r["values"][b]
        assert par[0] == -1 and dep[0] == 0
        for v in range(1, M + 1):
            assert 0 <= par[v] < v                       # topological, closed
            assert dep[v] == dep[par[v]] + 1
            assert val[v] <= val[par[v]]                  # probabilities multiply
        # siblings carry distinct tokens
        for p in set(par[1:].tolist()):
            kids = r["tokens"][b, 1:][par[1:] == p]
            assert len(set(kids.tolist())) == len(kids)
    # the budget keeps the M best nodes by value: the tree grown with every
    # node kept has the same M largest values
    n_all = K + (D - 1) * K * K
    r_all = oracle_mod.tree_grow(z, 0.8, n_all, dtype="f32")
    for b in range(B):
        best = np.sort(r_all["values"][b, 1:])[::-1][:M]
        assert np.array_equal(np.sort(r["values"][b, 1:])[::-1], best)


def _logp_rows(*rows, V=6):
    """Draft rows given as probabilities (the rest spread evenly): logits are
    their logs, so softmax at T = 1 returns them."""
    out = []
    for spec in rows:
        p = np.full(V, 0.0)
        for tok, pr in spec.items():
            p[tok] = pr
        rest = [x for x in range(V) if x not in spec]
        p[rest] = (1.0 - sum(spec.values())) / len(rest)
        out.append(np.log(p).astype(np.float32))
    return np.array(out)


def test_tree_grow_worked_example_frontier_by_value(oracle_mod):
    # root: a=0 (0.6), b=1 (0.3).  a's row: x=2 (0.5), y=3 (0.4); b's row:
    # u=4 (0.9), v=5 (0.05).  Candidates: a.x 0.30, a.y 0.24, b.u 0.27,
    # b.v 0.015 -> the depth-2 frontier is (a.x, b.u), not the first two
    # created (a.x, a.y).  Their rows (slots 0, 1) put token 5 and token 0 on top.
    K, D, V = 2, 3, 6
    z = np.zeros((1, D, K, V), np.float32)
    z[0, 0, 0] = _logp_rows({0: 0.6, 1: 0.3})[0]
    z[0, 0, 1] = z[0, 0, 0]                        # unused slot at layer 0
    z[0, 1] = _logp_rows({2: 0.5, 3: 0.4}, {4: 0.9, 5: 0.05})
    z[0, 2] = _logp_rows({5: 0.7, 1: 0.2}, {0: 0.8, 2: 0.1})
    M = 1 + K + K * K + K * K - 1                   # every node but the worst
    r = oracle_mod.tree_grow(z, 1.0, M, dtype="f32")
    tok, par = r["tokens"][0], r["parents"][0]
    path = lambda v: (tuple(path(par[v])) if par[v] > 0 else ()) + (int(tok[v]),)
    depth3_parents = {path(par[v]) for v in range(1, M + 1) if r["depth"][0, v] == 3}
    assert depth3_parents == {(0, 2), (1, 4)}
    vals = {path(v): r["values"][0, v] for v in range(1, M + 1)}
    assert (1, 4, 0) in vals and (0, 2, 5) in vals
    assert np.isclose(vals[(1, 4, 0)], np.log(0.3 * 0.9 * 0.8))
    assert np.isclose(vals[(0, 2, 5)], np.log(0.6 * 0.5 * 0.7))


def test_tree_grow_ties_take_the_lower_token(oracle_mod):
    z = np.zeros((1, 1, 2, 8), np.float32)
    z[0, 0, 0] = [0, 1, 3, 0, 0, 3, 2, 0]       # tokens 2 and 5 tie for the top
    r = oracle_mod.tree_grow(z, 1.0, 1, dtype="f32")
    assert r["tokens"][0, 1] == 2
    r = oracle_mod.tree_grow(z, 1.0, 2, dtype="f32")
    assert r["tokens"][0, 1:].tolist() == [2, 5]


# ---------------------------------------------------------------------------
# diagnostics that decide which sampling rows may differ, and how
# ---------------------------------------------------------------------------

def _worked_margin_case():
    """Two drafts over V = 4, T = 1, logits = ln(probability), worked by hand.

    position 0: p = (.1 .2 .3 .4), q = (.4 .3 .2 .1), draft token 0: p/q = 1/4;
                u = 0.3 rejects (0.3 * 0.4 >= 0.1), 0.05 from the threshold.
    position 1: p = q = (.1 .2 .3 .4), u = 0.99: 0.01 from the threshold p/q = 1,
                but never decided (position 0 rejects).
    residual of row 0: max(0, p - q) = (0 0 .1 .3), R = 0.4; u_sample = 0.5
                puts u*R = 0.2 between C_2 = 0.1 and C_3 = 0.4: token 3, 0.1 from
                C_2, i.e. 0.25 of R.
    bonus row 2: p = 1/4 each (C = .25 .5 .75 1; u*R = 0.5 exactly on C_1).
    """
    ln = lambda v: np.log(np.array(v, np.float64)).astype(np.float32)
    zt = np.stack([ln([.1, .2, .3, .4]), ln([.1, .2, .3, .4]), np.zeros(4, np.float32)])[None]
    zd = np.stack([ln([.4, .3, .2, .1]), ln([.1, .2, .3, .4])])[None]
    toks = np.array([[0, 3]], np.int32)
    ua = np.array([[0.3, 0.99]], np.float32)
    us = np.array([0.5], np.float32)
    return zt, zd, toks, ua, us


def test_margins_and_flag_probability_worked_example(oracle_mod):
    zt, zd, toks, ua, us = _worked_margin_case()
    r = oracle_mod.verify_sample(zt, zd, toks, ua, us, 1.0, window=0.01)
    assert r["accepted_len"][0] == 0 and r["out_tokens"][0].tolist() == [3, -1, -1]
    assert r["resid_mass"][0] == pytest.approx(0.4, rel=1e-6)
    # acceptance margin of the decided position only (not 0.01 of position 1)
    assert r["acc_margin"][0] == pytest.approx(abs(0.3 - 0.25), rel=1e-5)
    # CDF margin as a fraction of R: 0.1 / 0.4
    assert r["cdf_margin"][0] == pytest.approx(0.25, rel=1e-5)
    # flag chance at window 0.01: the acceptance window around 1/4 (0.02) and
    # the CDF boundaries 0, 1/4, 1 of the residual (0.01 + 0.02 + 0.01)
    assert r["flag_prob"][0] == pytest.approx(0.06, rel=1e-5)


def test_claim_violation_worked_example(oracle_mod):
    zt, zd, toks, ua, us = _worked_margin_case()

    def claim(n, t):
        v, R = oracle_mod.sample_claim(zt, zd, toks, ua, us, 1.0, np.array([n]), np.array([t]))
        return v[0], R[0]

    v, R = claim(0, 3)                 # the exact outcome
    assert v == 0.0 and R == pytest.approx(0.4, rel=1e-6)
    v, _ = claim(0, 2)                 # u*R = 0.2 lies 0.1 past [C_1, C_2) = [0, 0.1)
    assert v == pytest.approx(0.25, rel=1e-5)
    assert claim(0, 0)[0] == np.inf    # zero residual weight: never drawn
    # n = 1: accepts position 0 (0.05 from its threshold) and rejects position
    # 1 (0.01); row 1's residual is empty, so p of row 1 is drawn (reading R6):
    # u = 0.5 gives token 2, token 3's interval [0.6, 1) is 0.1 away
    v, R = claim(1, 3)
    assert v == pytest.approx(0.1, rel=1e-5) and R == 0.0
    v, _ = claim(1, 2)
    assert v == pytest.approx(0.05, rel=1e-5)
    # n = 2 (bonus): only position 0 is crossed; u*R = 0.5 is C_1 exactly, so
    # both neighbouring tokens sit at distance 0 from their interval
    assert claim(2, 2)[0] == pytest.approx(0.05, rel=1e-5)
    assert claim(2, 1)[0] == pytest.approx(0.05, rel=1e-5)
    assert claim(2, 0)[0] == pytest.approx(0.25, rel=1e-5)
    assert claim(3, 0)[0] == np.inf and claim(-1, 0)[0] == np.inf


def _gap_case():
    """D = 3 layers, K = 2, V = 4, T = 1, rows given as probabilities.

    layer 0 (root): (.6 .38 .01 .01) -> a = 0.6, b = 0.38
    layer 1: a's row (.5 .4 .05 .05) -> .30, .24; b's row (.7 .2 .05 .05) ->
             .266, .076; the frontier keeps .30 and .266 and drops .24: gap
             ln(.266/.24)
    layer 2: both frontier rows uniform -> .075, .075 (under .30) and .0665,
             .0665 (under .266): exact ties between siblings
    """
    ln = lambda v: np.log(np.array(v, np.float64)).astype(np.float32)
    z = np.zeros((1, 3, 2, 4), np.float32)
    z[0, 0, 0] = z[0, 0, 1] = ln([.6, .38, .01, .01])
    z[0, 1, 0] = ln([.5, .4, .05, .05])
    z[0, 1, 1] = ln([.7, .2, .05, .05])
    return z


def test_tree_grow_min_gap_worked_example(oracle_mod):
    z = _gap_case()
    gap = lambda M: oracle_mod.tree_grow(z, 1.0, M, dtype="f32")["min_gap"][0]
    frontier = np.log(.266 / .24)
    # every node kept: only the frontier cut
    assert gap(10) == pytest.approx(frontier, rel=1e-5)
    # M = 6 keeps .076 and drops .075: the final cut is the closer one
    assert gap(6) == pytest.approx(np.log(.076 / .075), rel=1e-5)
    # M = 7 splits the exact tie .075 / .075: the tie rule decides it, and the
    # nearest unequal pair across the cut is .076 (kept) and .075 (dropped)
    assert gap(7) == pytest.approx(np.log(.076 / .075), rel=1e-5)
    # M = 9 splits the tie .0665 / .0665: the nearest unequal pair is .075 / .0665
    assert gap(9) == pytest.approx(min(frontier, np.log(.075 / .0665)), rel=1e-5)
    # the cut between the tied siblings still follows creation order
    r = oracle_mod.tree_grow(z, 1.0, 7, dtype="f32")
    kept_l3 = [v for v in range(1, 8) if r["depth"][0, v] == 3]
    assert len(kept_l3) == 1 and r["tokens"][0, kept_l3[0]] == 0


# ---------------------------------------------------------------------------
# LM head fused with sampling verification
# ---------------------------------------------------------------------------

def _int_bf16(rng, shape, lo, hi):
    """Small integers as bf16 bits (exactly representable)."""
    return synth.f32_to_bf16_bits(rng.integers(lo, hi, size=shape).astype(np.float32))


def test_lm_head_sample_equals_plain_sampling_on_exact_logits(oracle_mod):
    # integer weights and features: every logit W h is a small integer, exact
    # in float32, so the fused oracle must equal plain sampling verification
    # of logits computed here by an integer matrix product
    rng = np.random.default_rng(3)
    B, k, d, V, T = 6, 3, 16, 40, 1.3
    W = _int_bf16(rng, (V, d), -2, 3)
    Ht = _int_bf16(rng, (B * (k + 1), d), -2, 3)
    Hd = _int_bf16(rng, (B * k, d), -2, 3)
    toks = rng.integers(0, V, (B, k)).astype(np.int32)
    ua = synth.uniforms_f32(rng, (B, k))
    us = synth.uniforms_f32(rng, (B,))
    r = oracle_mod.lm_head_sample(Ht, Hd, W, toks, ua, us, T)
    Wi = synth.bf16_bits_to_f32(W).astype(np.int64)
    zt = (synth.bf16_bits_to_f32(Ht).astype(np.int64) @ Wi.T).astype(np.float32).reshape(B, k + 1, V)
    zd = (synth.bf16_bits_to_f32(Hd).astype(np.int64) @ Wi.T).astype(np.float32).reshape(B, k, V)
    ref = oracle_mod.verify_sample(zt, zd, toks, ua, us, T, dtype="f32")
    for key in ("accepted_len", "out_tokens"):
        assert np.array_equal(r[key], ref[key]), key
    for key in ("p", "q", "resid_mass"):
        assert np.allclose(r[key], ref[key], rtol=1e-12, atol=0), key
    # a subset of sequences gives the same rows
    sub = oracle_mod.lm_head_sample(Ht, Hd, W, toks, ua, us, T, seqs=[4, 1])
    assert np.array_equal(sub["out_tokens"], ref["out_tokens"][[4, 1]])
    assert 0 < (r["accepted_len"] < k).sum() < B
