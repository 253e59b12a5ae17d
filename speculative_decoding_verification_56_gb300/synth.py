"""Seeded synthetic inputs for batched draft-token verification.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It builds *inputs only*: logits rows, draft tokens, uniforms and
draft trees.  It holds none of the verification arithmetic (no softmax, no
acceptance test, no residual, no inverse CDF).  Draft tokens are drawn from the
tempered draft distribution with the Gumbel-max construction (argmax of
logits/T plus Gumbel noise), which samples softmax(logits/T) exactly without
evaluating it.

Workload recipes (the pages measure on MT-Bench, HumanEval, GSM8K, Alpaca and
CNN/DailyMail; none of those items are used here, these seeded recipes stand in
for them):

* ``tiny``   : sampling, B=1, k=4, V=1000, fp32, T=1.0.  Target ~ N(0, 2^2)
               i.i.d.; draft = target of the same position + N(0, 1).
* ``peaked`` : sampling, B=8, k=5, V=32000, fp32, T=0.8.  Target ~ N(0, 3^2),
               1% of each row (without replacement) boosted by +8; draft =
               target + N(0, 0.5^2).
* ``zipf128k``: sampling and greedy, B=64, k=4, V=128256, bf16, T=1.0.  Target
               = N(0, 3^2) + Zipf(1.1) log-bias over a seeded per-sequence vocab
               permutation (bias of rank r is -1.1 ln r); draft = bf16(target +
               N(0, 1)).  Greedy drafts: 70% forced to the target argmax.
* ``zipf152k``: large-batch sampling, B=256, k=7, V=151936, bf16, T=0.7, same
               target recipe, draft = bf16(target + N(0, 1.5^2)).
* ``tree``   : draft-tree greedy, B=16 trees of N=60 nodes, depth <= 6,
               branching <= 4, V=128256, bf16 target rows ~ N(0, 3^2).  A child's
               token equals the argmax of its parent's row with probability 0.6,
               else it is uniform over the other V-1 tokens.

Seeds: logits and draft tokens come from ``seed``; the uniforms from
``seed + 1`` (numpy PCG64 in both cases).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPE_F32 = "f32"
DTYPE_BF16 = "bf16"

# ---------------------------------------------------------------------------
# bf16 storage helpers (bit manipulation only)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits.

    Inputs must be finite.  Works in place-friendly chunks to bound memory.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step]
        lsb = (u >> np.uint32(16)) & np.uint32(1)
        r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
        flat_out[s:s + step] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def logits_as_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Float32 view of stored logits (bf16 bits are widened exactly)."""
    if dtype == DTYPE_BF16:
        return bf16_bits_to_f32(arr)
    return np.asarray(arr, dtype=np.float32)


def uniforms_f32(rng: np.random.Generator, shape) -> np.ndarray:
    """U[0,1) drawn in float64 and rounded toward zero to float32 (so < 1)."""
    x = rng.random(shape)
    f = x.astype(np.float32)
    over = f.astype(np.float64) > x
    f[over] = np.nextafter(f[over], np.float32(0.0))
    return f


def _store(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == DTYPE_BF16:
        return f32_to_bf16_bits(x_f32)
    return np.ascontiguousarray(x_f32, dtype=np.float32)


def gumbel_max_tokens(rng: np.random.Generator, logits_f32: np.ndarray,
                      temperature: float) -> np.ndarray:
    """One exact draw from softmax(logits/T) per row via the Gumbel-max trick.

    ``logits_f32``: [..., V].  Rows are processed one at a time in float64.
    """
    lead = logits_f32.shape[:-1]
    V = logits_f32.shape[-1]
    rows = logits_f32.reshape(-1, V)
    out = np.empty(rows.shape[0], dtype=np.int32)
    for r in range(rows.shape[0]):
        u = rng.random(V)
        # open interval keeps both logs finite
        u = np.clip(u, np.finfo(np.float64).tiny, 1.0 - 2.0 ** -53)
        g = -np.log(-np.log(u))
        out[r] = int(np.argmax(rows[r].astype(np.float64) / temperature + g))
    return out.reshape(lead)


# ---------------------------------------------------------------------------
# Input containers
# ---------------------------------------------------------------------------


@dataclass
class ChainInputs:
    """Inputs of one chain verification call (sampling or greedy)."""

    name: str
    B: int
    k: int
    V: int
    dtype: str
    temperature: float
    target: np.ndarray          # [B, k+1, V] float32 or bf16 bits (uint16)
    draft: np.ndarray | None    # [B, k, V] same storage; None for greedy-only
    tokens: np.ndarray          # int32 [B, k]
    u_accept: np.ndarray        # float32 [B, k]
    u_sample: np.ndarray        # float32 [B]
    meta: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == DTYPE_BF16 else 4


@dataclass
class TreeInputs:
    """Inputs of one draft-tree greedy verification call."""

    name: str
    B: int
    N: int
    V: int
    dtype: str
    max_depth: int
    target: np.ndarray          # [B, N, V]; row v scores the children of node v
    tokens: np.ndarray          # int32 [B, N]; token of node 0 is ignored
    parents: np.ndarray         # int32 [B, N]; parents[:,0] = -1, parents[v] < v
    meta: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == DTYPE_BF16 else 4


# ---------------------------------------------------------------------------
# Logit recipes
# ---------------------------------------------------------------------------


def _gauss(rng, shape, sigma):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def _zipf_bias_rows(rng, B, V, s=1.1):
    """Per-sequence log-Zipf bias: bias[perm_b[r-1]] = -s * ln r, r = 1..V."""
    ranks = (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    bias = np.empty((B, V), dtype=np.float32)
    for b in range(B):
        perm = rng.permutation(V)
        bias[b, perm] = ranks
    return bias


def make_chain_logits(rng, B, k, V, dtype, recipe, target_sigma, draft_noise,
                      boost_frac=0.0, boost=0.0):
    """Target rows [B,k+1,V] and draft rows [B,k,V] (both as stored arrays)."""
    zt = _gauss(rng, (B, k + 1, V), target_sigma)
    if recipe == "peaked":
        nb = max(1, int(round(boost_frac * V)))
        for b in range(B):
            for i in range(k + 1):
                idx = rng.choice(V, size=nb, replace=False)
                zt[b, i, idx] += np.float32(boost)
    elif recipe == "zipf":
        bias = _zipf_bias_rows(rng, B, V)
        zt += bias[:, None, :]
    elif recipe != "gauss":
        raise ValueError(recipe)
    target = _store(zt, dtype)
    del zt
    zt_f = logits_as_f32(target[:, :k, :], dtype)
    zd = zt_f + _gauss(rng, (B, k, V), draft_noise)
    del zt_f
    draft = _store(zd, dtype)
    return target, draft


def make_chain_case(*, B, k, V, dtype=DTYPE_F32, temperature=1.0, recipe="gauss",
                    target_sigma=2.0, draft_noise=1.0, boost_frac=0.0, boost=0.0,
                    greedy_force=None, seed=0, name="case", with_draft=True):
    """Generic chain case.

    Draft tokens are exact samples of softmax(draft/T) (Gumbel-max).  With
    ``greedy_force=f`` the tokens are those of :func:`greedy_variant`.
    """
    rng = np.random.default_rng(seed)
    target, draft = make_chain_logits(rng, B, k, V, dtype, recipe, target_sigma,
                                      draft_noise, boost_frac, boost)
    tokens = np.zeros((B, k), dtype=np.int32)
    if k > 0:
        zd_f = logits_as_f32(draft, dtype)
        tokens = gumbel_max_tokens(rng, zd_f, temperature).astype(np.int32)
        del zd_f
    urng = np.random.default_rng(seed + 1)
    u_accept = uniforms_f32(urng, (B, k))
    u_sample = uniforms_f32(urng, (B,))
    case = ChainInputs(name=name, B=B, k=k, V=V, dtype=dtype,
                       temperature=float(temperature), target=target,
                       draft=draft if with_draft else None, tokens=tokens,
                       u_accept=u_accept, u_sample=u_sample,
                       meta=dict(recipe=recipe, seed=seed))
    if greedy_force is not None:
        case = greedy_variant(case, greedy_force)
        if not with_draft:
            case.draft = None
    return case


def greedy_variant(case: ChainInputs, force: float) -> ChainInputs:
    """Same logits; each draft token replaced, with probability ``force``, by
    the lowest-index argmax of the same position's target row (seed + 2)."""
    rng = np.random.default_rng(case.meta.get("seed", 0) + 2)
    k = case.k
    tokens = case.tokens.copy()
    if k > 0:
        zt_f = logits_as_f32(case.target[:, :k, :], case.dtype)
        amax = np.argmax(zt_f, axis=-1).astype(np.int32)
        del zt_f
        forced = rng.random((case.B, k)) < force
        tokens = np.where(forced, amax, tokens).astype(np.int32)
    meta = dict(case.meta, greedy_force=force)
    return ChainInputs(name=case.name + " greedy", B=case.B, k=k, V=case.V, dtype=case.dtype,
                       temperature=case.temperature, target=case.target, draft=case.draft,
                       tokens=tokens, u_accept=case.u_accept, u_sample=case.u_sample,
                       meta=meta)


def make_tree_parents(rng, N, max_depth=6, max_children=4):
    """Random rooted tree in topological order (parent index < child index)."""
    parents = np.full(N, -1, dtype=np.int32)
    depth = np.zeros(N, dtype=np.int32)
    nchild = np.zeros(N, dtype=np.int32)
    for v in range(1, N):
        cand = [u for u in range(v) if depth[u] < max_depth and nchild[u] < max_children]
        p = cand[int(rng.integers(len(cand)))]
        parents[v] = p
        depth[v] = depth[p] + 1
        nchild[p] += 1
    return parents


def make_tree_case(*, B, N, V, dtype=DTYPE_BF16, target_sigma=3.0, max_depth=6,
                   max_children=4, p_match=0.6, seed=0, name="tree", parents=None):
    rng = np.random.default_rng(seed)
    zt = _gauss(rng, (B, N, V), target_sigma)
    target = _store(zt, dtype)
    del zt
    zt_f = logits_as_f32(target, dtype)
    amax = np.argmax(zt_f, axis=-1).astype(np.int32)   # [B, N]
    del zt_f
    par = np.empty((B, N), dtype=np.int32)
    tok = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        par[b] = make_tree_parents(rng, N, max_depth, max_children) if parents is None \
            else np.asarray(parents, dtype=np.int32)
        tok[b, 0] = int(rng.integers(V))
        for v in range(1, N):
            a = int(amax[b, par[b, v]])
            if rng.random() < p_match:
                tok[b, v] = a
            else:
                t = int(rng.integers(V - 1)) if V > 1 else 0
                tok[b, v] = t + 1 if t >= a else t
    return TreeInputs(name=name, B=B, N=N, V=V, dtype=dtype, max_depth=max_depth,
                      target=target, tokens=tok, parents=par, meta=dict(seed=seed))


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------


def tiny(seed=0):
    return make_chain_case(B=1, k=4, V=1000, dtype=DTYPE_F32, temperature=1.0,
                           recipe="gauss", target_sigma=2.0, draft_noise=1.0,
                           seed=seed, name="tiny B=1 k=4 V=1000 f32")


def peaked(seed=0):
    return make_chain_case(B=8, k=5, V=32000, dtype=DTYPE_F32, temperature=0.8,
                           recipe="peaked", target_sigma=3.0, draft_noise=0.5,
                           boost_frac=0.01, boost=8.0, seed=seed,
                           name="peaked B=8 k=5 V=32000 f32")


def zipf128k(seed=0, greedy=False, B=64, k=4, V=128256):
    return make_chain_case(B=B, k=k, V=V, dtype=DTYPE_BF16, temperature=1.0,
                           recipe="zipf", target_sigma=3.0, draft_noise=1.0,
                           greedy_force=0.7 if greedy else None, seed=seed,
                           name=f"zipf B={B} k={k} V={V} bf16" + (" greedy" if greedy else ""))


def zipf152k(seed=0, B=256, k=7, V=151936):
    return make_chain_case(B=B, k=k, V=V, dtype=DTYPE_BF16, temperature=0.7,
                           recipe="zipf", target_sigma=3.0, draft_noise=1.5,
                           seed=seed, name=f"zipf B={B} k={k} V={V} bf16 T=0.7")


def tree(seed=0, B=16, N=60, V=128256):
    return make_tree_case(B=B, N=N, V=V, dtype=DTYPE_BF16, target_sigma=3.0,
                          max_depth=6, max_children=4, p_match=0.6, seed=seed,
                          name=f"tree B={B} N={N} V={V} bf16")


WORKLOADS = {
    "tiny": tiny,
    "peaked": peaked,
    "zipf128k": zipf128k,
    "zipf152k": zipf152k,
    "tree": tree,
}


# ---------------------------------------------------------------------------
# LM-head inputs: hidden states and LM-head weights (bf16 bits)
# ---------------------------------------------------------------------------

def make_lm_head_case(*, B, k, d, V, seed=0, peak=6.0, p_match=0.7, flat_frac=0.1):
    """Synthetic LM head W [V, d] ~ N(0, 1/d) and hidden states H [B*(k+1), d].
    Most rows point at a random 'intended' token j (h = peak * sqrt(d) *
    W[j] / |W[j]|^2 ... scaled so z_j ~ peak above the N(0, 1) background,
    plus N(0, 1) noise), like a confident LM; a fraction `flat_frac` of rows
    are pure noise (no clear winner).  Draft tokens equal the intended token
    with probability p_match, else a uniform token.  Returns (H bits, W bits,
    tokens, intended)."""
    rng = np.random.default_rng(seed)
    W_bits = np.empty((V, d), dtype=np.uint16)
    for v0 in range(0, V, 8192):  # in slices: the full-size head is 128256 x 4096
        v1 = min(V, v0 + 8192)
        W_bits[v0:v1] = f32_to_bf16_bits(
            (rng.standard_normal((v1 - v0, d), dtype=np.float32) / np.float32(np.sqrt(d))))
    rows = B * (k + 1)
    intended = rng.integers(0, V, rows)
    Hm = rng.standard_normal((rows, d))
    wj = bf16_bits_to_f32(W_bits[intended]).astype(np.float64)
    coef = peak / np.maximum((wj * wj).sum(1), 1e-12)
    flat = rng.random(rows) < flat_frac
    Hm = Hm + np.where(flat[:, None], 0.0, coef[:, None] * wj)
    H_bits = f32_to_bf16_bits(Hm.astype(np.float32))
    draft_int = intended.reshape(B, k + 1)[:, :k]
    tokens = np.where(rng.random((B, k)) < p_match, draft_int,
                      rng.integers(0, V, (B, k))).astype(np.int32)
    return H_bits, W_bits, tokens, intended.astype(np.int32)


class LmSampleInputs:
    """Inputs of the LM head fused with sampling verification: target hidden
    states [B*(k+1), d], drafted features [B*k, d] and the LM head [V, d] as
    bf16 bits; draft tokens, uniforms and the temperature."""

    def __init__(self, B, k, d, V, temperature, h_target, h_draft, w_lm, tokens, u_accept,
                 u_sample):
        self.B, self.k, self.d, self.V = B, k, d, V
        self.temperature = temperature
        self.h_target, self.h_draft, self.w_lm = h_target, h_draft, w_lm
        self.tokens, self.u_accept, self.u_sample = tokens, u_accept, u_sample


def make_lm_head_sample_case(*, B, k, d, V, seed=0, peak=6.0, p_match=0.7, flat_frac=0.1,
                             feature_noise=0.3, temperature=1.0):
    """The LM-head recipe of make_lm_head_case for the target hidden states,
    plus drafted features h_d = h_t + N(0, feature_noise^2) per element of the
    k drafted positions (a drafter that predicts the target's features with
    some error).  Draft tokens are the intended token of the position with
    probability p_match, else uniform; uniforms from seed + 1."""
    H_bits, W_bits, tokens, _ = make_lm_head_case(B=B, k=k, d=d, V=V, seed=seed, peak=peak,
                                                  p_match=p_match, flat_frac=flat_frac)
    rng = np.random.default_rng(seed + 7)
    Ht = bf16_bits_to_f32(H_bits).reshape(B, k + 1, d)
    Hd = Ht[:, :k] + feature_noise * rng.standard_normal((B, k, d)).astype(np.float32)
    Hd_bits = f32_to_bf16_bits(Hd.reshape(B * k, d).astype(np.float32))
    urng = np.random.default_rng(seed + 1)
    u_accept = uniforms_f32(urng, (B, k))
    u_sample = uniforms_f32(urng, (B,))
    return LmSampleInputs(B, k, d, V, float(temperature), H_bits, Hd_bits, W_bits, tokens,
                          u_accept, u_sample)


# ---------------------------------------------------------------------------
# Draft rows for tree growth
# ---------------------------------------------------------------------------

def make_grow_logits(*, B, D, K, V, dtype=DTYPE_BF16, sigma=3.0, zipf=True, seed=0):
    """Draft logits [B, D, K, V] (stored bits) for tree growth: Gaussian
    N(0, sigma^2) plus, with ``zipf``, the per-sequence Zipf(1.1) log-bias of
    the verification workloads (a peaked, LM-like distribution)."""
    rng = np.random.default_rng(seed)
    z = _gauss(rng, (B, D, K, V), sigma)
    if zipf:
        bias = _zipf_bias_rows(rng, B, V)
        z += bias[:, None, None, :]
    out = _store(z, dtype)
    del z
    return out
