"""GPU parity of the LM head fused with greedy verification (tcgen05 GEMM with
an argmax epilogue) against the float64 oracle.

The kernel's logits are float32 accumulations of exact bf16 products; the
oracle's are exact.  A row's argmax is compared exactly unless its top two
exact logits lie within a bound of the float32 accumulation error, in which
case either index is correct (the row is counted as flagged)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_56_gb300 as sv
from speculative_decoding_verification_56_gb300 import build, synth

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()
    sv.load_library()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _flag_bound(d, mag):
    # recursive float32 summation of d exact products: |error| <= d u sum|x_i y_i|
    # (for each of the two competing logits), with a safety factor of 4
    return 8.0 * d * U32 * mag


def _gpu(H, W, tok):
    out = sv.lm_head_verify_greedy(_bf16(H), _bf16(W), torch.from_numpy(tok).cuda())
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def _rows_argmax(H, W):
    """Per-row argmax from the GPU: every row as its own sequence with k = 0."""
    rows = H.shape[0]
    return _gpu(H, W, np.zeros((rows, 0), np.int32))["out_tokens"][:, 0]


@pytest.mark.parametrize("B,k,d,V,seed", [
    (1, 0, 64, 1, 0), (2, 3, 64, 300, 1), (3, 4, 128, 1000, 2), (4, 1, 72, 129, 3),
    (2, 2, 200, 5000, 4), (100, 4, 64, 700, 5),        # 500 rows: two halves of 256
    (1, 0, 8, 257, 6), (130, 4, 64, 700, 7),           # 650 rows: two row groups
    (41, 0, 96, 20000, 8),                             # 41 rows: halves of 32, one partly empty
    # three or more 256-entry vocabulary tiles per CTA pair, so the
    # accumulator slots rotate: 320 rows (two MMAs, three slots), 384 rows
    # (two MMAs, two slots), 256 and 64 rows (one MMA, two slots)
    (64, 4, 64, 60001, 10), (96, 3, 64, 60001, 11), (64, 3, 64, 60001, 12),
    (32, 1, 64, 60001, 13),
])
def test_lm_head_rows_and_chains(B, k, d, V, seed):
    H, W, tok, _ = synth.make_lm_head_case(B=B, k=k, d=d, V=V, seed=seed)
    res = oracle.lm_head_greedy(H, W, tok)
    flagged = res["gap"] <= _flag_bound(d, res["mag"])
    g_arg = _rows_argmax(H, W)
    assert np.array_equal(g_arg[~flagged], res["argmax"][~flagged])
    assert flagged.mean() <= 0.05
    out = _gpu(H, W, tok)
    seq_ok = ~flagged.reshape(B, k + 1).any(1)   # sequences with no flagged row
    assert np.array_equal(out["accepted_len"][seq_ok], res["accepted_len"][seq_ok])
    assert np.array_equal(out["out_tokens"][seq_ok], res["out_tokens"][seq_ok])


def test_lm_head_tie_picks_lowest_index():
    rng = np.random.default_rng(11)
    d, V = 64, 400
    H, W, _, intended = synth.make_lm_head_case(B=8, k=0, d=d, V=V, seed=11, flat_frac=0.0)
    for r, j in enumerate(intended):         # duplicate each intended row at a lower index
        lo = int(rng.integers(0, j + 1))
        W[lo] = W[j]
        intended[r] = lo
    res = oracle.lm_head_greedy(H, W, np.zeros((8, 0), np.int32))
    g = _rows_argmax(H, W)
    assert np.array_equal(res["argmax"], g)


@pytest.mark.slow
def test_lm_head_full_size_sampled_rows():
    # the greedy workload's shape: B=64, k=4, d=4096 (hidden), V=128256
    B, k, d, V = 64, 4, 4096, 128256
    H, W, tok, _ = synth.make_lm_head_case(B=B, k=k, d=d, V=V, seed=0)
    out = _gpu(H, W, tok)
    seqs = [0, 37]
    res = oracle.lm_head_greedy(H, W, tok, seqs=seqs)
    for b in seqs:
        rws = slice(b * (k + 1), (b + 1) * (k + 1))
        if (res["gap"][rws] <= _flag_bound(d, res["mag"][rws])).any():
            continue
        assert out["accepted_len"][b] == res["accepted_len"][b]
        assert np.array_equal(out["out_tokens"][b], res["out_tokens"][b])


# ---------------------------------------------------------------------------
# LM head fused with sampling verification
# ---------------------------------------------------------------------------
# The kernel's logits are float32 accumulations of exact bf16 products; the
# oracle's are exact (float64).  The decisions therefore compare within a
# wider window than on logits inputs: p, q and R within 1e-4 relative, and a
# row may differ from the oracle only where a uniform lies within 1e-4 of a
# decision boundary (the claim check), the flagged count bounded by the
# oracle's own flag probability at that window.
LM_WINDOW = 1e-4
LM_PQ_RTOL = 1e-4


class _F64Case:
    """The inputs of the claim check: the oracle's float64 logits."""

    def __init__(self, c, orc, seqs):
        self.B = len(seqs)
        self.target, self.draft = orc["zt"], orc["zd"]
        self.dtype = "f64"
        self.tokens = c.tokens[seqs]
        self.u_accept, self.u_sample = c.u_accept[seqs], c.u_sample[seqs]
        self.temperature = c.temperature


def _gpu_lm_sample(c):
    out = sv.lm_head_verify_sample(_bf16(c.h_target), _bf16(c.h_draft) if c.k else None,
                                   _bf16(c.w_lm), torch.from_numpy(c.tokens).cuda(),
                                   torch.from_numpy(c.u_accept).cuda(),
                                   torch.from_numpy(c.u_sample).cuda(), c.temperature)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def _lm_sample_parity(c, seqs=None):
    import parity_helpers as ph
    seqs = np.arange(c.B) if seqs is None else np.asarray(seqs)
    g = _gpu_lm_sample(c)
    o = oracle.lm_head_sample(c.h_target, c.h_draft, c.w_lm, c.tokens, c.u_accept, c.u_sample,
                              c.temperature, seqs=seqs, window=LM_WINDOW)
    s = ph.compare_sample(g, o, rows=seqs, case=_F64Case(c, o, seqs), window=LM_WINDOW,
                          pq_rtol=LM_PQ_RTOL)
    return s, g, o


@pytest.mark.parametrize("B,k,d,V,T,seed", [
    (2, 3, 64, 300, 1.0, 1), (3, 4, 128, 1000, 0.8, 2), (4, 0, 64, 500, 1.0, 3),
    (5, 2, 200, 5000, 1.2, 4), (100, 4, 64, 700, 1.0, 5),   # 500 target rows: two row groups
    (2, 1, 72, 129, 1.0, 6),                                # odd V: the draw's plain loads
    (6, 3, 96, 20000, 0.7, 7),
    (64, 4, 64, 60001, 1.0, 8),   # 320 target, 256 draft, 128 drawn rows; rotating slots
])
def test_lm_head_sample_matches_oracle(B, k, d, V, T, seed):
    c = synth.make_lm_head_sample_case(B=B, k=k, d=d, V=V, seed=seed, temperature=T,
                                       feature_noise=0.6, p_match=0.6)
    s, g, _ = _lm_sample_parity(c)
    assert s["rows"] == B


def test_lm_head_sample_both_outcomes():
    c = synth.make_lm_head_sample_case(B=40, k=4, d=64, V=2000, seed=9, feature_noise=0.8,
                                       p_match=0.6)
    s, g, _ = _lm_sample_parity(c)
    n = g["accepted_len"]
    assert (n < 4).any() and (n == 4).any()      # residual and bonus draws both occur


def test_lm_head_sample_launch_count():
    c = synth.make_lm_head_sample_case(B=2, k=2, d=64, V=300, seed=3)
    n0 = sv.spec_verify_launch_count()
    _gpu_lm_sample(c)
    # statistics GEMM, accept + gather, logits GEMM, clustered finish
    assert sv.spec_verify_launch_count() - n0 == 4


@pytest.mark.slow
def test_lm_head_sample_full_size_sampled_sequences():
    # the sampling workload's shape: B=64, k=4, hidden 4096, V=128256
    B, k, d, V = 64, 4, 4096, 128256
    c = synth.make_lm_head_sample_case(B=B, k=k, d=d, V=V, seed=0)
    s, g, _ = _lm_sample_parity(c, seqs=[0, 21, 63])
    n = g["accepted_len"]
    assert ((n >= 0) & (n <= k)).all()
    for b in range(B):
        assert (g["out_tokens"][b, :n[b]] == c.tokens[b, :n[b]]).all()
        assert 0 <= g["out_tokens"][b, n[b]] < V and (g["out_tokens"][b, n[b] + 1:] == -1).all()
