"""GPU parity of the kernels around the draft tree, through the C ABI, against
the oracle (bit-exact: these are integer results)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_56_gb300 as sv
from speculative_decoding_verification_56_gb300 import build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()
    sv.load_library()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


# ---------------------------------------------------------------------------
# tree attention mask
# ---------------------------------------------------------------------------

def _gpu_mask(par, with_depth=True):
    p = torch.from_numpy(np.ascontiguousarray(par, dtype=np.int32)).cuda()
    B, N = par.shape
    ws = sv.alloc_workspace(sv.SPEC_MODE_TREE_MASK, B, N, 1, sv.SPEC_DTYPE_F32)
    if with_depth:
        mask, depth = sv.tree_attention_mask(p, workspace=ws)
        depth = depth.cpu().numpy()
    else:
        mask = torch.empty(B, N, (N + 31) // 32, dtype=torch.int32, device="cuda")
        sv.spec_tree_attention_mask(p, mask, None, ws)
        depth = None
    torch.cuda.synchronize()
    flags = sv.spec_verify_read_flags(ws)
    return mask.cpu().numpy().view(np.uint32), depth, flags


def _random_parents(rng, B, N, max_depth=8, max_children=4):
    return np.stack([synth.make_tree_parents(rng, N, max_depth=max_depth,
                                             max_children=max_children)
                     for _ in range(B)]).astype(np.int32)


def _deep_parents(rng, B, N, span):
    """Parents drawn from the previous `span` nodes: deep, narrow trees."""
    par = np.empty((B, N), dtype=np.int32)
    par[:, 0] = -1
    for v in range(1, N):
        par[:, v] = rng.integers(max(0, v - span), v, size=B)
    return par


@pytest.mark.parametrize("B,N", [(1, 1), (3, 2), (2, 31), (2, 32), (2, 33), (16, 60), (4, 64),
                                 (4, 65), (2, 500), (1, 2048), (1, 3001)])
def test_tree_mask_random(B, N):
    rng = np.random.default_rng(1000 + N)
    par = _random_parents(rng, B, N) if N <= 600 else _deep_parents(rng, B, N, 40)
    m_o, d_o, bad = oracle.tree_mask(par)
    m_g, d_g, flags = _gpu_mask(par)
    assert not bad and flags == 0
    assert np.array_equal(m_g, m_o)
    assert np.array_equal(d_g, d_o)


def test_tree_mask_chain_and_star():
    N = 1500
    chain = np.array([[-1] + list(range(N - 1))], dtype=np.int32)
    star = np.array([[-1] + [0] * (N - 1)], dtype=np.int32)
    for par in (chain, star):
        m_o, d_o, _ = oracle.tree_mask(par)
        m_g, d_g, flags = _gpu_mask(par)
        assert flags == 0
        assert np.array_equal(m_g, m_o) and np.array_equal(d_g, d_o)


def test_tree_mask_workload_shape():
    # the tree-verification workload: 16 trees of 60 nodes, depth <= 6
    t = synth.tree(seed=0)
    m_o, d_o, _ = oracle.tree_mask(t.parents)
    m_g, d_g, _ = _gpu_mask(t.parents)
    assert np.array_equal(m_g, m_o) and np.array_equal(d_g, d_o)
    m_g2, _, _ = _gpu_mask(t.parents, with_depth=False)   # depth output omitted
    assert np.array_equal(m_g2, m_o)


def test_tree_mask_malformed_is_flagged_and_matches():
    rng = np.random.default_rng(7)
    par = _random_parents(rng, 4, 70)
    par[1, 20] = 25          # forward parent
    par[2, 33] = -3          # negative parent
    par[3, 5] = 5            # self parent
    m_o, d_o, bad = oracle.tree_mask(par)
    m_g, d_g, flags = _gpu_mask(par)
    assert bad and flags & sv.SPEC_FLAG_BAD_PARENT
    assert np.array_equal(m_g, m_o) and np.array_equal(d_g, d_o)
    assert (d_g[0] >= 0).all()


# ---------------------------------------------------------------------------
# KV commit of the accepted path
# ---------------------------------------------------------------------------

def _random_paths(rng, par, W):
    """A random root-to-node path per tree (as tree verification writes it)."""
    B, N = par.shape
    path = np.full((B, W), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        v = int(rng.integers(N))
        chain = [v]
        while chain[-1] != 0:
            chain.append(int(par[b, chain[-1]]))
        chain = chain[::-1][:W]
        acc[b] = len(chain) - 1
        path[b, :len(chain)] = chain
    return path, acc


def _gpu_kv(cache, base, acc, path, N):
    c = torch.from_numpy(np.ascontiguousarray(cache)).cuda()
    B = cache.shape[1]
    ws = sv.alloc_workspace(sv.SPEC_MODE_KV_COMMIT, B, N, 1, sv.SPEC_DTYPE_F32)
    new_len = torch.empty(B, dtype=torch.int32, device="cuda")
    sv.spec_kv_commit_path(c, torch.from_numpy(np.asarray(base, np.int32)).cuda(),
                           torch.from_numpy(np.asarray(acc, np.int32)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(path, np.int32)).cuda(), N,
                           new_len, ws)
    torch.cuda.synchronize()
    return c.cpu().numpy(), new_len.cpu().numpy(), sv.spec_verify_read_flags(ws)


@pytest.mark.parametrize("planes,B,N,E,W,seed", [
    (1, 1, 8, 8, 6, 0),          # 16-byte entries (bf16 x 8)
    (4, 5, 30, 64, 7, 1),
    (64, 16, 60, 1024, 7, 2),    # 32 layers x K/V, 8 heads x 128 bf16
    (3, 4, 200, 40, 40, 3),      # deep paths
    (2, 3, 300, 8, 120, 4),      # more moves than one staging pass holds
    (2, 2, 20, 40000, 10, 5),    # entries sliced across passes
])
def test_kv_commit_matches_oracle(planes, B, N, E, W, seed):
    rng = np.random.default_rng(seed)
    depth = W - 1
    if W >= 100:  # deep, mostly two-way trees: paths longer than one staging pass
        par = np.stack([np.concatenate([[-1, 0], np.arange(2, N) - rng.integers(1, 3, N - 2)])
                        for _ in range(B)]).astype(np.int32)
    else:
        par = np.stack([synth.make_tree_parents(rng, N, max_depth=depth, max_children=3)
                        for _ in range(B)]).astype(np.int32)
    base = rng.integers(1, 50, size=B).astype(np.int32)
    L = int(base.max()) + N + int(rng.integers(0, 5))
    cache = rng.integers(-30000, 30000, size=(planes, B, L, E), dtype=np.int16)
    path, acc = _random_paths(rng, par, W)
    want, want_len, bad = oracle.kv_commit(cache, base, acc, path, N)
    got, got_len, flags = _gpu_kv(cache, base, acc, path, N)
    assert not bad and flags == 0
    assert np.array_equal(got_len, want_len)
    assert np.array_equal(got, want)


def test_kv_commit_overlaps_chain_empty_and_malformed():
    rng = np.random.default_rng(9)
    planes, B, N, E, W = 3, 6, 10, 16, 6
    base = np.array([2, 3, 1, 4, 2, 9], dtype=np.int32)
    L = 20
    cache = rng.integers(-30000, 30000, size=(planes, B, L, E), dtype=np.int16)
    path = np.full((B, W), -1, dtype=np.int32)
    path[:, 0] = 0
    path[0, 1:4] = [2, 3, 5]        # overlapping moves
    path[1, 1:4] = [1, 2, 3]        # a chain: nothing moves
    acc = np.array([3, 3, 0, 2, 1, 1], dtype=np.int32)   # seq 2: empty path
    path[3, 1:3] = [4, 10]          # node outside [1, N): malformed
    path[4, 0] = 1                  # does not start at the root: malformed
    path[5, 1] = 1                  # tree past the cache end: malformed
    want, want_len, bad = oracle.kv_commit(cache, base, acc, path, N)
    got, got_len, flags = _gpu_kv(cache, base, acc, path, N)
    assert bad and flags & sv.SPEC_FLAG_BAD_PATH
    assert np.array_equal(got_len, want_len) and np.array_equal(got, want)
    assert np.array_equal(got[:, 1:3], cache[:, 1:3])      # chain and empty: untouched


def test_kv_commit_after_tree_verification():
    # the path written by spec_verify_tree_greedy drives the commit
    t = synth.tree(seed=1)
    out = sv.verify_tree_greedy(sv.to_device_logits(t.target, t.dtype),
                                torch.from_numpy(t.tokens).cuda(),
                                torch.from_numpy(t.parents).cuda(), t.max_depth)
    torch.cuda.synchronize()
    path = out["path_nodes"].cpu().numpy()
    acc = out["accepted_len"].cpu().numpy()
    rng = np.random.default_rng(3)
    planes, E = 8, 256
    base = (100 + np.arange(t.B)).astype(np.int32)
    L = int(base.max()) + t.N
    cache = rng.integers(-30000, 30000, size=(planes, t.B, L, E), dtype=np.int16)
    want, want_len, bad = oracle.kv_commit(cache, base, acc, path, t.N)
    got, got_len, flags = _gpu_kv(cache, base, acc, path, t.N)
    assert not bad and flags == 0
    assert np.array_equal(got_len, want_len) and np.array_equal(got, want)


# ---------------------------------------------------------------------------
# EAGLE-2 tree growth
# ---------------------------------------------------------------------------

# Node values are sums of float64 logarithms that the GPU and the oracle round
# differently (a few 1e-15 relative); two unequal values closer than this at a
# selection cut may swap.
GROW_GAP = 1e-9


def _gpu_grow(z, dtype, T, M):
    t = sv.to_device_logits(z, dtype)
    out = sv.tree_grow(t, T, M)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


@pytest.mark.parametrize("B,D,K,V,M,T,dtype,seed", [
    (1, 1, 1, 8, 1, 1.0, "f32", 0),
    (3, 2, 4, 100, 10, 1.0, "f32", 1),
    (4, 4, 3, 1000, 20, 0.7, "bf16", 2),
    (2, 6, 8, 20000, 59, 1.0, "bf16", 3),       # crosses 32 KB chunks
    (2, 3, 16, 33000, 100, 1.3, "f32", 4),
    (2, 5, 5, 5001, 40, 1.0, "bf16", 5),        # odd vocabulary: plain loads
])
def test_tree_grow_matches_oracle(B, D, K, V, M, T, dtype, seed):
    z = synth.make_grow_logits(B=B, D=D, K=K, V=V, dtype=dtype, seed=seed)
    ref = oracle.tree_grow(z, T, M, dtype=dtype)
    got = _gpu_grow(z, dtype, T, M)
    # a tree may differ only where two unequal values meet at a cut closer
    # than GROW_GAP (exact ties are decided by the tie rule and compared)
    ok = ref["min_gap"] > GROW_GAP
    assert ok.mean() >= 0.9
    for key in ("tokens", "parents", "depth"):
        assert np.array_equal(got[key][ok], ref[key][ok]), key
    assert np.allclose(got["values"][ok], ref["values"][ok], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("V", [2048, 20000])
def test_tree_grow_many_segments_per_cta(V):
    # 8 trees of 16 layers x 16 frontier rows over short rows (one or two
    # chunks each): every CTA of the streaming top-k closes several row
    # segments, so its four segment slots are reused within the CTA
    B, D, K, M = 8, 16, 16, 200
    z = synth.make_grow_logits(B=B, D=D, K=K, V=V, seed=31)
    ref = oracle.tree_grow(z, 1.0, M, dtype="bf16")
    got = _gpu_grow(z, "bf16", 1.0, M)
    ok = ref["min_gap"] > GROW_GAP
    assert ok.mean() >= 0.9, ref["min_gap"]
    for key in ("tokens", "parents", "depth"):
        assert np.array_equal(got[key][ok], ref[key][ok]), key
    assert np.allclose(got["values"][ok], ref["values"][ok], rtol=1e-6, atol=1e-6)


def test_tree_grow_full_workload():
    # the benchmark's grow workload: 16 trees, 6 layers x 8 frontier rows over
    # V = 128256 bf16, budget 59; exact ties between siblings (equal bf16
    # logits) are compared, since the tie rule decides them
    B, D, K, V, M = 16, 6, 8, 128256, 59
    z = synth.make_grow_logits(B=B, D=D, K=K, V=V, seed=0)
    ref = oracle.tree_grow(z, 1.0, M, dtype="bf16")
    got = _gpu_grow(z, "bf16", 1.0, M)
    ok = ref["min_gap"] > GROW_GAP
    assert ok.mean() >= 0.9, ref["min_gap"]
    for key in ("tokens", "parents", "depth"):
        assert np.array_equal(got[key][ok], ref[key][ok]), key
    assert np.allclose(got["values"][ok], ref["values"][ok], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("B,D,K,V,M,dtype", [
    (2, 4, 4, 20000, 12, "bf16"),
    (2, 3, 16, 40000, 32, "f32"),
])
def test_tree_grow_tied_block(B, D, K, V, M, dtype):
    # 3000 equal logits on top of every row: more tied candidates than the
    # top-k buffer holds, so the exact per-warp fallback ranks the chunk;
    # the K lowest indices of the block win
    z = synth.logits_as_f32(synth.make_grow_logits(B=B, D=D, K=K, V=V, dtype=dtype, seed=11), dtype)
    z[..., :3000] = z.max(axis=-1, keepdims=True) + 0.5
    if dtype == "bf16":
        z = synth.f32_to_bf16_bits(z)
    ref = oracle.tree_grow(z, 1.0, M, dtype=dtype)
    got = _gpu_grow(z, dtype, 1.0, M)
    assert set(np.unique(ref["tokens"][:, 1:])) <= set(range(K))
    ok = ref["min_gap"] > GROW_GAP
    assert ok.mean() >= 0.9
    for key in ("tokens", "parents", "depth"):
        assert np.array_equal(got[key][ok], ref[key][ok]), key
    assert np.allclose(got["values"][ok], ref["values"][ok], rtol=1e-6, atol=1e-6)


def test_tree_grow_largest_tree_and_budgets():
    # 16 layers x 16 frontier rows (3857 nodes, 241 draft rows per tree):
    # the node sort takes its shared-memory path; budgets 0, 1, all nodes
    B, D, K, V = 2, 16, 16, 3000
    z = synth.make_grow_logits(B=B, D=D, K=K, V=V, dtype="f32", seed=21)
    t = sv.to_device_logits(z, "f32")
    for M in (0, 1, 700, 3856):
        ref = oracle.tree_grow(z, 1.0, M, dtype="f32")
        out = sv.tree_grow(t, 1.0, M)
        torch.cuda.synchronize()
        got = {key: v.cpu().numpy() for key, v in out.items()}
        ok = ref["min_gap"] > GROW_GAP
        assert ok.mean() >= 0.9 or M == 0, (M, ref["min_gap"])
        for key in ("tokens", "parents", "depth"):
            assert np.array_equal(got[key][ok], ref[key][ok]), (M, key)
        assert np.allclose(got["values"][ok], ref["values"][ok], rtol=1e-6, atol=1e-6)


def test_tree_grow_empty_batch():
    z = synth.make_grow_logits(B=1, D=2, K=2, V=64, dtype="f32", seed=0)[:0]
    out = sv.tree_grow(sv.to_device_logits(z, "f32"), 1.0, 3)
    assert out["tokens"].shape == (0, 4)


@pytest.mark.parametrize("V", [1000, 1001])
def test_tree_grow_launch_count(V):
    # one top-k pass over every draft row, one tree kernel; on the bulk-copy
    # path (rows of whole 16-byte vectors) and the plain-load path
    z = synth.make_grow_logits(B=2, D=5, K=4, V=V, dtype="f32", seed=1)
    t = sv.to_device_logits(z, "f32")
    n0 = sv.spec_verify_launch_count()
    sv.tree_grow(t, 1.0, 20)
    torch.cuda.synchronize()
    assert sv.spec_verify_launch_count() - n0 == 2


def test_tree_grow_feeds_verification_and_mask():
    # the grown tree is a valid input of tree verification and of the mask
    B, D, K, V, M = 4, 6, 8, 128256, 59
    z = synth.make_grow_logits(B=B, D=D, K=K, V=V, seed=7)
    got = _gpu_grow(z, "bf16", 1.0, M)
    par = got["parents"]
    assert (par[:, 0] == -1).all()
    assert ((par[:, 1:] >= 0) & (par[:, 1:] < np.arange(1, M + 1))).all()
    m_o, d_o, bad = oracle.tree_mask(par)
    assert not bad and np.array_equal(d_o, got["depth"])
