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
