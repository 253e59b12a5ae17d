"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.  Rules and tolerances: parity_helpers.py."""
import numpy as np
import pytest
import torch

import oracle
import parity_helpers as ph
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
# helpers
# ---------------------------------------------------------------------------

def dev_chain(c):
    t = sv.to_device_logits(c.target, c.dtype)
    d = sv.to_device_logits(c.draft, c.dtype) if c.draft is not None else None
    return dict(t=t, d=d, tok=torch.from_numpy(np.ascontiguousarray(c.tokens)).cuda(),
                ua=torch.from_numpy(np.ascontiguousarray(c.u_accept)).cuda(),
                us=torch.from_numpy(np.ascontiguousarray(c.u_sample)).cuda())


def gpu_sample(c, ws=None, stream=None):
    x = dev_chain(c)
    out = sv.verify_sample(x["t"], x["d"], x["tok"], x["ua"], x["us"], c.temperature,
                           workspace=ws, stream=stream)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def gpu_greedy(c, ws=None):
    x = dev_chain(c)
    out = sv.verify_greedy(x["t"], x["tok"], workspace=ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def gpu_tree(t, max_depth=None, ws=None):
    md = t.max_depth if max_depth is None else max_depth
    out = sv.verify_tree_greedy(sv.to_device_logits(t.target, t.dtype),
                                torch.from_numpy(t.tokens).cuda(),
                                torch.from_numpy(t.parents).cuda(), md, workspace=ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def oracle_sample(c, rows=None):
    s = slice(None) if rows is None else rows
    return oracle.verify_sample(c.target[s], None if c.draft is None else c.draft[s],
                                c.tokens[s], c.u_accept[s], c.u_sample[s], c.temperature,
                                dtype=c.dtype)


def sample_parity(c, rows=None, allow_flags=None, ws=None):
    g = gpu_sample(c, ws=ws)
    o = oracle_sample(c, rows)
    return ph.compare_sample(g, o, rows=rows, allow_flags=allow_flags, case=c), g, o


# ---------------------------------------------------------------------------
# the named workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
def test_sample_tiny(seed):
    s, _, _ = sample_parity(synth.tiny(seed))
    assert s["flagged"] == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_sample_peaked(seed):
    sample_parity(synth.peaked(seed))


def test_sample_zipf128k_full():
    c = synth.zipf128k(seed=0)
    s, g, o = sample_parity(c)
    assert s["rows"] == 64
    # both outcomes of the accept test occur in this workload
    assert 0 < (g["accepted_len"] < c.k).sum() < c.B


def test_sample_zipf152k_full():
    # every one of the 256 sequences (3840 rows of 151936 logits) against the
    # float64 oracle
    c = synth.zipf152k(seed=0)
    s, g, _ = sample_parity(c)
    assert s["rows"] == c.B
    # properties that hold at any size
    n = g["accepted_len"]
    assert ((n >= 0) & (n <= c.k)).all()
    for b in range(c.B):
        assert (g["out_tokens"][b, :n[b]] == c.tokens[b, :n[b]]).all()
        assert 0 <= g["out_tokens"][b, n[b]] < c.V
        assert (g["out_tokens"][b, n[b] + 1:] == -1).all()
    assert np.isfinite(g["p"]).all() and (g["p"] >= 0).all() and (g["p"] <= 1).all()


def test_greedy_zipf128k_full():
    c = synth.zipf128k(seed=0, greedy=True)
    g = gpu_greedy(c)
    o = oracle.verify_greedy(c.target, c.tokens, dtype=c.dtype)
    ph.compare_exact(g, o, ["accepted_len", "out_tokens"])
    assert 0 < (g["accepted_len"] < c.k).sum() < c.B


def test_tree_full():
    t = synth.tree(seed=0)
    g = gpu_tree(t)
    o = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth, dtype=t.dtype)
    ph.compare_exact(g, o, ["accepted_len", "path_nodes", "out_tokens"])
    assert g["accepted_len"].max() >= 2


def test_sample_flag_rate_many_rows():
    c = synth.make_chain_case(B=20000, k=4, V=96, dtype="f32", temperature=1.0,
                              target_sigma=1.5, draft_noise=0.7, seed=11)
    s, _, _ = sample_parity(c)
    # the flagged count stays within the Poisson bound of the exact law's
    # own expectation (about 2.9 of these 20000 rows)
    assert s["flagged"] <= s["flag_allowance"]


# ---------------------------------------------------------------------------
# ragged, degenerate and boundary shapes
# ---------------------------------------------------------------------------

SHAPES = [  # dtype, V, B, k, T
    ("bf16", 1001, 3, 3, 1.0),        # scalar path (row bytes not a multiple of 16)
    ("f32", 17, 5, 2, 0.5),
    ("f32", 1, 4, 3, 1.0),            # one-token vocabulary: everything accepted
    ("bf16", 2 * 8192 + 8, 2, 4, 1.3),  # vector path, last chunk holds one vector
    ("f32", 3 * 4096 + 3, 2, 2, 0.9),   # scalar path over four chunks
    ("bf16", 8, 7, 1, 1.0),
    ("bf16", 5000, 10, 0, 1.0),       # k = 0: plain sampling from row 0
    ("f32", 300, 3, 0, 0.7),
    ("bf16", 40000, 1, 9, 2.0),
    ("bf16", 300000, 3, 2, 1.0),      # rows of 19 chunks: the two-kernel draw path
    ("f32", 140003, 2, 2, 0.8),       # scalar loads, 18 chunks, two-kernel draw path
    ("bf16", 16 * 16384, 2, 3, 1.0),  # exactly 16 chunks: the largest cluster draw
]


@pytest.mark.parametrize("dtype,V,B,k,T", SHAPES)
def test_sample_shapes(dtype, V, B, k, T):
    # large vocabularies use the peaked Zipf recipe of the real workloads: with
    # flat logits the CDF steps (~1/V) approach the 1e-6 flag window and most
    # rows would be flagged rather than compared
    recipe, sigma = ("zipf", 3.0) if V >= 100000 else ("gauss", 2.0)
    c = synth.make_chain_case(B=B, k=k, V=V, dtype=dtype, temperature=T, recipe=recipe,
                              target_sigma=sigma, draft_noise=1.0, seed=V + B + k)
    s, g, _ = sample_parity(c)
    if V == 1:
        assert (g["accepted_len"] == k).all() and (g["out_tokens"][:, k] == 0).all()


@pytest.mark.parametrize("dtype,V,B,k", [("bf16", 3 * 8192 + 100, 6, 3), ("f32", 17, 9, 4),
                                         ("bf16", 1001, 5, 0), ("f32", 4096, 4, 2)])
def test_greedy_ties_and_shapes(dtype, V, B, k):
    rng = np.random.default_rng(V)
    zt = rng.integers(-2, 3, size=(B, k + 1, V)).astype(np.float32)   # many ties
    stored = synth.f32_to_bf16_bits(zt) if dtype == "bf16" else zt
    g_ref = np.argmax(zt, axis=-1)
    toks = np.where(rng.random((B, k)) < 0.8, g_ref[:, :k], rng.integers(0, V, (B, k)))
    c = synth.ChainInputs("ties", B, k, V, dtype, 1.0, stored, None, toks.astype(np.int32),
                          np.zeros((B, k), np.float32), np.zeros(B, np.float32))
    g = gpu_greedy(c)
    o = oracle.verify_greedy(stored, c.tokens, dtype=dtype)
    ph.compare_exact(g, o, ["accepted_len", "out_tokens"])


def test_sample_identical_rows_accept_all():
    c = synth.make_chain_case(B=32, k=5, V=3000, dtype="bf16", seed=2)
    c.draft = c.target[:, :5].copy()
    s, g, _ = sample_parity(c, allow_flags=0)
    assert (g["accepted_len"] == 5).all() and (g["resid_mass"] == 0).all()


@pytest.mark.parametrize("V", [37, 40])   # plain loads; bulk copies (the one-kernel path)
def test_sample_zero_probabilities_and_fallback(V):
    base = np.random.default_rng(0).standard_normal((3, 3, V)).astype(np.float32)
    zt = base.copy()
    zd = base[:, :2].copy()
    zt[0, 0, 2] = -5000.0                      # seq 0: p(x_0) = 0 -> reject at 0
    zd[1, 1, 4] = -5000.0                      # seq 1: q(x_1) = 0 -> accept at 1
    zt[2, 0, 6] = -5000.0                      # seq 2: identical rows, p = q = 0 at x_0
    zd[2, 0] = zt[2, 0]
    toks = np.array([[2, 0], [1, 4], [6, 1]], np.int32)
    ua = np.array([[0.0, 0.5], [0.0, 0.99999994], [0.0, 0.0]], np.float32)
    us = np.array([0.3, 0.6, 0.8], np.float32)
    c = synth.ChainInputs("zero", 3, 2, V, "f32", 1.0, zt, zd, toks, ua, us)
    x = dev_chain(c)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, 3, 2, V, sv.SPEC_DTYPE_F32)
    out = sv.verify_sample(x["t"], x["d"], x["tok"], x["ua"], x["us"], 1.0, workspace=ws)
    flags = sv.spec_verify_read_flags(ws)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    o = oracle_sample(c)
    ph.compare_sample(g, o, allow_flags=0, case=c)
    assert g["accepted_len"][0] == 0 and g["accepted_len"][1] == 2
    assert o["fallback"][2] == 1 and flags & sv.SPEC_FLAG_RESIDUAL_FALLBACK


def test_sample_invalid_token_sets_flag():
    c = synth.make_chain_case(B=4, k=3, V=500, dtype="f32", seed=5)
    c.tokens[1, 1] = 500
    c.tokens[2, 0] = -3
    x = dev_chain(c)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, 4, 3, 500, sv.SPEC_DTYPE_F32)
    out = sv.verify_sample(x["t"], x["d"], x["tok"], x["ua"], x["us"], 1.0, workspace=ws)
    assert sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_TOKEN_RANGE
    assert sv.spec_verify_read_flags(ws) == 0            # cleared by the first read
    n = out["accepted_len"].cpu().numpy()
    assert n[2] == 0                                       # invalid token is rejected
    ok = np.array([0, 3])
    o = oracle.verify_sample(c.target[ok], c.draft[ok], c.tokens[ok], c.u_accept[ok],
                             c.u_sample[ok], 1.0)
    ph.compare_sample({k: v.cpu().numpy() for k, v in out.items()}, o, rows=ok, allow_flags=0,
                      case=c)


# ---------------------------------------------------------------------------
# trees
# ---------------------------------------------------------------------------

def test_tree_root_only_and_shapes():
    t = synth.make_tree_case(B=5, N=1, V=700, dtype="f32", seed=1)
    g = gpu_tree(t, max_depth=3)
    o = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, 3, dtype="f32")
    ph.compare_exact(g, o, ["accepted_len", "path_nodes", "out_tokens"])
    assert (g["accepted_len"] == 0).all()


@pytest.mark.parametrize("seed,N,V,depth,dtype", [(1, 12, 33, 4, "f32"), (2, 300, 2000, 9, "bf16"),
                                                 (3, 60, 8192 + 8, 6, "bf16")])
def test_tree_random(seed, N, V, depth, dtype):
    t = synth.make_tree_case(B=7, N=N, V=V, dtype=dtype, max_depth=depth, p_match=0.8,
                             seed=seed)
    g = gpu_tree(t)
    o = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, depth, dtype=dtype)
    ph.compare_exact(g, o, ["accepted_len", "path_nodes", "out_tokens"])


@pytest.mark.parametrize("dtype,V,noise", [("f32", 300, 0.0), ("bf16", 1000, 0.05)])
def test_sample_longest_draft(dtype, V, noise):
    # k at the interface's limit (256 drafts, 513 rows per sequence); with no
    # draft noise every draft is accepted and the bonus comes from row 256
    k = 256
    c = synth.make_chain_case(B=2, k=k, V=V, dtype=dtype, target_sigma=1.0, draft_noise=noise,
                              seed=31)
    s, g, _ = sample_parity(c, allow_flags=1)
    if noise == 0.0:
        assert (g["accepted_len"] == k).all()


def test_greedy_longest_draft():
    k = 256
    c = synth.make_chain_case(B=3, k=k, V=500, dtype="bf16", greedy_force=0.995, seed=32)
    g = gpu_greedy(c)
    o = oracle.verify_greedy(c.target, c.tokens, dtype="bf16")
    ph.compare_exact(g, o, ["accepted_len", "out_tokens"])
    assert g["accepted_len"].max() > 32


def test_tree_large_and_deep():
    # 3000 nodes (more than the resolve kernel keeps in shared memory: its
    # global-memory path) and paths hundreds of levels deep under the
    # interface's depth limit; most tokens follow the parent's argmax
    rng = np.random.default_rng(33)
    B, N, V, max_depth = 2, 3000, 64, 1024
    target = synth.make_tree_case(B=B, N=N, V=V, dtype="f32", seed=33).target
    g_arg = np.argmax(target, axis=-1)
    par = np.full((B, N), -1, np.int32)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        depth = np.zeros(N, np.int64)
        for v in range(1, N):
            while True:
                p = v - 1 if rng.random() < 0.7 else int(rng.integers(max(0, v - 40), v))
                if depth[p] < max_depth:
                    break
            par[b, v] = p
            depth[v] = depth[p] + 1
            tok[b, v] = g_arg[b, p] if rng.random() < 0.995 else int(rng.integers(0, V))
    t = synth.TreeInputs("deep", B, N, V, "f32", max_depth, target, tok, par)
    g = gpu_tree(t)
    o = oracle.verify_tree_greedy(target, tok, par, max_depth, dtype="f32")
    ph.compare_exact(g, o, ["accepted_len", "path_nodes", "out_tokens"])
    assert g["accepted_len"].max() > 100


def test_chain_tree_matches_gpu_greedy():
    c = synth.make_chain_case(B=20, k=6, V=5000, dtype="bf16", greedy_force=0.85, seed=4)
    par = np.tile(np.arange(-1, c.k, dtype=np.int32), (c.B, 1))
    tok = np.concatenate([np.zeros((c.B, 1), np.int32), c.tokens], axis=1)
    t = synth.TreeInputs("chain", c.B, c.k + 1, c.V, "bf16", c.k, c.target, tok, par)
    gt = gpu_tree(t)
    gg = gpu_greedy(c)
    assert (gt["accepted_len"] == gg["accepted_len"]).all()
    assert (gt["out_tokens"] == gg["out_tokens"]).all()


def test_tree_bad_parent_and_depth_flags():
    t = synth.make_tree_case(B=2, N=10, V=100, dtype="f32", max_depth=3, seed=8)
    t.parents[0, 5] = 7                      # parent after the child
    ws = sv.alloc_workspace(sv.SPEC_MODE_TREE_GREEDY, 2, 10, 100, sv.SPEC_DTYPE_F32)
    gpu_tree(t, max_depth=3, ws=ws)
    assert sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_BAD_PARENT
    t2 = synth.make_tree_case(B=2, N=10, V=100, dtype="f32", max_depth=5, seed=8,
                              parents=np.array([-1, 0, 1, 2, 3, 4, 0, 1, 2, 3]))
    gpu_tree(t2, max_depth=2, ws=ws)         # nodes 3.. are deeper than 2
    assert sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_DEPTH


# ---------------------------------------------------------------------------
# workspace reuse, determinism, streams, launch counting
# ---------------------------------------------------------------------------

def test_workspace_reuse_across_shapes_and_modes():
    big = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, 64, 4, 128256, sv.SPEC_DTYPE_BF16)
    c1 = synth.make_chain_case(B=9, k=2, V=20000, dtype="bf16", seed=1)
    c2 = synth.make_chain_case(B=3, k=6, V=777, dtype="f32", seed=2)
    t = synth.make_tree_case(B=4, N=30, V=9000, dtype="bf16", seed=3)
    for _ in range(2):
        sample_parity(c1, ws=big)
        sample_parity(c2, ws=big, allow_flags=0)
        g = gpu_tree(t, ws=big)
        o = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth, dtype="bf16")
        ph.compare_exact(g, o, ["accepted_len", "path_nodes", "out_tokens"])
        gg = gpu_greedy(c1, ws=big)
        og = oracle.verify_greedy(c1.target, c1.tokens, dtype="bf16")
        ph.compare_exact(gg, og, ["accepted_len", "out_tokens"])
    # garbage left in the workspace by other shapes does not leak into results
    big[256:].fill_(0xA5)
    sample_parity(c2, ws=big, allow_flags=0)


def test_inputs_written_by_the_kernel_just_before():
    # The first kernel of every call is a programmatic dependent launch: it
    # must see everything the preceding kernel in the stream wrote.  Here a
    # torch kernel writes the logits (and an extra one the draft tokens) right
    # before each call, with no synchronisation in between.
    c = synth.zipf128k(seed=4)
    o = oracle_sample(c)
    x = dev_chain(c)
    t_src, d_src, tok_src = x["t"], x["d"], x["tok"]
    t = torch.zeros_like(t_src)
    d = torch.zeros_like(d_src)
    tok = torch.zeros_like(tok_src)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, c.B, c.k, c.V, sv.SPEC_DTYPE_BF16)
    torch.cuda.synchronize()
    for _ in range(2):
        d.copy_(d_src)
        tok.copy_(tok_src)
        t.zero_()
        torch.add(t_src, 0, out=t)             # the kernel right before the call
        out = sv.verify_sample(t, d, tok, x["ua"], x["us"], c.temperature, workspace=ws)
        g = {k: v.cpu().numpy() for k, v in out.items()}
        ph.compare_sample(g, o, case=c)
        t.zero_()
        d.zero_()
        tok.zero_()
    cg = synth.greedy_variant(c, 0.7)
    og = oracle.verify_greedy(cg.target, cg.tokens, dtype=cg.dtype)
    gt = torch.from_numpy(cg.tokens).cuda()
    for _ in range(2):
        t.zero_()
        torch.add(t_src, 0, out=t)
        out = sv.verify_greedy(t, gt, workspace=ws)
        ph.compare_exact({k: v.cpu().numpy() for k, v in out.items()}, og,
                         ["accepted_len", "out_tokens"])


def test_back_to_back_calls_share_a_workspace():
    # The argmax streaming kernel reads its logits before waiting for the
    # call before it on the stream (the previous call's resolve kernel, which
    # reads the same workspace's records); its first record write must still
    # come after that kernel.  Greedy and tree calls on alternating inputs,
    # one workspace, one stream, no synchronisation until the end.
    c1 = synth.greedy_variant(synth.zipf128k(seed=7, B=16), 0.7)
    c2 = synth.greedy_variant(synth.zipf128k(seed=8, B=16), 0.5)
    t = synth.make_tree_case(B=8, N=40, V=128256, dtype="bf16", seed=9)
    nbytes = max(sv.spec_verify_workspace_bytes(sv.SPEC_MODE_GREEDY, 16, 4, 128256, sv.SPEC_DTYPE_BF16),
                 sv.spec_verify_workspace_bytes(sv.SPEC_MODE_TREE_GREEDY, 8, 40, 128256,
                                                sv.SPEC_DTYPE_BF16))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    xs = [(sv.to_device_logits(c.target, c.dtype), torch.from_numpy(c.tokens).cuda()) for c in (c1, c2)]
    tt = sv.to_device_logits(t.target, t.dtype)
    ttok, tpar = torch.from_numpy(t.tokens).cuda(), torch.from_numpy(t.parents).cuda()
    torch.cuda.synchronize()
    outs = []
    for i in range(6):
        outs.append(("g", i % 2, sv.verify_greedy(xs[i % 2][0], xs[i % 2][1], workspace=ws)))
        outs.append(("t", 0, sv.verify_tree_greedy(tt, ttok, tpar, t.max_depth, workspace=ws)))
    torch.cuda.synchronize()
    og = [oracle.verify_greedy(c.target, c.tokens, dtype=c.dtype) for c in (c1, c2)]
    ot = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth, dtype="bf16")
    for kind, j, out in outs:
        g = {k: v.cpu().numpy() for k, v in out.items()}
        if kind == "g":
            ph.compare_exact(g, og[j], ["accepted_len", "out_tokens"])
        else:
            ph.compare_exact(g, ot, ["accepted_len", "path_nodes", "out_tokens"])


def test_three_calls_on_three_streams():
    # the benchmark step's layout: sampling, greedy and tree calls forked onto
    # three streams, one workspace each, running at the same time
    c = synth.zipf128k(seed=5)
    cg = synth.greedy_variant(c, 0.7)
    t = synth.tree(seed=5)
    o = oracle_sample(c)
    og = oracle.verify_greedy(cg.target, cg.tokens, dtype=cg.dtype)
    ot = oracle.verify_tree_greedy(t.target, t.tokens, t.parents, t.max_depth, dtype=t.dtype)
    x = dev_chain(c)
    gt = torch.from_numpy(cg.tokens).cuda()
    tt = sv.to_device_logits(t.target, t.dtype)
    ttok, tpar = torch.from_numpy(t.tokens).cuda(), torch.from_numpy(t.parents).cuda()
    ws = {m: sv.alloc_workspace(m, Bm, km, c.V, sv.SPEC_DTYPE_BF16)
          for m, Bm, km in ((sv.SPEC_MODE_SAMPLE, c.B, c.k), (sv.SPEC_MODE_GREEDY, c.B, c.k),
                            (sv.SPEC_MODE_TREE_GREEDY, t.B, t.N))}
    streams = [torch.cuda.Stream() for _ in range(3)]
    torch.cuda.synchronize()
    for _ in range(3):
        fork = torch.cuda.Event()
        fork.record(torch.cuda.current_stream())
        for st in streams:
            st.wait_event(fork)
        gs = sv.verify_sample(x["t"], x["d"], x["tok"], x["ua"], x["us"], c.temperature,
                              workspace=ws[sv.SPEC_MODE_SAMPLE], stream=streams[0])
        gg = sv.verify_greedy(x["t"], gt, workspace=ws[sv.SPEC_MODE_GREEDY], stream=streams[1])
        gtr = sv.verify_tree_greedy(tt, ttok, tpar, t.max_depth,
                                    workspace=ws[sv.SPEC_MODE_TREE_GREEDY], stream=streams[2])
        torch.cuda.synchronize()
        ph.compare_sample({k: v.cpu().numpy() for k, v in gs.items()}, o, case=c)
        ph.compare_exact({k: v.cpu().numpy() for k, v in gg.items()}, og,
                         ["accepted_len", "out_tokens"])
        ph.compare_exact({k: v.cpu().numpy() for k, v in gtr.items()}, ot,
                         ["accepted_len", "path_nodes", "out_tokens"])


def test_deterministic_and_side_stream():
    c = synth.make_chain_case(B=16, k=4, V=50000, dtype="bf16", seed=6)
    a = gpu_sample(c)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = gpu_sample(c, stream=s)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_exp2_fma_accuracy():
    """The FMA-pipe 2^x against float64 exp2 and against the SFU's ex2."""
    x = np.concatenate([np.linspace(-126.0, 0.5, 200001), -np.abs(np.random.default_rng(0)
                        .standard_normal(100000)) * 8]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    yf = torch.empty_like(xd)
    ys = torch.empty_like(xd)
    lib = sv.load_library()
    assert lib.spec_verify_selftest_exp2(xd.data_ptr(), yf.data_ptr(), ys.data_ptr(), x.size,
                                         None) == 0
    torch.cuda.synchronize()
    ref = np.exp2(x.astype(np.float64))
    rel_f = np.abs(yf.cpu().numpy() / ref - 1)
    rel_s = np.abs(ys.cpu().numpy() / ref - 1)
    assert rel_f.max() < 2.5e-7, rel_f.max()
    assert rel_s.max() < 5e-7, rel_s.max()


def test_launch_count():
    # statistics + clustered finish for sampling; argmax + resolve for greedy,
    # on the bulk-copy path (rows of whole 16-byte vectors) and the other
    for V, n_sample in ((100, 2), (101, 2)):
        c = synth.make_chain_case(B=2, k=2, V=V, dtype="f32", seed=0)
        n0 = sv.spec_verify_launch_count()
        gpu_sample(c)
        assert sv.spec_verify_launch_count() - n0 == n_sample
        gpu_greedy(c)
        assert sv.spec_verify_launch_count() - n0 == n_sample + 2
