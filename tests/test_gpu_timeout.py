"""The bounded-wait path on the GPU.

Every wait of the verification kernels on their own bulk copies gives up
after a limit; the CTA then raises SPEC_FLAG_TIMEOUT, stops copying, waits
(with the default limit) for the copies it has in flight and finishes its
control flow.  Here the limit is set to 1 ns, which gives up whenever a copy
has not landed at the first look (the first copies of every CTA have not:
they were issued a few hundred ns earlier): the call must return, raise the
flag, and leave the context usable, with the next call (default limit)
matching the oracle again.  Nothing here faults or hangs the GPU: the copies
still land, and only the waits on them are cut short.
"""
import numpy as np
import pytest
import torch

import oracle
import parity_helpers as ph
import speculative_decoding_verification_56_gb300 as sv
from speculative_decoding_verification_56_gb300 import build, synth

pytestmark = pytest.mark.gpu

SHORT_NS = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()
    sv.load_library()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _inputs(c):
    return (sv.to_device_logits(c.target, c.dtype), sv.to_device_logits(c.draft, c.dtype),
            torch.from_numpy(c.tokens).cuda(), torch.from_numpy(c.u_accept).cuda(),
            torch.from_numpy(c.u_sample).cuda())


def _with_short_limit(fn):
    # evict the inputs from L2 first (a write larger than its 129 MB), so that
    # the first copies of every CTA come from HBM and cannot have landed when
    # the consumers first look
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush.fill_(1)
    sv.spec_verify_set_wait_limit_ns(SHORT_NS)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        sv.spec_verify_set_wait_limit_ns(0)
    return out


def test_sampling_timeout_sets_flag_and_next_call_matches():
    c = synth.zipf128k(seed=2)
    t, d, tok, ua, us = _inputs(c)
    ws = sv.alloc_workspace(sv.SPEC_MODE_SAMPLE, c.B, c.k, c.V, sv.SPEC_DTYPE_BF16)
    sv.spec_verify_read_flags(ws)                        # start from a clear flag word
    _with_short_limit(lambda: sv.verify_sample(t, d, tok, ua, us, c.temperature, workspace=ws))
    assert sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_TIMEOUT
    out = sv.verify_sample(t, d, tok, ua, us, c.temperature, workspace=ws)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    assert not sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_TIMEOUT
    o = oracle.verify_sample(c.target, c.draft, c.tokens, c.u_accept, c.u_sample, c.temperature,
                             dtype=c.dtype)
    ph.compare_sample(g, o, case=c)


def test_greedy_and_tree_timeout_set_flag_and_next_calls_match():
    c = synth.zipf128k(seed=3, greedy=True)
    t, _, tok, _, _ = _inputs(c)
    ws = sv.alloc_workspace(sv.SPEC_MODE_GREEDY, c.B, c.k, c.V, sv.SPEC_DTYPE_BF16)
    sv.spec_verify_read_flags(ws)
    _with_short_limit(lambda: sv.verify_greedy(t, tok, workspace=ws))
    assert sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_TIMEOUT
    out = sv.verify_greedy(t, tok, workspace=ws)
    o = oracle.verify_greedy(c.target, c.tokens, dtype=c.dtype)
    ph.compare_exact({k: v.cpu().numpy() for k, v in out.items()}, o,
                     ["accepted_len", "out_tokens"])
    assert not sv.spec_verify_read_flags(ws) & sv.SPEC_FLAG_TIMEOUT

    tr = synth.tree(seed=4)
    tt = sv.to_device_logits(tr.target, tr.dtype)
    ttok, tpar = torch.from_numpy(tr.tokens).cuda(), torch.from_numpy(tr.parents).cuda()
    wst = sv.alloc_workspace(sv.SPEC_MODE_TREE_GREEDY, tr.B, tr.N, tr.V, sv.SPEC_DTYPE_BF16)
    sv.spec_verify_read_flags(wst)
    _with_short_limit(lambda: sv.verify_tree_greedy(tt, ttok, tpar, tr.max_depth, workspace=wst))
    assert sv.spec_verify_read_flags(wst) & sv.SPEC_FLAG_TIMEOUT
    out = sv.verify_tree_greedy(tt, ttok, tpar, tr.max_depth, workspace=wst)
    o = oracle.verify_tree_greedy(tr.target, tr.tokens, tr.parents, tr.max_depth, dtype=tr.dtype)
    ph.compare_exact({k: v.cpu().numpy() for k, v in out.items()}, o,
                     ["accepted_len", "path_nodes", "out_tokens"])
