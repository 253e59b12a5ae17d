"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and rejects bad host arguments before touching the GPU.

No test here launches a kernel: every call below fails host validation (or is
the B = 0 no-op), which the library performs before any CUDA call.
"""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_56_gb300 as sv
from speculative_decoding_verification_56_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")

FAKE = 0x10000          # 64 KiB-aligned fake device address, never dereferenced
MISALIGNED = FAKE + 2


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("spec_verify_sample", "spec_verify_greedy", "spec_verify_tree_greedy",
              "spec_verify_workspace_bytes", "spec_verify_read_flags",
              "spec_verify_launch_count", "spec_status_string", "spec_verify_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(sv.LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), n


def test_abi_version_and_status_strings(lib):
    assert sv.spec_verify_abi_version() == 1
    assert sv.spec_status_string(0) == "ok"
    assert "workspace" in sv.spec_status_string(3)
    assert sv.spec_verify_launch_count() >= 0


def test_workspace_bytes(lib):
    ws = sv.spec_verify_workspace_bytes
    a = ws(sv.SPEC_MODE_SAMPLE, 64, 4, 128256, sv.SPEC_DTYPE_BF16)
    b = ws(sv.SPEC_MODE_SAMPLE, 128, 4, 128256, sv.SPEC_DTYPE_BF16)
    assert 0 < a < b and a % 256 == 0
    assert ws(sv.SPEC_MODE_GREEDY, 64, 4, 128256, sv.SPEC_DTYPE_BF16) > 0
    assert ws(sv.SPEC_MODE_TREE_GREEDY, 16, 60, 128256, sv.SPEC_DTYPE_BF16) > 0
    assert ws(sv.SPEC_MODE_SAMPLE, 1, 4, 0, sv.SPEC_DTYPE_F32) == 0            # V < 1
    assert ws(sv.SPEC_MODE_SAMPLE, 1, 4, 10, 7) == 0                            # dtype
    assert ws(sv.SPEC_MODE_TREE_GREEDY, 1, 0, 10, 0) == 0                       # N < 1
    assert ws(sv.SPEC_MODE_SAMPLE, 1 << 20, 1024, 1 << 26, 1) == 0              # index space
    assert ws(9, 1, 1, 10, 0) == 0


def _sample(lib, **over):
    a = dict(target=FAKE, draft=FAKE, dtype=0, tokens=FAKE, ua=FAKE, us=FAKE, T=1.0, B=2, k=3,
             V=64, acc=FAKE, out=FAKE, p=FAKE, q=FAKE, R=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return lib.spec_verify_sample(a["target"], a["draft"], a["dtype"], a["tokens"], a["ua"],
                                  a["us"], a["T"], a["B"], a["k"], a["V"], a["acc"], a["out"],
                                  a["p"], a["q"], a["R"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(T=0.0), 1), (dict(T=-1.0), 1), (dict(T=float("nan")), 1), (dict(T=float("inf")), 1),
    (dict(k=-1), 1), (dict(V=0), 1), (dict(dtype=5), 1), (dict(B=-1), 1),
    (dict(k=2000), 1),
    (dict(target=None), 1), (dict(draft=None), 1), (dict(tokens=None), 1), (dict(us=None), 1),
    (dict(acc=None), 1), (dict(p=None), 1), (dict(R=None), 1),
    (dict(target=MISALIGNED), 2), (dict(out=MISALIGNED), 2), (dict(dtype=1, draft=FAKE + 1), 2),
    (dict(ws=None), 3), (dict(wsb=1024), 3), (dict(ws=FAKE + 16), 2),
    (dict(B=0), 0),
])
def test_sample_host_validation(lib, over, status):
    assert _sample(lib, **over) == status


def test_sample_k0_allows_null_draft_arguments(lib):
    # passes the NULL checks and then fails on the workspace size, before CUDA
    assert _sample(lib, k=0, draft=None, tokens=None, ua=None, p=None, q=None, wsb=16) == 3


def test_greedy_and_tree_host_validation(lib):
    g = lib.spec_verify_greedy
    assert g(None, 1, FAKE, 4, 3, 100, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert g(FAKE, 1, None, 4, 3, 100, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert g(FAKE, 1, FAKE, 4, 3, 100, FAKE, FAKE, FAKE, 10, None) == 3
    assert g(FAKE + 1, 1, FAKE, 4, 3, 100, FAKE, FAKE, FAKE, 1 << 30, None) == 2
    assert g(FAKE, 1, FAKE, 0, 3, 100, FAKE, FAKE, FAKE, 0, None) == 0
    t = lib.spec_verify_tree_greedy
    args = [FAKE, 1, FAKE, FAKE, 4, 60, 1000, 6, FAKE, FAKE, FAKE, FAKE, 10, None]
    assert t(*args) == 3
    bad = list(args); bad[5] = 0
    assert t(*bad) == 1
    bad = list(args); bad[7] = -1
    assert t(*bad) == 1
    bad = list(args); bad[7] = 5000
    assert t(*bad) == 1
    bad = list(args); bad[3] = None
    assert t(*bad) == 1
    bad = list(args); bad[3] = FAKE + 2
    assert t(*bad) == 2


def test_noalloc_host_validation(lib):
    f = lib.spec_verify_greedy_noalloc
    assert f(None, 1, FAKE, 4, 3, 100, FAKE, FAKE, None) == 1
    assert f(FAKE, 9, FAKE, 4, 3, 100, FAKE, FAKE, None) == 1
    assert f(FAKE, 1, FAKE, 0, 3, 100, FAKE, FAKE, None) == 0          # B = 0: no work
    assert f(FAKE, 1, FAKE, 4096, 8, 1 << 20, FAKE, FAKE, None) == 5   # beyond the scratch


def test_tree_mask_host_validation(lib):
    f = lib.spec_tree_attention_mask
    assert lib.spec_verify_workspace_bytes(3, 16, 60, 0, 7) == 256   # flag header only
    assert lib.spec_verify_workspace_bytes(3, 16, 0, 0, 0) == 0
    assert lib.spec_verify_workspace_bytes(3, 16, 65537, 0, 0) == 0
    assert f(FAKE, -1, 60, FAKE, FAKE, FAKE, 256, None) == 1
    assert f(FAKE, 4, 0, FAKE, FAKE, FAKE, 256, None) == 1
    assert f(FAKE, 4, 65537, FAKE, FAKE, FAKE, 256, None) == 1
    assert f(None, 4, 60, FAKE, FAKE, FAKE, 256, None) == 1
    assert f(FAKE, 4, 60, None, FAKE, FAKE, 256, None) == 1
    assert f(FAKE + 2, 4, 60, FAKE, FAKE, FAKE, 256, None) == 2
    assert f(FAKE, 4, 60, FAKE, FAKE + 1, FAKE, 256, None) == 2
    assert f(FAKE, 4, 60, FAKE, FAKE, FAKE, 255, None) == 3
    assert f(FAKE, 4, 60, FAKE, FAKE, None, 256, None) == 3
    assert f(FAKE, 4, 60, FAKE, FAKE, FAKE + 16, 256, None) == 2
    assert f(FAKE, 0, 60, FAKE, FAKE, FAKE, 256, None) == 0            # B = 0: no work


def test_kv_commit_host_validation(lib):
    f = lib.spec_kv_commit_path
    ok = [FAKE, 4, 64, 1 << 24, 1 << 20, 2048, 512, 60, FAKE, FAKE, FAKE, 6, FAKE, FAKE, 256, None]

    def call(**kw):
        a = list(ok)
        names = ["cache", "B", "planes", "ps", "ss", "eb", "L", "N", "base", "acc", "path",
                 "md", "nl", "ws", "wsb", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)
    assert lib.spec_verify_workspace_bytes(4, 16, 60, 0, 0) == 256
    assert call(B=-1) == 1 and call(planes=0) == 1 and call(planes=65536) == 1
    assert call(eb=8) == 1 and call(N=0) == 1 and call(md=-1) == 1 and call(md=1025) == 1
    assert call(cache=None) == 1 and call(path=None) == 1 and call(nl=None) == 1
    assert call(cache=FAKE + 8) == 2 and call(eb=2056) == 2 and call(ps=(1 << 24) + 4) == 2
    assert call(base=FAKE + 2) == 2
    assert call(ws=None) == 3 and call(wsb=100) == 3 and call(ws=FAKE + 16) == 2
    assert call(B=0) == 0


def test_read_flags_validation(lib):
    v = ctypes.c_uint32(0)
    assert lib.spec_verify_read_flags(None, ctypes.byref(v), 0, None) == 1
    assert lib.spec_verify_read_flags(FAKE + 8, ctypes.byref(v), 0, None) == 2


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sv.load_library(str(tmp_path / "nope.so"))


def test_product_path_never_touches_the_oracle():
    pkg = os.path.dirname(sv.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "spec_oracle" not in text, f
                assert "libspecoracle" not in text, f


# ---------------------------------------------------------------------------
# EAGLE-2 tree growth and the fused LM head: host validation only
# ---------------------------------------------------------------------------

def _grow(lib, **over):
    a = dict(z=FAKE, dtype=1, T=1.0, B=2, D=3, K=4, V=1000, M=10, tok=FAKE, par=FAKE, dep=FAKE,
             val=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return lib.spec_tree_grow(a["z"], a["dtype"], a["T"], a["B"], a["D"], a["K"], a["V"], a["M"],
                              a["tok"], a["par"], a["dep"], a["val"], a["ws"], a["wsb"],
                              a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(dtype=7), 1), (dict(T=0.0), 1), (dict(T=float("nan")), 1), (dict(T=float("inf")), 1),
    (dict(B=-1), 1), (dict(D=0), 1), (dict(D=17), 1), (dict(K=0), 1), (dict(K=17), 1),
    (dict(V=3, K=4), 1),                                  # fewer tokens than children
    (dict(M=-1), 1), (dict(M=4 + 2 * 16 + 1), 1),         # budget past the tree's nodes
    (dict(K=16, V=3_000_000, dtype=0), 1),                # more than 2048 chunk lists
    (dict(z=0), 1), (dict(tok=0), 1), (dict(par=0), 1), (dict(dep=0), 1), (dict(val=0), 1),
    (dict(z=MISALIGNED, dtype=0), 2), (dict(val=MISALIGNED), 2),
    (dict(ws=0), 3), (dict(wsb=16), 3), (dict(ws=FAKE + 16), 2),
])
def test_tree_grow_rejects_bad_arguments(lib, over, status):
    assert _grow(lib, **over) == status


def test_tree_grow_empty_batch_is_a_no_op(lib):
    assert _grow(lib, B=0, z=0, tok=0, par=0, dep=0, val=0, ws=0, wsb=0) == 0


def test_tree_grow_workspace_grows_with_the_batch(lib):
    ws = sv.spec_verify_workspace_bytes
    a = ws(sv.SPEC_MODE_TREE_GROW, 16, 8, 128256, sv.SPEC_DTYPE_BF16)
    b = ws(sv.SPEC_MODE_TREE_GROW, 32, 8, 128256, sv.SPEC_DTYPE_BF16)
    assert 0 < a < b
    assert ws(sv.SPEC_MODE_TREE_GROW, 16, 17, 128256, sv.SPEC_DTYPE_BF16) == 0


def _lm(lib, **over):
    a = dict(h=FAKE, w=FAKE, tok=FAKE, B=2, k=3, d=64, V=1000, acc=FAKE, out=FAKE, ws=FAKE,
             wsb=1 << 30, stream=None)
    a.update(over)
    return lib.spec_lm_head_verify_greedy(a["h"], a["w"], a["tok"], a["B"], a["k"], a["d"],
                                          a["V"], a["acc"], a["out"], a["ws"], a["wsb"],
                                          a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(B=-1), 1), (dict(k=-1), 1), (dict(d=4), 1), (dict(d=68), 1), (dict(V=0), 1),
    (dict(h=0), 1), (dict(w=0), 1), (dict(acc=0), 1), (dict(out=0), 1), (dict(tok=0), 1),
    (dict(h=FAKE + 8), 2), (dict(w=FAKE + 8), 2), (dict(out=MISALIGNED), 2),
    (dict(ws=0), 3), (dict(wsb=16), 3),
])
def test_lm_head_rejects_bad_arguments(lib, over, status):
    assert _lm(lib, **over) == status


def test_lm_head_empty_batch_is_a_no_op(lib):
    assert _lm(lib, B=0, h=0, w=0, tok=0, acc=0, out=0, ws=0, wsb=0) == 0
