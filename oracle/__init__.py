"""Float64 CPU oracle for batched draft-token verification (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  The product path (the CUDA library and its binding) never
does.  The arithmetic lives in ``spec_oracle.c`` (plain loops, float64); this
module compiles it with gcc and marshals numpy arrays to it.

Functions and the passages they follow:

* :func:`verify_sample` -- rejection-sampling verification: "EAGLE-3
  speculative decoding review", sections "Speculative Decoding" (step 3, Accept
  or Reject) and "Does Using a Small Model's Answer Reduce Quality?" (eqs.
  A(x), p_residual); "EAGLE math", section "Vanilla speculative decoding";
  "Speculative decoding" wiki, section "The mechanism".
* :func:`verify_greedy` -- greedy verification: review page, "Does Using a
  Small Model's Answer Reduce Quality?" (greedy bullets).
* :func:`verify_tree_greedy` -- draft-tree greedy walk: review page, "EAGLE-2"
  and "The Complete EAGLE-3 Inference Process" (steps 3-4); "EAGLE math",
  "EAGLE-2: dynamic draft trees".
* :func:`expected_tokens`, :func:`speedup_model` -- "EAGLE math", sections
  "Vanilla speculative decoding" (E formula) and "The speedup math, worked".

Every function is pinned by tests against values that do not come from the
oracle itself (the worked example printed on the "EAGLE math" page, exact
enumeration of the emitted-token law, chi-square tests, the expected-length
closed form, brute-force tree search).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libspecoracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", 1: "invalid argument", 2: "non-finite logit", 3: "token out of range",
          4: "malformed tree", 5: "out of memory"}


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_verify_sample.argtypes = [P, P, I, P, P, P, D, I, I, I,
                                         P, P, P, P, P, P, P, P, D, P]
    lib.oracle_verify_sample.restype = I
    lib.oracle_sample_claim.argtypes = [P, P, I, P, P, P, D, I, I, I, P, P, P, P]
    lib.oracle_sample_claim.restype = I
    lib.oracle_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P]
    lib.oracle_verify_greedy.restype = I
    lib.oracle_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P]
    lib.oracle_verify_tree_greedy.restype = I
    lib.oracle_tree_mask.argtypes = [P, I, I, P, P]
    lib.oracle_tree_mask.restype = I
    LL = ctypes.c_longlong
    lib.oracle_kv_commit.argtypes = [P, P, ctypes.c_size_t, I, I, LL, LL, I, I, I, P, P, P, I, P]
    lib.oracle_kv_commit.restype = I
    lib.oracle_lm_head_greedy.argtypes = [P, P, P, I, I, I, I, P, I, P, P, P, P, P]
    lib.oracle_lm_head_greedy.restype = I
    lib.oracle_tree_grow.argtypes = [P, I, I, I, I, I, D, I, P, P, P, P, P]
    lib.oracle_tree_grow.restype = I
    lib.oracle_expected_tokens.argtypes = [D, I]
    lib.oracle_expected_tokens.restype = D
    lib.oracle_speedup_model.argtypes = [D, I, D]
    lib.oracle_speedup_model.restype = D
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def load_variant(lib_path):
    """Bind another compiled copy of the oracle source (used by the tests that
    plant mistakes in the oracle to show the pins catch them)."""
    return _bind(ctypes.CDLL(lib_path))


def _dtype_code(dtype: str) -> int:
    return {"f32": 0, "bf16": 1, "f64": 2}[dtype]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _logits(a, dtype):
    want = {"bf16": np.uint16, "f32": np.float32, "f64": np.float64}[dtype]
    return np.ascontiguousarray(a, dtype=want)


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        raise OracleError(f"oracle error {rc}: {ERRORS.get(rc, '?')}")


FLAG_WINDOW = 1e-6


def verify_sample(target, draft, tokens, u_accept, u_sample, temperature, dtype="f32", lib=None,
                  window=FLAG_WINDOW):
    """Sampling verification over a batch.  Returns a dict of numpy arrays.

    target [B, k+1, V], draft [B, k, V] (float32, or uint16 bf16 bits);
    tokens int32 [B, k]; u_accept float32 [B, k]; u_sample float32 [B].
    Besides the outputs of the method, the dict holds the diagnostics
    ``acc_margin``, ``cdf_margin`` (distance of the uniforms to the nearest
    decision boundary), ``fallback`` (reading R6 applied) and ``flag_prob``
    (chance that fresh uniforms put a margin below ``window``).
    """
    lib = lib or _load()
    target = _logits(target, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    draft = _logits(draft if draft is not None else np.zeros((B, 0, V)), dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, k)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    out = dict(
        accepted_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, k + 1), np.int32),
        p=np.zeros((B, k), np.float64),
        q=np.zeros((B, k), np.float64),
        resid_mass=np.zeros(B, np.float64),
        acc_margin=np.zeros(B, np.float64),
        cdf_margin=np.zeros(B, np.float64),
        fallback=np.zeros(B, np.int32),
        flag_prob=np.zeros(B, np.float64),
    )
    rc = lib.oracle_verify_sample(
        _ptr(target), _ptr(draft), _dtype_code(dtype), _ptr(tokens), _ptr(u_accept),
        _ptr(u_sample), float(temperature), B, k, V,
        _ptr(out["accepted_len"]), _ptr(out["out_tokens"]), _ptr(out["p"]), _ptr(out["q"]),
        _ptr(out["resid_mass"]), _ptr(out["acc_margin"]), _ptr(out["cdf_margin"]),
        _ptr(out["fallback"]), float(window), _ptr(out["flag_prob"]))
    _check(rc)
    return out


def sample_claim(target, draft, tokens, u_accept, u_sample, temperature, claim_len, claim_tok,
                 dtype="f32", lib=None):
    """How far a claimed outcome (accepted length, token drawn at that
    position) of sampling verification is from the exact float64 outcome:
    returns ``(violation, claim_R)`` per sequence.  ``violation`` is 0 for the
    exact outcome, +inf for an outcome no rounding can produce, else the
    largest distance of a uniform to the boundary the claim puts it across
    (acceptance scale, or CDF scale divided by R).  ``claim_R`` is the residual
    mass of the claimed distribution (0 for the bonus draw)."""
    lib = lib or _load()
    target = _logits(target, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    draft = _logits(draft if draft is not None else np.zeros((B, 0, V)), dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, k)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    cl = np.ascontiguousarray(claim_len, dtype=np.int32).reshape(B)
    ct = np.ascontiguousarray(claim_tok, dtype=np.int32).reshape(B)
    viol = np.zeros(B, np.float64)
    cR = np.zeros(B, np.float64)
    rc = lib.oracle_sample_claim(
        _ptr(target), _ptr(draft), _dtype_code(dtype), _ptr(tokens), _ptr(u_accept),
        _ptr(u_sample), float(temperature), B, k, V, _ptr(cl), _ptr(ct), _ptr(viol), _ptr(cR))
    _check(rc)
    return viol, cR


def verify_greedy(target, tokens, dtype="f32", lib=None):
    lib = lib or _load()
    target = _logits(target, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    out = dict(accepted_len=np.zeros(B, np.int32),
               out_tokens=np.zeros((B, k + 1), np.int32),
               argmax=np.zeros((B, k + 1), np.int32))
    rc = lib.oracle_verify_greedy(_ptr(target), _dtype_code(dtype), _ptr(tokens), B, k, V,
                                  _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
                                  _ptr(out["argmax"]))
    _check(rc)
    return out


def verify_tree_greedy(target, tokens, parents, max_depth, dtype="bf16", lib=None):
    lib = lib or _load()
    target = _logits(target, dtype)
    B, N, V = target.shape
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    parents = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    W = max_depth + 1
    out = dict(accepted_len=np.zeros(B, np.int32),
               path_nodes=np.zeros((B, W), np.int32),
               out_tokens=np.zeros((B, W), np.int32))
    rc = lib.oracle_verify_tree_greedy(_ptr(target), _dtype_code(dtype), _ptr(tokens),
                                       _ptr(parents), B, N, V, int(max_depth),
                                       _ptr(out["accepted_len"]), _ptr(out["path_nodes"]),
                                       _ptr(out["out_tokens"]))
    _check(rc)
    return out


def tree_mask(parents, lib=None):
    """Tree attention mask (reading R9 of spec_oracle.c): returns
    ``(mask, depth, malformed)`` with mask uint32 [B, N, ceil(N/32)] (node u
    of row v is bit u % 32 of word u // 32), depth int32 [B, N] and whether
    some chain met an invalid parent."""
    lib = lib or _load()
    par = np.ascontiguousarray(parents, dtype=np.int32)
    B, N = par.shape
    W = (N + 31) // 32
    mask = np.zeros((B, N, W), dtype=np.uint32)
    depth = np.zeros((B, N), dtype=np.int32)
    rc = lib.oracle_tree_mask(_ptr(par), B, N, _ptr(mask), _ptr(depth))
    if rc not in (0, 4):
        _check(rc)
    return mask, depth, rc == 4


def kv_commit(cache, base_len, accepted_len, path_nodes, N, lib=None):
    """KV commit of the accepted path (reading R10 of spec_oracle.c), out of
    place.  ``cache``: array [planes, B, L, E] of any dtype (E elements per
    entry).  Returns ``(new_cache, new_len, malformed)``."""
    lib = lib or _load()
    c = np.ascontiguousarray(cache)
    planes, B, L = c.shape[:3]
    eb = c[0, 0, 0].nbytes
    out = np.empty_like(c)
    path = np.ascontiguousarray(path_nodes, dtype=np.int32)
    base = np.ascontiguousarray(base_len, dtype=np.int32)
    acc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    new_len = np.zeros(B, dtype=np.int32)
    rc = lib.oracle_kv_commit(_ptr(c), _ptr(out), c.nbytes, B, planes, B * L * eb, L * eb, eb,
                              L, int(N), _ptr(base), _ptr(acc), _ptr(path), path.shape[1] - 1,
                              _ptr(new_len))
    if rc not in (0, 4):
        _check(rc)
    return out, new_len, rc == 4


def lm_head_greedy(hidden, w_lm, tokens, seqs=None, lib=None):
    """LM head fused with greedy verification (reading R11 of spec_oracle.c).
    ``hidden`` uint16 bf16 bits [B*(k+1), d], ``w_lm`` uint16 bf16 bits
    [V, d], ``tokens`` int32 [B, k]; ``seqs``: the sequences to evaluate
    (default all).  Returns dict(accepted_len [B], out_tokens [B, k+1],
    argmax, gap, mag [B*(k+1)]); entries of sequences not evaluated are -2 /
    NaN."""
    lib = lib or _load()
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B, k = tok.shape
    H = np.ascontiguousarray(hidden, dtype=np.uint16)
    Wm = np.ascontiguousarray(w_lm, dtype=np.uint16)
    V, d = Wm.shape
    assert H.shape == (B * (k + 1), d)
    res = dict(accepted_len=np.full(B, -2, np.int32),
               out_tokens=np.full((B, k + 1), -2, np.int32),
               argmax=np.full(B * (k + 1), -2, np.int32),
               gap=np.full(B * (k + 1), np.nan), mag=np.full(B * (k + 1), np.nan))
    sq = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    rc = lib.oracle_lm_head_greedy(_ptr(H), _ptr(Wm), _ptr(tok), B, k, d, V,
                                   None if sq is None else _ptr(sq), 0 if sq is None else len(sq),
                                   _ptr(res["accepted_len"]), _ptr(res["out_tokens"]),
                                   _ptr(res["argmax"]), _ptr(res["gap"]), _ptr(res["mag"]))
    _check(rc)
    return res


def _bf16_to_f64(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def lm_head_logits(hidden, w_lm):
    """Exact logits z = W_LM h in float64 of bf16 hidden states [rows, d] and
    a bf16 LM head [V, d] (raw 16-bit patterns): "EAGLE math", "EAGLE's move"
    (p = softmax(LM_head(f))).  The products of two bf16 values are exact in
    float64 and the sums are rounded in float64 (a library matrix product)."""
    return _bf16_to_f64(hidden) @ _bf16_to_f64(w_lm).T


def lm_head_sample(h_target, h_draft, w_lm, tokens, u_accept, u_sample, temperature, seqs=None,
                   lib=None, window=FLAG_WINDOW):
    """LM head fused with sampling verification (reading R13 of spec_oracle.c's
    header): the target rows' logits W_LM h_t and the draft rows' logits
    W_LM h_d, then sampling verification of them in float64
    (:func:`verify_sample` on float64 logits).  h_target [B*(k+1), d] and
    h_draft [B*k, d] bf16 bits, sequence-major; ``seqs`` selects the
    sequences to evaluate (default all).  Returns the verify_sample dict for
    those sequences, plus the float64 logits ``zt`` [S, k+1, V] and ``zd``
    [S, k, V]."""
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B, k = tok.shape
    V = np.asarray(w_lm).shape[0]
    sq = np.arange(B) if seqs is None else np.asarray(seqs, dtype=np.int64)
    Ht = np.asarray(h_target).reshape(B, k + 1, -1)[sq].reshape(len(sq) * (k + 1), -1)
    zt = lm_head_logits(Ht, w_lm).reshape(len(sq), k + 1, V)
    if k > 0:
        Hd = np.asarray(h_draft).reshape(B, k, -1)[sq].reshape(len(sq) * k, -1)
        zd = lm_head_logits(Hd, w_lm).reshape(len(sq), k, V)
    else:
        zd = np.zeros((len(sq), 0, V))
    out = verify_sample(zt, zd, tok[sq], np.asarray(u_accept)[sq], np.asarray(u_sample)[sq],
                        temperature, dtype="f64", lib=lib, window=window)
    out["zt"] = zt
    out["zd"] = zd
    return out


def tree_grow(logits, temperature, M, dtype="bf16", lib=None):
    """EAGLE-2 tree growth (reading R12 of spec_oracle.c).  ``logits``
    [B, D, K, V] draft rows by layer and frontier slot.  Returns dict with
    tokens, parents, depth [B, M+1] int32, values [B, M+1] float64 and
    min_gap [B] (smallest gap between a kept and a dropped value that are not
    equal, over every selection boundary; exact ties are decided by the tie
    rule)."""
    lib = lib or _load()
    z = _logits(logits, dtype)
    B, D, K, V = z.shape
    out = dict(tokens=np.zeros((B, M + 1), np.int32), parents=np.zeros((B, M + 1), np.int32),
               depth=np.zeros((B, M + 1), np.int32), values=np.zeros((B, M + 1)),
               min_gap=np.zeros(B))
    rc = lib.oracle_tree_grow(_ptr(z), _dtype_code(dtype), B, D, K, V, float(temperature), int(M),
                              _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["depth"]),
                              _ptr(out["values"]), _ptr(out["min_gap"]))
    _check(rc)
    return out


def expected_tokens(alpha: float, gamma: int, lib=None) -> float:
    return (lib or _load()).oracle_expected_tokens(float(alpha), int(gamma))


def speedup_model(alpha: float, gamma: int, c: float, lib=None) -> float:
    return (lib or _load()).oracle_speedup_model(float(alpha), int(gamma), float(c))


def sample_flags(res: dict, window: float = 1e-6) -> np.ndarray:
    """Rows whose outcome sits within ``window`` of an acceptance threshold or
    of a CDF boundary (oracle float64 values); such rows may legitimately
    differ between two correct implementations."""
    return (res["acc_margin"] < window) | (res["cdf_margin"] < window)
