"""Plain CPU oracle for batched lossless speculative verification.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; the
product path (``rejection_sampling_gb300``) never imports it.  The
arithmetic lives in ``spec_verify_oracle.c`` (scalar IEEE double, one row at
a time); this module only compiles it with gcc and marshals numpy arrays.

Rule being checked: Leviathan-style rejection sampling as stated in the Uno
article ("What 'lossless' actually has to mean"), truncated at the first
rejection (DFlash/DFlash2 guide, 4.4), with the target's bonus token after an
all-accept block (same guide, section 2), and the any-order variant of
"Self-Speculative Masked Diffusions" (key design 2).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_verify_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_spec_verify.so")
_lock = threading.Lock()
_lib = None

FLAG_ACCEPT_BAND = 1
FLAG_CDF_TIE = 2
FLAG_ZERO_RESID = 4
FLAG_INPUT_ERR = 8

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/ (gcc, strict IEEE, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    hdr = os.path.join(_HERE, "spec_verify_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_verify_dense.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P, P, I]
            lib.oracle_verify_sparse.argtypes = [P, P, I, P, P, I, P, P, P, I, I, I, P, P, P, P, P, P, I]
            lib.oracle_verify_anyorder.argtypes = [P, P, I, P, P, P, P, I, I, I, I, P, P, P, P, P, P, I]
            lib.oracle_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, I]
            lib.oracle_commit_confident.argtypes = [P, I, P, ctypes.c_double, I, I, I, P, P, P, P, I]
            lib.oracle_support_topk.argtypes = [P, I, I, I, ctypes.c_double, I, ctypes.c_double, P, P, P, I]
            lib.oracle_anyorder_rounds.argtypes = [P, P, I, P, P, P, P, P, P, I, I, I, I, P, P, P, P, I]
            lib.oracle_cosine_window.argtypes = [I, I, ctypes.c_double]
            for f in (lib.oracle_verify_dense, lib.oracle_verify_sparse, lib.oracle_verify_anyorder,
                      lib.oracle_verify_greedy, lib.oracle_commit_confident,
                      lib.oracle_support_topk, lib.oracle_anyorder_rounds, lib.oracle_cosine_window):
                f.restype = I
            lib.oracle_default_threads.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """Return (contiguous array, dtype code).  bf16 arrives as raw uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def verify_dense(target, draft, draft_ids, u_accept, u_sample, *, residual=True,
                 nthreads: int = 0) -> dict:
    """Dense verification of B rows.  target [B, g+1, V], draft [B, g, V]."""
    lib = _load()
    lt, dt = _logits(target)
    B, G1, V = lt.shape
    G = G1 - 1
    if G > 0:
        ld, dt2 = _logits(draft)
        assert dt2 == dt and ld.shape == (B, G, V)
    else:
        ld = None
    x = np.ascontiguousarray(draft_ids, dtype=np.int32).reshape(B, G)
    ua = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    us = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    out = dict(
        n_accepted=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, G + 1), np.int32),
        residual=np.zeros((B, V), np.float64) if residual else None,
        accept_prob=np.zeros((B, G), np.float64),
        resid_mass=np.zeros(B, np.float64),
        flags=np.zeros(B, np.uint32),
    )
    rc = lib.oracle_verify_dense(
        _ptr(lt), _ptr(ld), dt, _ptr(x), _ptr(ua), _ptr(us), B, G, V,
        _ptr(out["n_accepted"]), _ptr(out["out_tokens"]), _ptr(out["residual"]),
        _ptr(out["accept_prob"]), _ptr(out["resid_mass"]), _ptr(out["flags"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_verify_dense failed")
    return out


def verify_greedy(target, draft_ids, *, nthreads: int = 0) -> dict:
    """Greedy (T = 0) verification of B rows.  target [B, g+1, V]; draft_ids [B, g].
    DFlash/DFlash2 guide, 4.4 (greedy decoding); the C file states the reading."""
    lib = _load()
    lt, dt = _logits(target)
    B, G1, V = lt.shape
    G = G1 - 1
    x = np.ascontiguousarray(draft_ids, dtype=np.int32).reshape(B, G)
    out = dict(n_accepted=np.zeros(B, np.int32), out_tokens=np.zeros((B, G + 1), np.int32))
    rc = lib.oracle_verify_greedy(_ptr(lt), dt, _ptr(x), B, G, V, _ptr(out["n_accepted"]),
                                  _ptr(out["out_tokens"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_verify_greedy failed")
    return out


def commit_confident(logits, masked, tau: float, *, nthreads: int = 0) -> dict:
    """Confidence-threshold commit of B blocks ("SDAR" page, section 5).
    logits [B, W, V]; masked [B, W] (nonzero: still masked)."""
    lib = _load()
    lt, dt = _logits(logits)
    B, W, V = lt.shape
    m = np.ascontiguousarray(masked, dtype=np.int32).reshape(B, W)
    out = dict(commit=np.zeros((B, W), np.int32), tokens=np.zeros((B, W), np.int32),
               confidence=np.zeros((B, W), np.float64), flags=np.zeros(B, np.uint32))
    rc = lib.oracle_commit_confident(_ptr(lt), dt, _ptr(m), float(tau), B, W, V,
                                     _ptr(out["commit"]), _ptr(out["tokens"]),
                                     _ptr(out["confidence"]), _ptr(out["flags"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_commit_confident failed")
    return out


def support_topk(logits, T: float, K: int, top_p: float, *, nthreads: int = 0) -> dict:
    """Sparse support lists from dense logits [..., V]: temperature T, top-k K,
    top-p; ids ascending [..., K], probs [..., K]."""
    lib = _load()
    lt, dt = _logits(logits)
    shape = lt.shape
    V = shape[-1]
    N = int(np.prod(shape[:-1]))
    out = dict(ids=np.zeros(shape[:-1] + (K,), np.int32),
               probs=np.zeros(shape[:-1] + (K,), np.float64),
               flags=np.zeros(shape[:-1], np.uint32))
    rc = lib.oracle_support_topk(_ptr(lt), dt, N, V, float(T), int(K), float(top_p),
                                 _ptr(out["ids"]), _ptr(out["probs"]), _ptr(out["flags"]),
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_support_topk failed")
    return out


def verify_sparse(tgt_ids, tgt_probs, drf_ids, drf_probs, draft_tokens, u_accept, u_sample, V,
                  *, residual=True, nthreads: int = 0) -> dict:
    """Sparse top-k verification.  tgt_* [B, g+1, kt], drf_* [B, g, kd]."""
    lib = _load()
    tid = np.ascontiguousarray(tgt_ids, dtype=np.int32)
    tp = np.ascontiguousarray(tgt_probs, dtype=np.float32)
    B, G1, kt = tid.shape
    G = G1 - 1
    did = np.ascontiguousarray(drf_ids, dtype=np.int32)
    dp = np.ascontiguousarray(drf_probs, dtype=np.float32)
    kd = did.shape[2] if did.ndim == 3 and did.size else 1
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
    ua = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    us = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    out = dict(
        n_accepted=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, G + 1), np.int32),
        residual=np.zeros((B, kt), np.float64) if residual else None,
        accept_prob=np.zeros((B, G), np.float64),
        resid_mass=np.zeros(B, np.float64),
        flags=np.zeros(B, np.uint32),
    )
    rc = lib.oracle_verify_sparse(
        _ptr(tid), _ptr(tp), kt, _ptr(did) if G else None, _ptr(dp) if G else None, kd,
        _ptr(x), _ptr(ua), _ptr(us), B, G, int(V),
        _ptr(out["n_accepted"]), _ptr(out["out_tokens"]), _ptr(out["residual"]),
        _ptr(out["accept_prob"]), _ptr(out["resid_mass"]), _ptr(out["flags"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_verify_sparse failed")
    return out


def verify_anyorder(target, draft, order, draft_tokens, u_accept, u_sample, *, out_init=None,
                    residual=True, nthreads: int = 0) -> dict:
    """Any-order verification.  target/draft [B, D, V]; order [B, W]."""
    lib = _load()
    lt, dt = _logits(target)
    ld, dt2 = _logits(draft)
    assert dt == dt2 and lt.shape == ld.shape
    B, D, V = lt.shape
    sig = np.ascontiguousarray(order, dtype=np.int32)
    W = sig.shape[1]
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, D)
    ua = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, W)
    us = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    out_tokens = (np.full((B, D), -7, np.int32) if out_init is None
                  else np.array(out_init, dtype=np.int32, copy=True))
    out = dict(
        n_accepted=np.zeros(B, np.int32),
        out_tokens=out_tokens,
        residual=np.zeros((B, V), np.float64) if residual else None,
        accept_prob=np.zeros((B, W), np.float64),
        resid_mass=np.zeros(B, np.float64),
        flags=np.zeros(B, np.uint32),
    )
    rc = lib.oracle_verify_anyorder(
        _ptr(lt), _ptr(ld), dt, _ptr(sig), _ptr(tok), _ptr(ua), _ptr(us), B, D, W, V,
        _ptr(out["n_accepted"]), _ptr(out["out_tokens"]), _ptr(out["residual"]),
        _ptr(out["accept_prob"]), _ptr(out["resid_mass"]), _ptr(out["flags"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_verify_anyorder failed")
    return out


def anyorder_rounds(target, draft, order, revealed, window, draft_tokens, u_accept, u_sample, *,
                    tokens_init=None, nthreads: int = 0) -> dict:
    """Windowed multi-round any-order verification.  target [B, R, D, V],
    draft [B, D, V], order [B, D], revealed [B], window [B], draft_tokens
    [B, R, D], u_accept [B, R, D] (by sigma index), u_sample [B, R]."""
    lib = _load()
    lt, dt = _logits(target)
    ld, dt2 = _logits(draft)
    assert dt == dt2
    B, R, D, V = lt.shape
    assert ld.shape == (B, D, V)
    sig = np.ascontiguousarray(order, dtype=np.int32).reshape(B, D)
    i0 = np.ascontiguousarray(revealed, dtype=np.int32).reshape(B)
    win = np.ascontiguousarray(window, dtype=np.int32).reshape(B)
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, R, D)
    ua = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, R, D)
    us = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B, R)
    out = dict(tokens=(np.full((B, D), -7, np.int32) if tokens_init is None
                       else np.array(tokens_init, dtype=np.int32, copy=True)),
               n_revealed=np.zeros(B, np.int32),
               round_accepts=np.zeros((B, R), np.int32),
               flags=np.zeros(B, np.uint32))
    rc = lib.oracle_anyorder_rounds(_ptr(lt), _ptr(ld), dt, _ptr(sig), _ptr(i0), _ptr(win),
                                    _ptr(tok), _ptr(ua), _ptr(us), B, R, D, V,
                                    _ptr(out["tokens"]), _ptr(out["n_revealed"]),
                                    _ptr(out["round_accepts"]), _ptr(out["flags"]), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_anyorder_rounds failed")
    return out


def cosine_window(D: int, i: int, dtau: float) -> int:
    """W(i): the window of an outer step starting with i of D tokens revealed."""
    return int(_load().oracle_cosine_window(int(D), int(i), float(dtau)))
