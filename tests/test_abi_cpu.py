"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol the header declares, rejects bad arguments on the host before touching
CUDA, and sizes its workspace sanely."""
import ctypes
import os
import re

import pytest

import rejection_sampling_gb300 as rs
from rejection_sampling_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rs.load()


def _declared_functions():
    names = set()
    for h in ("spec_verify.h",):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"spec_verify_dense", "spec_verify_sparse", "spec_verify_anyorder",
            "spec_verify_workspace_size", "spec_verify_check"} <= declared
    assert declared == set(rs.EXPORTED)
    raw = ctypes.CDLL(rs.library_path())
    for name in declared:
        assert hasattr(raw, name), name


def test_abi_version_and_status_strings(lib):
    assert rs.abi_version() == 1
    assert rs.status_string(0) == "ok"
    assert "invalid" in rs.status_string(1)
    assert rs.status_string(99) == "unknown status"


def test_workspace_size(lib):
    assert rs.workspace_size(-1, 3, 10) == 0
    assert rs.workspace_size(1, 4, 32) >= 256
    a = rs.workspace_size(64, 7, 128256)
    b = rs.workspace_size(128, 7, 128256)
    assert 0 < a < b < 8 * a
    assert rs.workspace_size(0, 7, 128256) >= 256


def test_host_validation_without_gpu(lib):
    P = None
    # negative sizes, out-of-range gamma / vocab, bad dtype: rejected before any CUDA call
    assert lib.spec_verify_dense(P, P, 1, P, P, P, -1, 3, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_dense(P, P, 1, P, P, P, 2, 256, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_dense(P, P, 1, P, P, P, 2, 3, 0, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_dense(P, P, 7, P, P, P, 2, 3, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    # empty batch is a no-op
    assert lib.spec_verify_dense(P, P, 1, P, P, P, 0, 3, 10, P, P, P, P, P, 0, P) == rs.SV_OK
    # null pointers
    assert lib.spec_verify_dense(P, P, 1, P, P, P, 2, 3, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_sparse(P, P, 0, P, P, 4, P, P, P, 2, 3, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_sparse(P, P, 4, P, P, 4, P, P, P, 2, 32, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_anyorder(P, P, 0, P, P, P, P, 2, 8, 33, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_anyorder(P, P, 0, P, P, P, P, 2, 4, 8, 10, P, P, P, P, P, 0, P) == rs.SV_ERR_INVALID_ARG
    # any-order beyond the small-vocabulary kernel
    assert lib.spec_verify_anyorder(P, P, 0, P, P, P, P, 2, 32, 32, 5000, P, P, P, P, P, 0, P) == rs.SV_ERR_UNSUPPORTED
    assert lib.spec_verify_workspace_init(P, 0, P) == rs.SV_ERR_INVALID_ARG
    assert lib.spec_verify_check(P, 0, P) == rs.SV_ERR_INVALID_ARG


def test_host_validation_of_the_next_rows_without_gpu(lib):
    """Greedy, commit, support lists and the windowed rounds reject bad
    arguments on the host (before any CUDA call); empty batches are no-ops.
    Non-null "pointers" below are never dereferenced: every call that passes
    one fails a host check (a misaligned address or a too-small workspace)
    before anything could be launched."""
    P = None
    F = ctypes.c_float
    odd = 0x1001  # misaligned for every element size, never touched
    ok4 = 0x1000
    E = rs.SV_ERR_INVALID_ARG
    # greedy: sizes, dtype, nulls, alignment
    assert lib.spec_verify_greedy(P, 1, P, -1, 3, 10, P, P, P, 0, P) == E
    assert lib.spec_verify_greedy(P, 1, P, 2, -1, 10, P, P, P, 0, P) == E
    assert lib.spec_verify_greedy(P, 1, P, 2, 3, 0, P, P, P, 0, P) == E
    assert lib.spec_verify_greedy(P, 5, P, 2, 3, 10, P, P, P, 0, P) == E
    assert lib.spec_verify_greedy(P, 1, P, 0, 3, 10, P, P, P, 0, P) == rs.SV_OK
    assert lib.spec_verify_greedy(P, 1, P, 2, 3, 10, P, P, P, 0, P) == E
    assert lib.spec_verify_greedy(odd, 1, ok4, 2, 3, 10, ok4, ok4, 0x10000, 1 << 20, P) == E
    # commit: W in [1, 256], tau not NaN
    assert lib.spec_commit_confident(P, 1, P, F(0.9), 2, 0, 10, P, P, P, P, 0, P) == E
    assert lib.spec_commit_confident(P, 1, P, F(0.9), 2, 257, 10, P, P, P, P, 0, P) == E
    assert lib.spec_commit_confident(P, 1, P, F(float("nan")), 2, 4, 10, P, P, P, P, 0, P) == E
    assert lib.spec_commit_confident(P, 1, P, F(0.9), 0, 4, 10, P, P, P, P, 0, P) == rs.SV_OK
    assert lib.spec_commit_confident(P, 1, P, F(0.9), 2, 4, 10, P, P, P, P, 0, P) == E
    # support lists: 1 <= top_k <= min(256, V), temperature finite and > 0, top_p not NaN
    for T, K, V, top_p in ((1.0, 0, 100, 0.9), (1.0, 257, 1000, 0.9), (1.0, 11, 10, 0.9),
                           (0.0, 5, 100, 0.9), (float("inf"), 5, 100, 0.9),
                           (float("nan"), 5, 100, 0.9), (1.0, 5, 100, float("nan"))):
        assert lib.spec_support_topk(ok4, 1, 3, V, F(T), K, F(top_p), ok4, ok4, 0x10000, 1 << 20, P) == E
    assert lib.spec_support_topk(P, 1, 0, 100, F(1.0), 5, F(0.9), P, P, P, 0, P) == rs.SV_OK
    assert lib.spec_support_topk(odd, 1, 3, 100, F(1.0), 5, F(0.9), ok4, ok4, 0x10000, 1 << 20, P) == E
    assert lib.spec_support_topk(ok4, 1, 3, 100, F(1.0), 5, F(0.9), ok4, ok4, 0x10000, 16, P) == E
    # windowed rounds: R, D, V >= 1, size products, dtype, nulls
    args = lambda B, R, D, V, dt=0, p=P: (p, p, dt, p, p, p, p, p, p, B, R, D, V, p, p, p, p, 0, P)
    assert lib.spec_verify_anyorder_rounds(*args(2, 0, 8, 5)) == E
    assert lib.spec_verify_anyorder_rounds(*args(2, 3, 0, 5)) == E
    assert lib.spec_verify_anyorder_rounds(*args(2, 3, 8, 0)) == E
    assert lib.spec_verify_anyorder_rounds(*args(-1, 3, 8, 5)) == E
    assert lib.spec_verify_anyorder_rounds(*args(2, 3, 8, 5, dt=9)) == E
    assert lib.spec_verify_anyorder_rounds(*args(4, 1 << 12, 1 << 20, 5)) == E  # B R D beyond 2^31
    assert lib.spec_verify_anyorder_rounds(*args(0, 3, 8, 5)) == rs.SV_OK
    assert lib.spec_verify_anyorder_rounds(*args(2, 3, 8, 5)) == E  # null pointers
