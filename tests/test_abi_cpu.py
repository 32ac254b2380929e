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
