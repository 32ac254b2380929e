"""GPU parity for the confidence-threshold commit: spec_commit_confident
through the C ABI against the oracle on the same seeded inputs.  Commit flags
and tokens are bit-exact except in blocks the oracle flags (a masked
position's confidence within 1e-6 of tau, or the fallback's top two
confidences within 1e-6 relative); confidences agree within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
import rejection_sampling_gb300 as rs
from rejection_sampling_gb300 import workloads as wl
from parity_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rs.build()
    rs.load()
    oracle.build()
    yield
    torch.cuda.synchronize()


def run_commit(logits, masked, tau):
    r = rs.spec_commit_confident(to_dev(logits), to_dev(masked), tau, confidence=True)
    torch.cuda.synchronize()
    return r.commit.cpu().numpy(), r.tokens.cpu().numpy(), r.confidence.cpu().numpy()


def commit_parity(logits, masked, tau, min_clean=0.9):
    c, t, f = run_commit(logits, masked, tau)
    o = oracle.commit_confident(logits, masked, tau)
    flagged = (o["flags"] & 3) != 0
    assert (~flagged).mean() >= min_clean
    clean = ~flagged
    np.testing.assert_array_equal(c[clean], o["commit"][clean])
    np.testing.assert_array_equal(t[clean], o["tokens"][clean])
    m = masked != 0
    err = (o["commit"] == -1).any(axis=1)
    sel = m & ~err[:, None]
    np.testing.assert_allclose(f[sel], o["confidence"][sel], rtol=1e-5, atol=0)
    assert np.isnan(f[~m]).all()
    return c, o


@pytest.mark.parametrize("B,W,V,dtype", [
    (3, 4, 20000, "bf16"),     # several pieces per row, ragged last piece
    (5, 4, 30001, "f32"),      # odd V: rows not 16-byte aligned (plain loads)
    (100, 8, 1000, "bf16"),    # many blocks, one piece per row
    (2, 1, 5000, "bf16"),      # one position per block
    (1, 256, 2048, "bf16"),    # the widest block
    (9, 4, 33, "f32"),         # tiny rows
])
def test_commit_parity(B, W, V, dtype):
    d = wl.commit_inputs(B, W, V, dtype=dtype, seed=B * 13 + W + V % 71)
    commit_parity(d["logits"], d["masked"], d["tau"])


def test_commit_sdar_shape_b64_w4_v151936():
    d = wl.commit_inputs(64, 4, 151936, dtype="bf16", seed=0)
    c, o = commit_parity(d["logits"], d["masked"], d["tau"])
    # the threshold and the fallback both occur
    m = d["masked"] != 0
    assert ((c == 1).sum(axis=1) >= 1)[m.any(axis=1)].all()


@pytest.mark.parametrize("tau", [-1.0, 1.0, 0.5])
def test_commit_thresholds(tau):
    d = wl.commit_inputs(32, 4, 9000, dtype="bf16", seed=5)
    # with tau = 1 most confidences sit within 1e-6 of it (flagged blocks are
    # compared by the properties below only)
    c, o = commit_parity(d["logits"], d["masked"], tau, min_clean=0.0)
    m = d["masked"] != 0
    if tau < 0:
        assert ((c == 1) == m).all()
    if tau >= 1:
        assert ((c == 1).sum(axis=1) == m.any(axis=1)).all()


def test_commit_input_errors_flag_blocks():
    d = wl.commit_inputs(6, 4, 7000, dtype="f32", seed=7)
    lt, m = d["logits"].copy(), d["masked"].copy()
    m[0, :] = 1
    lt[0, 1, 5] = np.nan
    m[1, 2] = 1
    lt[1, 2, :] = -np.inf
    m[2, :] = 1
    lt[2, 3, 6999] = np.inf
    m[3, 3] = 0
    lt[3, 3, 0] = np.nan  # not masked: not read, no error
    c, t, f = run_commit(lt, m, d["tau"])
    o = oracle.commit_confident(lt, m, d["tau"])
    np.testing.assert_array_equal(c[:3], o["commit"][:3])
    assert (c[:3] == -1).all() and (t[:3] == -1).all()
    assert (c[3:] >= 0).all()
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    assert rs.check() == rs.SV_OK


def test_commit_leaves_the_workspace_zero():
    dev = torch.device("cuda", torch.cuda.current_device())
    rs.check()
    d = wl.commit_inputs(8, 4, 60000, dtype="bf16", seed=9)
    commit_parity(d["logits"], d["masked"], d["tau"])
    sp = int(torch.cuda.current_stream(dev).cuda_stream)
    ws = rs.get_workspace(rs.workspace_size(8, 3, 60000), dev, sp)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
