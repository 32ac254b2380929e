"""GPU parity for sparse support lists (temperature, top-k, top-p):
spec_support_topk through the C ABI against the oracle on the same seeded
logits.  The top-k set is decided by exact comparisons, so ids must match on
every row; probabilities agree within 1e-5 (relative, absolute below 1e-12)
on rows whose top-p cut is not within 1e-6 of top_p (flagged by the oracle,
where one entry more or less may be kept)."""
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


def run_support(logits, T, K, P):
    r = rs.spec_support_topk(to_dev(logits), T, K, P)
    torch.cuda.synchronize()
    return r.ids.cpu().numpy(), r.probs.cpu().numpy()


def support_parity(logits, T, K, P, min_clean=0.9):
    ids, probs = run_support(logits, T, K, P)
    o = oracle.support_topk(logits, T, K, P)
    np.testing.assert_array_equal(ids, o["ids"])
    clean = o["flags"] == 0
    assert clean.mean() >= min_clean
    np.testing.assert_allclose(probs[clean], o["probs"][clean], rtol=1e-5, atol=1e-12)
    assert rs.check() == rs.SV_OK
    return ids, probs, o


def _normal_rows(N, V, dtype, seed, sigma=3.0):
    a = np.random.default_rng(seed).normal(0, sigma, size=(N, V)).astype(np.float32)
    return wl.bf16_bits(a) if dtype == "bf16" else a


@pytest.mark.parametrize("N,V,K,T,P,dtype", [
    (16, 151936, 50, 1.0, 0.95, "bf16"),   # the Uno article's test setting
    (20, 30001, 128, 0.7, 0.9, "f32"),     # odd V: unaligned rows
    (8, 5000, 256, 1.3, 1.0, "bf16"),      # the largest top_k, no top-p cut
    (33, 100, 1, 1.0, 0.5, "f32"),         # top_k = 1
    (5, 64, 64, 1.0, 0.8, "bf16"),         # top_k = V
    (300, 2048, 32, 0.5, 0.95, "bf16"),    # many short rows
])
def test_support_parity(N, V, K, T, P, dtype):
    support_parity(_normal_rows(N, V, dtype, seed=N + V + K), T, K, P)


def test_support_headline_rows():
    # the 64 x (8 + 7) target and draft rows of the dense headline workload
    d = wl.make("dense_b64_g7_v128256", seed=0)
    support_parity(d["target"].reshape(-1, d["V"]), 1.0, 64, 0.95)
    support_parity(d["draft"].reshape(-1, d["V"]), 1.0, 64, 0.95)


def test_support_ties_go_to_the_smaller_id():
    # logits on a coarse grid: many equal values at the top-k boundary
    rng = np.random.default_rng(4)
    a = rng.integers(0, 12, size=(24, 9000)).astype(np.float32)
    # (the top 100 are all equal: top_p 0.905 cuts after 91 entries, clear of
    # the 1e-6 band that an exact 0.9 would hit)
    support_parity(a, 1.0, 100, 0.905, min_clean=0.5)
    support_parity(wl.bf16_bits(a), 0.8, 64, 1.0, min_clean=0.5)


def test_support_input_errors():
    a = _normal_rows(6, 4000, "f32", seed=5)
    a[0, 17] = np.nan
    a[1, :] = -np.inf
    a[2, 3999] = np.inf
    ids, probs = run_support(a, 1.0, 20, 0.9)
    assert (ids[:3] == -1).all() and np.isnan(probs[:3]).all()
    assert (ids[3:] >= 0).all()
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    assert rs.check() == rs.SV_OK


def test_support_feeds_sparse_verification():
    # dense logits -> support lists -> sparse verification, all on the GPU,
    # against the same composition of the oracles (same uniforms)
    B, G, V, T, K, P = 32, 3, 20000, 0.9, 64, 0.95
    d = wl.dense_inputs(B, G, V, dtype="bf16", seed=12, target_sigma=3.0, draft_noise=0.5)
    tgt = rs.spec_support_topk(to_dev(d["target"]), T, K, P)
    drf = rs.spec_support_topk(to_dev(d["draft"]), T, K, P)
    ot = oracle.support_topk(d["target"], T, K, P)
    od = oracle.support_topk(d["draft"], T, K, P)
    rng = np.random.default_rng(3)
    x = np.empty((B, G), np.int32)
    for b in range(B):
        for j in range(G):
            x[b, j] = rng.choice(od["ids"][b, j], p=od["probs"][b, j] / od["probs"][b, j].sum())
    r = rs.spec_verify_sparse(tgt.ids, tgt.probs, drf.ids, drf.probs, to_dev(x), to_dev(d["u_accept"]),
                              to_dev(d["u_sample"]), V)
    torch.cuda.synchronize()
    o = oracle.verify_sparse(ot["ids"], ot["probs"].astype(np.float32), od["ids"],
                             od["probs"].astype(np.float32), x, d["u_accept"], d["u_sample"], V)
    clean = (ot["flags"] == 0).all(axis=1) & (od["flags"] == 0).all(axis=1) & (o["flags"] == 0)
    assert clean.mean() > 0.7
    n = r.n_accepted.cpu().numpy()
    tok = r.out_tokens.cpu().numpy()
    np.testing.assert_array_equal(n[clean], o["n_accepted"][clean])
    np.testing.assert_array_equal(tok[clean], o["out_tokens"][clean])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_support_sorted_rows(dtype):
    # ascending rows: every element clears the running threshold, so the
    # candidate buffers fill and are cut back to the top k many times;
    # descending rows: the first elements already hold the answer.  Rounding
    # makes the top entries equal, so top_p is kept off multiples of 1/K.
    V = 70000
    base = np.linspace(-20.0, 20.0, V, dtype=np.float32)
    rows = np.stack([base, base[::-1], np.round(base), np.round(base[::-1]) * 0.5])
    a = wl.bf16_bits(rows) if dtype == "bf16" else rows
    for K in (1, 50, 200):
        support_parity(a, 1.0, K, 0.913, min_clean=0.5)


def test_support_full_960_rows():
    # the support workload at full size: all 960 target and draft rows of a
    # headline batch (one full wave of CTAs and part of a second)
    d = wl.make("dense_b64_g7_v128256", seed=1)
    rows = np.concatenate([d["target"].reshape(-1, d["V"]), d["draft"].reshape(-1, d["V"])])
    support_parity(rows, 1.0, 50, 0.95)


def test_support_input_errors_in_the_last_wave():
    # errors in the last rows of a 960-row call (CTAs of the second wave): a
    # NaN early and one late in the row, +inf, a row of -inf
    N, V = 960, 60000
    a = _normal_rows(N, V, "f32", seed=9)
    a[N - 1, 100] = np.nan
    a[N - 2, 7000] = np.nan
    a[N - 3, V - 1] = np.inf
    a[N - 4, :] = -np.inf
    b = wl.bf16_bits(a)
    ids, probs = run_support(b, 1.0, 50, 0.95)
    assert (ids[N - 4:] == -1).all() and np.isnan(probs[N - 4:]).all()
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    o = oracle.support_topk(b[:N - 4], 1.0, 50, 0.95)
    np.testing.assert_array_equal(ids[:N - 4], o["ids"])
    assert rs.check() == rs.SV_OK
