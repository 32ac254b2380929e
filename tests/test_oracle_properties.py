"""Oracle properties fixed by the pages or by mathematics.

 * q = p  =>  every draft accepted (ratio 1 > u for every u in [0, 1)).
 * disjoint supports  =>  reject at position 0 and the residual is p itself
   (Uno's fragment: q_on_clean = 0 everywhere on the target support).
 * gamma = 0  =>  plain categorical sampling from p_0, checked against
   numpy's cumsum + searchsorted on scipy's softmax.
 * sigma = identity  =>  any-order equals dense without the bonus token.
 * sparse lists covering the whole vocabulary  =>  the dense rule.
 * emitted count in [1, gamma + 1] (DFlash/DFlash2 guide, section 2).
 * the reported residual is a distribution (sums to 1 within 1e-12).
 * flags, input errors and thread-count invariance.
"""
import numpy as np
import pytest
from scipy.special import softmax

from rejection_sampling_gb300 import workloads as wl

ACC, TIE, ZERO, ERR = 1, 2, 4, 8


def _dense(oracle_mod, d, **kw):
    return oracle_mod.verify_dense(d["target"], d["draft"], d["draft_ids"], d["u_accept"],
                                   d["u_sample"], **kw)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_q_equals_p_accepts_everything(oracle_mod, dtype):
    d = wl.dense_inputs(64, 6, 300, dtype=dtype, seed=3)
    d["draft"] = np.ascontiguousarray(d["target"][:, :6])
    d["draft_ids"] = wl.gumbel_argmax(np.random.default_rng(1), d["draft"]).astype(np.int32)
    d["u_accept"][:, 0] = np.float32(np.nextafter(np.float32(1), np.float32(0)))  # largest u < 1
    out = _dense(oracle_mod, d)
    assert (out["n_accepted"] == 6).all()
    assert (out["accept_prob"] == 1.0).all()
    assert (out["out_tokens"][:, :6] == d["draft_ids"]).all()


def test_disjoint_supports_reject_at_zero_and_residual_is_p(oracle_mod):
    rng = np.random.default_rng(4)
    B, G, V = 32, 3, 50
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    lt[:, :, 25:] = -np.inf  # target support {0..24}
    ld[:, :, :25] = -np.inf  # draft support {25..49}
    x = wl.gumbel_argmax(rng, ld).astype(np.int32)
    out = oracle_mod.verify_dense(lt, ld, x, rng.random((B, G), dtype=np.float32),
                                  rng.random(B, dtype=np.float32))
    assert (out["n_accepted"] == 0).all()
    assert (out["accept_prob"] == 0).all()
    p0 = softmax(lt[:, 0].astype(np.float64), axis=-1)
    np.testing.assert_allclose(out["residual"], p0, rtol=1e-12, atol=1e-15)
    assert (out["out_tokens"][:, 0] < 25).all()
    assert (out["out_tokens"][:, 1:] == -1).all()


def test_gamma0_is_categorical_sampling(oracle_mod):
    rng = np.random.default_rng(7)
    B, V = 2000, 1000
    lt = rng.normal(0, 3, (B, 1, V)).astype(np.float32)
    us = rng.random(B, dtype=np.float32)
    out = oracle_mod.verify_dense(lt, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                                  np.zeros((B, 0), np.float32), us)
    p = softmax(lt[:, 0].astype(np.float64), axis=-1)
    c = np.cumsum(p, axis=-1)
    want = np.array([np.searchsorted(c[b], us[b] * c[b, -1], side="right") for b in range(B)])
    ok = (out["flags"] & TIE) == 0
    assert ok.mean() > 0.95
    assert (out["out_tokens"][ok, 0] == want[ok]).all()
    assert (out["n_accepted"] == 0).all()
    np.testing.assert_allclose(out["residual"], p, rtol=1e-12, atol=1e-15)


def test_sigma_identity_equals_dense_without_bonus(oracle_mod):
    d = wl.dense_inputs(256, 8, 40, dtype="f32", seed=9, target_sigma=2.0, draft_noise=0.8)
    G = 8
    den = _dense(oracle_mod, d)
    order = np.broadcast_to(np.arange(G, dtype=np.int32), (256, G)).copy()
    any_ = oracle_mod.verify_anyorder(np.ascontiguousarray(d["target"][:, :G]), d["draft"], order,
                                      d["draft_ids"], d["u_accept"], d["u_sample"])
    assert (any_["n_accepted"] == den["n_accepted"]).all()
    rej = den["n_accepted"] < G
    assert (any_["out_tokens"][rej] == den["out_tokens"][rej, :G]).all()
    np.testing.assert_array_equal(any_["residual"][rej], den["residual"][rej])
    acc = ~rej
    assert (any_["out_tokens"][acc] == d["draft_ids"][acc]).all()
    np.testing.assert_array_equal(any_["accept_prob"], den["accept_prob"])


def test_sparse_full_support_equals_dense(oracle_mod):
    rng = np.random.default_rng(12)
    B, G, V = 400, 4, 24
    lt = rng.normal(0, 2, (B, G + 1, V))
    ld = lt[:, :G] + rng.normal(0, 1, (B, G, V))
    tp = softmax(lt, axis=-1).astype(np.float32)
    dp = softmax(ld, axis=-1).astype(np.float32)
    ids_t = np.broadcast_to(np.arange(V, dtype=np.int32), (B, G + 1, V)).copy()
    ids_d = np.broadcast_to(np.arange(V, dtype=np.int32), (B, G, V)).copy()
    x = wl.gumbel_argmax(rng, np.log(dp.astype(np.float64))).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    sp = oracle_mod.verify_sparse(ids_t, tp, ids_d, dp, x, ua, us, V)
    # the same distributions as logits (fp32 log of the fp32 probabilities)
    den = oracle_mod.verify_dense(np.log(tp).astype(np.float32), np.log(dp).astype(np.float32), x,
                                  ua, us)
    clean = (sp["flags"] == 0) & (den["flags"] == 0)
    assert clean.mean() > 0.97
    assert (sp["n_accepted"][clean] == den["n_accepted"][clean]).all()
    assert (sp["out_tokens"][clean] == den["out_tokens"][clean]).all()
    np.testing.assert_allclose(sp["accept_prob"], den["accept_prob"], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(sp["residual"][clean], den["residual"][clean], rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("name", ["dense_v32_g4", "dense_v151936_g15"])
def test_emitted_count_and_residual_normalised(oracle_mod, name):
    d = wl.make(name, seed=1)
    out = _dense(oracle_mod, d)
    G = d["gamma"]
    n = out["n_accepted"]
    assert ((n >= 0) & (n <= G)).all()
    emitted = (out["out_tokens"] >= 0).sum(-1)
    assert (emitted == n + 1).all()  # tau = n + 1 in [1, gamma + 1]
    assert np.abs(out["residual"].sum(-1) - 1).max() < 1e-12


def test_sparse_and_anyorder_workloads_well_formed(oracle_mod):
    s = wl.make("sparse_b256_g15_k64", seed=2, B=32)
    o = oracle_mod.verify_sparse(s["tgt_ids"], s["tgt_probs"], s["drf_ids"], s["drf_probs"],
                                 s["draft_tokens"], s["u_accept"], s["u_sample"], s["V"])
    assert (o["flags"] & ERR == 0).all()
    assert np.abs(o["residual"].sum(-1) - 1).max() < 1e-12
    assert ((o["out_tokens"] >= 0).sum(-1) == o["n_accepted"] + 1).all()
    a = wl.make("anyorder_b4096_w32_v33", seed=2, B=64)
    o = oracle_mod.verify_anyorder(a["target"], a["draft"], a["order"], a["draft_tokens"],
                                   a["u_accept"], a["u_sample"])
    assert (o["flags"] & ERR == 0).all()
    rej = o["n_accepted"] < a["W"]
    assert np.abs(o["residual"][rej].sum(-1) - 1).max() < 1e-12
    assert (o["out_tokens"] != -7).all()  # D == W: every position is in the window


def test_accept_band_flag(oracle_mod):
    # p uniform on 4, q uniform on {1,2}: accept prob of x = 1 is exactly 1/2
    lt = np.zeros((4, 2, 4), np.float32)
    ld = np.full((4, 1, 4), -np.inf, np.float32)
    ld[:, :, 1:3] = 0
    x = np.ones((4, 1), np.int32)
    ua = np.array([[0.5 - 4e-7], [0.5 + 4e-7], [0.5 - 3e-6], [0.5 + 3e-6]], np.float32)
    out = oracle_mod.verify_dense(lt, ld, x, ua, np.full(4, 0.3, np.float32))
    assert (out["flags"] & ACC).tolist() == [ACC, ACC, 0, 0]
    assert out["n_accepted"].tolist() == [1, 0, 1, 0]


def test_flags_only_count_consumed_decisions(oracle_mod):
    # position 0 rejects clearly; position 1's decision sits on the band but is never used
    lt = np.zeros((1, 3, 4), np.float32)
    ld = np.full((1, 2, 4), -np.inf, np.float32)
    ld[0, 0, 0] = 0  # q0 = point mass at 0
    ld[0, 1, 1:3] = 0
    x = np.array([[3, 1]], np.int32)  # q0(3) = 0 -> reject; pos 1 ratio 1/2
    out = oracle_mod.verify_dense(lt, ld, x, np.array([[0.4, 0.5]], np.float32),
                                  np.array([0.3], np.float32))
    assert out["n_accepted"][0] == 0 and out["flags"][0] == 0


def test_dense_input_errors(oracle_mod):
    d = wl.dense_inputs(6, 3, 20, dtype="f32", seed=5)
    d["target"][0, 1, 4] = np.nan
    d["draft"][1, 2, :] = -np.inf
    d["draft_ids"][2, 0] = 20
    d["draft_ids"][3, 1] = -1
    d["target"][4, 3, 0] = np.inf  # bonus row is validated too
    out = _dense(oracle_mod, d)
    assert out["n_accepted"].tolist()[:5] == [-1] * 5
    assert (out["flags"][:5] == ERR).all() and out["flags"][5] & ERR == 0
    assert (out["out_tokens"][:5] == -1).all()
    assert out["n_accepted"][5] >= 0


def test_sparse_input_errors(oracle_mod):
    s = wl.make("sparse_b256_g15_k64", seed=3, B=5, gamma=3)
    s["tgt_ids"][0, 0, [3, 4]] = s["tgt_ids"][0, 0, [4, 3]]  # unsorted
    s["drf_ids"][1, 1, 5] = s["drf_ids"][1, 1, 4]  # duplicate
    s["tgt_ids"][2, 3, -1] = s["V"]  # out of range (bonus list)
    s["draft_tokens"][3, 2] = -5
    o = oracle_mod.verify_sparse(s["tgt_ids"], s["tgt_probs"], s["drf_ids"], s["drf_probs"],
                                 s["draft_tokens"], s["u_accept"], s["u_sample"], s["V"])
    assert o["n_accepted"].tolist()[:4] == [-1] * 4 and o["n_accepted"][4] >= 0


def test_anyorder_input_errors(oracle_mod):
    a = wl.anyorder_inputs(4, 6, 4, 9, seed=8)
    a["order"][0, 1] = a["order"][0, 0]  # repeated position
    a["order"][1, 2] = 6  # out of range
    a["draft_tokens"][2, a["order"][2, 3]] = 9  # token out of range at a window position
    o = oracle_mod.verify_anyorder(a["target"], a["draft"], a["order"], a["draft_tokens"],
                                   a["u_accept"], a["u_sample"])
    assert o["n_accepted"].tolist()[:3] == [-1] * 3 and o["n_accepted"][3] >= 0


def test_thread_count_invariance(oracle_mod):
    d = wl.dense_inputs(24, 5, 3000, dtype="bf16", seed=6)
    a = _dense(oracle_mod, d, nthreads=1)
    b = _dense(oracle_mod, d, nthreads=7)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k])
