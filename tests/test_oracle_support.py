"""Pins for the sparse-support oracle (temperature, top-k, top-p; Uno article's
test setting and DFlash/DFlash2 guide Q3).

The pins: exact hand cases, numpy/scipy re-derivations of each stage, and the
link to the verification rule itself -- sparse verification on the lists must
equal dense verification on the scaled logits with everything outside the kept
set at -inf (both oracles, the same uniforms)."""
import numpy as np
import pytest
from scipy.special import softmax

from rejection_sampling_gb300 import workloads as wl


def _log_weights(w):
    return np.log(np.asarray(w, np.float64)).astype(np.float32)[None, :]


def test_support_hand_cases(oracle_mod):
    # (the logits are the fp32 roundings of log w, so masses agree with the
    # exact ratios to ~1e-8 relative)
    # weights 1, 4, 2, 8, 1 (logits their logs, T = 1): the top-3 set is ids
    # {3, 1, 2} with mass 8/14, 4/14, 2/14; top-p 0.6 keeps 3 and 1 (8/14 <
    # 0.6 <= 12/14), renormalised to 2/3 and 1/3; id 2 stays listed at 0
    lt = _log_weights([1, 4, 2, 8, 1])
    a = oracle_mod.support_topk(lt, 1.0, 3, 1.0)
    assert a["ids"][0].tolist() == [1, 2, 3]
    np.testing.assert_allclose(a["probs"][0], [4 / 14, 2 / 14, 8 / 14], rtol=1e-7)
    b = oracle_mod.support_topk(lt, 1.0, 3, 0.6)
    assert b["ids"][0].tolist() == [1, 2, 3]
    np.testing.assert_allclose(b["probs"][0], [1 / 3, 0.0, 2 / 3], rtol=1e-7, atol=1e-15)
    # ties: ids 0 and 4 share the smallest weight; with K = 4 the smaller id wins
    c = oracle_mod.support_topk(lt, 1.0, 4, 1.0)
    assert c["ids"][0].tolist() == [0, 1, 2, 3]
    # temperature 2 halves the log-weights: masses sqrt(8), 2, sqrt(2) over the top 3
    d = oracle_mod.support_topk(lt, 2.0, 3, 1.0)
    z = np.sqrt(8) + 2 + np.sqrt(2)
    np.testing.assert_allclose(d["probs"][0], [2 / z, np.sqrt(2) / z, np.sqrt(8) / z], rtol=1e-7)


@pytest.mark.parametrize("T,K,P", [(1.0, 64, 1.0), (0.7, 50, 0.95), (1.3, 200, 0.9), (1.0, 1, 0.5)])
def test_support_against_numpy(oracle_mod, T, K, P):
    rng = np.random.default_rng(int(T * 10) + K)
    N, V = 12, 3000
    lt = wl.bf16_bits(rng.normal(0, 3, size=(N, V)).astype(np.float32))
    vals = wl.bf16_bits_to_f32(lt).astype(np.float64)
    out = oracle_mod.support_topk(lt, T, K, P)
    for r in range(N):
        order = np.lexsort((np.arange(V), -vals[r]))  # value descending, then id ascending
        top = order[:K]
        p = softmax(vals[r, top] / T)
        c = np.cumsum(p)
        keep = K if P >= 1 else int(np.searchsorted(c, P, side="left")) + 1
        keep = min(keep, K)
        want = np.zeros(K)
        want[:keep] = p[:keep] / p[:keep].sum()
        by_id = np.argsort(top)
        assert out["ids"][r].tolist() == top[by_id].tolist()
        if out["flags"][r] == 0:
            np.testing.assert_allclose(out["probs"][r], want[by_id], rtol=1e-9, atol=1e-15)


@pytest.mark.parametrize("seed", [0, 1])
def test_sparse_verify_on_the_support_equals_dense_verify_on_masked_logits(oracle_mod, seed):
    # the lists are just a truncated distribution: verifying with them must be
    # verifying the dense distribution whose logits outside the kept set are -inf
    B, G, V, T, K, P = 16, 3, 800, 0.8, 40, 0.9
    d = wl.dense_inputs(B, G, V, dtype="f32", seed=seed, target_sigma=2.0, draft_noise=0.7)
    st = oracle_mod.support_topk(d["target"], T, K, P)
    sd = oracle_mod.support_topk(d["draft"], T, K, P)
    clean = (st["flags"] == 0).all(axis=1) & (sd["flags"] == 0).all(axis=1)

    def masked(logits, sup):
        out = np.full(logits.shape, -np.inf, np.float32)
        for idx in np.ndindex(logits.shape[:-1]):
            ids = sup["ids"][idx][sup["probs"][idx] > 0]
            out[idx + (ids,)] = logits[idx + (ids,)] / np.float32(T)
        return out

    mt, md = masked(d["target"], st), masked(d["draft"], sd)
    rng = np.random.default_rng(seed + 10)
    # draft tokens from the truncated draft distribution
    x = np.empty((B, G), np.int32)
    for b in range(B):
        for j in range(G):
            x[b, j] = rng.choice(sd["ids"][b, j], p=sd["probs"][b, j])
    dense = oracle_mod.verify_dense(mt, md, x, d["u_accept"], d["u_sample"], residual=False)
    sparse = oracle_mod.verify_sparse(st["ids"], st["probs"].astype(np.float32), sd["ids"],
                                      sd["probs"].astype(np.float32), x, d["u_accept"],
                                      d["u_sample"], V)
    ok = clean & (dense["flags"] == 0) & (sparse["flags"] == 0)
    assert ok.mean() > 0.7
    np.testing.assert_array_equal(dense["n_accepted"][ok], sparse["n_accepted"][ok])
    np.testing.assert_array_equal(dense["out_tokens"][ok], sparse["out_tokens"][ok])


def test_support_input_errors(oracle_mod):
    lt = np.random.default_rng(3).normal(0, 1, size=(4, 100)).astype(np.float32)
    lt[0, 5] = np.nan
    lt[1, :] = -np.inf
    lt[2, 7] = np.inf
    out = oracle_mod.support_topk(lt, 1.0, 10, 0.9)
    assert (out["ids"][:3] == -1).all() and np.isnan(out["probs"][:3]).all()
    assert (out["flags"][:3] & 8).all() and out["ids"][3].min() >= 0
