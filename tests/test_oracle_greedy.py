"""Pins for the greedy (T = 0) oracle.

The page's condition for greedy acceptance (DFlash/DFlash2 guide, 4.4) is lost
in extraction; the oracle takes the T -> 0 limit of the stochastic rule.  The
pins check it against hand-derived cases, against that limit computed by the
stochastic (dense) oracle itself, and against numpy's argmax.
"""
import json
import os

import numpy as np
import pytest

from rejection_sampling_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "greedy_cases.json")
CASES = json.load(open(GOLDEN))["greedy"]


def _f32(rows):
    return np.array([[-np.inf if v == "-inf" else float(v) for v in r] for r in rows], np.float32)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_greedy_hand_cases(oracle_mod, case):
    V, G = case["V"], case["gamma"]
    lt = _f32(case["target"]).reshape(1, G + 1, V)
    out = oracle_mod.verify_greedy(lt, np.array(case["draft_ids"], np.int32).reshape(1, G))
    assert int(out["n_accepted"][0]) == case["expect"]["n"]
    assert out["out_tokens"][0].tolist() == case["expect"]["tokens"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_greedy_is_the_zero_temperature_limit_of_the_dense_rule(oracle_mod, seed):
    # Integer logits with a unique maximum per row, scaled by 1000: in fp64
    # softmax every non-maximal entry underflows to exactly 0, so the
    # stochastic rule (accept with min(1, p/q), resample from max(p - q, 0),
    # bonus from p) must give the greedy result for ANY uniforms.
    rng = np.random.default_rng(seed)
    B, G, V = 40, 5, 23
    base = rng.integers(0, 20, size=(B, G + 1, V)).astype(np.float64)
    am = rng.integers(0, V, size=(B, G + 1))
    for b in range(B):
        for j in range(G + 1):
            base[b, j, am[b, j]] = 25.0  # unique maximum
    lt = (base * 1000.0).astype(np.float32)
    ld = rng.normal(0, 1, size=(B, G, V)).astype(np.float32)
    # drafts: the argmax most of the time, otherwise another id
    x = np.where(rng.random((B, G)) < 0.7, am[:, :G], rng.integers(0, V, size=(B, G))).astype(np.int32)
    ua = rng.random((B, G)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    dense = oracle_mod.verify_dense(lt, ld, x, ua, us, residual=False)
    greedy = oracle_mod.verify_greedy(lt, x)
    np.testing.assert_array_equal(dense["n_accepted"], greedy["n_accepted"])
    np.testing.assert_array_equal(dense["out_tokens"], greedy["out_tokens"])
    assert (greedy["n_accepted"] < G).any() and (greedy["n_accepted"] == G).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_matches_numpy_argmax(oracle_mod, dtype):
    rng = np.random.default_rng(7)
    d = wl.greedy_inputs(30, 4, 301, dtype=dtype, seed=3, draft_noise=1.0)
    lt = d["target"]
    vals = wl.bf16_bits_to_f32(lt) if dtype == "bf16" else lt
    out = oracle_mod.verify_greedy(lt, d["draft_ids"])
    am = np.argmax(vals, axis=-1)  # numpy returns the first maximum
    x = d["draft_ids"]
    for b in range(30):
        miss = np.nonzero(x[b] != am[b, :4])[0]
        n = int(miss[0]) if len(miss) else 4
        assert out["n_accepted"][b] == n
        assert out["out_tokens"][b, :n].tolist() == x[b, :n].tolist()
        assert out["out_tokens"][b, n] == am[b, n]
        assert (out["out_tokens"][b, n + 1:] == -1).all()
    del rng


def test_greedy_input_errors(oracle_mod):
    d = wl.greedy_inputs(5, 3, 50, dtype="f32", seed=4)
    lt, x = d["target"].copy(), d["draft_ids"].copy()
    lt[0, 2, 7] = np.nan
    lt[1, 3, :] = -np.inf
    x[2, 1] = 50
    lt[3, 0, 3] = np.inf
    out = oracle_mod.verify_greedy(lt, x)
    assert out["n_accepted"][:4].tolist() == [-1] * 4
    assert (out["out_tokens"][:4] == -1).all()
    assert out["n_accepted"][4] >= 0
