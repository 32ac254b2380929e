"""Pins for the confidence-threshold commit oracle ("SDAR" page, section 5).

The pins: hand-derived cases with exactly known confidences, the confidence
against scipy's softmax, the extreme thresholds, the committed tokens against
the greedy oracle's argmax, and input errors."""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

from rejection_sampling_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "commit_cases.json")
CASES = json.load(open(GOLDEN))["commit"]


def _f32(rows):
    return np.array([[-np.inf if v == "-inf" else float(v) for v in r] for r in rows], np.float32)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_commit_hand_cases(oracle_mod, case):
    W = len(case["masked"])
    lt = _f32(case["logits"]).reshape(1, W, case["V"])
    out = oracle_mod.commit_confident(lt, np.array([case["masked"]], np.int32), case["tau"])
    e = case["expect"]
    assert out["commit"][0].tolist() == e["commit"]
    assert out["tokens"][0].tolist() == e["tokens"]
    want = np.array([np.nan if v == "nan" else v for v in e["confidence"]], float)
    np.testing.assert_allclose(out["confidence"][0], want, rtol=0, atol=1e-15)


def _inputs(seed, dtype="f32"):
    return wl.commit_inputs(24, 4, 700, dtype=dtype, seed=seed, masked_frac=0.75)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_commit_confidence_and_tokens_against_libraries(oracle_mod, dtype):
    d = _inputs(1, dtype)
    vals = wl.bf16_bits_to_f32(d["logits"]) if dtype == "bf16" else d["logits"]
    out = oracle_mod.commit_confident(d["logits"], d["masked"], d["tau"])
    p = softmax(vals.astype(np.float64), axis=-1)
    conf = p.max(axis=-1)
    m = d["masked"] != 0
    np.testing.assert_allclose(out["confidence"][m], conf[m], rtol=1e-12)
    assert np.isnan(out["confidence"][~m]).all()
    am = np.argmax(vals, axis=-1)
    c = out["commit"] == 1
    assert (out["tokens"][c] == am[c]).all() and (out["tokens"][~c] == -1).all()
    # the rule itself, from the library confidences
    for b in range(d["B"]):
        mb = m[b]
        if not mb.any():
            assert not c[b].any()
            continue
        above = mb & (conf[b] > d["tau"])
        if above.any():
            assert (c[b] == above).all()
        else:
            first = int(np.argmax(np.where(mb, conf[b], -1.0)))
            assert c[b].tolist() == [i == first for i in range(4)]


def test_commit_extreme_thresholds(oracle_mod):
    d = _inputs(2)
    m = d["masked"] != 0
    low = oracle_mod.commit_confident(d["logits"], d["masked"], -1.0)
    assert ((low["commit"] == 1) == m).all()  # every masked position clears tau < 0
    high = oracle_mod.commit_confident(d["logits"], d["masked"], 1.0)
    per_block = (high["commit"] == 1).sum(axis=1)
    assert (per_block == m.any(axis=1)).all()  # exactly one per block with a masked position


def test_commit_tokens_are_the_greedy_argmax(oracle_mod):
    d = _inputs(3, "bf16")
    out = oracle_mod.commit_confident(d["logits"], d["masked"], d["tau"])
    B, W, V = d["logits"].shape
    g = oracle_mod.verify_greedy(d["logits"].reshape(B * W, 1, V), np.zeros((B * W, 0), np.int32))
    am = g["out_tokens"][:, 0].reshape(B, W)
    c = out["commit"] == 1
    assert (out["tokens"][c] == am[c]).all()


def test_commit_input_errors(oracle_mod):
    d = _inputs(4)
    lt, m = d["logits"].copy(), d["masked"].copy()
    m[0, :] = 1
    lt[0, 1, 5] = np.nan
    m[1, :] = 0
    m[1, 2] = 1
    lt[1, 2, :] = -np.inf
    m[2, 3] = 0
    lt[2, 3, 0] = np.nan  # not masked: not read, no error
    out = oracle_mod.commit_confident(lt, m, d["tau"])
    assert (out["commit"][:2] == -1).all() and (out["tokens"][:2] == -1).all()
    assert out["flags"][0] & 8 and out["flags"][1] & 8
    assert not out["flags"][2] & 8
