"""Oracle against hand-derived cases (tests/golden/hand_cases.json).

Each case's expected outputs were worked out by hand from the rule on the
pages (see the "derivation" string in each case); the logits use only 0 and
-inf so every probability and threshold is an exact dyadic number.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
CASES = json.load(open(GOLDEN))


def _f32(rows):
    def conv(v):
        return -np.inf if v == "-inf" else float(v)
    return np.array([[conv(v) for v in r] for r in rows], dtype=np.float32)


def _check(out, exp, tokens_key="tokens"):
    assert int(out["n_accepted"][0]) == exp["n"]
    assert out["out_tokens"][0].tolist() == exp[tokens_key]
    np.testing.assert_allclose(out["accept_prob"][0], np.array(exp["accept_prob"], float), rtol=0, atol=1e-12)
    assert abs(out["resid_mass"][0] - exp["resid_mass"]) < 1e-12
    np.testing.assert_allclose(out["residual"][0], np.array(exp["residual"], float), rtol=0, atol=1e-12)
    assert int(out["flags"][0]) == exp["flags"]


@pytest.mark.parametrize("case", CASES["dense"], ids=[c["name"] for c in CASES["dense"]])
def test_dense_hand_cases(oracle_mod, case):
    V, G = case["V"], case["gamma"]
    lt = _f32(case["target"]).reshape(1, G + 1, V)
    ld = _f32(case["draft"]).reshape(1, G, V) if G else np.zeros((1, 0, V), np.float32)
    out = oracle_mod.verify_dense(lt, ld, np.array([case["draft_ids"]], np.int32).reshape(1, G),
                                  np.array([case["u_accept"]], np.float32).reshape(1, G),
                                  np.array([case["u_sample"]], np.float32))
    _check(out, case["expect"])


@pytest.mark.parametrize("case", CASES["dense"], ids=[c["name"] for c in CASES["dense"]])
def test_dense_hand_cases_bf16(oracle_mod, case):
    """0 and -inf are exact in bf16: the bf16 path must give identical results."""
    from rejection_sampling_gb300.workloads import bf16_bits
    V, G = case["V"], case["gamma"]
    lt = bf16_bits(_f32(case["target"])).reshape(1, G + 1, V)
    ld = bf16_bits(_f32(case["draft"]).reshape(1, G, V)) if G else np.zeros((1, 0, V), np.uint16)
    out = oracle_mod.verify_dense(lt, ld, np.array([case["draft_ids"]], np.int32).reshape(1, G),
                                  np.array([case["u_accept"]], np.float32).reshape(1, G),
                                  np.array([case["u_sample"]], np.float32))
    _check(out, case["expect"])


@pytest.mark.parametrize("case", CASES["sparse"], ids=[c["name"] for c in CASES["sparse"]])
def test_sparse_hand_cases(oracle_mod, case):
    G = case["gamma"]
    out = oracle_mod.verify_sparse(
        np.array([case["tgt_ids"]], np.int32), np.array([case["tgt_probs"]], np.float32),
        np.array([case["drf_ids"]], np.int32), np.array([case["drf_probs"]], np.float32),
        np.array([case["draft_tokens"]], np.int32), np.array([case["u_accept"]], np.float32),
        np.array([case["u_sample"]], np.float32), case["V"])
    _check(out, case["expect"])


@pytest.mark.parametrize("case", CASES["anyorder"], ids=[c["name"] for c in CASES["anyorder"]])
def test_anyorder_hand_cases(oracle_mod, case):
    D, V = case["D"], case["V"]
    lt = _f32(case["target"]).reshape(1, D, V)
    ld = _f32(case["draft"]).reshape(1, D, V)
    out = oracle_mod.verify_anyorder(lt, ld, np.array([case["order"]], np.int32),
                                     np.array([case["draft_tokens"]], np.int32),
                                     np.array([case["u_accept"]], np.float32),
                                     np.array([case["u_sample"]], np.float32))
    _check(out, case["expect"])
