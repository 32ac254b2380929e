"""The seeded input generators: shapes, determinism and bf16 rounding."""
import numpy as np
import torch

from rejection_sampling_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 100_000), rng.normal(0, 1e-3, 1000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1e30, -1e-30])]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(wl.bf16_bits(x), want)
    back = wl.bf16_bits_to_f32(want)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_named_workload_shapes_and_determinism():
    a = wl.make("dense_v32_g4")
    assert a["target"].shape == (1, 5, 32) and a["draft"].shape == (1, 4, 32)
    assert a["target"].dtype == np.float32
    b = wl.make("dense_v32_g4")
    for k in ("target", "draft", "draft_ids", "u_accept", "u_sample"):
        np.testing.assert_array_equal(a[k], b[k])
    s = wl.make("sparse_b256_g15_k64", B=4)
    assert s["tgt_ids"].shape == (4, 16, 64) and s["drf_ids"].shape == (4, 15, 64)
    assert (np.diff(s["tgt_ids"], axis=-1) > 0).all() and (np.diff(s["drf_ids"], axis=-1) > 0).all()
    overlap = [len(np.intersect1d(s["tgt_ids"][0, j], s["drf_ids"][0, j])) for j in range(15)]
    assert overlap == [32] * 15
    np.testing.assert_allclose(s["tgt_probs"].sum(-1), 1, atol=1e-6)
    o = wl.make("anyorder_b4096_w32_v33", B=8)
    assert o["target"].shape == (8, 32, 33) and o["order"].shape == (8, 32)
    assert all(sorted(r) == list(range(32)) for r in o["order"].tolist())
    u = wl.make("dense_v32_g4", repeats=1000)["u_accept"]
    assert u.dtype == np.float32 and (u >= 0).all() and (u < 1).all()


def test_spikes_present():
    d = wl.dense_inputs(1, 2, 5000, dtype="f32", seed=1, spikes=8, spike_height=12.0)
    assert ((d["target"][0] > 10).sum(-1) >= 8).all()


def test_next_row_generators():
    # greedy: drafts are the argmax of the noisy target, so ids are in range
    g = wl.make("greedy_b64_g7_v128256", B=3)
    assert g["target"].shape == (3, 8, 128256) and g["draft_ids"].shape == (3, 7)
    assert (g["draft_ids"] >= 0).all() and (g["draft_ids"] < 128256).all()
    # commit: one spike per position, a 0/1 mask, tau in (0, 1)
    c = wl.commit_inputs(5, 4, 3000, dtype="f32", seed=2)
    assert c["logits"].shape == (5, 4, 3000) and set(np.unique(c["masked"])) <= {0, 1}
    assert 0 < c["tau"] < 1
    assert ((c["logits"] > 9).sum(-1) >= 1).all()
    # support: the headline's target and draft rows stacked
    s = wl.make("support_b64_g7_v128256", seed=0, B=2)
    assert s["logits"].shape == (2 * 8 + 2 * 7, 128256) and s["K"] == 50
    # rounds: shapes, ranges and determinism
    r1 = wl.rounds_inputs(6, 3, 20, 9, dtype="f32", seed=4, wmax=7)
    r2 = wl.rounds_inputs(6, 3, 20, 9, dtype="f32", seed=4, wmax=7)
    assert r1["target"].shape == (6, 3, 20, 9) and r1["draft"].shape == (6, 20, 9)
    assert r1["draft_tokens"].shape == (6, 3, 20) and r1["u_accept"].shape == (6, 3, 20)
    assert r1["u_sample"].shape == (6, 3)
    assert all(sorted(o) == list(range(20)) for o in r1["order"].tolist())
    assert (r1["revealed"] >= 0).all() and (r1["revealed"] < 20).all()
    assert (r1["window"] >= 1).all() and (r1["window"] <= 7).all()
    assert (r1["draft_tokens"] >= 0).all() and (r1["draft_tokens"] < 9).all()
    for k in ("target", "draft", "order", "revealed", "window", "draft_tokens", "u_accept", "u_sample"):
        np.testing.assert_array_equal(r1[k], r2[k])
    # the per-round draft tokens are fresh draws, not one draw repeated
    assert (r1["draft_tokens"][:, 0] != r1["draft_tokens"][:, 1]).any()
    t8 = wl.make("rounds_b4096_r4_d256_v27", seed=0, B=4)
    assert t8["target"].shape == (4, 4, 256, 27) and t8["dtau"] == 0.05 and "window" not in t8
