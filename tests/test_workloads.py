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
