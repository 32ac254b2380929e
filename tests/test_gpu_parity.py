"""GPU parity: the CUDA kernels through the C ABI against the fp64 oracle on
the same seeded inputs (see tests/parity_util.py for the bar)."""
import numpy as np
import pytest
import torch

import oracle
import rejection_sampling_gb300 as rs
from rejection_sampling_gb300 import workloads as wl
from parity_util import (check_accept_prob, check_anyorder_flagged, check_anyorder_residual,
                         check_dense_residual, compare_dense_like, to_dev, softmax64, widen)

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


def run_dense(d, residual=True, accept_prob=True):
    r = rs.spec_verify_dense(to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["draft_ids"]),
                             to_dev(d["u_accept"]), to_dev(d["u_sample"]), residual=residual,
                             accept_prob=accept_prob)
    torch.cuda.synchronize()
    return (r.n_accepted.cpu().numpy(), r.out_tokens.cpu().numpy(),
            None if r.residual is None else r.residual.cpu().numpy(),
            None if r.accept_prob is None else r.accept_prob.cpu().numpy())


def oracle_dense(d, residual=True):
    return oracle.verify_dense(d["target"], d["draft"], d["draft_ids"], d["u_accept"],
                               d["u_sample"], residual=residual)


def dense_parity(d, min_clean=0.8, residual=True):
    n, tok, res, acc = run_dense(d, residual=residual)
    o = oracle_dense(d, residual=True)
    compare_dense_like(n, tok, o, d["draft_ids"], d["u_sample"], d["gamma"], min_clean=min_clean)
    check_accept_prob(acc, o["accept_prob"])
    if residual:
        check_dense_residual(res, n, o, d["target"], d["draft"], d["gamma"])
    assert rs.check() == rs.SV_OK
    return n, tok, o


# ---------------------------------------------------------------------------
# dense, large vocabularies (statistics kernel + row kernel); every case here
# has (gamma + 1) * V too large for one warp's shared-memory block, or more
# than 32 positions
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,G,V,dtype", [
    (3, 7, 20000, "bf16"),     # several units per row, ragged last piece
    (9, 40, 1024, "bf16"),     # exactly one piece per row
    (2, 0, 50000, "bf16"),     # gamma = 0: plain categorical draw from p_0
    (1, 15, 70001, "bf16"),    # odd V: rows not 16-byte aligned -> plain-copy path
    (5, 3, 30000, "f32"),
    (4, 2, 12289, "f32"),      # odd V in fp32 (unaligned rows)
    (2, 40, 3000, "bf16"),     # gamma + 1 > 32 routes to the fused kernel
    (70, 2, 5000, "bf16"),     # many rows, small clusters
    (3, 4, 200000, "bf16"),    # 196 pieces per row: block-wide draw over on-chip masses
    (2, 3, 530001, "f32"),     # 1036 pieces per row, unaligned: masses in the workspace
    (1, 255, 2048, "bf16"),    # the largest gamma: 256 positions per row
    (400, 33, 1024, "bf16"),   # more rows than SMs: one CTA per row
])
def test_dense_fused_parity(B, G, V, dtype):
    d = wl.dense_inputs(B, G, V, dtype=dtype, seed=B * 1000 + G * 10 + V % 97, target_sigma=3.0,
                        draft_noise=0.5)
    dense_parity(d, min_clean=0.5)


def test_dense_full_block16_v151936():
    d = wl.make("dense_v151936_g15", seed=0)
    dense_parity(d, min_clean=0.0)


def test_dense_full_b64_v128256():
    d = wl.make("dense_b64_g7_v128256", seed=0)
    n, tok, o = dense_parity(d, min_clean=0.8)
    # tau in [1, gamma + 1]
    assert ((tok >= 0).sum(-1) == n + 1).all()


@pytest.mark.parametrize("path", ["fused", "split"])
def test_dense_forced_paths(path, monkeypatch):
    """Both large-vocabulary paths on the headline and the 16-position
    workloads (the automatic choice takes the two-kernel path for the first and
    the single-pass kernel for the second; the switch forces the other)."""
    monkeypatch.setenv("SPEC_VERIFY_DENSE_KERNELS", path)
    dense_parity(wl.make("dense_b64_g7_v128256", seed=5), min_clean=0.8)
    dense_parity(wl.make("dense_v151936_g15", seed=1), min_clean=0.0)
    dense_parity(wl.dense_inputs(5, 3, 30000, dtype="f32", seed=77, target_sigma=3.0,
                                 draft_noise=0.5), min_clean=0.5)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_dense_b64_v128256_more_seeds(seed):
    d = wl.make("dense_b64_g7_v128256", seed=seed)
    dense_parity(d, min_clean=0.8, residual=False)


# ---------------------------------------------------------------------------
# dense, small vocabulary (warp per row)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,G,V,dtype", [
    (1, 4, 32, "f32"), (300, 4, 32, "f32"), (200, 31, 33, "f32"), (100, 0, 100, "bf16"),
    (64, 6, 257, "bf16"), (50, 2, 1000, "f32"),
    (9, 1, 4096, "bf16"),      # few long rows: the warp computes each row's statistics
    (400, 1, 4096, "bf16"),    # the same, many rows
    (50, 30, 384, "f32"),      # one lane per row, sums over more than 256 terms
    (3, 0, 12287, "f32"),      # the longest row one warp holds
])
def test_dense_small_parity(B, G, V, dtype):
    d = wl.dense_inputs(B, G, V, dtype=dtype, seed=G * 7 + V, target_sigma=2.0, draft_noise=1.0)
    dense_parity(d, min_clean=0.9)


def test_dense_v32_exact_law_million_repeats():
    """1e6 rows with the same logits and fresh (x ~ q, u): the GPU's output law
    equals Leviathan's closed form; every unflagged row equals the oracle."""
    from scipy.stats import chisquare
    R = 1_000_000
    d = wl.make("dense_v32_g4", seed=0, repeats=R)
    n, tok, _, _ = run_dense(d, residual=False, accept_prob=False)
    o = oracle_dense(d, residual=False)
    compare_dense_like(n, tok, o, d["draft_ids"], d["u_sample"], 4, min_clean=0.99)
    p = softmax64(d["target"][0])
    q = softmax64(d["draft"][0])
    alpha = np.minimum(p[:4], q).sum(-1)
    probs = np.array([np.prod(alpha[:m]) * (1 - alpha[m]) for m in range(4)] + [np.prod(alpha)])
    counts = np.bincount(n, minlength=5)
    assert chisquare(counts, probs * R)[1] > 1e-3
    for j in range(5):  # token at every reached position ~ p_j
        y = tok[n >= j, j]
        c = np.bincount(y, minlength=32).astype(float)
        e = p[j] * len(y)
        k = e >= 5
        obs = np.append(c[k], c[~k].sum())
        ex = np.append(e[k], e[~k].sum())
        if ex[-1] == 0:
            obs, ex = obs[:-1], ex[:-1]
        assert chisquare(obs, ex * obs.sum() / ex.sum())[1] > 1e-4, j


# ---------------------------------------------------------------------------
# sparse top-k
# ---------------------------------------------------------------------------
def _sparse_run(s):
    r = rs.spec_verify_sparse(to_dev(s["tgt_ids"]), to_dev(s["tgt_probs"]), to_dev(s["drf_ids"]),
                              to_dev(s["drf_probs"]), to_dev(s["draft_tokens"]),
                              to_dev(s["u_accept"]), to_dev(s["u_sample"]), s["V"], residual=True,
                              accept_prob=True)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in r]


def _sparse_parity(s):
    n, tok, res, acc = _sparse_run(s)
    o = oracle.verify_sparse(s["tgt_ids"], s["tgt_probs"], s["drf_ids"], s["drf_probs"],
                             s["draft_tokens"], s["u_accept"], s["u_sample"], s["V"])

    def to_index(b, nn, y):
        return int(np.searchsorted(s["tgt_ids"][b, nn], y))

    compare_dense_like(n, tok, o, s["draft_tokens"], s["u_sample"], s["gamma"], min_clean=0.95,
                       to_index=to_index)
    check_accept_prob(acc, o["accept_prob"])
    np.testing.assert_allclose(res, o["residual"], rtol=1e-5, atol=1e-7)
    assert rs.check() == rs.SV_OK


def test_sparse_full_b256_k64():
    _sparse_parity(wl.make("sparse_b256_g15_k64", seed=0))


@pytest.mark.parametrize("B,G,k", [(32, 0, 64), (16, 3, 5), (8, 31, 200), (40, 7, 33)])
def test_sparse_shapes(B, G, k):
    _sparse_parity(wl.sparse_inputs(B, G, 151936, k=k, seed=B + G + k))


# ---------------------------------------------------------------------------
# any-order
# ---------------------------------------------------------------------------
def _anyorder_parity(a, min_clean=0.95):
    B, D = a["B"], a["D"]
    init = np.full((B, D), -7, np.int32)
    r = rs.spec_verify_anyorder(to_dev(a["target"]), to_dev(a["draft"]), to_dev(a["order"]),
                                to_dev(a["draft_tokens"]), to_dev(a["u_accept"]),
                                to_dev(a["u_sample"]), out_tokens=to_dev(init), residual=True,
                                accept_prob=True)
    torch.cuda.synchronize()
    n, tok, res, acc = [t.cpu().numpy() for t in r]
    o = oracle.verify_anyorder(a["target"], a["draft"], a["order"], a["draft_tokens"],
                               a["u_accept"], a["u_sample"], out_init=init)
    clean = o["flags"] == 0
    assert clean.mean() >= min_clean
    assert (n[clean] == o["n_accepted"][clean]).all()
    assert (tok[clean] == o["out_tokens"][clean]).all()
    check_accept_prob(acc, o["accept_prob"])
    check_anyorder_residual(res, n, o, a["target"], a["draft"], a["order"], a["W"])
    check_anyorder_flagged(n, tok, o, a["draft_tokens"], a["order"], a["u_sample"], init)
    assert rs.check() == rs.SV_OK


def test_anyorder_full_b4096_w32_v33():
    _anyorder_parity(wl.make("anyorder_b4096_w32_v33", seed=0))


@pytest.mark.parametrize("B,D,W,V,dtype", [
    (64, 48, 16, 33, "f32"), (64, 32, 32, 27, "bf16"), (32, 8, 5, 200, "f32"),
    # whole-window fp32 blocks copied in two groups (D = W, 16-byte multiples):
    (50, 12, 12, 33, "f32"),    # a lane per row's statistics
    (40, 4, 4, 101, "f32"),     # few long rows: the warp takes each row's statistics
    (40, 8, 8, 1001, "f32"),
])
def test_anyorder_shapes(B, D, W, V, dtype):
    _anyorder_parity(wl.anyorder_inputs(B, D, W, V, dtype=dtype, seed=D + W + V))


# ---------------------------------------------------------------------------
# special cases and edges
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V", [32, 20000])
def test_q_equals_p_accepts_everything(V):
    d = wl.dense_inputs(8, 5, V, dtype="bf16", seed=4)
    d["draft"] = np.ascontiguousarray(d["target"][:, :5])
    d["draft_ids"] = wl.gumbel_argmax(np.random.default_rng(0), d["draft"]).astype(np.int32)
    n, tok, _, acc = run_dense(d, residual=False)
    assert (n == 5).all() and (acc == 1.0).all()
    assert (tok[:, :5] == d["draft_ids"]).all()


@pytest.mark.parametrize("V", [50, 30000])
def test_disjoint_supports_reject_at_zero(V):
    rng = np.random.default_rng(5)
    B, G = 6, 3
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    lt[:, :, V // 2:] = -np.inf
    ld[:, :, :V // 2] = -np.inf
    d = dict(target=lt, draft=ld, draft_ids=wl.gumbel_argmax(rng, ld).astype(np.int32),
             u_accept=rng.random((B, G), dtype=np.float32), u_sample=rng.random(B, dtype=np.float32),
             gamma=G)
    n, tok, o = dense_parity(d, min_clean=0.5)
    assert (n == 0).all() and (tok[:, 0] < V // 2).all()


@pytest.mark.parametrize("V", [40, 9000])
def test_input_errors_flag_rows(V):
    d = wl.dense_inputs(5, 3, V, dtype="f32", seed=6)
    d["target"][0, 1, 4] = np.nan
    d["draft"][1, 2, :] = -np.inf
    d["draft_ids"][2, 0] = V
    d["target"][3, 3, 0] = np.inf
    n, tok, res, acc = run_dense(d)
    assert n[:4].tolist() == [-1] * 4 and n[4] >= 0
    assert (tok[:4] == -1).all()
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    assert rs.check() == rs.SV_OK  # the status word was cleared
    o = oracle_dense(d)
    assert (tok[4] == o["out_tokens"][4]).all() or o["flags"][4]


def test_empty_batch_and_argument_errors():
    dev = torch.device("cuda")
    z = torch.empty(0, 4, 100, dtype=torch.bfloat16, device=dev)
    r = rs.spec_verify_dense(z, torch.empty(0, 3, 100, dtype=torch.bfloat16, device=dev),
                             torch.empty(0, 3, dtype=torch.int32, device=dev),
                             torch.empty(0, 3, device=dev), torch.empty(0, device=dev))
    assert r.n_accepted.numel() == 0
    with pytest.raises(rs.SpecVerifyError):
        t = torch.zeros(1, 300, 100, dtype=torch.bfloat16, device=dev)  # gamma = 299 > 255
        rs.spec_verify_dense(t, t[:, :299], torch.zeros(1, 299, dtype=torch.int32, device=dev),
                             torch.zeros(1, 299, device=dev), torch.zeros(1, device=dev))


def test_repeated_calls_reuse_workspace_and_graph_replay():
    d = wl.dense_inputs(6, 7, 25000, dtype="bf16", seed=8)
    args = [to_dev(d[k]) for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")]
    first = rs.spec_verify_dense(*args)
    for _ in range(3):  # the workspace counters reset themselves
        again = rs.spec_verify_dense(*args)
        assert torch.equal(first.n_accepted, again.n_accepted)
        assert torch.equal(first.out_tokens, again.out_tokens)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        warm = rs.spec_verify_dense(*args)  # creates this stream's workspace outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cap = rs.spec_verify_dense(*args)
    for _ in range(3):
        cap.n_accepted.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(cap.n_accepted, first.n_accepted)
        assert torch.equal(cap.out_tokens, first.out_tokens)
    assert torch.equal(warm.out_tokens, first.out_tokens)


def test_workspace_returns_to_zero_across_geometries():
    """Every successful call leaves the whole workspace zero (apart from the
    sticky status word), so calls of different sizes can share it."""
    from rejection_sampling_gb300 import _binding as bnd
    dev = torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.Stream()
    cases = [(3, 7, 20000, "bf16", True, False), (9, 1, 4096, "bf16", False, False),
             (5, 3, 30000, "f32", True, True), (2, 40, 3000, "bf16", False, False),
             (1, 15, 70001, "bf16", True, False), (12, 3, 9000, "f32", False, True)]
    for (B, G, V, dt, resid, bad) in cases:
        d = wl.dense_inputs(B, G, V, dtype=dt, seed=B + V)
        if bad:
            d["draft_ids"][0, 0] = V  # one invalid row
        with torch.cuda.stream(s):
            rs.spec_verify_dense(to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["draft_ids"]),
                                 to_dev(d["u_accept"]), to_dev(d["u_sample"]), residual=resid,
                                 stream=s)
        s.synchronize()
        ws = bnd._ws_cache[(dev.index, s.cuda_stream)].cpu().numpy()
        status = ws[12:16].view(np.uint32)[0]
        ws[12:16] = 0
        assert not ws.any(), (B, G, V, np.nonzero(ws)[0][:10])
        assert status == (1 if bad else 0)
        assert rs.check(dev, s) == (rs.SV_ERR_DEVICE_INPUT if bad else rs.SV_OK)
