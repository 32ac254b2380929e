"""GPU parity for windowed multi-round any-order verification:
spec_verify_anyorder_rounds through the C ABI against the oracle on the same
seeded inputs.  Every output is an integer; decisions and draws agree bit for
bit except in sequences the oracle flags (an accept uniform within 1e-6 of
min(1, p/q), or a draw within 1e-6 T of a CDF boundary), which are compared
by what they must still satisfy."""
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


def run_rounds(d, window, tokens_init):
    r = rs.spec_verify_anyorder_rounds(
        to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["order"]), to_dev(d["revealed"]),
        to_dev(np.asarray(window, np.int32)), to_dev(d["draft_tokens"]), to_dev(d["u_accept"]),
        to_dev(d["u_sample"]), tokens=to_dev(np.asarray(tokens_init, np.int32)))
    torch.cuda.synchronize()
    return r.tokens.cpu().numpy(), r.n_revealed.cpu().numpy(), r.round_accepts.cpu().numpy()


def rounds_parity(d, window, min_clean=0.9):
    B, D = d["B"], d["D"]
    init = np.full((B, D), -3, np.int32)
    tok, n, racc = run_rounds(d, window, init)
    o = oracle.anyorder_rounds(d["target"], d["draft"], d["order"], d["revealed"], window,
                               d["draft_tokens"], d["u_accept"], d["u_sample"], tokens_init=init)
    clean = (o["flags"] & 7) == 0
    assert clean.mean() >= min_clean
    np.testing.assert_array_equal(n[clean], o["n_revealed"][clean])
    np.testing.assert_array_equal(racc[clean], o["round_accepts"][clean])
    np.testing.assert_array_equal(tok[clean], o["tokens"][clean])
    # every sequence, flagged or not: progress and bookkeeping hold
    ok = n >= 0
    assert (ok == (o["n_revealed"] >= 0)).all()
    e = np.minimum(D, d["revealed"] + np.asarray(window))
    assert (n[ok] <= e[ok]).all()
    assert ((n[ok] > d["revealed"][ok]) | (d["revealed"][ok] == D)).all()
    assert rs.check() == rs.SV_OK
    return tok, n, racc, o


@pytest.mark.parametrize("B,R,D,V,dtype,wmax", [
    (64, 4, 32, 33, "f32", 32),       # the any-order shape, every window length
    (64, 4, 40, 32, "f32", 32),       # the one-group fast path at its limits (V, R, window)
    (128, 3, 256, 27, "bf16", 24),    # text8-like
    (16, 2, 40, 1000, "f32", 40),     # rows longer than a warp's stride
    (6, 2, 20, 50000, "bf16", 12),    # a large vocabulary
    (40, 1, 16, 7, "f32", 16),        # one round
    (8, 6, 9, 2, "f32", 9),           # two symbols, many rounds
    (12, 3, 24, 512, "bf16", 24),     # the largest vocabulary a lane reduces alone
    (12, 3, 24, 513, "f32", 24),      # the smallest one a warp reduces per position
])
def test_rounds_parity(B, R, D, V, dtype, wmax):
    d = wl.rounds_inputs(B, R, D, V, dtype=dtype, seed=B + R + D + V % 97, wmax=wmax)
    rounds_parity(d, d["window"])


def test_rounds_cosine_windows_text8_like():
    d = wl.make("rounds_b4096_r4_d256_v27", seed=1, B=512)
    window = np.array([oracle.cosine_window(d["D"], int(i), d["dtau"]) for i in d["revealed"]], np.int32)
    tok, n, racc, o = rounds_parity(d, window)
    assert (racc[:, 0] >= 0).all()  # every window has at least one position


@pytest.mark.parametrize("V,D", [(5, 1500), (600, 1200)])
def test_rounds_long_windows(V, D):
    # windows of more than a thousand positions: for small vocabularies groups
    # of 32 lanes (draft statistics kept for the first group only), for large
    # ones groups of eight warps (draft statistics kept for the first 1024
    # window positions); a near-identical target runs deep into the window
    d = wl.rounds_inputs(4, 3, D, V, dtype="f32", seed=11, target_noise=1e-3)
    d["revealed"][:] = [0, 0, 100, D - 1]
    window = np.array([D, D - 300, D - 100, 1], np.int32)
    tok, n, racc, o = rounds_parity(d, window, min_clean=0.5)
    assert n.max() > 1024


def test_rounds_input_errors():
    d = wl.rounds_inputs(6, 2, 5, 4, dtype="f32", seed=3, wmax=5)
    window = np.full(6, 5, np.int32)
    d["revealed"][:] = 0
    d["order"][0, 3] = d["order"][0, 1]            # repeated sigma entry
    d["revealed"][1] = 6                           # revealed count out of range
    window[2] = 0                                  # empty window
    d["draft_tokens"][3, 0, d["order"][3, 0]] = 4  # first verified draft token out of range
    d["revealed"][4] = 5                           # nothing left to verify: no error
    d["target"][5, 0, d["order"][5, 0], 0] = np.nan
    init = np.full((6, 5), 9, np.int32)
    tok, n, racc = run_rounds(d, window, init)
    o = oracle.anyorder_rounds(d["target"], d["draft"], d["order"], d["revealed"], window,
                               d["draft_tokens"], d["u_accept"], d["u_sample"], tokens_init=init)
    np.testing.assert_array_equal(n, o["n_revealed"])
    np.testing.assert_array_equal(racc, o["round_accepts"])
    np.testing.assert_array_equal(tok, o["tokens"])
    assert n.tolist() == [-1, -1, -1, -1, 5, -1]
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    assert rs.check() == rs.SV_OK


def test_rounds_decode_loop_reveals_every_position():
    # the driver a sampler runs: outer steps of one window each (windows from
    # the cosine schedule), fresh per-step logits, until the sequence is
    # complete; the GPU and the oracle walk the same steps
    B, R, D, V, dtau = 32, 3, 48, 11, 0.1
    rng = np.random.default_rng(5)
    tok_g = np.full((B, D), -1, np.int32)
    tok_o = tok_g.copy()
    i = np.zeros(B, np.int32)
    order = np.stack([rng.permutation(D) for _ in range(B)]).astype(np.int32)
    steps = 0
    while (i < D).any():
        d = wl.rounds_inputs(B, R, D, V, dtype="f32", seed=100 + steps)
        d["order"], d["revealed"] = order, i.copy()
        window = np.array([max(1, rs.spec_anyorder_window(D, int(k), dtau)) for k in i], np.int32)
        tok_g, n_g, _ = run_rounds(d, window, tok_g)
        o = oracle.anyorder_rounds(d["target"], d["draft"], order, i, window, d["draft_tokens"],
                                   d["u_accept"], d["u_sample"], tokens_init=tok_o)
        assert (o["flags"] & 7 == 0).all(), "a flagged decision in the loop; pick another seed"
        np.testing.assert_array_equal(n_g, o["n_revealed"])
        tok_o = o["tokens"]
        np.testing.assert_array_equal(tok_g, tok_o)
        assert ((n_g > i) | (i == D)).all()
        i = np.maximum(n_g, i)
        steps += 1
        assert steps <= 60
    assert (tok_g >= 0).all() and (tok_g < V).all()
