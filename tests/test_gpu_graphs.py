"""CUDA-graph capture and replay of the greedy, commit, support-list and
windowed-rounds calls: each call leaves its workspace as it found it, so a
captured call replays to the eager result every time."""
import numpy as np
import pytest
import torch

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
    yield
    torch.cuda.synchronize()


def _capture_and_replay(fn, outputs_of, reset):
    """Run fn eagerly, warm it on a side stream, capture it there, replay it
    three times (outputs reset before each) and compare with the eager run."""
    eager = [t.clone() for t in outputs_of(fn())]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()  # this stream's workspace and the per-device attributes, outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cap = fn()
    for _ in range(3):
        reset(cap)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outputs_of(cap), eager):
            if a.is_floating_point():  # bit for bit (NaN marks positions with no value)
                a, b = a.view(torch.int32), b.view(torch.int32)
            assert torch.equal(a, b)
    assert rs.check() == rs.SV_OK


def test_graph_greedy():
    d = wl.greedy_inputs(5, 3, 30000, dtype="bf16", seed=21)
    args = [to_dev(d[k]) for k in ("target", "draft_ids")]
    _capture_and_replay(lambda: rs.spec_verify_greedy(*args),
                        lambda r: (r.n_accepted, r.out_tokens),
                        lambda r: (r.n_accepted.fill_(-9), r.out_tokens.fill_(-9)))


def test_graph_commit():
    d = wl.commit_inputs(6, 4, 30000, dtype="bf16", seed=22)
    args = [to_dev(d["logits"]), to_dev(d["masked"])]
    _capture_and_replay(lambda: rs.spec_commit_confident(*args, d["tau"], confidence=True),
                        lambda r: (r.commit, r.tokens, r.confidence),
                        lambda r: (r.commit.fill_(-9), r.tokens.fill_(-9), r.confidence.fill_(0)))


def test_graph_support():
    a = wl.bf16_bits(np.random.default_rng(23).normal(0, 3, size=(40, 50000)).astype(np.float32))
    lg = to_dev(a)
    _capture_and_replay(lambda: rs.spec_support_topk(lg, 0.8, 50, 0.95),
                        lambda r: (r.ids, r.probs),
                        lambda r: (r.ids.fill_(-9), r.probs.fill_(0)))


@pytest.mark.parametrize("V", [27, 700])  # the lane-per-position and warp-per-position kernels
def test_graph_rounds(V):
    q = wl.rounds_inputs(24, 3, 48, V, dtype="f32", seed=24, wmax=30)
    args = [to_dev(q[k]) for k in ("target", "draft", "order", "revealed", "window", "draft_tokens",
                                  "u_accept", "u_sample")]
    tok = torch.full((24, 48), -1, dtype=torch.int32, device=args[0].device)

    def run():
        tok.fill_(-1)
        return rs.spec_verify_anyorder_rounds(*args, tokens=tok)

    _capture_and_replay(run,
                        lambda r: (r.tokens, r.n_revealed, r.round_accepts),
                        lambda r: (r.n_revealed.fill_(-9), r.round_accepts.fill_(-9)))
