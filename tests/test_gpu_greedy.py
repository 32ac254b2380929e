"""GPU parity for greedy (T = 0) verification: spec_verify_greedy through the C
ABI against the oracle on the same seeded inputs.  Every output is an integer
decided by exact comparisons of the (widened) logits, so the bar is bit-exact
n_accepted and out_tokens on every row."""
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


def run_greedy(target, draft_ids):
    r = rs.spec_verify_greedy(to_dev(target), to_dev(draft_ids))
    torch.cuda.synchronize()
    return r.n_accepted.cpu().numpy(), r.out_tokens.cpu().numpy()


def greedy_parity(d):
    n, tok = run_greedy(d["target"], d["draft_ids"])
    o = oracle.verify_greedy(d["target"], d["draft_ids"])
    np.testing.assert_array_equal(n, o["n_accepted"])
    np.testing.assert_array_equal(tok, o["out_tokens"])
    assert rs.check() == rs.SV_OK
    return n


@pytest.mark.parametrize("B,G,V,dtype,noise", [
    (3, 7, 20000, "bf16", 0.3),      # several pieces per row, ragged last piece
    (1, 15, 151936, "bf16", 0.3),    # one long block
    (5, 3, 30001, "f32", 0.3),       # odd V: rows not 16-byte aligned (plain loads)
    (7, 4, 12287, "bf16", 0.3),      # odd V in bf16
    (2, 0, 50000, "bf16", 0.3),      # gamma = 0: the argmax alone
    (400, 1, 1000, "bf16", 0.5),     # many rows, one piece each
    (1, 255, 2048, "bf16", 0.0),     # the largest gamma; noise 0: drafts all accepted
    (9, 4, 33, "f32", 1.0),          # tiny rows
    (4, 2, 1, "f32", 1.0),           # V = 1: every draft is id 0
])
def test_greedy_parity(B, G, V, dtype, noise):
    d = wl.greedy_inputs(B, G, V, dtype=dtype, seed=B * 100 + G * 7 + V % 89, draft_noise=noise)
    greedy_parity(d)


def test_greedy_full_b64_v128256():
    d = wl.greedy_inputs(64, 7, 128256, dtype="bf16", seed=0)
    n = greedy_parity(d)
    assert (n >= 0).all()


def test_greedy_ties_take_the_smallest_id():
    # equal maxima in different pieces and in the same vector: the smallest id
    rng = np.random.default_rng(11)
    B, G, V = 6, 3, 40000
    lt = rng.normal(0, 1, size=(B, G + 1, V)).astype(np.float32)
    for b in range(B):
        for j in range(G + 1):
            ids = sorted(rng.choice(V, size=3, replace=False))
            lt[b, j, ids] = 50.0
    x = np.zeros((B, G), np.int32)
    for b in range(B):
        for j in range(G):
            m = np.nonzero(lt[b, j] == 50.0)[0]
            # even rows draft the first tied id everywhere (all accepted); odd
            # rows draft a later tied id somewhere (rejected there)
            x[b, j] = m[0] if (b % 2 == 0 or (b + j) % 3) else m[-1]
    d = dict(target=wl.bf16_bits(lt), draft_ids=x)
    n = greedy_parity(d)
    assert (n < G).any() and (n == G).any()


def test_greedy_input_errors_flag_rows():
    d = wl.greedy_inputs(5, 3, 9000, dtype="f32", seed=6)
    t, x = d["target"].copy(), d["draft_ids"].copy()
    t[0, 2, 4] = np.nan
    t[1, 3, :] = -np.inf
    x[2, 0] = 9000
    t[3, 0, 8999] = np.inf
    n, tok = run_greedy(t, x)
    o = oracle.verify_greedy(t, x)
    np.testing.assert_array_equal(n, o["n_accepted"])
    np.testing.assert_array_equal(tok, o["out_tokens"])
    assert n[:4].tolist() == [-1] * 4 and n[4] >= 0
    assert rs.check() == rs.SV_ERR_DEVICE_INPUT
    assert rs.check() == rs.SV_OK  # the status word is cleared by the check


def test_greedy_leaves_the_workspace_zero_and_shares_it_with_dense():
    dev = torch.device("cuda", torch.cuda.current_device())
    rs.check()  # clear a status bit an earlier test may have left
    g = wl.greedy_inputs(3, 5, 70000, dtype="bf16", seed=8)
    greedy_parity(g)
    sp = int(torch.cuda.current_stream(dev).cuda_stream)
    ws = rs.get_workspace(rs.workspace_size(3, 5, 70000), dev, sp)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
    # a dense call of another shape on the same workspace, then greedy again
    d = wl.dense_inputs(2, 3, 90000, dtype="bf16", seed=9)
    r = rs.spec_verify_dense(to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["draft_ids"]),
                             to_dev(d["u_accept"]), to_dev(d["u_sample"]))
    torch.cuda.synchronize()
    o = oracle.verify_dense(d["target"], d["draft"], d["draft_ids"], d["u_accept"], d["u_sample"],
                            residual=False)
    assert (r.n_accepted.cpu().numpy() == o["n_accepted"]).mean() >= 0.5
    greedy_parity(g)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
