"""Pins for the windowed multi-round any-order oracle and its cosine window
("Self-Speculative Masked Diffusions", key design 4; the any-order rule of key
design 2).

The pins: one round is the single-round any-order oracle (itself pinned by
hand cases and the exact law); R rounds are that oracle chained over the
shrinking window; exact hand cases; the law of every revealed token (the
target distribution of the round that revealed it); the window's closed forms;
input errors."""
import math

import numpy as np
import pytest

NEG = -np.inf


@pytest.fixture(scope="module")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def _case(rng, B, R, D, V, sigma_t=2.0, noise=0.6):
    ld = rng.normal(0, sigma_t, size=(B, D, V)).astype(np.float32)
    lt = (ld[:, None] + rng.normal(0, noise, size=(B, R, D, V))).astype(np.float32)
    order = np.stack([rng.permutation(D) for _ in range(B)]).astype(np.int32)
    q = np.exp(ld - ld.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    cdf = np.cumsum(q, -1)
    u = rng.random((B, R, D, 1))
    x = np.minimum((u > cdf[:, None]).sum(-1), V - 1).astype(np.int32)  # x ~ q, every round
    ua = rng.random((B, R, D)).astype(np.float32)
    us = rng.random((B, R)).astype(np.float32)
    return lt, ld, order, x, ua, us


def test_one_round_is_the_single_round_rule(oracle_mod):
    rng = np.random.default_rng(1)
    B, D, V = 64, 12, 7
    lt, ld, order, x, ua, us = _case(rng, B, 1, D, V)
    for i0, W in ((0, D), (3, 5), (9, 40)):
        e = min(D, i0 + W)
        o = oracle_mod.anyorder_rounds(lt, ld, order, np.full(B, i0), np.full(B, W), x, ua, us,
                                       tokens_init=np.full((B, D), -5))
        s = oracle_mod.verify_anyorder(lt[:, 0], ld, order[:, i0:e], x[:, 0], ua[:, 0, i0:e], us[:, 0],
                                       out_init=np.full((B, D), -5), residual=False)
        n = s["n_accepted"]
        np.testing.assert_array_equal(o["round_accepts"][:, 0], n)
        np.testing.assert_array_equal(o["n_revealed"], i0 + np.where(n < e - i0, n + 1, n))
        np.testing.assert_array_equal(o["tokens"], s["out_tokens"].clip(min=-5) * (s["out_tokens"] != -1)
                                      + (s["out_tokens"] == -1) * -5)


def test_rounds_are_single_rounds_chained(oracle_mod):
    rng = np.random.default_rng(2)
    B, R, D, V = 48, 4, 10, 5
    lt, ld, order, x, ua, us = _case(rng, B, R, D, V, noise=1.2)
    i0 = rng.integers(0, D, size=B).astype(np.int32)
    win = rng.integers(1, D + 1, size=B).astype(np.int32)
    o = oracle_mod.anyorder_rounds(lt, ld, order, i0, win, x, ua, us, tokens_init=np.full((B, D), -5))
    for b in range(B):
        e = min(D, int(i0[b]) + int(win[b]))
        i = int(i0[b])
        tok = np.full(D, -5, np.int32)
        racc = []
        for r in range(R):
            if i >= e:
                racc.append(-1)
                continue
            s = oracle_mod.verify_anyorder(lt[b:b + 1, r], ld[b:b + 1], order[b:b + 1, i:e], x[b:b + 1, r],
                                           ua[b:b + 1, r, i:e], us[b:b + 1, r],
                                           out_init=tok[None], residual=False)
            n = int(s["n_accepted"][0])
            tok = s["out_tokens"][0].copy()
            tok[tok == -1] = -5  # positions the round left masked stay as they were
            racc.append(n)
            i = i + n + 1 if n < e - i else e
        assert o["n_revealed"][b] == i, b
        np.testing.assert_array_equal(o["round_accepts"][b], racc)
        np.testing.assert_array_equal(o["tokens"][b], tok)


def test_hand_cases(oracle_mod):
    # V = 2, logits in {0, -inf}: every probability is 0, 1/2 or 1.
    # sigma = [2, 0, 1], i0 = 0, window 3, R = 2.
    #   round 0: pos 2 target (.5,.5), draft (.5,.5), x = 1: ratio 1, u .5 < 1 accept;
    #            pos 0 target (1,0), draft (0,1), x = 1: ratio 0, reject; the
    #            residual max(p - q, 0) = (1, 0), u_s .25 -> token 0.
    #   round 1: pos 1 target (0,1), draft (1,0), x = 0: ratio 0, reject;
    #            residual (0, 1) -> token 1.  Window closed: 3 revealed.
    lt = np.full((1, 2, 3, 2), NEG, np.float32)
    ld = np.full((1, 3, 2), NEG, np.float32)
    lt[0, 0, 2] = [0, 0]
    lt[0, 0, 0] = [0, NEG]
    lt[0, 0, 1] = [0, 0]
    lt[0, 1, 1] = [NEG, 0]
    lt[0, 1, 0] = [0, 0]
    lt[0, 1, 2] = [0, 0]
    ld[0, 2] = [0, 0]
    ld[0, 0] = [NEG, 0]
    ld[0, 1] = [0, NEG]
    order = np.array([[2, 0, 1]], np.int32)
    x = np.array([[[1, 0, 1], [1, 0, 1]]], np.int32)  # [r, position]
    ua = np.array([[[0.5, 0.5, 0.5], [0.5, 0.5, 0.5]]], np.float32)  # [r, sigma index]
    us = np.array([[0.25, 0.75]], np.float32)
    o = oracle_mod.anyorder_rounds(lt, ld, order, [0], [3], x, ua, us)
    assert o["n_revealed"].tolist() == [3]
    assert o["round_accepts"].tolist() == [[1, 0]]
    assert o["tokens"].tolist() == [[0, 1, 1]]
    assert o["flags"].tolist() == [0]
    # the same with the draft agreeing at pos 0 (q = p = (1, 0), x = 0):
    ld2 = ld.copy()
    ld2[0, 0] = [0, NEG]
    x2 = x.copy()
    x2[0, 0, 0] = 0
    # round 0: pos 2 accepted, pos 0 (p = q = (1,0), x = 0) accepted, pos 1
    # target (.5,.5), draft (1,0), x = 0: ratio .5, u .5 not < .5 -> reject;
    # residual (0, .5) -> token 1.  One round fills the window; round 1 unused.
    o = oracle_mod.anyorder_rounds(lt, ld2, order, [0], [3], x2, ua, us)
    assert o["round_accepts"].tolist() == [[2, -1]]
    assert o["tokens"].tolist() == [[0, 1, 1]]
    assert o["flags"].tolist() == [1]  # u exactly at min(1, ratio): the accept band flag
    # a window of 1 starting at i0 = 2 (sigma index 2 = position 1): round 0
    # verifies only position 1: target (.5,.5) vs draft (1,0), x = 0, u .25 < .5: accepted
    ua3 = ua.copy()
    ua3[0, 0, 2] = 0.25
    o = oracle_mod.anyorder_rounds(lt, ld2, order, [2], [1], x2, ua3, us, tokens_init=[[9, 9, 9]])
    assert o["round_accepts"].tolist() == [[1, -1]]
    assert o["n_revealed"].tolist() == [3]
    assert o["tokens"].tolist() == [[9, 0, 9]]


def test_law_of_revealed_tokens(oracle_mod):
    # Every reached position is revealed with the target law of that round
    # (accepted with min(p, q), else resampled from max(p - q, 0)), so a
    # position revealed in round r carries p_r.  Targets differ per round.
    rng = np.random.default_rng(7)
    N, R, D, V = 120000, 3, 3, 3
    ld1 = rng.normal(0, 1.0, size=(D, V)).astype(np.float32)
    lt1 = (ld1[None] + rng.normal(0, 1.5, size=(R, D, V))).astype(np.float32)
    lt = np.broadcast_to(lt1, (N, R, D, V))
    ld = np.broadcast_to(ld1, (N, D, V))
    order = np.broadcast_to(np.array([1, 2, 0], np.int32), (N, D))
    q = np.exp(ld1.astype(np.float64))
    q /= q.sum(-1, keepdims=True)
    cdf = np.cumsum(q, -1)
    x = np.minimum((rng.random((N, R, D, 1)) > cdf[None, None]).sum(-1), V - 1).astype(np.int32)
    ua = rng.random((N, R, D)).astype(np.float32)
    us = rng.random((N, R)).astype(np.float32)
    o = oracle_mod.anyorder_rounds(lt, ld, order, np.zeros(N), np.full(N, D), x, ua, us)
    assert (o["n_revealed"] == D).all()  # R = D rounds always reveal the whole window
    p = np.exp(lt1.astype(np.float64))
    p /= p.sum(-1, keepdims=True)
    # the round that revealed sigma index k
    ends = np.cumsum(np.where(o["round_accepts"] >= 0, o["round_accepts"] + 1, 0), axis=1)
    for k in range(D):
        pos = [1, 2, 0][k]
        rk = (ends <= k).sum(axis=1)  # rounds that ended before index k
        for r in range(R):
            sel = rk == r
            m = int(sel.sum())
            if m < 2000:
                continue
            freq = np.bincount(o["tokens"][sel, pos], minlength=V) / m
            sd = np.sqrt(p[r, pos] * (1 - p[r, pos]) / m)
            assert (np.abs(freq - p[r, pos]) < 5 * sd + 1e-12).all(), (k, r, freq, p[r, pos])


def test_cosine_window_closed_forms(oracle_mod):
    cw = oracle_mod.cosine_window
    # from i = 0, a third of the schedule's time: D (1 - cos(pi/6)) = D (1 - sqrt(3)/2)
    assert cw(1000, 0, 1 / 3) == math.ceil(1000 * (1 - math.sqrt(3) / 2))
    # i = D/2 sits at t = 2/3 (cos(pi/3) = 1/2): a third more reaches t = 1
    assert cw(1000, 500, 1 / 3) == 500
    # dtau >= 1 reveals the rest; dtau = 0 still reveals one; done when i = D
    assert [cw(64, i, 1.0) for i in (0, 5, 63)] == [64, 59, 1]
    assert [cw(64, i, 0.0) for i in (0, 30, 63)] == [1, 1, 1]
    assert cw(64, 64, 0.1) == 0
    assert cw(0, 0, 0.1) == -1


@pytest.mark.parametrize("D,dtau", [(256, 0.01), (256, 0.083), (1024, 0.05), (37, 0.2)])
def test_cosine_schedule_covers_the_sequence(oracle_mod, D, dtau):
    # the outer steps i <- i + W(i) stay ahead of the cosine schedule
    # D (1 - cos(pi s dtau / 2)) and finish within ceil(1 / dtau) steps
    i, steps, widths = 0, 0, []
    while i < D:
        w = oracle_mod.cosine_window(D, i, dtau)
        assert 1 <= w <= D - i
        widths.append(w)
        i += w
        steps += 1
        assert i >= D * (1 - math.cos(math.pi * min(1.0, steps * dtau) / 2)) - 1e-6
    assert steps <= math.ceil(1 / dtau - 1e-12)
    # the window grows through the schedule (early steps reveal little)
    assert widths[0] <= widths[len(widths) // 2]


def test_input_errors(oracle_mod):
    rng = np.random.default_rng(3)
    B, R, D, V = 6, 2, 5, 4
    lt, ld, order, x, ua, us = _case(rng, B, R, D, V)
    i0 = np.zeros(B, np.int32)
    win = np.full(B, D, np.int32)
    order[0, 3] = order[0, 1]           # repeated sigma entry inside the window
    i0[1] = D + 1                       # revealed count out of range
    win[2] = 0                          # empty window
    x[3, 0, order[3, 0]] = V            # the first verified draft token out of range
    i0[4] = D                           # nothing left: no round runs, no error
    lt[5, 0, order[5, 0], 0] = np.nan   # the first verified target row has a NaN
    o = oracle_mod.anyorder_rounds(lt, ld, order, i0, win, x, ua, us, tokens_init=np.full((B, D), 9))
    assert o["n_revealed"].tolist()[:4] == [-1, -1, -1, -1]
    assert o["n_revealed"][4] == D and o["n_revealed"][5] == -1
    assert (o["round_accepts"][[0, 1, 2, 3, 5]] == -1).all()
    assert (o["round_accepts"][4] == -1).all()
    assert (o["tokens"][4] == 9).all()
    assert (o["tokens"][[3, 5]] == -1).all()  # the window's positions
    assert (o["tokens"][0, order[0]] == -1).all()  # (row 0: the positions sigma lists)
    assert (o["flags"][[0, 1, 2, 3, 5]] & 8).all() and o["flags"][4] == 0


def test_unreached_rows_are_not_read(oracle_mod):
    # a NaN row past the first rejection of the last round run is never used
    rng = np.random.default_rng(4)
    B, R, D, V = 1, 1, 4, 3
    lt, ld, order, x, ua, us = _case(rng, B, R, D, V)
    order[0] = [0, 1, 2, 3]
    ua[0, 0, 1] = 0.999999  # position 1: rejected unless the ratio exceeds this
    lt[0, 0, 1] = [0, NEG, NEG]
    ld[0, 1] = [0, 0, 0]
    x[0, 0, 1] = 1          # p(1) = 0: rejected
    ua[0, 0, 0] = 0.0       # position 0 accepted (u = 0 < min(1, ratio) unless ratio 0)
    lt[0, 0, 0] = ld[0, 0]
    lt[0, 0, 3, 2] = np.nan  # never reached
    o = oracle_mod.anyorder_rounds(lt, ld, order, [0], [D], x, ua, us)
    assert o["round_accepts"].tolist() == [[1]] and o["n_revealed"].tolist() == [2]
    assert o["flags"][0] & 8 == 0


def test_round_bookkeeping_invariants(oracle_mod):
    # on random inputs: each round reveals its accepted drafts plus, unless it
    # closed the window, the resampled position; the revealed positions are
    # exactly sigma[i0, n); nothing else changes; the rounds run form a prefix
    rng = np.random.default_rng(9)
    B, R, D, V = 200, 5, 24, 6
    lt, ld, order, x, ua, us = _case(rng, B, R, D, V, noise=1.0)
    i0 = rng.integers(0, D + 1, size=B).astype(np.int32)
    win = rng.integers(1, D + 3, size=B).astype(np.int32)
    init = np.full((B, D), -5, np.int32)
    o = oracle_mod.anyorder_rounds(lt, ld, order, i0, win, x, ua, us, tokens_init=init)
    assert (o["n_revealed"] >= 0).all()
    for b in range(B):
        e = min(D, int(i0[b]) + int(win[b]))
        ra = o["round_accepts"][b]
        ran = ra >= 0
        assert (np.diff(ran.astype(int)) <= 0).all()  # a prefix of the rounds ran
        i = int(i0[b])
        for r in np.nonzero(ran)[0]:
            i += int(ra[r]) + (1 if i + int(ra[r]) < e else 0)
            assert i <= e
        assert i == o["n_revealed"][b]
        assert (i == e) or ran.all()  # stopped early only by closing the window
        revealed = set(order[b, i0[b]:i].tolist())
        for pos in range(D):
            if pos in revealed:
                assert 0 <= o["tokens"][b, pos] < V
            else:
                assert o["tokens"][b, pos] == -5
