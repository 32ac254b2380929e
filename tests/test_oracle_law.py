"""The oracle's output law against Leviathan's theorem.

The pages state the theorem the rule rests on: running the rule reproduces
samples from the target distribution p exactly, whatever q is (Uno article,
"What 'lossless' actually has to mean"; DFlash/DFlash2 guide, FAQ Q1), and a
speculative step accepts with probability 1 - TV(p, q) = sum min(p, q) (Uno
article, "Numbers that don't quite agree with each other", citing Leviathan et
al. Corollary 3.6).  The closed form used here, with m accepted drafts:

    P(n = m, y_0..y_m) = prod_{i<m} min(p_i, q_i)(y_i)
                         * ( max(p_m - q_m, 0)(y_m)   if m < gamma
                             p_gamma(y_gamma)         if m = gamma )

Two kinds of check:
  * exact enumeration: dyadic p, q (every accept threshold and every residual
    CDF boundary is a multiple of 1/4; 1/8 for the sparse lists), all draft
    tuples x weighted by q, and a midpoint grid over each uniform (8 points;
    16 for the sparse lists) pushed through the oracle; no grid point sits on
    a threshold, so the grid integral equals the closed form exactly;
  * Monte Carlo on random logits (x ~ q by Gumbel-max, seeded uniforms) with
    binomial / chi-square bounds.
"""
import itertools
from fractions import Fraction as Fr

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

from rejection_sampling_gb300.workloads import dense_inputs, gumbel_argmax

NG = 8  # grid points per uniform: every threshold below is a multiple of 1/4


def _grid(ng=NG):
    return (np.arange(ng, dtype=np.float64) + 0.5) / ng


def _log32(p):
    with np.errstate(divide="ignore"):
        return np.log(np.array([float(v) for v in p], np.float64)).astype(np.float32)


def _closed_form(ps, qs, bonus):
    """Law over outcomes (n, (y_0..y_n)) for fixed per-position p_j, q_j (Fractions)."""
    G = len(qs)
    V = len(ps[0])
    law = {}
    for m in range(G + 1):
        emitted = m + 1 if (m < G or bonus is not None) else m
        for ys in itertools.product(range(V), repeat=emitted):
            w = Fr(1)
            for i in range(m):
                w *= min(ps[i][ys[i]], qs[i][ys[i]])
            if m < G:
                w *= max(ps[m][ys[m]] - qs[m][ys[m]], Fr(0))
            elif bonus is not None:
                w *= bonus[ys[m]]
            if w:
                law[(m, ys)] = law.get((m, ys), Fr(0)) + w
    return law


def _accumulate(n, toks, weights):
    """Sum weights per outcome (n, tokens[:n+1]) -> dict.  toks [R, L] uses -1 past n."""
    L = toks.shape[1]
    keys = n.astype(np.int64) + 1
    base = int(toks.max()) + 2
    for i in range(L):
        keys = keys * base + (toks[:, i].astype(np.int64) + 1)
    uk, inv = np.unique(keys, return_inverse=True)
    w = np.bincount(inv, weights=weights)
    law = {}
    for k, wk in zip(uk, w):
        if wk == 0:
            continue
        ts = []
        kk = int(k)
        for _ in range(L):
            ts.append(kk % base - 1)
            kk //= base
        nn = kk - 1
        ts = ts[::-1]
        law[(nn, tuple(t for t in ts if t >= 0))] = wk
    return law


def _enumerate_dense(oracle_mod, ps, qs, bonus):
    G, V = len(qs), len(ps[0])
    xs = list(itertools.product(range(V), repeat=G))
    g = _grid()
    grids = np.stack(np.meshgrid(*([g] * (G + 1)), indexing="ij"), -1).reshape(-1, G + 1)
    R = len(xs) * len(grids)
    lt1 = np.stack([_log32(p) for p in ps] + [_log32(bonus)])
    ld1 = np.stack([_log32(q) for q in qs])
    lt = np.broadcast_to(lt1, (R, G + 1, V)).copy()
    ld = np.broadcast_to(ld1, (R, G, V)).copy()
    x = np.repeat(np.array(xs, np.int32), len(grids), axis=0)
    u = np.tile(grids, (len(xs), 1)).astype(np.float32)
    out = oracle_mod.verify_dense(lt, ld, x, u[:, :G], u[:, G], residual=False)
    wx = [np.prod([float(qs[i][xx[i]]) for i in range(G)]) for xx in xs]
    weights = np.repeat(np.array(wx), len(grids)) / len(grids)
    return _accumulate(out["n_accepted"], out["out_tokens"], weights)


def _assert_laws_equal(got, want):
    keys = set(got) | set(want)
    for k in keys:
        g = got.get(k, 0.0)
        w = float(want.get(k, Fr(0)))
        assert abs(g - w) < 1e-12, (k, g, w)


# dyadic distributions: every threshold lands on a multiple of 1/4
P0 = [Fr(1, 2), Fr(1, 4), Fr(1, 8), Fr(1, 8)]
Q0 = [Fr(1, 4)] * 4
P1 = [Fr(1, 8), Fr(3, 8), Fr(3, 8), Fr(1, 8)]
Q1 = [Fr(1, 2), Fr(1, 8), Fr(1, 8), Fr(1, 4)]
P2 = [Fr(1, 4), Fr(1, 4), Fr(1, 2), Fr(0)]


def test_closed_form_is_a_distribution_with_marginal_p():
    law = _closed_form([P0, P1], [Q0, Q1], P2)
    assert sum(law.values()) == 1
    first = [sum(w for (m, ys), w in law.items() if ys[0] == y) for y in range(4)]
    assert first == P0  # Leviathan: the first emitted token is distributed as p_0


def test_dense_exact_enumeration(oracle_mod):
    got = _enumerate_dense(oracle_mod, [P0, P1], [Q0, Q1], P2)
    _assert_laws_equal(got, _closed_form([P0, P1], [Q0, Q1], P2))


def test_dense_exact_enumeration_gamma1(oracle_mod):
    got = _enumerate_dense(oracle_mod, [P1], [Q1], P0)
    _assert_laws_equal(got, _closed_form([P1], [Q1], P0))


def test_sparse_exact_enumeration(oracle_mod):
    # target / draft lists with dyadic probabilities (ids sorted)
    t_ids = [[1, 3, 4, 6], [0, 2, 5, 7], [1, 2, 3, 4]]
    t_pr = [[Fr(3, 8), Fr(1, 4), Fr(1, 4), Fr(1, 8)], [Fr(1, 4)] * 4,
            [Fr(1, 8), Fr(1, 8), Fr(1, 4), Fr(1, 2)]]
    d_ids = [[1, 2, 3, 6], [2, 5, 8, 9]]
    d_pr = [[Fr(1, 8), Fr(1, 4), Fr(1, 2), Fr(1, 8)], [Fr(1, 2), Fr(1, 4), Fr(1, 8), Fr(1, 8)]]
    V, G, k = 10, 2, 4
    dense_p = [[Fr(0)] * V for _ in range(3)]
    dense_q = [[Fr(0)] * V for _ in range(2)]
    for j in range(3):
        for i, pr in zip(t_ids[j], t_pr[j]):
            dense_p[j][i] = pr
    for j in range(2):
        for i, pr in zip(d_ids[j], d_pr[j]):
            dense_q[j][i] = pr
    want = _closed_form(dense_p[:2], dense_q, dense_p[2])

    xs = list(itertools.product(range(k), range(k)))  # indices into the draft lists
    g = _grid(16)
    grids = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    R = len(xs) * len(grids)
    tid = np.broadcast_to(np.array(t_ids, np.int32), (R, 3, k)).copy()
    tp = np.broadcast_to(np.array([[float(v) for v in r] for r in t_pr], np.float32), (R, 3, k)).copy()
    did = np.broadcast_to(np.array(d_ids, np.int32), (R, 2, k)).copy()
    dp = np.broadcast_to(np.array([[float(v) for v in r] for r in d_pr], np.float32), (R, 2, k)).copy()
    x = np.repeat(np.array([[d_ids[0][a], d_ids[1][b]] for a, b in xs], np.int32), len(grids), axis=0)
    u = np.tile(grids, (len(xs), 1)).astype(np.float32)
    out = oracle_mod.verify_sparse(tid, tp, did, dp, x, u[:, :2], u[:, 2], V, residual=False)
    wx = np.repeat(np.array([float(d_pr[0][a] * d_pr[1][b]) for a, b in xs]), len(grids)) / len(grids)
    got = _accumulate(out["n_accepted"], out["out_tokens"], wx)
    _assert_laws_equal(got, want)


def test_anyorder_exact_enumeration(oracle_mod):
    # positions 0..2 with sigma = (2, 0, 1); no bonus token
    P_pos = {2: P0, 0: P1, 1: [Fr(1, 2), Fr(1, 2), Fr(0), Fr(0)]}
    Q_pos = {2: Q0, 0: Q1, 1: [Fr(1, 4)] * 4}
    sigma = [2, 0, 1]
    V, D = 4, 3
    ps = [P_pos[s] for s in sigma]
    qs = [Q_pos[s] for s in sigma]
    want_seq = _closed_form(ps, qs, None)  # outcomes in window order
    lt1 = np.stack([_log32(P_pos[d]) for d in range(D)])
    ld1 = np.stack([_log32(Q_pos[d]) for d in range(D)])
    xs = list(itertools.product(range(V), repeat=3))  # tokens at window indices
    g = _grid()
    grids = np.stack(np.meshgrid(g, g, g, g, indexing="ij"), -1).reshape(-1, 4)
    R = len(xs) * len(grids)
    lt = np.broadcast_to(lt1, (R, D, V)).copy()
    ld = np.broadcast_to(ld1, (R, D, V)).copy()
    tok_pos = np.zeros((len(xs), D), np.int32)
    for r, xx in enumerate(xs):
        for i, s in enumerate(sigma):
            tok_pos[r, s] = xx[i]
    tok = np.repeat(tok_pos, len(grids), axis=0)
    u = np.tile(grids, (len(xs), 1)).astype(np.float32)
    order = np.broadcast_to(np.array(sigma, np.int32), (R, 3)).copy()
    out = oracle_mod.verify_anyorder(lt, ld, order, tok, u[:, :3], u[:, 3], residual=False)
    wx = np.repeat(np.array([float(qs[0][a] * qs[1][b] * qs[2][c]) for a, b, c in xs]), len(grids)) / len(grids)
    # tokens in window order (n accepted, then the resample if n < W, then -1)
    win = out["out_tokens"][:, sigma]
    got = _accumulate(out["n_accepted"], win, wx)
    _assert_laws_equal(got, want_seq)


# ---------------------------------------------------------------------------
# Monte Carlo on random logits (x ~ q, seeded uniforms)
# ---------------------------------------------------------------------------
def _chi2_pvalue(counts, probs):
    """Chi-square p-value of counts against probs, pooling cells expected < 5."""
    exp = probs * counts.sum()
    keep = exp >= 5
    obs, ex = counts[keep], exp[keep]
    if (~keep).any() and exp[~keep].sum() > 0:
        obs = np.append(obs, counts[~keep].sum())
        ex = np.append(ex, exp[~keep].sum())
    return chisquare(obs, ex * obs.sum() / ex.sum())[1]


def _mc_batch(R=200_000, seed=11):
    return dense_inputs(1, 4, 32, dtype="f32", seed=seed, target_sigma=2.0, draft_noise=1.0,
                        repeats=R)


@pytest.fixture(scope="module")
def mc(oracle_mod):
    d = _mc_batch()
    out = oracle_mod.verify_dense(d["target"], d["draft"], d["draft_ids"], d["u_accept"],
                                  d["u_sample"], residual=False)
    p = softmax(d["target"][0].astype(np.float64), axis=-1)
    q = softmax(d["draft"][0].astype(np.float64), axis=-1)
    return d, out, p, q


def test_mc_acceptance_equals_one_minus_tv(mc):
    d, out, p, q = mc
    alpha = np.minimum(p[0], q[0]).sum()  # = 1 - TV(p0, q0)
    acc0 = (out["n_accepted"] > 0).mean()
    R = len(out["n_accepted"])
    sd = np.sqrt(alpha * (1 - alpha) / R)
    assert abs(acc0 - alpha) < 5 * sd, (acc0, alpha, sd)


def test_mc_accept_count_distribution(mc):
    d, out, p, q = mc
    G = 4
    alpha = np.minimum(p[:G], q).sum(-1)
    probs = [np.prod(alpha[:m]) * (1 - alpha[m]) for m in range(G)] + [np.prod(alpha)]
    counts = np.bincount(out["n_accepted"], minlength=G + 1)
    R = counts.sum()
    _, pval = chisquare(counts, np.array(probs) * R)
    assert pval > 1e-3, (counts, np.array(probs) * R)


def test_mc_first_token_is_distributed_as_p0(mc):
    d, out, p, q = mc
    y0 = out["out_tokens"][:, 0]
    assert _chi2_pvalue(np.bincount(y0, minlength=32), p[0]) > 1e-3


def test_mc_every_reached_position_is_distributed_as_p(mc):
    """Token emitted at position j, given position j was reached (n >= j), ~ p_j."""
    d, out, p, q = mc
    for j in range(1, 5):
        reached = out["n_accepted"] >= j
        y = out["out_tokens"][reached, j]
        pval = _chi2_pvalue(np.bincount(y, minlength=32), p[j])
        assert pval > 1e-4, (j, pval)


def test_mc_resample_after_rejection_follows_residual(mc):
    d, out, p, q = mc
    rej = out["n_accepted"] == 0
    y = out["out_tokens"][rej, 0]
    r = np.maximum(p[0] - q[0], 0)
    r /= r.sum()
    counts = np.bincount(y, minlength=32)
    assert counts[r == 0].sum() == 0
    assert _chi2_pvalue(counts, r) > 1e-3


def test_gumbel_draft_sampler_matches_softmax():
    """The workload generator's draft sampler draws x ~ softmax(l)."""
    rng = np.random.default_rng(5)
    l = rng.normal(0, 2, size=16)
    x = gumbel_argmax(rng, np.broadcast_to(l, (100_000, 16)).copy())
    counts = np.bincount(x, minlength=16)
    _, pval = chisquare(counts, softmax(l) * len(x))
    assert pval > 1e-3
