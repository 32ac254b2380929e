"""Helpers for GPU-vs-oracle parity tests.

The bar (spec tolerances):
  * n_accepted and out_tokens bit-exact on every row the oracle does not flag
    (flags: an accept test within 1e-6 of its threshold, an inverse-CDF draw
    within 1e-6 (in units of the sample uniform) of a boundary, a zero
    residual);
  * on flagged rows, the GPU result must still be a valid outcome: the
    accepted prefix equals the drafts, and when n agrees the token lies on the
    oracle's CDF within the tie band;
  * probabilities (accept probabilities, residual distribution) within 1e-5
    relative -- for the residual, relative to the operands p(y) + q(y) of the
    subtraction that produced it.
"""
import numpy as np
import torch

TIE_BAND = 1e-6
PROB_RTOL = 1e-5


def to_dev(a, dev="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def cdf_consistent(w, u, y, band=2 * TIE_BAND):
    """Is token index y a valid inverse-CDF draw of the normalised weights w at
    u, allowing ties within `band`?"""
    if y < 0 or y >= len(w):
        return False
    c = np.cumsum(w)
    lo = c[y - 1] if y > 0 else 0.0
    hi = c[y]
    return (lo - band <= u < hi + band) and (w[y] > 0 or hi - lo < band)


def compare_dense_like(gpu_n, gpu_tok, ora, draft_ids, u_s, G, *, min_clean=0.8,
                       to_index=None):
    """Row-wise comparison.  Returns (clean rows, flagged rows)."""
    on, ot, fl = ora["n_accepted"], ora["out_tokens"], ora["flags"]
    clean = fl == 0
    assert clean.mean() >= min_clean, f"only {clean.mean():.3f} of rows unflagged"
    bad = np.nonzero(clean & ((gpu_n != on) | (gpu_tok != ot).any(-1)))[0]
    assert bad.size == 0, (
        f"{bad.size} unflagged rows differ, first {bad[:5]}: gpu n={gpu_n[bad[:5]]} "
        f"oracle n={on[bad[:5]]} gpu tok={gpu_tok[bad[:3]]} oracle tok={ot[bad[:3]]}")
    # flagged rows: still valid outcomes
    for b in np.nonzero(~clean)[0]:
        n = int(gpu_n[b])
        if fl[b] & 8:  # input error rows must agree exactly
            assert n == -1 and (gpu_tok[b] == -1).all()
            continue
        assert 0 <= n <= G
        assert (gpu_tok[b, :n] == draft_ids[b, :n]).all()
        assert (gpu_tok[b, n + 1:] == -1).all()
        if n == on[b] and ora.get("residual") is not None and ora["residual"] is not None:
            w = ora["residual"][b]
            y = int(gpu_tok[b, n])
            if to_index is not None:  # sparse: vocabulary id -> index in the target list
                y = to_index(b, n, y)
            if not (fl[b] & 4):
                assert cdf_consistent(w, float(u_s[b]), y), (b, y, int(ot[b, n]))
    return int(clean.sum()), int((~clean).sum())


def softmax64(rows):
    r = rows.astype(np.float64)
    m = r.max(-1, keepdims=True)
    e = np.exp(r - m)
    return e / e.sum(-1, keepdims=True)


def widen(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def check_accept_prob(gpu_a, ora_a):
    m = np.isfinite(ora_a)
    np.testing.assert_allclose(gpu_a[m], ora_a[m], rtol=PROB_RTOL, atol=1e-9)


def check_dense_residual(gpu_res, gpu_n, ora, target, draft, G):
    """residual_out within 1e-5 of the operands p + q (divided by T), on rows
    where the GPU and the oracle stopped at the same position."""
    lt = widen(target)
    ld = widen(draft) if G else None
    for b in range(len(ora["n_accepted"])):
        n = int(ora["n_accepted"][b])
        if n != int(gpu_n[b]):
            continue
        if n < 0:
            assert (gpu_res[b] == 0).all()
            continue
        w = ora["residual"][b]
        T = ora["resid_mass"][b]
        p = softmax64(lt[b, n])
        q = softmax64(ld[b, n]) if (n < G and not (ora["flags"][b] & 4)) else np.zeros_like(p)
        atol = PROB_RTOL * (p + q) / T + 1e-12
        err = np.abs(gpu_res[b].astype(np.float64) - w)
        assert (err <= atol + PROB_RTOL * np.abs(w)).all(), (b, err.max())


def check_anyorder_residual(gpu_res, gpu_n, ora, target, draft, order, W):
    """Any-order residual_out within 1e-5 of the operands p + q (divided by T)
    at the stop position sigma(n), on rows where the GPU and the oracle
    stopped at the same window index; all-zero on rows that accepted the
    whole window (no bonus) and on input-error rows."""
    lt, ld = widen(target), widen(draft)
    for b in range(len(ora["n_accepted"])):
        n = int(ora["n_accepted"][b])
        if n != int(gpu_n[b]):
            continue
        if n < 0 or n == W:
            assert (gpu_res[b] == 0).all(), b
            continue
        s = int(order[b, n])
        w = ora["residual"][b]
        T = ora["resid_mass"][b]
        p = softmax64(lt[b, s])
        q = softmax64(ld[b, s]) if not (ora["flags"][b] & 4) else np.zeros_like(p)
        atol = PROB_RTOL * (p + q) / T + 1e-12
        err = np.abs(gpu_res[b].astype(np.float64) - w)
        assert (err <= atol + PROB_RTOL * np.abs(w)).all(), (b, err.max())


def check_anyorder_flagged(gpu_n, gpu_tok, ora, draft_tokens, order, u_s, init):
    """Rows the oracle flags must still hold a valid any-order outcome: the
    accepted prefix (in sigma order) keeps the draft tokens, the token at
    sigma(n) lies on the oracle's CDF within the tie band, the rest of the
    window is -1, and positions outside the window are untouched.  Input-error
    rows must agree exactly (n = -1, the window -1)."""
    fl = ora["flags"]
    B, W = order.shape
    for b in np.nonzero(fl != 0)[0]:
        sig = order[b]
        outside = np.ones(gpu_tok.shape[1], bool)
        outside[sig] = False
        assert (gpu_tok[b, outside] == init[b, outside]).all(), b
        n = int(gpu_n[b])
        if fl[b] & 8:
            assert n == -1 and (gpu_tok[b, sig] == -1).all(), b
            continue
        assert 0 <= n <= W, (b, n)
        assert (gpu_tok[b, sig[:n]] == draft_tokens[b, sig[:n]]).all(), b
        assert (gpu_tok[b, sig[n + 1:]] == -1).all(), b
        if n < W:
            y = int(gpu_tok[b, sig[n]])
            assert y >= 0, b
            if n == int(ora["n_accepted"][b]) and not (fl[b] & 4):
                assert cdf_consistent(ora["residual"][b], float(u_s[b]), y), (b, y)
