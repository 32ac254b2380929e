"""Seeded synthetic inputs for speculative verification.

This module only *generates* inputs; it holds none of the verification
arithmetic (no softmax, no ratio, no residual, no inverse CDF).  Draft tokens
are drawn with the Gumbel-max trick, x = argmax(l + G) with G ~ Gumbel(0, 1),
which samples x ~ softmax(l) without computing a softmax.  Draft tokens are
always sampled from the *rounded* draft logits, so q is exactly the
distribution the draft came from (the Uno article's I-DLM lesson: a q that is
not the sampling distribution breaks losslessness).

All randomness comes from ``numpy.random.default_rng(seed)`` (PCG64).  bf16
tensors are produced by round-to-nearest-even from fp32 and returned as raw
uint16 bits; fp32 tensors as float32.  The same arrays feed the oracle and the
GPU library.

Workloads (sizes and distributions of the five verification workloads):

=========================  ===================================================
``dense_v32_g4``           B=1, gamma=4, V=32, fp32; target ~ N(0, 2^2),
                           draft = target + N(0, 1^2); seed 0.  ``repeats``
                           replicates the logits over rows with fresh x, u.
``dense_v151936_g15``      B=1, gamma=15, V=151936, bf16; target ~ N(0, 3^2)
                           plus +12 at 8 distinct random ids per row;
                           draft = target + N(0, 0.7^2).
``dense_b64_g7_v128256``   B=64, gamma=7, V=128256, bf16; target ~ N(0, 3^2),
                           draft = target + N(0, 0.5^2).
``sparse_b256_g15_k64``    B=256, gamma=15, V=151936, k=64 (id, prob) lists,
                           Zipf(1.1) ids, 50% target/draft id overlap.
``anyorder_b4096_w32_v33`` B=4096, D=W=32, V=33, fp32; draft ~ N(0, 2^2),
                           target = draft + N(0, 0.4^2); sigma a random
                           permutation per sequence.
``greedy_b64_g7_v128256``  greedy (T = 0) verification on the headline shape:
                           B=64, gamma=7, V=128256, bf16 target ~ N(0, 3^2);
                           draft ids = argmax of target + N(0, 0.5^2).
``support_b64_g7_v128256`` sparse support lists (temperature 1, top-k 50,
                           top-p 0.95) for the 64 x (8 + 7) target and draft
                           rows of ``dense_b64_g7_v128256``.
``commit_b64_w4_v151936``  confidence-threshold commit: 64 blocks of 4
                           positions (SDAR block length), V=151936, bf16
                           logits ~ N(0, 3^2) plus one spike of height
                           U(10, 40) per position; 3/4 of the positions still
                           masked; tau = 0.9.
=========================  ===================================================
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits", "bf16_bits_to_f32", "gumbel_argmax", "dense_inputs", "greedy_inputs", "commit_inputs",
    "sparse_inputs", "anyorder_inputs", "WORKLOADS", "make",
]


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 by round-to-nearest-even; returns the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    # keep infinities exact (the add above cannot overflow finite inputs of this range)
    inf_mask = np.isinf(x)
    if inf_mask.any():
        out[inf_mask] = (u[inf_mask] >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32 (16-bit shift)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _as_f64(logits: np.ndarray) -> np.ndarray:
    if logits.dtype == np.uint16:
        return bf16_bits_to_f32(logits).astype(np.float64)
    return logits.astype(np.float64)


# ---------------------------------------------------------------------------
# sampling helpers (input generation only)
# ---------------------------------------------------------------------------
def gumbel_argmax(rng: np.random.Generator, log_weights: np.ndarray, chunk_rows: int = 64) -> np.ndarray:
    """x ~ Categorical(softmax(log_weights)) along the last axis, by Gumbel-max.

    -inf entries are never chosen.  Processes rows in chunks to bound memory.
    """
    lw = np.asarray(log_weights)
    lead = lw.shape[:-1]
    V = lw.shape[-1]
    flat = lw.reshape(-1, V)
    out = np.empty(flat.shape[0], dtype=np.int32)
    for s in range(0, flat.shape[0], chunk_rows):
        blk = _as_f64(flat[s:s + chunk_rows]) if flat.dtype == np.uint16 else flat[s:s + chunk_rows].astype(np.float64)
        u = rng.random(blk.shape)
        g = -np.log(-np.log(np.maximum(u, 1e-300)))
        out[s:s + chunk_rows] = np.argmax(blk + g, axis=-1)
    return out.reshape(lead)


def _uniform_f32(rng: np.random.Generator, shape) -> np.ndarray:
    """fp32 uniforms in [0, 1)."""
    return rng.random(shape, dtype=np.float32)


# ---------------------------------------------------------------------------
# dense
# ---------------------------------------------------------------------------
def dense_inputs(B: int, gamma: int, V: int, *, dtype: str = "bf16", seed: int = 0,
                 target_sigma: float = 3.0, draft_noise: float = 0.5, spikes: int = 0,
                 spike_height: float = 12.0, repeats: int = 1) -> dict:
    """Dense verification inputs.

    target [B*repeats, gamma+1, V], draft [B*repeats, gamma, V] (draft = first
    gamma target rows + noise), draft_ids sampled from the rounded draft logits,
    u_accept [.., gamma], u_sample [..].  ``repeats > 1`` replicates the same
    logits over rows with fresh draft ids and uniforms (an exact-law batch).
    """
    rng = np.random.default_rng(seed)
    lt = rng.normal(0.0, target_sigma, size=(B, gamma + 1, V)).astype(np.float32)
    if spikes:
        for b in range(B):
            for j in range(gamma + 1):
                ids = rng.choice(V, size=min(spikes, V), replace=False)
                lt[b, j, ids] += np.float32(spike_height)
    ld = (lt[:, :gamma] + rng.normal(0.0, draft_noise, size=(B, gamma, V))).astype(np.float32)
    if dtype == "bf16":
        lt_q, ld_q = bf16_bits(lt), bf16_bits(ld)
    elif dtype == "f32":
        lt_q, ld_q = lt, ld
    else:
        raise ValueError(dtype)
    if repeats > 1:
        lt_q = np.repeat(lt_q, repeats, axis=0)
        ld_q = np.repeat(ld_q, repeats, axis=0)
    Bt = B * repeats
    if gamma > 0:
        if repeats > 1:
            # same draft logits in every repeat: sample per repeat block
            draft_ids = np.empty((Bt, gamma), np.int32)
            base = _as_f64(ld_q[::repeats])  # [B, gamma, V]
            step = max(1, (1 << 21) // max(1, gamma * V))
            for b in range(B):
                for r0 in range(0, repeats, step):
                    r1 = min(repeats, r0 + step)
                    u = rng.random((r1 - r0, gamma, V))
                    g = -np.log(-np.log(np.maximum(u, 1e-300)))
                    draft_ids[b * repeats + r0:b * repeats + r1] = np.argmax(base[b][None] + g, axis=-1)
        else:
            draft_ids = gumbel_argmax(rng, ld_q).astype(np.int32)
    else:
        draft_ids = np.zeros((Bt, 0), np.int32)
    return dict(kind="dense", dtype=dtype, B=Bt, gamma=gamma, V=V,
                target=np.ascontiguousarray(lt_q), draft=np.ascontiguousarray(ld_q),
                draft_ids=np.ascontiguousarray(draft_ids, dtype=np.int32),
                u_accept=_uniform_f32(rng, (Bt, gamma)), u_sample=_uniform_f32(rng, (Bt,)))


def greedy_inputs(B: int, gamma: int, V: int, *, dtype: str = "bf16", seed: int = 0,
                  target_sigma: float = 3.0, draft_noise: float = 0.5) -> dict:
    """Greedy (T = 0) verification inputs.

    target [B, gamma+1, V] ~ N(0, target_sigma^2); a greedy drafter's ids:
    draft_ids[b, j] = the id of the largest draft logit, the draft logits being
    the target's + N(0, draft_noise^2) (a drafter that agrees with the target
    up to noise).  No uniforms: greedy verification consumes none.
    """
    rng = np.random.default_rng(seed)
    lt = rng.normal(0.0, target_sigma, size=(B, gamma + 1, V)).astype(np.float32)
    ld = (lt[:, :gamma] + rng.normal(0.0, draft_noise, size=(B, gamma, V))).astype(np.float32)
    if dtype == "bf16":
        lt_q, ld_q = bf16_bits(lt), bf16_bits(ld)
    elif dtype == "f32":
        lt_q, ld_q = lt, ld
    else:
        raise ValueError(dtype)
    draft_ids = np.argmax(_as_f64(ld_q), axis=-1).astype(np.int32) if gamma else np.zeros((B, 0), np.int32)
    return dict(kind="greedy", dtype=dtype, B=B, gamma=gamma, V=V,
                target=np.ascontiguousarray(lt_q), draft_ids=np.ascontiguousarray(draft_ids))


def commit_inputs(B: int, W: int, V: int, *, dtype: str = "bf16", seed: int = 0,
                  sigma: float = 3.0, spike_lo: float = 10.0, spike_hi: float = 40.0,
                  masked_frac: float = 0.75, tau: float = 0.9) -> dict:
    """Confidence-threshold commit inputs: B blocks of W positions.

    logits [B, W, V] ~ N(0, sigma^2) plus one spike per position at a random
    id, its height uniform in [spike_lo, spike_hi] (so the positions' largest
    probabilities spread over (0, 1)); masked [B, W] int32, each position still
    masked with probability masked_frac; threshold tau.
    """
    rng = np.random.default_rng(seed)
    lt = rng.normal(0.0, sigma, size=(B, W, V)).astype(np.float32)
    ids = rng.integers(0, V, size=(B, W))
    h = rng.uniform(spike_lo, spike_hi, size=(B, W)).astype(np.float32)
    np.put_along_axis(lt, ids[..., None], np.take_along_axis(lt, ids[..., None], -1) + h[..., None], -1)
    if dtype == "bf16":
        lq = bf16_bits(lt)
    elif dtype == "f32":
        lq = lt
    else:
        raise ValueError(dtype)
    masked = (rng.random((B, W)) < masked_frac).astype(np.int32)
    return dict(kind="commit", dtype=dtype, B=B, W=W, V=V, tau=float(tau),
                logits=np.ascontiguousarray(lq), masked=masked)


# ---------------------------------------------------------------------------
# sparse top-k lists
# ---------------------------------------------------------------------------
def _zipf_rank_cdf(V: int, s: float) -> np.ndarray:
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def _draw_distinct(rng, cdf, perm, k, exclude=None, batch=None):
    """k distinct ids: iid Zipf rank draws mapped through perm, first k distinct
    (the law of sequential sampling without replacement)."""
    batch = batch or max(4 * k, 64)
    chosen = []
    seen = set() if exclude is None else set(int(e) for e in exclude)
    while len(chosen) < k:
        ranks = np.searchsorted(cdf, rng.random(batch), side="right")
        ranks = np.minimum(ranks, len(cdf) - 1)
        for r in ranks:
            i = int(perm[r])
            if i not in seen:
                seen.add(i)
                chosen.append(i)
                if len(chosen) == k:
                    break
    return np.array(chosen, dtype=np.int64)


def sparse_inputs(B: int, gamma: int, V: int, k: int = 64, *, seed: int = 0, s: float = 1.1,
                  overlap: float = 0.5) -> dict:
    """Sparse (id, prob) support lists, each sorted by id.

    Target list per (row, position): k distinct ids by Zipf(s) over vocab ranks
    (rank -> id through a fixed seeded permutation), probs proportional to
    Zipf(s) over the list's draw rank, normalised.  Draft list: round(overlap*k)
    ids kept from the target list plus fresh Zipf ids, with its own Zipf(s)
    probs under a random rank order.  Draft token ~ draft list.  Position gamma
    holds the bonus target list.
    """
    rng = np.random.default_rng(seed)
    cdf = _zipf_rank_cdf(V, s)
    perm = rng.permutation(V)
    zipf_k = np.arange(1, k + 1, dtype=np.float64) ** (-s)
    zipf_k /= zipf_k.sum()
    keep = int(round(overlap * k))
    tid = np.empty((B, gamma + 1, k), np.int32)
    tp = np.empty((B, gamma + 1, k), np.float32)
    did = np.empty((B, gamma, k), np.int32)
    dp = np.empty((B, gamma, k), np.float32)
    x = np.empty((B, gamma), np.int32)
    for b in range(B):
        for j in range(gamma + 1):
            ids = _draw_distinct(rng, cdf, perm, k)
            order = np.argsort(ids, kind="stable")
            tid[b, j] = ids[order]
            tp[b, j] = zipf_k[order].astype(np.float32)
            if j == gamma:
                continue
            kept = rng.choice(ids, size=keep, replace=False)
            fresh = _draw_distinct(rng, cdf, perm, k - keep, exclude=ids)
            dids = np.concatenate([kept, fresh])
            dprob = zipf_k[rng.permutation(k)]
            o = np.argsort(dids, kind="stable")
            did[b, j] = dids[o]
            dp[b, j] = dprob[o].astype(np.float32)
            x[b, j] = did[b, j][gumbel_argmax(rng, np.log(dp[b, j].astype(np.float64))[None])[0]]
    return dict(kind="sparse", B=B, gamma=gamma, V=V, kt=k, kd=k, tgt_ids=tid, tgt_probs=tp,
                drf_ids=did, drf_probs=dp, draft_tokens=x,
                u_accept=_uniform_f32(rng, (B, gamma)), u_sample=_uniform_f32(rng, (B,)))


# ---------------------------------------------------------------------------
# any-order
# ---------------------------------------------------------------------------
def anyorder_inputs(B: int, D: int, W: int, V: int, *, dtype: str = "f32", seed: int = 0,
                    draft_sigma: float = 2.0, target_noise: float = 0.4) -> dict:
    """Any-order inputs: draft ~ N(0, draft_sigma^2), target = draft + noise,
    [B, D, V] in sequence-position order; order [B, W] = the first W entries
    of a random permutation of 0..D-1 per sequence; a draft token at every
    position sampled from the rounded draft logits."""
    rng = np.random.default_rng(seed)
    ld = rng.normal(0.0, draft_sigma, size=(B, D, V)).astype(np.float32)
    lt = (ld + rng.normal(0.0, target_noise, size=(B, D, V))).astype(np.float32)
    if dtype == "bf16":
        lt, ld = bf16_bits(lt), bf16_bits(ld)
    order = np.stack([rng.permutation(D)[:W] for _ in range(B)]).astype(np.int32)
    tok = gumbel_argmax(rng, ld, chunk_rows=8192).astype(np.int32)
    return dict(kind="anyorder", dtype=dtype, B=B, D=D, W=W, V=V, target=lt, draft=ld,
                order=order, draft_tokens=tok,
                u_accept=_uniform_f32(rng, (B, W)), u_sample=_uniform_f32(rng, (B,)))


def rounds_inputs(B: int, R: int, D: int, V: int, *, dtype: str = "f32", seed: int = 0,
                  draft_sigma: float = 2.0, target_noise: float = 0.4, wmax: int = 0) -> dict:
    """Windowed multi-round any-order inputs.

    draft [B, D, V] ~ N(0, draft_sigma^2) (one non-causal pass); target
    [B, R, D, V] = draft + fresh N(0, target_noise^2) per round (the causal
    recompute of each round); order [B, D] a random permutation per sequence;
    revealed [B] uniform in [0, D); draft_tokens [B, R, D] sampled afresh per
    round from the rounded draft logits; u_accept [B, R, D], u_sample [B, R].
    With wmax > 0 also window [B] uniform in [1, wmax]; otherwise the caller
    derives the windows (for instance from the cosine schedule).
    """
    rng = np.random.default_rng(seed)
    ld = rng.normal(0.0, draft_sigma, size=(B, D, V)).astype(np.float32)
    lt = (ld[:, None] + rng.normal(0.0, target_noise, size=(B, R, D, V))).astype(np.float32)
    if dtype == "bf16":
        lt, ld = bf16_bits(lt), bf16_bits(ld)
    elif dtype != "f32":
        raise ValueError(dtype)
    order = np.stack([rng.permutation(D) for _ in range(B)]).astype(np.int32)
    revealed = rng.integers(0, D, size=B).astype(np.int32)
    tok = np.stack([gumbel_argmax(rng, ld, chunk_rows=8192) for _ in range(R)], axis=1).astype(np.int32)
    d = dict(kind="rounds", dtype=dtype, B=B, R=R, D=D, V=V, target=np.ascontiguousarray(lt),
             draft=ld, order=order, revealed=revealed, draft_tokens=np.ascontiguousarray(tok),
             u_accept=_uniform_f32(rng, (B, R, D)), u_sample=_uniform_f32(rng, (B, R)))
    if wmax > 0:
        d["window"] = rng.integers(1, wmax + 1, size=B).astype(np.int32)
    return d


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    "dense_v32_g4": dict(kind="dense", B=1, gamma=4, V=32, dtype="f32", target_sigma=2.0,
                         draft_noise=1.0),
    "dense_v151936_g15": dict(kind="dense", B=1, gamma=15, V=151936, dtype="bf16",
                              target_sigma=3.0, draft_noise=0.7, spikes=8, spike_height=12.0),
    "dense_b64_g7_v128256": dict(kind="dense", B=64, gamma=7, V=128256, dtype="bf16",
                                 target_sigma=3.0, draft_noise=0.5),
    "sparse_b256_g15_k64": dict(kind="sparse", B=256, gamma=15, V=151936, k=64),
    "anyorder_b4096_w32_v33": dict(kind="anyorder", B=4096, D=32, W=32, V=33, dtype="f32"),
    "greedy_b64_g7_v128256": dict(kind="greedy", B=64, gamma=7, V=128256, dtype="bf16",
                                  target_sigma=3.0, draft_noise=0.5),
    "commit_b64_w4_v151936": dict(kind="commit", B=64, W=4, V=151936, dtype="bf16"),
    "support_b64_g7_v128256": dict(kind="support", B=64, gamma=7, V=128256, dtype="bf16"),
    # text8-like character model (27 symbols), 256 positions, 4 verification
    # rounds per draft, windows from the cosine schedule with dtau = 0.05
    "rounds_b4096_r4_d256_v27": dict(kind="rounds", B=4096, R=4, D=256, V=27, dtype="f32",
                                     dtau=0.05),
}


def make(name: str, seed: int = 0, **override) -> dict:
    """Build a named workload (``override`` may shrink B etc. for quick cases)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    kind = cfg.pop("kind")
    if kind == "dense":
        B, g, V = cfg.pop("B"), cfg.pop("gamma"), cfg.pop("V")
        d = dense_inputs(B, g, V, seed=seed, **cfg)
    elif kind == "sparse":
        B, g, V = cfg.pop("B"), cfg.pop("gamma"), cfg.pop("V")
        d = sparse_inputs(B, g, V, seed=seed, **cfg)
    elif kind == "greedy":
        B, g, V = cfg.pop("B"), cfg.pop("gamma"), cfg.pop("V")
        d = greedy_inputs(B, g, V, seed=seed, **cfg)
    elif kind == "commit":
        B, W, V = cfg.pop("B"), cfg.pop("W"), cfg.pop("V")
        d = commit_inputs(B, W, V, seed=seed, **cfg)
    elif kind == "support":
        # the headline's target and draft rows, preprocessed with the Uno
        # article's test setting (temperature 1, top-k 50, top-p 0.95)
        B, g, V = cfg.pop("B"), cfg.pop("gamma"), cfg.pop("V")
        dd = dense_inputs(B, g, V, seed=seed, dtype=cfg.pop("dtype"))
        rows = np.concatenate([dd["target"].reshape(-1, V), dd["draft"].reshape(-1, V)])
        d = dict(kind="support", dtype=dd["dtype"], N=rows.shape[0], V=V, K=50, T=1.0,
                 top_p=0.95, logits=np.ascontiguousarray(rows))
    elif kind == "rounds":
        dtau = cfg.pop("dtau")
        B, R, D, V = cfg.pop("B"), cfg.pop("R"), cfg.pop("D"), cfg.pop("V")
        d = rounds_inputs(B, R, D, V, seed=seed, **cfg)
        d["dtau"] = dtau  # the windows come from the cosine schedule (computed by the caller)
    else:
        B, D, W, V = cfg.pop("B"), cfg.pop("D"), cfg.pop("W"), cfg.pop("V")
        d = anyorder_inputs(B, D, W, V, seed=seed, **cfg)
    d["name"] = name
    return d
