/*
 * spec_verify_oracle.h -- plain CPU oracle for lossless speculative verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The GPU
 * library never links, includes or calls it, and shares no code with it.
 *
 * Everything is computed in IEEE double, one row at a time, in the order the
 * pages state the algorithm:
 *   - accept draft x with probability min(1, p(x)/q(x)); on rejection resample
 *     from max(p - q, 0) renormalised  (Uno article, "What 'lossless' actually
 *     has to mean": the rule and Uno's _sparse_verify_tensors fragment);
 *   - the block is truncated at the first rejection  (DFlash/DFlash2 guide,
 *     4.4 "Mathematical Losslessness Guarantee");
 *   - when all gamma drafts are accepted the target's bonus token is emitted,
 *     so 1 <= emitted <= gamma + 1  (DFlash/DFlash2 guide, section 2
 *     "Speculative Decoding Speedup Formulation");
 *   - any-order variant: verify in generation order sigma, resample the first
 *     rejected position from max(0, target - draft) and end the round
 *     (Self-Speculative Masked Diffusions, key design 2).
 *
 * Readings where the pages are silent are listed with each function below.
 */
#ifndef SPEC_VERIFY_ORACLE_H
#define SPEC_VERIFY_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Per-row flag bits written to flags[b]. */
enum {
  ORACLE_FLAG_ACCEPT_BAND = 1u, /* some evaluated accept test had |u - min(1,p/q)| < 1e-6 */
  ORACLE_FLAG_CDF_TIE = 2u,     /* emitted token's CDF boundary within 1e-6*T of u_s*T   */
  ORACLE_FLAG_ZERO_RESID = 4u,  /* residual mass T <= 0 after a rejection: sampled from p */
  ORACLE_FLAG_INPUT_ERR = 8u    /* invalid input row: n = -1, tokens = -1                 */
};

#define ORACLE_ACCEPT_BAND 1e-6 /* absolute, in units of the accept uniform          */
#define ORACLE_TIE_BAND 1e-6    /* relative to T, i.e. in units of the sample uniform */

/*
 * Dense verification.
 *   target_logits [B, gamma+1, V]   (dtype ORACLE_F32 or ORACLE_BF16 raw bits)
 *   draft_logits  [B, gamma, V]
 *   draft_ids     [B, gamma]  int32 in [0, V)
 *   u_accept      [B, gamma]  fp32 in [0, 1)
 *   u_sample      [B]         fp32 in [0, 1)
 * Outputs (caller-owned host arrays):
 *   n_accepted [B]; out_tokens [B, gamma+1] (x_0..x_{n-1}, resample/bonus, then -1)
 *   residual_out [B, V] or NULL: the distribution the emitted token was drawn
 *     from (r / T after a rejection, p_gamma for the bonus)
 *   accept_prob [B, gamma] or NULL: min(1, p_j(x_j)/q_j(x_j)) for every j
 *   resid_mass [B] or NULL: T (1 for a bonus draw, the sum of p_gamma)
 *   flags [B] or NULL: ORACLE_FLAG_* bits
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_verify_dense(const void* target_logits, const void* draft_logits, int dtype,
                        const int32_t* draft_ids, const float* u_accept, const float* u_sample,
                        int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                        double* residual_out, double* accept_prob, double* resid_mass,
                        uint32_t* flags, int nthreads);

/*
 * Sparse top-k verification (Uno's sampler on (id, prob) support lists).
 *   tgt_ids/tgt_probs [B, gamma+1, kt]  sorted strictly ascending by id
 *   drf_ids/drf_probs [B, gamma, kd]    sorted strictly ascending by id
 *   draft_tokens [B, gamma]; u_accept [B, gamma]; u_sample [B]
 * Outputs as for dense; residual_out is [B, kt] (on the target support, list
 * order).  p and q are the listed probabilities as given (no renormalisation);
 * the draw after a rejection is over r = max(p - q_on_clean, 0) renormalised,
 * the bonus draw is over the target list of position gamma normalised by its
 * sum.
 */
int oracle_verify_sparse(const int32_t* tgt_ids, const float* tgt_probs, int kt,
                         const int32_t* drf_ids, const float* drf_probs, int kd,
                         const int32_t* draft_tokens, const float* u_accept, const float* u_sample,
                         int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                         double* residual_out, double* accept_prob, double* resid_mass,
                         uint32_t* flags, int nthreads);

/*
 * Any-order (masked-diffusion self-speculative) verification.
 *   target_logits, draft_logits [B, D, V] in sequence-position order
 *   order [B, W]: sigma, the window positions in verification order, a
 *     permutation of W distinct positions in [0, D)
 *   draft_tokens [B, D]; u_accept [B, W] (in window order); u_sample [B]
 * Outputs: n_accepted [B] in [0, W]; out_tokens [B, D]: for window index i,
 *   out[b, sigma_i] = draft token (i < n), resample (i == n), -1 (i > n);
 *   positions outside the window are left untouched.  No bonus token.
 *   residual_out [B, V] or NULL (zeros when n == W); accept_prob [B, W].
 */
int oracle_verify_anyorder(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* order, const int32_t* draft_tokens,
                           const float* u_accept, const float* u_sample, int B, int D, int W,
                           int V, int32_t* n_accepted, int32_t* out_tokens, double* residual_out,
                           double* accept_prob, double* resid_mass, uint32_t* flags,
                           int nthreads);

/* Greedy (T = 0) verification ("DFlash/DFlash2 guide", 4.4: under greedy
 * decoding a draft token is accepted if and only if it is the target's
 * choice; the condition's formula is lost from the page, and the reading
 * taken is the T -> 0 limit of the stochastic rule, see the .c file).
 *   target_logits [B, gamma+1, V] (dtype), draft_ids [B, gamma];
 *   n_accepted [B] (-1 on an input error), out_tokens [B, gamma+1]
 *   (x_0..x_{n-1}, the target argmax at n, then -1).
 */
int oracle_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_ids, int B,
                         int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                         int nthreads);

/* Confidence-threshold commit of a block-diffusion pass ("SDAR" page,
 * section 5, decoding timeline): every masked position of a block has a full
 * distribution p_i = softmax(logits[b, i]); its confidence is max_y p_i(y)
 * and its candidate token the argmax (the smallest id on ties).  Masked
 * positions whose confidence clears tau (conf > tau) are committed; if none
 * does, the single most confident masked position is (the smallest index on
 * ties), so every pass makes progress.
 *   logits [B, W, V] (dtype); masked [B, W] int32 (nonzero: still masked);
 *   commit [B, W] int32 (1 committed, 0 not, -1 on an input error in the
 *   block); tokens [B, W] int32 (the argmax where committed, else -1);
 *   confidence [B, W] or NULL (NaN where not masked); flags [B] or NULL:
 *   ORACLE_FLAG_ACCEPT_BAND when a masked position's confidence is within
 *   1e-6 of tau, ORACLE_FLAG_CDF_TIE when the fallback's top two confidences
 *   are within 1e-6 relative, ORACLE_FLAG_INPUT_ERR on an input error (a
 *   masked row with NaN, +inf or no finite logit).  A block with no masked
 *   position commits nothing.
 */
int oracle_commit_confident(const void* logits, int dtype, const int32_t* masked, double tau,
                            int B, int W, int V, int32_t* commit, int32_t* tokens,
                            double* confidence, uint32_t* flags, int nthreads);

/* Sparse support from dense logits: temperature, top-k, top-p (the Uno
 * article's test setting, top-k 50 / top-p 0.95; DFlash/DFlash2 guide, Q3:
 * temperature scaling of both logit sets before the acceptance ratio).  For
 * each of the N rows: the K largest logits (the smaller id first on ties)
 * with p_i = softmax(l / T) renormalised over those K; sorted by p (ties:
 * smaller id first), the smallest prefix whose cumulative mass reaches
 * top_p (at least one) is kept and renormalised, the rest of the K get 0.
 *   logits [N, V] (dtype), 1 <= K <= V, T > 0;
 *   ids [N, K] int32 ascending, probs [N, K] double;
 *   flags [N] or NULL: ORACLE_FLAG_CDF_TIE when the cumulative mass at the
 *   cut is within 1e-6 of top_p (either side), ORACLE_FLAG_INPUT_ERR (ids
 *   -1, probs NaN) for a row with NaN, +inf or no finite logit.
 */
int oracle_support_topk(const void* logits, int dtype, int N, int V, double T, int K,
                        double top_p, int32_t* ids, double* probs, uint32_t* flags,
                        int nthreads);

/* Windowed multi-round any-order verification ("Self-Speculative Masked
 * Diffusions", key design 4): one non-causal pass drafts the window, several
 * causal verification rounds run on it.  Round r verifies the still-masked
 * window positions in sigma order against round r's target logits with
 * round r's draft tokens, ends at its first rejection with a resample from
 * max(p - q, 0) (revealed too), and the next round starts after it; a round
 * that accepts every remaining draft closes the window.  No bonus token.
 *   target_logits [B, R, D, V]  round r's target logits per sequence position
 *   draft_logits  [B, D, V]     the window's draft logits (every round)
 *   order [B, D]  sigma; revealed [B] = i0 (sigma[0, i0) already revealed);
 *   window [B] >= 1: the window is sigma[i0, min(D, i0 + window))
 *   draft_tokens [B, R, D]      round r's draft token per sequence position
 *   u_accept [B, R, D]          round r's accept uniform, by sigma index
 *   u_sample [B, R]             round r's residual uniform
 * Outputs: tokens [B, D] (each revealed token at its position; others left
 * as they are; the window's positions -1 on an input error); n_revealed [B]
 * (i0 + the tokens the rounds revealed, -1 on an input error);
 * round_accepts [B, R] (drafts accepted in round r, -1 for rounds not run);
 * flags [B] or NULL (accept band, CDF tie, zero residual, input error).
 */
int oracle_anyorder_rounds(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* order, const int32_t* revealed, const int32_t* window,
                           const int32_t* draft_tokens, const float* u_accept,
                           const float* u_sample, int B, int R, int D, int V, int32_t* tokens,
                           int32_t* n_revealed, int32_t* round_accepts, uint32_t* flags,
                           int nthreads);

/* The window W(i) of an outer step starting with i of D tokens revealed
 * (same page, key design 4: it grows with i, cosine-shaped, set by dtau):
 * the positions a cosine-schedule masked-diffusion sampler (revealed
 * fraction 1 - cos(pi t / 2) at time t) reveals over the next dtau of its
 * time, at least 1 and at most D - i; 0 when i >= D, -1 on bad arguments. */
int oracle_cosine_window(int D, int i, double dtau);

/* Threads the oracle would use for nthreads <= 0 (all online host cores). */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif
