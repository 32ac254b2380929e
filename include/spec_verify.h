/*
 * spec_verify.h -- C ABI of the GB300 batched lossless speculative-verification
 * library (libspec_verify.so, CUDA kernels for sm_103a).
 *
 * The operation (Leviathan-style rejection sampling) as the pages state it:
 *   - a drafter proposes gamma tokens x_j with distribution q_j; the target
 *     scores every position in one parallel pass and gives p_j
 *     (DFlash/DFlash2 guide, 4.4 "Mathematical Losslessness Guarantee");
 *   - x_j is accepted with probability min(1, p_j(x_j)/q_j(x_j)); at the first
 *     rejection the block is truncated and a replacement is drawn from the
 *     renormalised residual max(p - q, 0)  (Uno article, "What 'lossless'
 *     actually has to mean", and Uno's _sparse_verify_tensors fragment:
 *     ratio = p/q where q > 0 else 0, accept iff u < min(1, ratio));
 *   - if all gamma drafts are accepted the target's bonus token is drawn from
 *     p_gamma, so every call emits between 1 and gamma + 1 tokens per row
 *     (DFlash/DFlash2 guide, section 2, tau in [1, gamma + 1]);
 *   - any-order variant: positions are verified in a generation order sigma,
 *     the first rejection is resampled from max(0, target - draft) and ends
 *     the round, no bonus token (Self-Speculative Masked Diffusions, key
 *     design 2).
 *
 * Randomness is supplied by the caller: one accept uniform per draft position
 * and one sample uniform per row, each in [0, 1).  For fixed inputs the
 * results are a deterministic function of those uniforms: the inverse CDF
 * walks the vocabulary (sparse: the sorted list) in ascending id order and
 * returns the smallest id whose inclusive prefix mass exceeds u_sample * T.
 *
 * Conventions for every entry point
 *   - All pointers are DEVICE pointers owned by the caller (cudaMalloc,
 *     cudaMallocAsync or a framework allocator); the library allocates no
 *     memory.  Its only state is a per-device cache of launch attributes (set
 *     on the first call on each device) and, for spec_verify_dense_static
 *     alone, a fixed device scratch array.  Calls are asynchronous on
 *     `stream` (the legacy default stream if 0).
 *   - Tensors are dense, row-major, contiguous, with the shapes given below.
 *     int32 / fp32 arrays need 4-byte alignment, bf16 arrays 2-byte
 *     alignment.  Logit rows whose byte length is a multiple of 16, with
 *     16-byte aligned base pointers, take the fast path (16-byte cp.async
 *     copies into shared memory); other rows are read element by element.
 *   - Host-side argument errors (null pointers, non-positive sizes, sizes out
 *     of range, a workspace that is too small) return SV_ERR_INVALID_ARG
 *     synchronously and launch nothing.  A failed launch returns SV_ERR_CUDA.
 *   - Device-side input errors (a draft id or sigma entry out of range, a
 *     repeated sigma entry, an unsorted or repeated list id, a logit row that
 *     contains NaN or +inf or is entirely -inf) do not stop the call: the
 *     offending row gets n_accepted = -1 and out_tokens = -1, and a bit is
 *     set in the workspace status word that spec_verify_check() reports.
 *   - Waits between thread blocks: the dense kernels are programmatic
 *     dependents (griddepcontrol.wait) of whatever precedes them on the
 *     stream and read nothing that grid writes before it has completed; the
 *     CTAs of a thread-block cluster meet at cluster barriers.  One kernel
 *     polls memory written by another grid: the row kernel of the two-kernel
 *     dense path waits for its row's piece count, which the statistics
 *     kernel's warps raise as they store the row's statistics.  Its launch as
 *     a programmatic dependent makes every statistics block resident before
 *     any row block starts, so the count always completes.  The single-pass
 *     dense kernel waits on its own bulk copies into shared memory.  Each of
 *     these waits gives up after about one second: the row then gets
 *     n_accepted = -1 and out_tokens = -1 and the timeout bit is set, which
 *     spec_verify_check reports as SV_ERR_TIMEOUT.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t (a CUstream_st pointer). */
struct CUstream_st;
typedef struct CUstream_st* sv_stream_t;

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,  /* rejected on the host, nothing launched           */
  SV_ERR_UNSUPPORTED = 2,  /* valid request this build cannot run (e.g. no GPU) */
  SV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed             */
  SV_ERR_DEVICE_INPUT = 4, /* spec_verify_check: some row had invalid inputs   */
  SV_ERR_TIMEOUT = 5,      /* spec_verify_check: a bounded wait ran out */
  SV_ERR_SCRATCH_LIMIT = 6 /* spec_verify_dense_static: sizes need more scratch
                              than SV_STATIC_SCRATCH_BYTES; nothing launched  */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Largest sizes accepted by the entry points. */
#define SV_MAX_VOCAB (1 << 24)
#define SV_MAX_GAMMA 255  /* dense: gamma; any-order: W (and D <= SV_MAX_GAMMA * 64) */
#define SV_MAX_LIST 4096  /* sparse: kt, kd */
#define SV_MAX_TOPK 256   /* spec_support_topk: top_k */

/* ABI version of this header; spec_verify_abi_version() returns it. */
#define SV_ABI_VERSION 1
int spec_verify_abi_version(void);

/*
 * Workspace: device scratch for the per-row counters, partial statistics and
 * the status word.  spec_verify_workspace_size(B, gamma_or_W, V) bytes are
 * enough for any of the three calls with those sizes (B rows, gamma drafts
 * or a window of W, vocabulary V).  The workspace must be zeroed once before
 * first use -- spec_verify_workspace_init() does that on `stream` -- and each
 * successful call leaves every byte of it (apart from the sticky status word)
 * at zero again, so one workspace serves calls of any sizes that fit it, and
 * a call can be replayed (e.g. from a CUDA graph) without re-initialising.
 * One workspace must not be used by two calls that may run at the same time.
 */
size_t spec_verify_workspace_size(int B, int gamma_or_W, int V);
sv_status spec_verify_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream);

/*
 * spec_verify_dense -- dense logits over the full vocabulary.
 *   target_logits [B, gamma+1, V]  (dtype SV_F32 or SV_BF16); row j < gamma
 *                                  scores draft j, row gamma is the bonus row
 *   draft_logits  [B, gamma, V]    same dtype; may be NULL when gamma == 0
 *   draft_ids     [B, gamma] int32 in [0, V): the drafted tokens x_j, which
 *                                  must have been sampled from softmax(draft)
 *   u_accept      [B, gamma] fp32 uniforms in [0, 1), one per draft
 *   u_sample      [B]        fp32 uniform in [0, 1) for the one draw per row
 * Outputs:
 *   n_accepted    [B] int32: accepted drafts n in [0, gamma] (-1: bad input)
 *   out_tokens    [B, gamma+1] int32: x_0..x_{n-1}, then the resampled token
 *                 (n < gamma) or the bonus token (n == gamma), then -1
 *   residual_out  [B, V] fp32 or NULL: the distribution the emitted token was
 *                 drawn from (max(p_n - q_n, 0)/T, or p_gamma for the bonus)
 *   accept_prob_out [B, gamma] fp32 or NULL: min(1, p_j(x_j)/q_j(x_j)) for
 *                 every j (all positions are scored, as in the parallel pass)
 * Softmax, gather, ratio test, first-reject scan and the inverse-CDF draw run
 * in fp32, with partial sums combined and prefixed in float-float (pairs of
 * fp32 carrying ~48 significant bits); bf16 inputs are widened exactly.
 * Paths (chosen per call, the same results up to rounding):
 *   - (gamma + 1) * V small enough for one warp: a warp per row;
 *   - rows of a 16-byte multiple with 16-byte aligned bases, and a grid that
 *     is resident all at once: one pass, a thread-block cluster per (row,
 *     position) holding both rows in shared memory, the draw taken from
 *     shared memory (a rejected or bonus position draws speculatively; the
 *     row's first rejection keeps its draw);
 *   - otherwise two kernels: the first reads every logit once (statistics,
 *     gather), the second takes the decisions and reads the two rows of each
 *     row's stop position again (residual masses and the draw).
 *   The environment variable SPEC_VERIFY_DENSE_KERNELS=split or =fused
 *   forces the two-kernel or the single-pass path (measurement switch).
 */
int spec_verify_dense(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_ids, const float* u_accept, const float* u_sample,
                      int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                      float* residual_out, float* accept_prob_out, void* workspace,
                      size_t ws_bytes, sv_stream_t stream);

/*
 * spec_verify_sparse -- Uno-style sparse support lists (Uno article, "What
 * 'lossless' actually has to mean", _sparse_verify_tensors).
 *   tgt_ids, tgt_probs [B, gamma+1, kt]: target ("clean") support per
 *       position, ids strictly ascending in [0, V); probs fp32 >= 0 as given
 *       (not renormalised); position gamma is the bonus list
 *   drf_ids, drf_probs [B, gamma, kd]: draft support per position, same rules
 *   draft_tokens [B, gamma] int32; u_accept [B, gamma]; u_sample [B]
 * p_spec / q_spec are the listed probabilities at the draft token (0 when
 * absent); after a rejection the draw is over the target list with weights
 * max(p - q_on_clean, 0), q_on_clean being the draft probability of the same
 * id; the bonus draw is over the target list of position gamma.
 * Outputs: n_accepted [B]; out_tokens [B, gamma+1] (vocabulary ids);
 *   residual_out [B, kt] fp32 or NULL (on the target support, list order);
 *   accept_prob_out [B, gamma] fp32 or NULL.
 * Limits: 1 <= kt, kd <= SV_MAX_LIST; gamma <= 31.
 */
int spec_verify_sparse(const int32_t* tgt_ids, const float* tgt_probs, int kt,
                       const int32_t* drf_ids, const float* drf_probs, int kd,
                       const int32_t* draft_tokens, const float* u_accept, const float* u_sample,
                       int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                       float* residual_out, float* accept_prob_out, void* workspace,
                       size_t ws_bytes, sv_stream_t stream);

/*
 * spec_verify_anyorder -- masked-diffusion self-speculative verification
 * (Self-Speculative Masked Diffusions, key design 2).
 *   target_logits, draft_logits [B, D, V] in sequence-position order
 *   order        [B, W] int32: sigma, the W window positions (distinct, in
 *                [0, D)) in verification order
 *   draft_tokens [B, D] int32: the non-causal draft's token at each position
 *   u_accept     [B, W] fp32 in window order; u_sample [B]
 * Outputs: n_accepted [B] in [0, W] (-1: bad input); out_tokens [B, D]:
 *   out[b, sigma_i] = draft token for i < n, the resample for i == n, -1 for
 *   i > n; positions outside the window are not written.  No bonus token:
 *   an all-accept round emits W tokens.  residual_out [B, V] or NULL (zeros
 *   when n == W); accept_prob_out [B, W] or NULL.
 * Limits: W <= 32, V <= 1024 (small-vocabulary kernel).
 */
int spec_verify_anyorder(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* order, const int32_t* draft_tokens,
                         const float* u_accept, const float* u_sample, int B, int D, int W,
                         int V, int32_t* n_accepted, int32_t* out_tokens, float* residual_out,
                         float* accept_prob_out, void* workspace, size_t ws_bytes,
                         sv_stream_t stream);

/*
 * spec_verify_anyorder_rounds -- windowed multi-round any-order verification
 * (Self-Speculative Masked Diffusions, key design 4: one non-causal pass
 * drafts the window, several causal verification rounds run on it).  For
 * sequence b the window is sigma[i0, e), i0 = revealed[b],
 * e = min(D, i0 + window[b]).  Round r (r = 0 .. R-1) starts at sigma index
 * i_r (i_0 = i0): it verifies positions s = sigma[k], k = i_r, i_r + 1, ...
 * in order with p = softmax(target_logits[b, r, s]),
 * q = softmax(draft_logits[b, s]), x = draft_tokens[b, r, s] and
 * u = u_accept[b, r, k] (accept iff u < min(1, p(x)/q(x)), ratio 0 when
 * q(x) = 0); at the first rejection it draws the replacement from
 * max(p - q, 0) renormalised by inverse CDF over ascending ids with
 * u_sample[b, r] and i_{r+1} = that index + 1; a round that accepts every
 * remaining draft closes the window.  No bonus token.
 *   target_logits [B, R, D, V] and draft_logits [B, D, V], fp32 or bf16, in
 *     sequence-position order (only the rows the rounds reach are read);
 *   order [B, D] sigma; revealed [B]; window [B] (>= 1; see
 *     spec_anyorder_window); draft_tokens [B, R, D]; u_accept [B, R, D]
 *     (indexed by sigma index); u_sample [B, R]; uniforms in [0, 1).
 * Outputs: tokens [B, D]: each revealed token at its position, other
 *   entries untouched; n_revealed [B] = i0 + the tokens the rounds revealed;
 *   round_accepts [B, R]: drafts accepted by round r, -1 for rounds not run.
 *   An input error (revealed outside [0, D], window < 1, a sigma entry in the
 *   window out of range or repeated, or -- where a round reaches it -- a
 *   draft token out of range or a logit row with NaN, +inf or no finite
 *   entry) gives n_revealed -1, round_accepts -1 and -1 at the window's
 *   positions, and sets the status bit.
 * Workspace: the status word only (any workspace of at least 256 bytes).
 * Host errors: B, D, V < 0 or 0 (B = 0 is a no-op), R < 1, D * V or
 * B * R * D beyond 2^31, dtype, null or misaligned pointers.
 */
int spec_verify_anyorder_rounds(const void* target_logits, const void* draft_logits,
                                sv_dtype dtype, const int32_t* order, const int32_t* revealed,
                                const int32_t* window, const int32_t* draft_tokens,
                                const float* u_accept, const float* u_sample, int B, int R, int D,
                                int V, int32_t* tokens, int32_t* n_revealed,
                                int32_t* round_accepts, void* workspace, size_t ws_bytes,
                                sv_stream_t stream);

/*
 * spec_anyorder_window -- the window W(i) of an outer step that starts with
 * i of D tokens revealed (same page, key design 4: it grows with i,
 * cosine-shaped, set by dtau).  Reading taken: the positions a
 * cosine-schedule masked-diffusion sampler, revealed fraction
 * f(t) = 1 - cos(pi t / 2) at time t in [0, 1], reveals over the next dtau
 * of its time: W = ceil(D f(min(1, t(i) + dtau)) - 1e-9) - i with
 * f(t(i)) = i / D, at least 1 and at most D - i.  Host function (no device
 * work); returns 0 when i >= D and -1 for D < 1 or i < 0.
 */
int spec_anyorder_window(int D, int revealed, float dtau);

/*
 * spec_verify_greedy -- greedy (temperature 0) verification (DFlash/DFlash2
 * guide, 4.4: under greedy decoding a draft token is accepted if and only if
 * it is the target's choice; the page's formula is lost, and this is the
 * T -> 0 limit of spec_verify_dense's rule).  With a_j = the id of the
 * largest target logit at position j (the smallest such id on ties):
 *   n = the first j < gamma with draft_ids[b, j] != a_j, gamma if none;
 *   out_tokens[b] = x_0 .. x_{n-1}, a_n, then -1 (a_gamma is the bonus token
 *   when every draft is accepted; DFlash/DFlash2 guide, section 2).
 *   target_logits [B, gamma+1, V] (fp32 or bf16); draft_ids [B, gamma] int32.
 * No uniforms and no draft logits are read.  Outputs: n_accepted [B] in
 * [0, gamma] (-1: a target row with NaN, +inf or no finite logit, or a draft
 * id out of range; every token of the row is then -1).  Workspace: as for
 * spec_verify_dense, spec_verify_workspace_size(B, gamma, V) bytes, zero
 * again after the call.  Limits as spec_verify_dense.
 */
int spec_verify_greedy(const void* target_logits, sv_dtype dtype, const int32_t* draft_ids,
                       int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                       void* workspace, size_t ws_bytes, sv_stream_t stream);

/*
 * spec_commit_confident -- confidence-threshold commit of one block-diffusion
 * pass ("SDAR" page, section 5, decoding timeline: positions whose
 * confidence clears a threshold tau are committed, at least the most
 * confident one, so every pass makes progress).  For every position i still
 * masked in block b: confidence c_i = the largest probability of
 * softmax(logits[b, i]) and token a_i = its argmax (the smallest id on ties).
 * Masked positions with c_i > tau are committed; if none is, the most
 * confident masked position is (the smallest index on ties).
 *   logits [B, W, V] (fp32 or bf16); masked [B, W] int32 (nonzero: still
 *   masked; the logits of other positions are not read); tau: threshold.
 * Outputs: commit [B, W] int32 (1 committed, 0 not, -1 in a block with an
 *   input error: a masked row with NaN, +inf or no finite logit);
 *   tokens [B, W] int32 (a_i where committed, else -1); confidence [B, W]
 *   fp32 or NULL (c_i; NaN where not masked or on an input error).
 * Workspace: spec_verify_workspace_size(B, W - 1, V) bytes, zero again after
 * the call.  Limits: W <= 256, V <= SV_MAX_VOCAB.
 */
int spec_commit_confident(const void* logits, sv_dtype dtype, const int32_t* masked, float tau,
                          int B, int W, int V, int32_t* commit, int32_t* tokens,
                          float* confidence, void* workspace, size_t ws_bytes,
                          sv_stream_t stream);

/*
 * spec_support_topk -- sparse support lists from dense logits: temperature,
 * top-k, top-p (the Uno article's test setting, top-k 50 / top-p 0.95;
 * DFlash/DFlash2 guide, Q3: both logit sets are temperature scaled before the
 * acceptance ratio).  For each of the N rows of logits [N, V] (fp32 or bf16):
 * the top_k largest logits (the smaller id first on ties) with probabilities
 * softmax(l / temperature) renormalised over them; in decreasing probability
 * the shortest prefix whose cumulative mass reaches top_p (at least one
 * entry) is kept and renormalised, the rest get probability 0.
 * Outputs: ids [N, top_k] int32 in ascending id order, probs [N, top_k] fp32
 *   -- the lists spec_verify_sparse takes (target rows as tgt_ids/tgt_probs,
 *   draft rows as drf_ids/drf_probs).  A row with NaN, +inf or no finite
 *   logit gets ids -1 and probs NaN, and the status bit is set.
 * Workspace: at least 256 bytes (the status word).  Limits: 1 <= top_k <=
 * min(256, V); temperature > 0.
 */
int spec_support_topk(const void* logits, sv_dtype dtype, int N, int V, float temperature,
                      int top_k, float top_p, int32_t* ids, float* probs, void* workspace,
                      size_t ws_bytes, sv_stream_t stream);

/*
 * spec_verify_check -- synchronise `stream`, read and clear the workspace
 * status word.  Returns SV_OK, SV_ERR_TIMEOUT (a dense row's statistics or
 * bulk copies did not arrive within the bounded wait; that row carries
 * n_accepted = -1), SV_ERR_DEVICE_INPUT (some row of an earlier call had
 * invalid inputs; those rows carry n_accepted = -1), or SV_ERR_CUDA.
 */
int spec_verify_check(void* workspace, size_t ws_bytes, sv_stream_t stream);

/* Static string for a status code. */
const char* spec_verify_status_string(int status);

/*
 * spec_verify_dense_static -- spec_verify_dense for callers that cannot
 * allocate device memory.  (Library plumbing: the paper has no counterpart.)
 *
 * Who needs it: code that must not call cudaMalloc or any other allocator
 * where it verifies -- inside host callbacks or allocator hooks, plug-ins
 * whose host runtime owns every allocation, loops that may not touch the
 * allocator after start-up.  Such callers own their inputs and outputs but
 * cannot provide the workspace, so this call takes its scratch from a fixed
 * device array inside the library and allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 *
 * Arguments, layouts, outputs and results: exactly those of spec_verify_dense
 * without the workspace; the same kernels run.
 *
 * The scratch: a file-scope device array of SV_STATIC_SCRATCH_BYTES (4 MiB),
 * which every GPU that loads the library holds until the process exits.  A
 * call uses what the path it takes needs (see spec_verify_dense): 256 bytes
 * on the warp-per-row path; 256 + 2 x 4 B + 32 B (gamma + 1) bytes (each
 * part rounded up to 256 bytes) on the single-pass path (17 KB at B = 64,
 * gamma = 7); on the two-kernel path 32 bytes per 2 KB piece of every row
 * and position plus small terms (2.0 MiB at B = 64, gamma = 7, V = 128256
 * bf16).  Larger needs return SV_ERR_SCRATCH_LIMIT and launch nothing: sizes
 * that exceed the array on every path are refused on the host before any
 * CUDA call, the rest once the path is known.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current) and keeps it.
 *     That look-up may load the library's device code, so make the first
 *     call on each device before any stream capture.
 *   - Every call shares the array.  A call clears the part it uses on
 *     `stream` before its kernels run, so state left by an earlier call never
 *     leaks in; calls whose work may overlap on the GPU (other streams, other
 *     host threads) race on the array and must be ordered by the caller.
 *   - Errors: host-side argument errors as spec_verify_dense (nothing
 *     launched).  There is no status word to query: rows with invalid inputs
 *     (and rows whose statistics or bulk copies did not arrive within the
 *     bounded wait) carry n_accepted = -1.
 */
#define SV_STATIC_SCRATCH_BYTES (4u << 20)
int spec_verify_dense_static(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                             const int32_t* draft_ids, const float* u_accept,
                             const float* u_sample, int B, int gamma, int V,
                             int32_t* n_accepted, int32_t* out_tokens, float* residual_out,
                             float* accept_prob_out, sv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
