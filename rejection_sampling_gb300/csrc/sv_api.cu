// sv_api.cu -- host side of the C ABI declared in include/spec_verify.h:
// argument validation, kernel selection, workspace layout, status word.
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace {

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The small warp-per-row kernel handles R <= 32 rows per warp if the staged
// block fits in 96 KB of shared memory.
int small_vstride(int V) { return (V % 2) ? V : V + 1; }
bool small_fits(int R, int V) {
  return R >= 1 && R <= 32 && sv::small_smem_per_warp(R, small_vstride(V)) <= 96 * 1024;
}

size_t dense_ws_bytes(long long B, int G, int V, int es) {
  const sv::DenseGeom g = sv::dense_geom(V, es);
  return sv::dense_layout(B, G, g).total;
}

sv_status launch_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// Which path takes a large-vocabulary dense call.  By default the
// single-pass cluster kernel when its whole grid is resident at once, else
// the two-kernel path (statistics kernel + row kernel).  The environment
// variable SPEC_VERIFY_DENSE_KERNELS=split or =fused forces one of them (the
// fused kernel still needs 16-byte rows): a measurement and diagnosis switch,
// read on every call.
enum DensePath { kPathAuto = 0, kPathSplit = 1, kPathFused = 2 };
int dense_path_env() {
  const char* v = getenv("SPEC_VERIFY_DENSE_KERNELS");
  if (!v) return kPathAuto;
  if (strcmp(v, "split") == 0) return kPathSplit;
  if (strcmp(v, "fused") == 0) return kPathFused;
  return kPathAuto;
}

// cluster size (> 0) if the fused kernel takes this call, 0 if the two-kernel
// path does, -1 on a CUDA error
int dense_fused_choice(const void* tl, const void* dl, int B, int gamma, int V, int es, int* L) {
  const int path = dense_path_env();
  if (path == kPathSplit) return 0;
  if (!(((size_t)V * es) % 16 == 0 && aligned_to(tl, 16) && (gamma == 0 || aligned_to(dl, 16))))
    return 0;
  return sv::fused_plan(B, gamma, V, es, path != kPathFused, L);
}


}  // namespace

namespace sv {
// Workspace bytes that spec_verify_dense touches for these arguments (the
// path it will take): 0 on a CUDA error.
size_t dense_workspace_need(const void* target_logits, const void* draft_logits, int es, int B,
                            int gamma, int V) {
  if (small_fits(gamma + 1, V)) return sizeof(WsHeader);
  int L = 0;
  const int C = dense_fused_choice(target_logits, draft_logits, B, gamma, V, es, &L);
  if (C < 0) return 0;
  if (C > 0) return fused_layout(B, gamma).total;
  return dense_layout(B, gamma, dense_geom(V, es)).total;
}
size_t dense_workspace_floor(int B, int gamma, int V) {
  if (small_fits(gamma + 1, V)) return sizeof(WsHeader);
  // the single-pass layout is the smaller of the two large-vocabulary ones
  return fused_layout(B, gamma).total;
}
}  // namespace sv

extern "C" {

int spec_verify_abi_version(void) { return SV_ABI_VERSION; }

size_t spec_verify_workspace_size(int B, int gamma_or_W, int V) {
  if (B < 0 || gamma_or_W < 0 || V <= 0) return 0;
  // fp32 rows need the most pieces, so they bound both dtypes
  const size_t d = dense_ws_bytes(B, gamma_or_W, V, 4);
  return d > sizeof(sv::WsHeader) ? d : sizeof(sv::WsHeader);
}

sv_status spec_verify_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!workspace || ws_bytes < sizeof(sv::WsHeader)) return SV_ERR_INVALID_ARG;
  return launch_status(cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream));
}

int spec_verify_dense(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_ids, const float* u_accept, const float* u_sample,
                      int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                      float* residual_out, float* accept_prob_out, void* workspace,
                      size_t ws_bytes, sv_stream_t stream) {
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || !u_sample || !n_accepted || !out_tokens || !workspace) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_logits || !draft_ids || !u_accept)) return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(target_logits, es) || (draft_logits && !aligned_to(draft_logits, es)))
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(u_sample, 4) || !aligned_to(n_accepted, 4) || !aligned_to(out_tokens, 4) ||
      (draft_ids && !aligned_to(draft_ids, 4)) || (u_accept && !aligned_to(u_accept, 4)) ||
      (residual_out && !aligned_to(residual_out, 4)) ||
      (accept_prob_out && !aligned_to(accept_prob_out, 4)) || !aligned_to(workspace, 256))
    return SV_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(sv::WsHeader)) return SV_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  sv::WsHeader* hdr = reinterpret_cast<sv::WsHeader*>(workspace);

  if (small_fits(gamma + 1, V)) {
    sv::SmallParams p;
    memset(&p, 0, sizeof p);
    p.lt = static_cast<const unsigned char*>(target_logits);
    p.ld = static_cast<const unsigned char*>(draft_logits);
    p.x = draft_ids;
    p.order = nullptr;
    p.u_acc = u_accept;
    p.u_s = u_sample;
    p.n_out = n_accepted;
    p.tok_out = out_tokens;
    p.resid_out = residual_out;
    p.acc_out = accept_prob_out;
    p.status = &hdr->status;
    p.B = B;
    p.V = V;
    p.R = gamma + 1;
    p.G = gamma;
    p.D = 0;
    p.anyorder = 0;
    p.bf16 = (dtype == SV_BF16);
    p.vstride = small_vstride(V);
    p.flat = !p.bf16 && p.vstride == V && ((size_t)(gamma + 1) * V * 4) % 16 == 0 &&
             ((size_t)gamma * V * 4) % 16 == 0 && aligned_to(target_logits, 16) &&
             (gamma == 0 || aligned_to(draft_logits, 16));
    return launch_status(sv::launch_small(p, s));
  }

  {
    int Ls = 0;
    const int C = dense_fused_choice(target_logits, draft_logits, B, gamma, V, es, &Ls);
    if (C < 0) return SV_ERR_CUDA;
    if (C > 0) {  // one pass: a thread-block cluster per (row, position)
      const sv::FusedLayout FL = sv::fused_layout(B, gamma);
      if (ws_bytes < FL.total) return SV_ERR_INVALID_ARG;
      unsigned char* ws = static_cast<unsigned char*>(workspace);
      sv::FusedParams f;
      memset(&f, 0, sizeof f);
      f.lt = static_cast<const unsigned char*>(target_logits);
      f.ld = static_cast<const unsigned char*>(draft_logits);
      f.x = draft_ids;
      f.u_acc = u_accept;
      f.u_s = u_sample;
      f.n_out = n_accepted;
      f.tok_out = out_tokens;
      f.acc_out = accept_prob_out;
      f.status = &hdr->status;
      f.cnt = reinterpret_cast<uint32_t*>(ws + FL.cnt);
      f.rej = reinterpret_cast<uint32_t*>(ws + FL.rej);
      f.rec = reinterpret_cast<sv::UnitRec*>(ws + FL.rec);
      f.B = B;
      f.G = gamma;
      f.V = V;
      f.bf16 = (dtype == SV_BF16);
      f.L = Ls;
      f.keep_stop = residual_out != nullptr;
      if (sv::launch_dense_fused(f, C, s) != cudaSuccess) return SV_ERR_CUDA;
      if (residual_out && sv::launch_dense_fused_resid_out(f, residual_out, s) != cudaSuccess)
        return SV_ERR_CUDA;
      return SV_OK;
    }
  }

  const sv::DenseGeom g = sv::dense_geom(V, es);
  const sv::DenseLayout L = sv::dense_layout(B, gamma, g);
  if (ws_bytes < L.total) return SV_ERR_INVALID_ARG;
  // pieces are numbered with 31-bit indices in places
  if ((long long)B * (gamma + 1) * g.np >= (1ll << 31) - 1) return SV_ERR_INVALID_ARG;
  sv::DenseParams p;
  memset(&p, 0, sizeof p);
  p.lt = static_cast<const unsigned char*>(target_logits);
  p.ld = static_cast<const unsigned char*>(draft_logits);
  p.x = draft_ids;
  p.u_acc = u_accept;
  p.u_s = u_sample;
  p.n_out = n_accepted;
  p.tok_out = out_tokens;
  p.acc_out = accept_prob_out;
  p.ws = static_cast<unsigned char*>(workspace);
  p.L = L;
  p.g = g;
  p.B = B;
  p.G = gamma;
  p.V = V;
  p.bf16 = (dtype == SV_BF16);
  p.aligned = ((size_t)V * es) % 16 == 0 && aligned_to(target_logits, 16) &&
              (!draft_logits || aligned_to(draft_logits, 16));
  p.keep_stop = residual_out != nullptr;
  if (sv::launch_dense(p, s) != cudaSuccess) return SV_ERR_CUDA;
  if (residual_out && sv::launch_dense_resid_out(p, residual_out, s) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

int spec_verify_greedy(const void* target_logits, sv_dtype dtype, const int32_t* draft_ids,
                       int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                       void* workspace, size_t ws_bytes, sv_stream_t stream) {
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || !n_accepted || !out_tokens || !workspace) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && !draft_ids) return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(target_logits, es) || !aligned_to(n_accepted, 4) || !aligned_to(out_tokens, 4) ||
      (draft_ids && !aligned_to(draft_ids, 4)) || !aligned_to(workspace, 256))
    return SV_ERR_INVALID_ARG;
  const sv::DenseGeom g = sv::dense_geom(V, es);
  const sv::DenseLayout L = sv::dense_layout(B, gamma, g);
  if (ws_bytes < L.total) return SV_ERR_INVALID_ARG;
  if ((long long)B * (gamma + 1) * g.np >= (1ll << 31) - 1) return SV_ERR_INVALID_ARG;
  sv::DenseParams p;
  memset(&p, 0, sizeof p);
  p.lt = static_cast<const unsigned char*>(target_logits);
  p.x = draft_ids;
  p.n_out = n_accepted;
  p.tok_out = out_tokens;
  p.ws = static_cast<unsigned char*>(workspace);
  p.L = L;
  p.g = g;
  p.B = B;
  p.G = gamma;
  p.V = V;
  p.bf16 = (dtype == SV_BF16);
  p.aligned = ((size_t)V * es) % 16 == 0 && aligned_to(target_logits, 16);
  return launch_status(sv::launch_greedy(p, (cudaStream_t)stream));
}

int spec_commit_confident(const void* logits, sv_dtype dtype, const int32_t* masked, float tau,
                          int B, int W, int V, int32_t* commit, int32_t* tokens,
                          float* confidence, void* workspace, size_t ws_bytes,
                          sv_stream_t stream) {
  if (B < 0 || W < 1 || W > SV_MAX_GAMMA + 1 || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (tau != tau) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !masked || !commit || !tokens || !workspace) return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(logits, es) || !aligned_to(masked, 4) || !aligned_to(commit, 4) ||
      !aligned_to(tokens, 4) || (confidence && !aligned_to(confidence, 4)) ||
      !aligned_to(workspace, 256))
    return SV_ERR_INVALID_ARG;
  const sv::DenseGeom g = sv::dense_geom(V, es);
  const sv::DenseLayout L = sv::dense_layout(B, W - 1, g);
  if (ws_bytes < L.total) return SV_ERR_INVALID_ARG;
  if ((long long)B * W * g.np >= (1ll << 31) - 1) return SV_ERR_INVALID_ARG;
  sv::DenseParams p;
  memset(&p, 0, sizeof p);
  p.lt = static_cast<const unsigned char*>(logits);
  p.x = masked;
  p.tok_out = tokens;
  p.ws = static_cast<unsigned char*>(workspace);
  p.L = L;
  p.g = g;
  p.B = B;
  p.G = W - 1;
  p.V = V;
  p.bf16 = (dtype == SV_BF16);
  p.aligned = ((size_t)V * es) % 16 == 0 && aligned_to(logits, 16);
  return launch_status(sv::launch_commit(p, tau, commit, confidence, (cudaStream_t)stream));
}

int spec_support_topk(const void* logits, sv_dtype dtype, int N, int V, float temperature,
                      int top_k, float top_p, int32_t* ids, float* probs, void* workspace,
                      size_t ws_bytes, sv_stream_t stream) {
  if (N < 0 || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > SV_MAX_TOPK || top_k > V) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(temperature < INFINITY) || top_p != top_p) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (N == 0) return SV_OK;
  if (!logits || !ids || !probs || !workspace || ws_bytes < sizeof(sv::WsHeader)) return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(logits, es) || !aligned_to(ids, 4) || !aligned_to(probs, 4) ||
      !aligned_to(workspace, 256))
    return SV_ERR_INVALID_ARG;
  sv::WsHeader* hdr = reinterpret_cast<sv::WsHeader*>(workspace);
  const int aligned = ((size_t)V * es) % 16 == 0 && aligned_to(logits, 16);
  return launch_status(sv::launch_support(static_cast<const unsigned char*>(logits), N, V, top_k,
                                          dtype == SV_BF16, aligned, temperature, top_p, ids,
                                          probs, &hdr->status, (cudaStream_t)stream));
}

int spec_verify_sparse(const int32_t* tgt_ids, const float* tgt_probs, int kt,
                       const int32_t* drf_ids, const float* drf_probs, int kd,
                       const int32_t* draft_tokens, const float* u_accept, const float* u_sample,
                       int B, int gamma, int V, int32_t* n_accepted, int32_t* out_tokens,
                       float* residual_out, float* accept_prob_out, void* workspace,
                       size_t ws_bytes, sv_stream_t stream) {
  if (B < 0 || gamma < 0 || gamma > 31 || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (kt < 1 || kt > SV_MAX_LIST || (gamma > 0 && (kd < 1 || kd > SV_MAX_LIST)))
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!tgt_ids || !tgt_probs || !u_sample || !n_accepted || !out_tokens || !workspace)
    return SV_ERR_INVALID_ARG;
  if (gamma > 0 && (!drf_ids || !drf_probs || !draft_tokens || !u_accept)) return SV_ERR_INVALID_ARG;
  const void* ptrs[] = {tgt_ids, tgt_probs, drf_ids, drf_probs, draft_tokens, u_accept,
                        u_sample, n_accepted, out_tokens, residual_out, accept_prob_out};
  for (const void* q : ptrs)
    if (q && !aligned_to(q, 4)) return SV_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(sv::WsHeader) || !aligned_to(workspace, 256)) return SV_ERR_INVALID_ARG;
  sv::SparseParams p;
  memset(&p, 0, sizeof p);
  p.tid = tgt_ids;
  p.tp = tgt_probs;
  p.did = drf_ids;
  p.dp = drf_probs;
  p.x = draft_tokens;
  p.u_acc = u_accept;
  p.u_s = u_sample;
  p.n_out = n_accepted;
  p.tok_out = out_tokens;
  p.resid_out = residual_out;
  p.acc_out = accept_prob_out;
  p.status = &reinterpret_cast<sv::WsHeader*>(workspace)->status;
  p.B = B;
  p.G = gamma;
  p.V = V;
  p.kt = kt;
  p.kd = gamma > 0 ? kd : 1;
  return launch_status(sv::launch_sparse(p, (cudaStream_t)stream));
}

int spec_verify_anyorder(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* order, const int32_t* draft_tokens,
                         const float* u_accept, const float* u_sample, int B, int D, int W,
                         int V, int32_t* n_accepted, int32_t* out_tokens, float* residual_out,
                         float* accept_prob_out, void* workspace, size_t ws_bytes,
                         sv_stream_t stream) {
  if (B < 0 || W < 1 || W > 32 || D < W || D > SV_MAX_GAMMA * 64 || V < 1 || V > SV_MAX_VOCAB)
    return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (!small_fits(W, V)) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !order || !draft_tokens || !u_accept || !u_sample ||
      !n_accepted || !out_tokens || !workspace)
    return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(target_logits, es) || !aligned_to(draft_logits, es)) return SV_ERR_INVALID_ARG;
  const void* ptrs[] = {order, draft_tokens, u_accept, u_sample, n_accepted, out_tokens,
                        residual_out, accept_prob_out};
  for (const void* q : ptrs)
    if (q && !aligned_to(q, 4)) return SV_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(sv::WsHeader) || !aligned_to(workspace, 256)) return SV_ERR_INVALID_ARG;
  sv::SmallParams p;
  memset(&p, 0, sizeof p);
  p.lt = static_cast<const unsigned char*>(target_logits);
  p.ld = static_cast<const unsigned char*>(draft_logits);
  p.x = draft_tokens;
  p.order = order;
  p.u_acc = u_accept;
  p.u_s = u_sample;
  p.n_out = n_accepted;
  p.tok_out = out_tokens;
  p.resid_out = residual_out;
  p.acc_out = accept_prob_out;
  p.status = &reinterpret_cast<sv::WsHeader*>(workspace)->status;
  p.B = B;
  p.V = V;
  p.R = W;
  p.G = W;
  p.D = D;
  p.anyorder = 1;
  p.bf16 = (dtype == SV_BF16);
  p.vstride = small_vstride(V);
  p.flat = !p.bf16 && p.vstride == V && D == W && ((size_t)D * V * 4) % 16 == 0 &&
           aligned_to(target_logits, 16) && aligned_to(draft_logits, 16);
  return launch_status(sv::launch_small(p, (cudaStream_t)stream));
}

int spec_verify_check(void* workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!workspace || ws_bytes < sizeof(sv::WsHeader)) return SV_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  sv::WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  if (h.status) {
    sv::WsHeader* d = reinterpret_cast<sv::WsHeader*>(workspace);
    if (cudaMemsetAsync(&d->status, 0, sizeof(uint32_t), s) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  }
  if (h.status & sv::kStatusTimeout) return SV_ERR_TIMEOUT;
  if (h.status & sv::kStatusInputErr) return SV_ERR_DEVICE_INPUT;
  return SV_OK;
}

const char* spec_verify_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported request";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_DEVICE_INPUT: return "invalid input rows (n_accepted = -1)";
    case SV_ERR_TIMEOUT: return "bounded device wait expired; re-initialise the workspace";
    case SV_ERR_SCRATCH_LIMIT: return "sizes need more than the library's static scratch";
    default: return "unknown status";
  }
}


int spec_verify_anyorder_rounds(const void* target_logits, const void* draft_logits,
                                sv_dtype dtype, const int32_t* order, const int32_t* revealed,
                                const int32_t* window, const int32_t* draft_tokens,
                                const float* u_accept, const float* u_sample, int B, int R, int D,
                                int V, int32_t* tokens, int32_t* n_revealed,
                                int32_t* round_accepts, void* workspace, size_t ws_bytes,
                                sv_stream_t stream) {
  if (B < 0 || R < 1 || D < 1 || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if ((long long)D * V > (1ll << 31) || (long long)B * R * D > (1ll << 31)) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !order || !revealed || !window || !draft_tokens ||
      !u_accept || !u_sample || !tokens || !n_revealed || !round_accepts || !workspace)
    return SV_ERR_INVALID_ARG;
  const int es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned_to(target_logits, es) || !aligned_to(draft_logits, es)) return SV_ERR_INVALID_ARG;
  const void* ptrs[] = {order, revealed, window, draft_tokens, u_accept, u_sample,
                        tokens, n_revealed, round_accepts};
  for (const void* q : ptrs)
    if (!aligned_to(q, 4)) return SV_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(sv::WsHeader) || !aligned_to(workspace, 256)) return SV_ERR_INVALID_ARG;
  sv::RoundsParams p;
  memset(&p, 0, sizeof p);
  p.lt = static_cast<const unsigned char*>(target_logits);
  p.ld = static_cast<const unsigned char*>(draft_logits);
  p.bf16 = dtype == SV_BF16;
  p.order = order;
  p.i0 = revealed;
  p.win = window;
  p.x = draft_tokens;
  p.u_acc = u_accept;
  p.u_s = u_sample;
  p.B = B;
  p.R = R;
  p.D = D;
  p.V = V;
  p.tok_out = tokens;
  p.n_out = n_revealed;
  p.racc_out = round_accepts;
  p.status = &reinterpret_cast<sv::WsHeader*>(workspace)->status;
  return launch_status(sv::launch_rounds(p, (cudaStream_t)stream));
}

int spec_anyorder_window(int D, int revealed, float dtau) {
  if (D < 1 || revealed < 0) return -1;
  if (revealed >= D) return 0;
  const double half_pi = 1.57079632679489661923;
  // the schedule time at which `revealed` of D tokens are out: 1 - cos(t pi/2) = i/D
  const double t = acos(1.0 - (double)revealed / (double)D) / half_pi;
  const double t1 = fmin(1.0, t + (dtau > 0.f ? (double)dtau : 0.0));
  long long end = (long long)ceil((double)D * (1.0 - cos(half_pi * t1)) - 1e-9);
  if (end > D) end = D;
  const long long w = end - revealed;
  return (int)(w < 1 ? 1 : w);
}

}  // extern "C"
