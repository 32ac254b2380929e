// sv_static.cu -- spec_verify_dense_static: dense verification for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they verify: code running inside a host callback or a custom allocator's
// own hooks, plug-ins loaded by a runtime that owns every allocation and
// forbids others, and embedded inference loops that must never touch the
// allocator after start-up.  They still own their inputs and outputs; what
// they cannot provide is the workspace.  This entry point takes its scratch
// from a fixed device array compiled into the library instead.
//
// The array is a file-scope __device__ object of SV_STATIC_SCRATCH_BYTES, so
// every GPU that loads the library holds it until the process exits.  In
// host code the array's name only stands for the symbol; its device address
// is looked up with cudaGetSymbolAddress once per device (with that device
// current) on the first call there, and kept.  That look-up may load the
// library's device code, so the first call on each device should come before
// any stream capture.
//
// Every call shares the one array: it clears the part it uses on the stream
// before the kernels run (so nothing a previous call left behind, finished
// or not, can leak in), and two calls whose work overlaps on the GPU -- on
// different streams, or from different host threads -- race on it.  The part
// a call uses is what the path it takes needs: the header alone for short
// vocabularies (the warp-per-row kernel), the per-row words and per-position
// records of the single-pass kernel, or the piece records of the two-kernel
// path; only the last depends on V.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace {

static __device__ __align__(256) unsigned char sv_static_scratch[SV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// device address of the scratch array on the current device (set-up on first use)
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, sv_static_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int spec_verify_dense_static(const void* target_logits, const void* draft_logits,
                                        sv_dtype dtype, const int32_t* draft_ids,
                                        const float* u_accept, const float* u_sample, int B,
                                        int gamma, int V, int32_t* n_accepted,
                                        int32_t* out_tokens, float* residual_out,
                                        float* accept_prob_out, sv_stream_t stream) {
  // the same argument rules as spec_verify_dense, checked before anything is launched
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  // sizes whose workspace exceeds the array on every path are refused first,
  // on the host alone (no CUDA call)
  if (sv::dense_workspace_floor(B, gamma, V) > (size_t)SV_STATIC_SCRATCH_BYTES)
    return SV_ERR_SCRATCH_LIMIT;
  if (!target_logits || !u_sample || !n_accepted || !out_tokens) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_logits || !draft_ids || !u_accept)) return SV_ERR_INVALID_ARG;
  const size_t es = (dtype == SV_BF16) ? 2 : 4;
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)))
    return SV_ERR_INVALID_ARG;
  if (!aligned(u_sample, 4) || !aligned(n_accepted, 4) || !aligned(out_tokens, 4) ||
      (draft_ids && !aligned(draft_ids, 4)) || (u_accept && !aligned(u_accept, 4)) ||
      (residual_out && !aligned(residual_out, 4)) ||
      (accept_prob_out && !aligned(accept_prob_out, 4)))
    return SV_ERR_INVALID_ARG;

  // the workspace bytes of the path this call takes (the same choice
  // spec_verify_dense makes from the same arguments)
  const size_t need = sv::dense_workspace_need(target_logits, draft_logits, (int)es, B, gamma, V);
  if (need == 0) return SV_ERR_CUDA;
  if (need > (size_t)SV_STATIC_SCRATCH_BYTES) return SV_ERR_SCRATCH_LIMIT;

  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != SV_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // the counters, records and status word must start at zero
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return SV_ERR_CUDA;
  return spec_verify_dense(target_logits, draft_logits, dtype, draft_ids, u_accept, u_sample, B,
                           gamma, V, n_accepted, out_tokens, residual_out, accept_prob_out,
                           scratch, need, stream);
}
