// sv_internal.h -- private declarations shared by the host API and the
// kernels: workspace layout, kernel parameter blocks, launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sv {

// ---------------------------------------------------------------------------
// status word bits (workspace header)
// ---------------------------------------------------------------------------
enum : uint32_t { kStatusInputErr = 1u, kStatusTimeout = 2u };

struct WsHeader {
  unsigned long long reserved0;
  uint32_t reserved1;
  uint32_t status;  // kStatus* bits, sticky until spec_verify_check
  uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ---------------------------------------------------------------------------
// dense kernels: geometry and workspace layout
// ---------------------------------------------------------------------------
constexpr int kPieceBytes = 2048;  // one warp's slice of a logit row

struct DenseGeom {
  int es;   // element size in bytes (2: bf16, 4: fp32)
  int pe;   // elements per piece
  int np;   // pieces per row
  int np4;  // np rounded up to a multiple of 4 (16-byte aligned rows of masses)
};

inline DenseGeom dense_geom(int V, int es) {
  DenseGeom g;
  g.es = es;
  g.pe = kPieceBytes / es;
  g.np = (V + g.pe - 1) / g.pe;
  g.np4 = (g.np + 3) / 4 * 4;
  return g;
}

// Statistics of one piece of a (row, position): S = sum 2^(v*log2e - c) over
// the piece's elements, c = log2e * (max logit), target and draft; tx / dx are
// the target and draft logits at the draft token when the piece holds it
// (kNoTokenBits otherwise).
struct UnitPart {
  float St_hi, St_lo, Sd_hi, Sd_lo;  // float-float sums
  float ct, cd;
  float tx, dx;
};

// a quiet NaN with a payload that no bf16 logit (low half zero) and no fp32
// logit of a valid row (NaN rows are input errors) can take
constexpr uint32_t kNoTokenBits = 0x7FC0BAD0u;

// Per row: what the residual / bonus draw uses.  mode 0: residual
// max(p_n - q_n, 0); mode 1: draw from p (bonus, or the zero-residual
// fallback); mode 2: input error.
struct StopInfo {
  int32_t n;
  int32_t mode;
  float ct, cd;
  float invSt, invSd;
  double T;
};

struct DenseLayout {  // byte offsets into the workspace
  size_t upart, stop, rmass, rcnt, total;
};

// per row: the count of its pieces whose statistics are written, one counter
// per 128-byte line (the row kernel's waits poll them while the statistics
// grid streams)
constexpr int kRowCountStride = 32;  // uint32 words

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline DenseLayout dense_layout(long long B, int G, const DenseGeom& g) {
  DenseLayout L;
  size_t o = sizeof(WsHeader);
  L.upart = o;
  o = align_up(o + sizeof(UnitPart) * (size_t)B * (size_t)(G + 1) * (size_t)g.np, 256);
  L.stop = o;
  o = align_up(o + sizeof(StopInfo) * (size_t)B, 256);
  L.rmass = o;
  o = align_up(o + sizeof(float) * (size_t)B * (size_t)g.np4, 256);
  L.rcnt = o;
  o = align_up(o + sizeof(uint32_t) * kRowCountStride * (size_t)B, 256);
  L.total = o;
  return L;
}

struct DenseParams {
  const unsigned char* lt;  // [B, G+1, V]
  const unsigned char* ld;  // [B, G, V]
  const int32_t* x;         // [B, G]
  const float* u_acc;       // [B, G]
  const float* u_s;         // [B]
  int32_t* n_out;           // [B]
  int32_t* tok_out;         // [B, G+1]
  float* acc_out;           // [B, G] or null
  unsigned char* ws;
  DenseLayout L;
  DenseGeom g;
  int B, G, V;
  int bf16;       // 1: bf16 logits, 0: fp32
  int aligned;    // 1: rows 16-byte aligned -> 16-byte vector loads
  int keep_stop;  // 1: residual_out requested; its kernel reads and clears stop[]
  long long stats_warps;  // warps of the statistics grid (their piece ranges locate the records)
};

// ---------------------------------------------------------------------------
// dense, single pass: one thread-block cluster per (row, position) unit
// ---------------------------------------------------------------------------
// Outcome of one unit, written by the CTA that finished it (32 bytes).
struct UnitRec {
  uint32_t flags;      // kRec* bits
  int32_t token;       // the draw at this position (kRecDrawn)
  float ct, cd;        // log2e * max of the target / draft row
  float invSt, invSd;  // 1 / sum 2^(v log2e - c) of the target / draft row
  float T_hi, T_lo;    // total mass of the distribution the draw walked
};
static_assert(sizeof(UnitRec) == 32, "unit record is 32 bytes");
enum : uint32_t {
  kRecAccept = 1u,   // the draft token was accepted
  kRecErr = 2u,      // input error in this unit
  kRecPDraw = 4u,    // the draw used p (bonus, or a zero residual)
  kRecDrawn = 8u,    // token holds a draw
  kRecTimeout = 16u  // a bulk copy did not land within the bounded wait
};

struct FusedLayout {  // byte offsets into the workspace
  size_t cnt, rej, rec, total;
};
inline FusedLayout fused_layout(long long B, int G) {
  FusedLayout L;
  size_t o = sizeof(WsHeader);
  L.cnt = o;  // per row: units that have finished
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.rej = o;  // per row: G + 1 - j of the earliest rejection seen so far (0: none)
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.rec = o;  // [B, G + 1] unit records
  o = align_up(o + sizeof(UnitRec) * (size_t)B * (size_t)(G + 1), 256);
  L.total = o;
  return L;
}

struct FusedParams {
  const unsigned char* lt;  // [B, G+1, V]
  const unsigned char* ld;  // [B, G, V]
  const int32_t* x;         // [B, G]
  const float* u_acc;       // [B, G]
  const float* u_s;         // [B]
  int32_t* n_out;           // [B]
  int32_t* tok_out;         // [B, G+1]
  float* acc_out;           // [B, G] or null
  uint32_t* status;         // workspace status word
  uint32_t* cnt;            // [B]
  uint32_t* rej;            // [B]
  UnitRec* rec;             // [B, G+1]
  int B, G, V;
  int bf16;
  int L;          // elements of a row per cluster rank (a multiple of 16 / element size)
  int keep_stop;  // residual_out follows: the stop record of each row is kept for it
};

// Cluster size of the single-pass kernel for these sizes, with the slice
// length in *L_out; 0: the call goes to the two-kernel path (rows not a
// multiple of 16 bytes, slices too long, or -- with single_wave -- a grid
// that is not resident all at once); -1: CUDA error.
int fused_plan(long long B, int G, int V, int es, bool single_wave, int* L_out);
cudaError_t launch_dense_fused(const FusedParams& p, int C, cudaStream_t s);
cudaError_t launch_dense_fused_resid_out(const FusedParams& p, float* resid_out, cudaStream_t s);
// workspace bytes the dense call touches on the path it takes (0: CUDA error)
size_t dense_workspace_need(const void* target_logits, const void* draft_logits, int es, int B,
                            int gamma, int V);
// the least of those over every path these sizes can take (host only, no CUDA call)
size_t dense_workspace_floor(int B, int gamma, int V);

// ---------------------------------------------------------------------------
// small-vocabulary warp-per-row kernel (dense and any-order)
// ---------------------------------------------------------------------------
struct SmallParams {
  const unsigned char* lt;
  const unsigned char* ld;
  const int32_t* x;      // dense: draft ids [B, G]; any-order: tokens [B, D]
  const int32_t* order;  // any-order: [B, W]; dense: null
  const float* u_acc;
  const float* u_s;
  int32_t* n_out;
  int32_t* tok_out;
  float* resid_out;
  float* acc_out;
  uint32_t* status;
  int B, V;
  int R;      // positions handled by the warp (dense: G+1 target rows; any-order: W)
  int G;      // dense: gamma; any-order: W (number of accept tests)
  int D;      // any-order: sequence length; dense: unused
  int anyorder;
  int bf16;
  int vstride;  // shared-memory row stride in floats (odd)
  int flat;     // 1: fp32 row blocks staged whole, in source order, by 16-byte copies
};

// ---------------------------------------------------------------------------
// sparse top-k kernel
// ---------------------------------------------------------------------------
struct SparseParams {
  const int32_t* tid;
  const float* tp;
  const int32_t* did;
  const float* dp;
  const int32_t* x;
  const float* u_acc;
  const float* u_s;
  int32_t* n_out;
  int32_t* tok_out;
  float* resid_out;
  float* acc_out;
  uint32_t* status;
  int B, G, V, kt, kd;
};

// a launch configuration with programmatic stream serialisation (the kernel
// starts with griddepcontrol.wait); `attr` holds the one attribute
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  c.attrs = attr;
  c.numAttrs = 1;
  return c;
}

// launchers (return the CUDA error of the launch)
// the two dense kernels (statistics + row decisions, then residual + draw)
cudaError_t launch_dense(const DenseParams& p, cudaStream_t s);
cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s);
cudaError_t launch_greedy(const DenseParams& p, cudaStream_t s);  // greedy: target logits and ids only
// confidence-threshold commit: p.lt = logits [B, W, V], p.x = masked [B, W],
// p.G = W - 1, p.tok_out = tokens [B, W]
cudaError_t launch_commit(const DenseParams& p, float tau, int32_t* commit, float* confidence,
                          cudaStream_t s);
// sparse support lists (temperature, top-k, top-p) from dense logits [N, V]
// windowed multi-round any-order verification (one CTA per sequence)
struct RoundsParams {
  const unsigned char* lt;  // target logits [B, R, D, V]
  const unsigned char* ld;  // draft logits [B, D, V]
  int bf16;
  const int32_t* order;     // sigma [B, D]
  const int32_t* i0;        // revealed count [B]
  const int32_t* win;       // window length [B]
  const int32_t* x;         // draft tokens [B, R, D]
  const float* u_acc;       // [B, R, D], by sigma index
  const float* u_s;         // [B, R]
  int B, R, D, V;
  int32_t* tok_out;         // [B, D]
  int32_t* n_out;           // [B]
  int32_t* racc_out;        // [B, R]
  uint32_t* status;
};
cudaError_t launch_rounds(const RoundsParams& p, cudaStream_t s);

cudaError_t launch_support(const unsigned char* lt, int N, int V, int K, int bf16, int aligned,
                           float temperature, float top_p, int32_t* ids, float* probs,
                           uint32_t* status, cudaStream_t s);
cudaError_t launch_small(const SmallParams& p, cudaStream_t s);
size_t small_smem_per_warp(int R, int vstride);
cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s);

}  // namespace sv
