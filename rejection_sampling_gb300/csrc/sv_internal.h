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
  unsigned long long ticket;  // dense persistent kernel: next work ticket
  uint32_t exit_cnt;          // CTAs that finished (last one resets ticket)
  uint32_t status;            // kStatus* bits, sticky until spec_verify_check
  uint32_t abort;             // set when a bounded wait ran out
  uint32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ---------------------------------------------------------------------------
// dense persistent kernel: geometry and workspace layout
// ---------------------------------------------------------------------------
constexpr int kPieceBytes = 4096;     // one pipeline stage: one row slice for statistics
constexpr int kResidRowBytes = 2048;  // residual stage: 2 KB target + 2 KB draft slice
constexpr int kUnitPieces = 8;        // row pieces per work unit

struct DenseGeom {
  int es;    // element size in bytes (2: bf16, 4: fp32)
  int pe;    // elements per statistics piece
  int re;    // elements per residual piece (per row)
  int np_s;  // statistics pieces per row
  int np_r;  // residual pieces per row
  int nc_s;  // statistics units per (row, position)
  int nc_r;  // residual units per row
};

inline DenseGeom dense_geom(int V, int es) {
  DenseGeom g;
  g.es = es;
  g.pe = kPieceBytes / es;
  g.re = kResidRowBytes / es;
  g.np_s = (V + g.pe - 1) / g.pe;
  g.np_r = (V + g.re - 1) / g.re;
  g.nc_s = (g.np_s + kUnitPieces - 1) / kUnitPieces;
  g.nc_r = (g.np_r + kUnitPieces - 1) / kUnitPieces;
  return g;
}

// Combined statistics of one work unit (up to 8 target + 8 draft pieces):
// S = sum 2^(v*log2e - c) over the unit's elements, c = log2e * (max logit).
struct UnitPart {
  double St, Sd;
  float ct, cd;
  float pad[2];
};

// Per (row, position) result of the accept test.
struct PosInfo {
  double St, Sd;  // normalisers relative to ct, cd
  float ct, cd;
  int32_t accept;
  int32_t err;
};

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
  size_t cnt_pos, cnt_row, cnt_res, ready, upart, pos, stop, rmass, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline DenseLayout dense_layout(long long B, int G, const DenseGeom& g) {
  DenseLayout L;
  size_t o = sizeof(WsHeader);
  L.cnt_pos = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B * (size_t)(G + 1), 256);
  L.cnt_row = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.cnt_res = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.ready = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.upart = o;
  o = align_up(o + sizeof(UnitPart) * (size_t)B * (size_t)(G + 1) * (size_t)g.nc_s, 256);
  L.pos = o;
  o = align_up(o + sizeof(PosInfo) * (size_t)B * (size_t)(G + 1), 256);
  L.stop = o;
  o = align_up(o + sizeof(StopInfo) * (size_t)B, 256);
  L.rmass = o;
  o = align_up(o + sizeof(float) * (size_t)B * (size_t)g.np_r, 256);
  L.total = o;
  return L;
}

#if defined(__CUDACC__)
#define SV_HD __host__ __device__ __forceinline__
#else
#define SV_HD inline
#endif

// Ticket order of the dense persistent kernel.  Round r holds the statistics
// units of row r (if r < B) followed by the residual units of row r - lag (if
// r >= lag); Us = (G+1) * nc_s statistics units and Ur = nc_r residual units
// per row.  Returns whether ticket t is a residual unit, its row, and its
// index within that row's units of that kind.
SV_HD void dense_ticket_row(long long t, long long B, int G, int nc_s, int nc_r, int lag,
                            int* resid, int* b, long long* rem) {
  const long long Us = (long long)(G + 1) * nc_s, Ur = nc_r, lg = lag;
  const long long LA = lg < B ? lg : B;
  const long long tA = LA * Us;
  const long long nB = B > lg ? B - lg : 0;
  const long long tB = tA + nB * (Us + Ur);
  if (t < tA) {
    *resid = 0;
    *b = (int)(t / Us);
    *rem = t % Us;
  } else if (t < tB) {
    const long long t2 = t - tA;
    const long long r = lg + t2 / (Us + Ur);
    const long long q = t2 % (Us + Ur);
    if (q < Us) {
      *resid = 0;
      *b = (int)r;
      *rem = q;
    } else {
      *resid = 1;
      *b = (int)(r - lg);
      *rem = q - Us;
    }
  } else {
    const long long t2 = t - tB;
    *resid = 1;
    *b = (int)((B - LA) + t2 / Ur);
    *rem = t2 % Ur;
  }
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
  long long tickets;  // total work units
  long long wait_bound;
  int B, G, V;
  int bf16;     // 1: bf16 logits, 0: fp32
  int aligned;  // 1: rows 16-byte aligned -> bulk copies
  int lag;      // residual units of row r are scheduled after statistics of row r + lag
};

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

// launchers (return the CUDA error of the launch)
cudaError_t launch_dense(const DenseParams& p, int grid, cudaStream_t s);
cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s);
int dense_ctas_per_sm();
size_t dense_smem_bytes();
cudaError_t launch_small(const SmallParams& p, cudaStream_t s);
size_t small_smem_per_warp(int R, int vstride);
cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s);

}  // namespace sv
