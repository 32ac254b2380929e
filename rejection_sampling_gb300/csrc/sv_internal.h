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
  unsigned long long ticket;  // dense persistent kernel: next statistics ticket
  uint32_t exit_cnt;          // CTAs that finished (the last one resets the counters)
  uint32_t status;            // kStatus* bits, sticky until spec_verify_check
  uint32_t abort;             // set when a bounded wait ran out
  uint32_t rq_head;           // residual queue: next entry to claim
  uint32_t rq_reserve;        // residual queue: entries reserved by row finalisers
  uint32_t timeout_site;      // first wait that ran out (diagnostics; 0 = none)
  uint32_t timeout_info;      // site-specific detail (slot, entry, ...)
  uint32_t pad[55];
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
  int np_r4; // np_r rounded up to a multiple of 4 (16-byte aligned rows of masses)
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
  g.np_r4 = (g.np_r + 3) / 4 * 4;
  g.nc_s = (g.np_s + kUnitPieces - 1) / kUnitPieces;
  g.nc_r = (g.np_r + kUnitPieces - 1) / kUnitPieces;
  return g;
}

// Combined statistics of one work unit (up to 8 target + 8 draft pieces):
// S = sum 2^(v*log2e - c) over the unit's elements, c = log2e * (max logit).
struct UnitPart {
  float St_hi, St_lo, Sd_hi, Sd_lo;  // float-float sums
  float ct, cd;
  float pad[2];
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
  size_t cnt_row, cnt_res, rq, upart, stop, rmass, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline DenseLayout dense_layout(long long B, int G, const DenseGeom& g) {
  DenseLayout L;
  size_t o = sizeof(WsHeader);
  L.cnt_row = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.cnt_res = o;
  o = align_up(o + sizeof(uint32_t) * (size_t)B, 256);
  L.rq = o;  // one 64-bit entry per residual unit; 0 = not yet published
  o = align_up(o + sizeof(unsigned long long) * (size_t)B * (size_t)g.nc_r, 256);
  L.upart = o;
  o = align_up(o + sizeof(UnitPart) * (size_t)B * (size_t)(G + 1) * (size_t)g.nc_s, 256);
  L.stop = o;
  o = align_up(o + sizeof(StopInfo) * (size_t)B, 256);
  L.rmass = o;
  o = align_up(o + sizeof(float) * (size_t)B * (size_t)g.np_r4, 256);
  L.total = o;
  return L;
}

#if defined(__CUDACC__)
#define SV_HD __host__ __device__ __forceinline__
#else
#define SV_HD inline
#endif

// Division of n < 2^31 by a fixed d >= 1 with one 64-bit multiply and a
// shift: q = (n * m) >> (32 + sh), m = ceil(2^(32+sh) / d), sh = ceil(log2 d)
// (Granlund and Montgomery's round-up method; exact because n * (m - 2^(32+sh)/d)
// < 2^31 <= 2^(32+sh)/d for d <= 2^sh).
struct FastDiv {
  unsigned long long m;
  unsigned d;
  int sh;
};

inline FastDiv make_fastdiv(unsigned d) {
  FastDiv f;
  f.d = d;
  int sh = 0;
  while ((1ull << sh) < d) ++sh;
  f.sh = sh;
  const unsigned long long num = 1ull << (32 + sh);
  f.m = num / d + ((num % d) ? 1ull : 0ull);
  return f;
}

SV_HD unsigned fdiv(unsigned n, const FastDiv& f) {
  return (unsigned)(((unsigned long long)n * f.m) >> (32 + f.sh));
}

// Statistics tickets are numbered row by row: ticket t is row b = t / Us,
// position j and unit c with t - b * Us = j * nc_s + c (Us = (G+1) * nc_s).
// Residual units are not ticketed: a row's finaliser publishes them to the
// residual queue.
SV_HD void dense_ticket(long long t, int G, int nc_s, int* b, int* j, int* c) {
  const long long Us = (long long)(G + 1) * nc_s;
  const long long bb = t / Us, rem = t - bb * Us;
  *b = (int)bb;
  *j = (int)(rem / nc_s);
  *c = (int)(rem - (long long)(*j) * nc_s);
}

struct TicketConsts {
  FastDiv div_us, div_ncs;
};

inline TicketConsts make_ticket_consts(int G, int nc_s) {
  TicketConsts k;
  k.div_us = make_fastdiv((unsigned)((G + 1) * nc_s));
  k.div_ncs = make_fastdiv((unsigned)nc_s);
  return k;
}

// dense_ticket for t < 2^31 with the precomputed dividers
SV_HD void dense_ticket_fast(unsigned t, const TicketConsts& k, int* b, int* j, int* c) {
  const unsigned bb = fdiv(t, k.div_us);
  const unsigned rem = t - bb * k.div_us.d;
  const unsigned jj = fdiv(rem, k.div_ncs);
  *b = (int)bb;
  *j = (int)jj;
  *c = (int)(rem - jj * k.div_ncs.d);
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
  long long tickets;  // statistics units: B * (G+1) * nc_s
  int small_tickets;  // 1: every ticket fits in 31 bits (32-bit decode)
  unsigned resid_units;  // B * nc_r
  TicketConsts tk;
  long long wait_bound;
  int B, G, V;
  int bf16;       // 1: bf16 logits, 0: fp32
  int aligned;    // 1: rows 16-byte aligned -> bulk copies
  int keep_stop;  // 1: residual_out requested; its kernel reads and clears stop[]
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
