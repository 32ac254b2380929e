// sv_greedy.cu -- greedy (T = 0) verification for any vocabulary size.
//
// Under greedy decoding a draft token is accepted if and only if it is the
// target's own choice (DFlash/DFlash2 guide, 4.4; the condition's formula did
// not survive on the page, and the reading taken is the T -> 0 limit of the
// stochastic rule of the Uno article, "What 'lossless' actually has to
// mean"): with a_j = argmax_y target[b, j, y] (the smallest such y when ids
// tie),
//   n       = first j < gamma with x_j != a_j (gamma if none),
//   token n = a_n (the replacement, or the bonus a_gamma when n = gamma;
//             DFlash/DFlash2 guide, section 2).
// Only the target logits are read; no uniform is consumed.
//
// Design (two kernels per call, one HBM pass over the target logits).
//  * A target row is cut into 2 KB pieces, numbered (b, j, k) row-major.
//  * greedy_stats_kernel: a persistent grid, one CTA of 24 warps per SM;
//    every warp takes one contiguous range of pieces and streams it through
//    a private three-stage ring of 2 KB shared-memory stages filled by
//    16-byte cp.async (plain loads when rows are not 16-byte aligned).  Each
//    piece is reduced to (max, first index of the max, bad) -- bad: the piece
//    holds a NaN or +inf -- and folded into the running values of the
//    (b, j) segment the warp is in; each segment of a range ends in one
//    record at its first piece.
//  * greedy_row_kernel: one CTA per row, a programmatic dependent of the
//    statistics kernel.  A warp per position combines the position's records
//    (found from the statistics warps' ranges), giving a_j; the first
//    mismatch and the tokens follow.  The CTA clears the records it read, so
//    the workspace is all zero again after the call.
#include <climits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kGWarps = 24;  // warps per statistics CTA
constexpr int kGThreads = 32 * kGWarps;
constexpr int kGStages = 3;  // ring depth per warp (2 KB stages)
constexpr size_t kGSmem = (size_t)kGWarps * kGStages * kPieceBytes;
constexpr int kGRowWarps = 16;  // warps per row CTA
constexpr int kGMaxPos = 256;   // positions per row (gamma + 1 <= 256)
constexpr uint32_t kNegInf2 = 0xFF80FF80u;  // two bf16 -inf
constexpr uint32_t kNegInfF = 0xFF800000u;  // fp32 -inf

// one segment's running argmax (16 bytes, at the segment's first piece slot)
struct ArgRec {
  float m;   // maximum
  int idx;   // first id holding it (INT_MAX while the maximum is -inf)
  int bad;   // a NaN or +inf was seen
  int pad;
};

__device__ __forceinline__ const unsigned char* target_row(const DenseParams& P, int b, int j) {
  return P.lt + ((size_t)b * (P.G + 1) + j) * (size_t)P.V * P.g.es;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// this lane's 16-byte vectors lane + 32 i of a 2 KB piece with `ne` valid
// elements; elements past `ne` read as -inf
__device__ __forceinline__ void load_vectors(const unsigned char* base, int ne, int bf16,
                                             int aligned, int lane, uint4 (&r)[4]) {
  const int epv = bf16 ? 8 : 4;
  const uint32_t ninf = bf16 ? kNegInf2 : kNegInfF;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    if (aligned) {
      r[i] = (vi * epv < ne) ? __ldcs(reinterpret_cast<const uint4*>(base) + vi)
                             : make_uint4(ninf, ninf, ninf, ninf);
      continue;
    }
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (bf16) {
        const int e0 = vi * 8 + 2 * q;
        const uint16_t* h = reinterpret_cast<const uint16_t*>(base);
        const uint32_t lo = (e0 < ne) ? h[e0] : 0xFF80u;
        const uint32_t hi = (e0 + 1 < ne) ? h[e0 + 1] : 0xFF80u;
        w[q] = lo | (hi << 16);
      } else {
        const int e = vi * 4 + q;
        w[q] = (e < ne) ? reinterpret_cast<const uint32_t*>(base)[e] : kNegInfF;
      }
    }
    r[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// maxima that propagate NaN (max.NaN): a NaN anywhere makes the result NaN
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// (max, first index of the max, bad) of a piece, on every lane.  Element e
// of vector vi is id vi * epv + e of the piece.  The maximum comes first, by
// packed maxima that propagate NaN; then only the lanes holding it look for
// its first id among their elements, and the warp keeps the smallest.  The
// piece is bad when the maximum is NaN (a NaN anywhere) or +inf.
__device__ __forceinline__ void piece_argmax(const uint4 (&r)[4], int bf16, int lane, float& m,
                                             int& idx, int& bad) {
  float lm;
  if (bf16) {
    uint32_t mx = kNegInf2;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mx = bf16x2_max_nan(mx, bf16x2_max_nan(bf16x2_max_nan(r[i].x, r[i].y),
                                             bf16x2_max_nan(r[i].z, r[i].w)));
    lm = fmax_nan(bf16_lo(mx), bf16_hi(mx));
  } else {
    lm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      lm = fmax_nan(lm, fmax_nan(fmax_nan(__uint_as_float(r[i].x), __uint_as_float(r[i].y)),
                                 fmax_nan(__uint_as_float(r[i].z), __uint_as_float(r[i].w))));
  }
  float wm = lm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmax_nan(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  bad = (wm != wm) || (wm == INFINITY);
  int bi = INT_MAX;
  if (!bad && lm == wm) {  // this lane holds the maximum: its first id with it
#pragma unroll
    for (int i = 3; i >= 0; --i) {  // scanned backwards, so the last hit is the first id
      const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
      if (bf16) {
#pragma unroll
        for (int e = 7; e >= 0; --e)
          if (((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1])) == wm) bi = (lane + 32 * i) * 8 + e;
      } else {
#pragma unroll
        for (int e = 3; e >= 0; --e)
          if (__uint_as_float(w[e]) == wm) bi = (lane + 32 * i) * 4 + e;
      }
    }
  }
  bi = (int)__reduce_min_sync(0xffffffffu, (unsigned)bi);
  m = wm;
  idx = bi;
}

struct GItem {  // piece k of row-position (b, j)
  int b, j, k;
};
__device__ __forceinline__ GItem gitem_at(long long w, int G, int np) {
  const long long r = w / np;
  GItem it;
  it.k = (int)(w - r * np);
  it.b = (int)(r / (G + 1));
  it.j = (int)(r - (long long)it.b * (G + 1));
  return it;
}
__device__ __forceinline__ void gitem_next(GItem& it, int G, int np) {
  if (++it.k == np) {
    it.k = 0;
    if (++it.j == G + 1) {
      it.j = 0;
      ++it.b;
    }
  }
}

struct GSeg {
  long long w0;  // record slot: the segment's first piece
  int b, j;
  float m;
  int idx, bad;
};
__device__ __forceinline__ void gseg_begin(GSeg& s, const GItem& it, long long w) {
  s.w0 = w;
  s.b = it.b;
  s.j = it.j;
  s.m = -INFINITY;
  s.idx = INT_MAX;
  s.bad = 0;
}
__device__ __forceinline__ void gseg_write(const DenseParams& P, const GSeg& s, int lane) {
  if (lane == 0) {
    ArgRec* rec = reinterpret_cast<ArgRec*>(P.ws + P.L.upart) + s.w0;
    *reinterpret_cast<int4*>(rec) = make_int4(__float_as_int(s.m), s.idx, s.bad, 0);
  }
}
// fold piece `it` into the segment; pieces arrive in increasing id order, so
// a strictly greater maximum replaces the running one and a tie keeps it
__device__ __forceinline__ void gseg_add(GSeg& s, const GItem& it, const uint4 (&r)[4], int bf16,
                                         int pe, int lane) {
  float m;
  int idx, bad;
  piece_argmax(r, bf16, lane, m, idx, bad);
  if (m > s.m) {
    s.m = m;
    s.idx = it.k * pe + idx;
  }
  s.bad |= bad;
}

__global__ void __launch_bounds__(kGThreads, 1) greedy_stats_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // a programmatic dependent of whatever precedes it on the stream: nothing
  // is read before that grid has completed (it may have written the logits)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = P.G, np = P.g.np, pe = P.g.pe, epv = P.bf16 ? 8 : 4;
  const long long W = (long long)P.B * (G + 1) * np;
  const long long nwt = (long long)gridDim.x * kGWarps;
  const long long gw = (long long)blockIdx.x * kGWarps + warp;
  const long long lo = gw * W / nwt, hi = (gw + 1) * W / nwt;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lo >= hi) return;
  const uint32_t ninf = P.bf16 ? kNegInf2 : kNegInfF;
  GSeg seg;
  GItem out = gitem_at(lo, G, np);
  gseg_begin(seg, out, lo);

  if (!P.aligned) {  // rows not 16-byte aligned: plain loads, no ring
    for (long long w = lo; w < hi; ++w, gitem_next(out, G, np)) {
      if (out.b != seg.b || out.j != seg.j) {
        gseg_write(P, seg, lane);
        gseg_begin(seg, out, w);
      }
      const int ne = min(pe, P.V - out.k * pe);
      uint4 r[4];
      load_vectors(target_row(P, out.b, out.j) + (size_t)out.k * kPieceBytes, ne, P.bf16, 0, lane, r);
      gseg_add(seg, out, r, P.bf16, pe, lane);
    }
    gseg_write(P, seg, lane);
    return;
  }

  unsigned char* ring = smem_raw + (size_t)warp * kGStages * kPieceBytes;
  GItem in = out;
  long long wi = lo;
  auto issue = [&](int s) {
    const int ne = min(pe, P.V - in.k * pe);
    const unsigned char* src = target_row(P, in.b, in.j) + (size_t)in.k * kPieceBytes;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = lane + 32 * i;
      if (vi * epv < ne) cp_async16(ring + s * kPieceBytes + 16 * vi, src + 16 * vi);
    }
  };
#pragma unroll
  for (int s = 0; s < kGStages - 1; ++s) {
    if (wi < hi) {
      issue(s);
      gitem_next(in, G, np);
      ++wi;
    }
    cp_async_commit();
  }
  int slot = 0, islot = kGStages - 1;
  for (long long w = lo; w < hi; ++w) {
    if (out.b != seg.b || out.j != seg.j) {
      gseg_write(P, seg, lane);
      gseg_begin(seg, out, w);
    }
    if (wi < hi) {
      issue(islot);
      gitem_next(in, G, np);
      ++wi;
    }
    cp_async_commit();
    cp_async_wait_group<kGStages - 1>();
    const unsigned char* stage = ring + slot * kPieceBytes;
    const int ne = min(pe, P.V - out.k * pe);
    uint4 r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = lane + 32 * i;
      r[i] = (vi * epv < ne) ? *reinterpret_cast<const uint4*>(stage + 16 * vi)
                             : make_uint4(ninf, ninf, ninf, ninf);
    }
    gseg_add(seg, out, r, P.bf16, pe, lane);
    gitem_next(out, G, np);
    slot = (slot + 1 == kGStages) ? 0 : slot + 1;
    islot = (islot + 1 == kGStages) ? 0 : islot + 1;
  }
  gseg_write(P, seg, lane);
  cp_async_wait_group<0>();
}

// Row b: a warp per position combines the position's records into a_j, then
// the first mismatch and the tokens.  Clears the records it read.
__global__ void __launch_bounds__(32 * kGRowWarps) greedy_row_kernel(const __grid_constant__ DenseParams P) {
  __shared__ int s_n, s_err;
  __shared__ int s_arg[kGMaxPos];
  __shared__ int s_x[kGMaxPos];  // the row's draft tokens
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x, G = P.G, np = P.g.np;
  if (threadIdx.x == 0) {
    s_n = G;
    s_err = 0;
  }
  // the draft tokens first: an input, not a result of the statistics grid
  // (this grid starts once every statistics CTA has passed its own wait for
  // the grids before it; read from L2)
  for (int j = threadIdx.x; j < G; j += blockDim.x) s_x[j] = __ldcg(P.x + (size_t)b * G + j);
  // the statistics grid's records must be complete and visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  ArgRec* rec = reinterpret_cast<ArgRec*>(P.ws + P.L.upart);
  // the statistics grid gave warp g the pieces [lo(g), lo(g + 1)), lo(g) =
  // g W / nwt; a segment record sits at the first piece of each segment
  const long long W = (long long)P.B * (G + 1) * np, nwt = P.stats_warps;
  // the range arithmetic in 32 bits when every product fits (a 64-bit
  // division is a long software sequence on each row's critical path)
  const bool idx32 = (unsigned long long)(nwt + 1) * (unsigned long long)(W + 1) < (1ull << 32);
  const unsigned W32 = (unsigned)W, n32 = (unsigned)nwt;
  for (int j = warp; j <= G; j += kGRowWarps) {
    const int xj = (j < G) ? s_x[j] : 0;
    const long long P0 = ((long long)b * (G + 1) + j) * np, P1 = P0 + np;
    const long long g0 = idx32 ? (long long)(((unsigned)(P0 + 1) * n32 + W32 - 1) / W32) - 1
                               : ((P0 + 1) * nwt + W - 1) / W - 1;
    const long long g1 = idx32 ? (long long)(((unsigned)P1 * n32 + W32 - 1) / W32) - 1
                               : (P1 * nwt + W - 1) / W - 1;
    float m = -INFINITY;
    int idx = INT_MAX, bad = 0;
    for (long long g = g0 + lane; g <= g1; g += 32) {
      const long long l0 = idx32 ? (long long)((unsigned)g * W32 / n32) : g * W / nwt;
      const long long l1 = idx32 ? (long long)((unsigned)(g + 1) * W32 / n32) : (g + 1) * W / nwt;
      if (l1 <= l0) continue;  // an empty range writes nothing
      int4* rp = reinterpret_cast<int4*>(rec + (l0 > P0 ? l0 : P0));
      const int4 v = __ldcg(rp);
      *rp = make_int4(0, 0, 0, 0);
      const float rm = __int_as_float(v.x);
      if (rm > m || (rm == m && v.y < idx)) {
        m = rm;
        idx = v.y;
      }
      bad |= v.z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (om > m || (om == m && oi < idx)) {
        m = om;
        idx = oi;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const int err = bad || !(m > -INFINITY) || (j < G && (xj < 0 || xj >= P.V));
      s_arg[j] = idx;
      if (err) atomicOr(&s_err, 1);
      else if (j < G && xj != idx) atomicMin(&s_n, j);
    }
  }
  __syncthreads();
  const int err = s_err, n = s_n;
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  for (int j = threadIdx.x; j <= G; j += blockDim.x) {
    int v = -1;
    if (!err) v = (j < n) ? s_x[j] : (j == n ? s_arg[n] : -1);
    tok[j] = v;
  }
  if (threadIdx.x == 0) {
    P.n_out[b] = err ? -1 : n;
    if (err) atomicOr(&reinterpret_cast<WsHeader*>(P.ws)->status, kStatusInputErr);
  }
}

// ---------------------------------------------------------------------------
// Confidence-threshold commit of a block-diffusion pass ("SDAR" page,
// section 5, decoding timeline).  For every masked position i of block b:
// confidence c_i = max_y p_i(y) = 1 / S_i, S_i = sum_y 2^((l_y - max l) log2e),
// token a_i = argmax (smallest id on ties); masked positions with c_i > tau
// are committed, and when none clears tau the most confident one is (the
// smallest index on ties), so every pass makes progress.
//  * commit_stats_kernel: the greedy statistics kernel's sweep over the
//    logits [B, W, V], only over the pieces of masked positions: each CTA
//    lists the masked positions (a block-wide compaction of the flags, for
//    up to 8192 positions; beyond that every piece is swept and unmasked
//    ones are skipped) and the warps take equal shares of their pieces.  Per
//    piece S = sum 2^((v - m) log2e) (ex2.approx) joins (max, first id, bad);
//    segments fold (m, S) with one rescale (float-float) and leave a marked
//    record at their first piece's slot.
//  * commit_row_kernel: one CTA per block; a warp per masked position
//    collects the marked records in its position's slots into (c_i, a_i)
//    and zeroes them; thread 0 applies the threshold.
// ---------------------------------------------------------------------------
struct ConfRec {  // one segment (32 bytes, at the segment's first piece slot)
  float m;        // maximum
  float s_hi, s_lo;  // sum 2^((v - m) log2e), float-float
  int idx;        // first id holding the maximum
  int bad;        // a NaN or +inf was seen
  int live;       // 1: a record is here (the workspace is zero elsewhere)
  int pad[2];
};

// A segment's running statistics, per lane: the lane's maximum, the first
// id holding it, an integer reference point c >= log2e * max and the sum
// S = sum 2^(v log2e - c) of the lane's elements (float-float); the lanes are
// combined once, when the warp's range leaves the segment.
struct CSeg {
  long long w0;
  int b, j;
  float m;  // this lane's maximum
  float c;  // this lane's reference point
  ff S;     // this lane's sum, relative to c
  int idx, bad;
  bool live;  // the position is masked (a record will be written)
};

__device__ __forceinline__ bool is_masked(const DenseParams& P, int b, int j) {
  return __ldg(P.x + (size_t)b * (P.G + 1) + j) != 0;
}

constexpr int kCMaxList = 8192;  // positions whose masked subset is listed in shared memory
constexpr int kCSlots = 5;       // record slots per lane in flight in the commit row kernel
// The commit statistics kernel's geometry (the greedy sweep's: measured
// against 12 x 8, 16 x 6 and 24 x 4 warps x stages, all slower)
constexpr int kCWarps = 24;
constexpr int kCThreads = 32 * kCWarps;
constexpr int kCStages = 3;  // 2 KB stages per warp
constexpr size_t kCSmem = (size_t)kCWarps * kCStages * kPieceBytes;

// Pieces in the order the statistics warps sweep them: every piece of the
// batch (all = 1), or only the pieces of masked positions, position list[m]
// for m = 0, 1, ... (all = 0), so that the warps' shares hold equal work.
struct CItem {
  int b, j, k, m;
};
__device__ __forceinline__ CItem citem_at(long long q, int all, const int* list, int Wn, int np) {
  CItem it;
  const long long r = q / np;
  it.k = (int)(q - r * np);
  const int pos = all ? (int)r : list[r];
  it.m = (int)r;
  it.b = pos / Wn;
  it.j = pos - it.b * Wn;
  return it;
}
__device__ __forceinline__ void citem_next(CItem& it, int all, const int* list, int M, int Wn, int np) {
  if (++it.k < np) return;
  it.k = 0;
  ++it.m;
  if (all) {
    if (++it.j == Wn) {
      it.j = 0;
      ++it.b;
    }
  } else if (it.m < M) {
    it.b = list[it.m] / Wn;
    it.j = list[it.m] - it.b * Wn;
  }
}
// the record slot of a piece: its index among all pieces of the batch
__device__ __forceinline__ long long citem_slot(const CItem& it, int Wn, int np) {
  return ((long long)it.b * Wn + it.j) * np + it.k;
}

__device__ __forceinline__ void cseg_begin(CSeg& s, const DenseParams& P, const CItem& it, long long w) {
  s.w0 = w;
  s.b = it.b;
  s.j = it.j;
  s.m = -INFINITY;
  s.c = -INFINITY;
  s.S = ff{0.f, 0.f};
  s.idx = INT_MAX;
  s.bad = 0;
  s.live = is_masked(P, it.b, it.j);
}
// every lane: the lanes are combined -- the maximum, the smallest first id
// among the lanes holding it, the sums moved exactly to the largest reference
// point and added, then expressed relative to the maximum (one exp2f) -- and
// lane 0 writes the record
__device__ __forceinline__ void cseg_write(const DenseParams& P, const CSeg& s, int lane) {
  if (!s.live) return;
  const int bad = __any_sync(0xffffffffu, s.bad);
  const float M = ord2f(__reduce_max_sync(0xffffffffu, f2ord(s.m)));
  const int idx = (int)__reduce_min_sync(0xffffffffu, (unsigned)((s.m == M && !bad) ? s.idx : INT_MAX));
  const float C = ord2f(__reduce_max_sync(0xffffffffu, f2ord(s.c)));
  ff S = warp_sum_ff(ff_mul_f(s.S, scale_exact(s.c, C)));
  if (M > -INFINITY && !bad) S = ff_mul_f(S, exp2f(C - M * kLog2e));
  if (lane == 0) {
    int4* q = reinterpret_cast<int4*>(reinterpret_cast<ConfRec*>(P.ws + P.L.upart) + s.w0);
    q[0] = make_int4(__float_as_int(M), __float_as_int(S.hi), __float_as_int(S.lo), idx);
    q[1] = make_int4(bad, 1, 0, 0);  // .y = 1 marks a record
  }
}
// This lane's elements of a piece folded into its segment statistics.  The
// lane's elements come in increasing id order (pieces in order; in a piece,
// vectors lane + 32 i, elements in order), so a strictly greater maximum takes
// over and ties keep the earlier id; the first id is searched only when the
// lane's maximum grows.  A NaN or +inf marks the lane bad.
__device__ __forceinline__ void cseg_add(CSeg& s, const CItem& it, const uint4 (&r)[4], int bf16,
                                         int pe, int lane) {
  if (s.bad) return;  // the segment is an error; nothing more to add
  float pm;
  if (bf16) {
    uint32_t mx = kNegInf2;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mx = bf16x2_max_nan(mx, bf16x2_max_nan(bf16x2_max_nan(r[i].x, r[i].y),
                                             bf16x2_max_nan(r[i].z, r[i].w)));
    pm = fmax_nan(bf16_lo(mx), bf16_hi(mx));
  } else {
    pm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      pm = fmax_nan(pm, fmax_nan(fmax_nan(__uint_as_float(r[i].x), __uint_as_float(r[i].y)),
                                 fmax_nan(__uint_as_float(r[i].z), __uint_as_float(r[i].w))));
  }
  if (pm != pm || pm == INFINITY) {
    s.bad = 1;
    return;
  }
  if (pm == -INFINITY) return;
  if (pm > s.m) {  // a new maximum for this lane: its first id, then the reference point
    int bi = INT_MAX;
#pragma unroll
    for (int i = 3; i >= 0; --i) {  // scanned backwards, so the last hit is the first id
      const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
      if (bf16) {
#pragma unroll
        for (int e = 7; e >= 0; --e)
          if (((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1])) == pm) bi = (lane + 32 * i) * 8 + e;
      } else {
#pragma unroll
        for (int e = 3; e >= 0; --e)
          if (__uint_as_float(w[e]) == pm) bi = (lane + 32 * i) * 4 + e;
      }
    }
    s.m = pm;
    s.idx = it.k * pe + bi;
    const float c = ref_point(pm);
    if (c > s.c) {
      s.S = ff_mul_f(s.S, scale_exact(s.c, c));
      s.c = c;
    }
  }
  const float cc = s.c;
  // four running sums as two packed pairs (one fma and one add per pair)
  const f32x2 L2 = f2_pack(kLog2e, kLog2e), nc = f2_pack(-cc, -cc);
  f32x2 a01 = f2_pack(0.f, 0.f), a23 = a01;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      a01 = f2_add(a01, f2_exp2_shift(f2_bf16(r[i].x), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift(f2_bf16(r[i].y), L2, nc));
      a01 = f2_add(a01, f2_exp2_shift(f2_bf16(r[i].z), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift(f2_bf16(r[i].w), L2, nc));
    } else {
      a01 = f2_add(a01, f2_exp2_shift(f2_pack(__uint_as_float(r[i].x), __uint_as_float(r[i].y)), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift(f2_pack(__uint_as_float(r[i].z), __uint_as_float(r[i].w)), L2, nc));
    }
  }
  float a0, a1, a2, a3;
  f2_unpack(a01, a0, a1);
  f2_unpack(a23, a2, a3);
  s.S = ff_add_f(s.S, __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3)));
}

__global__ void __launch_bounds__(kCThreads, 1) commit_stats_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_list[kCMaxList];
  __shared__ int s_wsum[kCWarps];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, Wn = G + 1, np = P.g.np, pe = P.g.pe, epv = P.bf16 ? 8 : 4;
  const int npos = P.B * Wn;
  // the masked positions in order (a block-wide compaction of the flags)
  const int all = npos > kCMaxList;
  int M = npos;
  if (!all) {
    const int C = (npos + kCThreads - 1) / kCThreads;
    const int p0 = min(npos, tid * C), p1 = min(npos, p0 + C);
    int cnt = 0;
    for (int p = p0; p < p1; ++p) cnt += (__ldg(P.x + p) != 0);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    M = 0;
    for (int w2 = 0; w2 < kCWarps; ++w2) {
      const int v = s_wsum[w2];
      if (w2 < warp) base += v;
      M += v;
    }
    int o = base + incl - cnt;
    for (int p = p0; p < p1; ++p)
      if (__ldg(P.x + p) != 0) s_list[o++] = p;
    __syncthreads();
  }
  const long long W = (long long)M * np;
  const long long nwt = (long long)gridDim.x * kCWarps;
  const long long gw = (long long)blockIdx.x * kCWarps + warp;
  const long long lo = gw * W / nwt, hi = (gw + 1) * W / nwt;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lo >= hi) return;
  const uint32_t ninf = P.bf16 ? kNegInf2 : kNegInfF;
  CSeg seg;
  CItem out = citem_at(lo, all, s_list, Wn, np);
  cseg_begin(seg, P, out, citem_slot(out, Wn, np));

  if (!P.aligned) {
    for (long long w = lo; w < hi; ++w, citem_next(out, all, s_list, M, Wn, np)) {
      if (out.b != seg.b || out.j != seg.j) {
        cseg_write(P, seg, lane);
        cseg_begin(seg, P, out, citem_slot(out, Wn, np));
      }
      if (!seg.live) continue;
      const int ne = min(pe, P.V - out.k * pe);
      uint4 r[4];
      load_vectors(target_row(P, out.b, out.j) + (size_t)out.k * kPieceBytes, ne, P.bf16, 0, lane, r);
      cseg_add(seg, out, r, P.bf16, pe, lane);
    }
    cseg_write(P, seg, lane);
    return;
  }

  unsigned char* ring = smem_raw + (size_t)warp * kCStages * kPieceBytes;
  CItem in = out;
  long long wi = lo;
  auto issue = [&](int s) {  // a full sweep does not read the unmasked positions' pieces
    if (all && !is_masked(P, in.b, in.j)) return;
    const int ne = min(pe, P.V - in.k * pe);
    const unsigned char* src = target_row(P, in.b, in.j) + (size_t)in.k * kPieceBytes;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = lane + 32 * i;
      if (vi * epv < ne) cp_async16(ring + s * kPieceBytes + 16 * vi, src + 16 * vi);
    }
  };
#pragma unroll
  for (int s = 0; s < kCStages - 1; ++s) {
    if (wi < hi) {
      issue(s);
      citem_next(in, all, s_list, M, Wn, np);
      ++wi;
    }
    cp_async_commit();
  }
  int slot = 0, islot = kCStages - 1;
  for (long long w = lo; w < hi; ++w) {
    if (out.b != seg.b || out.j != seg.j) {
      cseg_write(P, seg, lane);
      cseg_begin(seg, P, out, citem_slot(out, Wn, np));
    }
    if (wi < hi) {
      issue(islot);
      citem_next(in, all, s_list, M, Wn, np);
      ++wi;
    }
    cp_async_commit();
    cp_async_wait_group<kCStages - 1>();
    if (seg.live) {
      const unsigned char* stage = ring + slot * kPieceBytes;
      const int ne = min(pe, P.V - out.k * pe);
      uint4 r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int vi = lane + 32 * i;
        r[i] = (vi * epv < ne) ? *reinterpret_cast<const uint4*>(stage + 16 * vi)
                               : make_uint4(ninf, ninf, ninf, ninf);
      }
      cseg_add(seg, out, r, P.bf16, pe, lane);
    }
    citem_next(out, all, s_list, M, Wn, np);
    slot = (slot + 1 == kCStages) ? 0 : slot + 1;
    islot = (islot + 1 == kCStages) ? 0 : islot + 1;
  }
  cseg_write(P, seg, lane);
  cp_async_wait_group<0>();
}

__global__ void __launch_bounds__(32 * kGRowWarps) commit_row_kernel(const __grid_constant__ DenseParams P,
                                                                    float tau, int32_t* commit,
                                                                    float* confidence) {
  __shared__ float s_conf[kGMaxPos];
  __shared__ int s_tok[kGMaxPos];
  __shared__ int s_msk[kGMaxPos];  // the block's mask flags
  __shared__ int s_err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x, G = P.G, Wn = G + 1, np = P.g.np;
  if (threadIdx.x == 0) s_err = 0;
  // the mask flags first: an input, not a result of the statistics grid (this
  // grid starts once every statistics CTA has passed its own wait for the
  // grids before it; read from L2)
  for (int j = threadIdx.x; j < Wn; j += blockDim.x) s_msk[j] = __ldcg(P.x + (size_t)b * Wn + j) != 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  ConfRec* rec = reinterpret_cast<ConfRec*>(P.ws + P.L.upart);
  for (int j = warp; j < Wn; j += kGRowWarps) {
    const bool masked = s_msk[j] != 0;
    if (!masked) {  // no record was written for it
      if (lane == 0) {
        s_conf[j] = -1.f;
        s_tok[j] = -1;
      }
      continue;
    }
    // the position's records sit at the first piece of each segment that
    // covers it, marked; every other slot of its range is zero
    const long long P0 = ((long long)b * Wn + j) * np;
    float m = -INFINITY;
    ff S{0.f, 0.f};
    int idx = INT_MAX, bad = 0;
    // five slots per lane in flight at once: one round for the 148-149
    // pieces of a 128k-152k vocabulary
    for (int k0 = lane; k0 < np; k0 += kCSlots * 32) {
      int4 v0[kCSlots], v1[kCSlots];
#pragma unroll
      for (int u = 0; u < kCSlots; ++u) {
        v1[u] = make_int4(0, 0, 0, 0);
        if (k0 + 32 * u < np) {
          const int4* rp = reinterpret_cast<const int4*>(rec + P0 + k0 + 32 * u);
          v0[u] = __ldcg(rp);
          v1[u] = __ldcg(rp + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < kCSlots; ++u) {
        if (v1[u].y != 1) continue;
        int4* rp = reinterpret_cast<int4*>(rec + P0 + k0 + 32 * u);
        rp[0] = make_int4(0, 0, 0, 0);
        rp[1] = make_int4(0, 0, 0, 0);
        bad |= v1[u].x;
        const float rm = __int_as_float(v0[u].x);
        const ff rs{__int_as_float(v0[u].y), __int_as_float(v0[u].z)};
        if (rm == -INFINITY) continue;
        if (rm > m) {
          S = ff_add(ff_mul_f(S, (m == -INFINITY) ? 0.f : exp2f((m - rm) * kLog2e)), rs);
          m = rm;
          idx = v0[u].w;
        } else {
          S = ff_add(S, ff_mul_f(rs, exp2f((rm - m) * kLog2e)));
          if (rm == m && v0[u].w < idx) idx = v0[u].w;
        }
      }
    }
    // warp: rescale every lane's sum to the warp maximum, then add
    const float M = warp_max(m);
    S = warp_sum_ff(ff_mul_f(S, (m == -INFINITY) ? 0.f : exp2f((m - M) * kLog2e)));
    int ci = (m == M) ? idx : INT_MAX;
    ci = (int)__reduce_min_sync(0xffffffffu, (unsigned)ci);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const float Sf = ff_to_f(S);
      // S is at least the maximum's own term, ex2 of the rounding residual of
      // m log2e: 1 within a few units in the last place, so 1/S can exceed 1
      // by as much; the confidence is clamped to 1
      const int err = bad || !(M > -INFINITY) || !(Sf > 0.f) || !(Sf < INFINITY);
      if (err) atomicOr(&s_err, 1);
      s_conf[j] = err ? -1.f : fminf(__fdiv_rn(1.f, Sf), 1.f);
      s_tok[j] = ci;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int err = s_err;
    int32_t* cm = commit + (size_t)b * Wn;
    int32_t* tk = P.tok_out + (size_t)b * Wn;
    float* cf = confidence ? confidence + (size_t)b * Wn : nullptr;
    int any = 0, best = -1;
    float bc = -1.f;
    for (int j = 0; j < Wn; ++j) {
      const float c = s_conf[j];
      const bool masked = s_msk[j] != 0;
      const int on = !err && masked && c > tau;
      cm[j] = err ? -1 : on;
      tk[j] = on ? s_tok[j] : -1;
      if (cf) cf[j] = (err || !masked) ? __int_as_float(0x7fc00000) : c;
      any |= on;
      if (masked && c > bc) {
        bc = c;
        best = j;
      }
    }
    if (!err && !any && best >= 0) {  // progress: the most confident position
      cm[best] = 1;
      tk[best] = s_tok[best];
    }
    if (err) atomicOr(&reinterpret_cast<WsHeader*>(P.ws)->status, kStatusInputErr);
  }
}

}  // namespace

cudaError_t launch_commit(const DenseParams& p, float tau, int32_t* commit, float* confidence,
                          cudaStream_t s) {
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(commit_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCSmem);
    if (e != cudaSuccess) return e;
    sms[dev] = n;
  }
  const long long pieces = (long long)p.B * (p.G + 1) * p.g.np;
  long long grid = sms[dev];
  if (grid * kCWarps > pieces) grid = (pieces + kCWarps - 1) / kCWarps;
  DenseParams q = p;
  q.stats_warps = grid * kCWarps;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t k1 = {};
  k1.gridDim = dim3((unsigned)grid, 1, 1);
  k1.blockDim = dim3(kCThreads, 1, 1);
  k1.dynamicSmemBytes = kCSmem;
  k1.stream = s;
  k1.attrs = attr;
  k1.numAttrs = 1;
  e = cudaLaunchKernelEx(&k1, commit_stats_kernel, q);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t k2 = {};
  k2.gridDim = dim3((unsigned)p.B, 1, 1);
  k2.blockDim = dim3(32 * kGRowWarps, 1, 1);
  k2.stream = s;
  k2.attrs = attr;
  k2.numAttrs = 1;
  return cudaLaunchKernelEx(&k2, commit_row_kernel, q, tau, commit, confidence);
}

cudaError_t launch_greedy(const DenseParams& p, cudaStream_t s) {
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {  // once per device: SM count and the ring's shared memory
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(greedy_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGSmem);
    if (e != cudaSuccess) return e;
    sms[dev] = n;
  }
  const long long pieces = (long long)p.B * (p.G + 1) * p.g.np;
  long long grid = sms[dev];
  if (grid * kGWarps > pieces) grid = (pieces + kGWarps - 1) / kGWarps;
  DenseParams q = p;
  q.stats_warps = grid * kGWarps;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t k1 = {};
  k1.gridDim = dim3((unsigned)grid, 1, 1);
  k1.blockDim = dim3(kGThreads, 1, 1);
  k1.dynamicSmemBytes = kGSmem;
  k1.stream = s;
  k1.attrs = attr;
  k1.numAttrs = 1;
  e = cudaLaunchKernelEx(&k1, greedy_stats_kernel, q);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t k2 = {};
  k2.gridDim = dim3((unsigned)p.B, 1, 1);
  k2.blockDim = dim3(32 * kGRowWarps, 1, 1);
  k2.stream = s;
  k2.attrs = attr;
  k2.numAttrs = 1;
  return cudaLaunchKernelEx(&k2, greedy_row_kernel, q);
}

}  // namespace sv
