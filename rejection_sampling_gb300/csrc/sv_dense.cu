// sv_dense.cu -- dense verification for large vocabularies: two streaming
// kernels, one HBM pass over every logit plus one pass over the two rows of
// each row's stop position.
//
// Computes, for every row b (DFlash/DFlash2 guide, 4.4; Uno article, "What
// 'lossless' actually has to mean"):
//   p_j = softmax(target[b, j]), q_j = softmax(draft[b, j]) for all positions,
//   a_j = min(1, p_j(x_j) / q_j(x_j))  (0 where q_j(x_j) = 0),
//   n   = first j with u_accept[b, j] >= a_j (gamma if none),
//   token n = inverse CDF of max(p_n - q_n, 0) (n < gamma) or of p_gamma
//   (bonus, DFlash/DFlash2 guide section 2) at u_sample[b].
//
// Design.
//  * A logit row is cut into 2 KB pieces; a CTA of 16 warps takes 16
//    consecutive pieces (a 32 KB chunk), one warp per piece.
//  * dense_stats_kernel: one CTA per (row b, position j, chunk c), launched
//    row by row.  Each warp loads its target piece and the same draft piece
//    straight into registers (16-byte loads, all in flight together), reduces
//    each to (c, S) -- c = log2e * max (max.bf16x2), S = sum 2^(v log2e - c)
//    (ex2.approx) -- and the warp holding the draft token x_j picks up the two
//    logits there.  Warp 0 combines the 16 pieces in float-float and writes
//    the chunk's partial.  The CTA that completes a row (a per-row arrival
//    counter) finalises it: combines every position's partials, forms the
//    ratios, runs the accept tests, finds n and writes the stop record, the
//    accept probabilities and every token but the one drawn at n.  Rows
//    complete in launch order, so all but the last rows' finalisations
//    overlap the stream of later rows.
//  * dense_resid_kernel: one CTA per (row b, chunk c) recomputes
//    r(y) = max(p_n(y) - q_n(y), 0) (or p_gamma) over its chunk of the stop
//    position's two rows and writes one mass per piece.  The CTA completing
//    the row draws the token: a float-float prefix over the piece masses picks
//    the piece, then a prefix over the piece's fp32 values picks y.
//  * No thread ever waits for another CTA: hand-offs are last-arriver
//    counters, which the finishing CTA resets, and every array a call reads is
//    written earlier in the same call.  The workspace is all zero again after
//    every call.
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kWarps = kChunkPieces;  // warps per CTA, one piece each
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxG = 256;            // positions per row (gamma + 1 <= 256)

// ---------------------------------------------------------------------------
// workspace accessors
// ---------------------------------------------------------------------------
__device__ __forceinline__ WsHeader* hdr_of(const DenseParams& P) {
  return reinterpret_cast<WsHeader*>(P.ws);
}
template <class T>
__device__ __forceinline__ T* ws_at(const DenseParams& P, size_t off) {
  return reinterpret_cast<T*>(P.ws + off);
}
// 32-byte records written by other CTAs: read around L1
template <class T>
__device__ __forceinline__ T ldcg32(const T* p) {
  static_assert(sizeof(T) == 32, "32-byte record");
  const int4* q = reinterpret_cast<const int4*>(p);
  int4 a = __ldcg(q), b = __ldcg(q + 1);
  T out;
  int4* o = reinterpret_cast<int4*>(&out);
  o[0] = a;
  o[1] = b;
  return out;
}
template <class T>
__device__ __forceinline__ void zero32(T* p) {
  static_assert(sizeof(T) == 32, "32-byte record");
  int4* q = reinterpret_cast<int4*>(p);
  q[0] = make_int4(0, 0, 0, 0);
  q[1] = make_int4(0, 0, 0, 0);
}

__device__ __forceinline__ const unsigned char* target_row(const DenseParams& P, int b, int j) {
  return P.lt + ((size_t)b * (P.G + 1) + j) * (size_t)P.V * P.g.es;
}
__device__ __forceinline__ const unsigned char* draft_row(const DenseParams& P, int b, int j) {
  return P.ld + ((size_t)b * P.G + j) * (size_t)P.V * P.g.es;
}
__device__ __forceinline__ float load_logit(const unsigned char* row, int y, int bf16) {
  if (bf16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[y]);
  return reinterpret_cast<const float*>(row)[y];
}

// fp32 scale 2^(c - C) for combining partial sums (0 for an all -inf part)
__device__ __forceinline__ float part_scale(float c, float C) {
  return (c == -INFINITY) ? 0.f : exp2f(c - C);
}

// r(y) from fp32 logits; identical operations wherever it is evaluated so the
// masses and the final walk see bit-identical values.
__device__ __forceinline__ float resid_val(float t, float d, float ct, float cd, float invSt,
                                           float invSd, int mode) {
  const float p = __fmul_rn(ex2(__fmaf_rn(t, kLog2e, -ct)), invSt);
  if (mode != 0) return p;
  const float q = __fmul_rn(ex2(__fmaf_rn(d, kLog2e, -cd)), invSd);
  const float r = __fsub_rn(p, q);
  return r > 0.f ? r : 0.f;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// streaming 16-byte load: no L1 allocation (every byte is read once here)
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

constexpr uint32_t kNegInf2 = 0xFF80FF80u;  // two bf16 -inf
constexpr uint32_t kNegInfF = 0xFF800000u;  // fp32 -inf

// ---------------------------------------------------------------------------
// one 2 KB piece per warp: lane holds 16-byte vectors lane + 32 i, i < 4
// (8 bf16 or 4 fp32 elements each); elements past `ne` read as -inf
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_piece(const unsigned char* base, int ne, int bf16,
                                           int aligned, int lane, uint4 (&r)[4]) {
  const int epv = bf16 ? 8 : 4;
  const uint32_t ninf = bf16 ? kNegInf2 : kNegInfF;
  if (aligned) {  // row bytes are a multiple of 16: every vector is whole
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = lane + 32 * i;
      r[i] = (vi * epv < ne) ? ld_stream(base + 16 * (size_t)vi) : make_uint4(ninf, ninf, ninf, ninf);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
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

// (c, S) of a piece: c = log2e * max, S = sum 2^(v log2e - c); an all -inf
// piece gives c = -inf, S = 0 (its exponentials use c = 0, so a NaN still
// poisons S)
__device__ __forceinline__ void piece_stats(const uint4 (&r)[4], int bf16, float& c_out,
                                            float& s_out) {
  float m;
  if (bf16) {
    uint32_t mx = kNegInf2;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(r[i].x, r[i].y), bf16x2_max(r[i].z, r[i].w)));
    m = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(r[i].x), __uint_as_float(r[i].y)),
                         fmaxf(__uint_as_float(r[i].z), __uint_as_float(r[i].w))));
  }
  m = warp_max(m);
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (bf16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a0 += ex2(fmaf(bf16_lo(r[i].x), kLog2e, -c));
      a1 += ex2(fmaf(bf16_hi(r[i].x), kLog2e, -c));
      a2 += ex2(fmaf(bf16_lo(r[i].y), kLog2e, -c));
      a3 += ex2(fmaf(bf16_hi(r[i].y), kLog2e, -c));
      a0 += ex2(fmaf(bf16_lo(r[i].z), kLog2e, -c));
      a1 += ex2(fmaf(bf16_hi(r[i].z), kLog2e, -c));
      a2 += ex2(fmaf(bf16_lo(r[i].w), kLog2e, -c));
      a3 += ex2(fmaf(bf16_hi(r[i].w), kLog2e, -c));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a0 += ex2(fmaf(__uint_as_float(r[i].x), kLog2e, -c));
      a1 += ex2(fmaf(__uint_as_float(r[i].y), kLog2e, -c));
      a2 += ex2(fmaf(__uint_as_float(r[i].z), kLog2e, -c));
      a3 += ex2(fmaf(__uint_as_float(r[i].w), kLog2e, -c));
    }
  }
  s_out = warp_sum((a0 + a1) + (a2 + a3));
  c_out = (m == -INFINITY) ? -INFINITY : c;
}

// fp32 bits of element xl (0 <= xl < ne) of the piece, on every lane
__device__ __forceinline__ uint32_t piece_element(const uint4 (&r)[4], int xl, int bf16, int lane) {
  const int vx = bf16 ? (xl >> 3) : (xl >> 2);
  const int owner = vx & 31, iv = vx >> 5, e = bf16 ? (xl & 7) : (xl & 3);
  uint32_t out = 0;
  if (lane == owner) {
    uint4 vv = r[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
      if (i == iv) vv = r[i];
    const int wi = bf16 ? (e >> 1) : e;
    const uint32_t w = wi == 0 ? vv.x : wi == 1 ? vv.y : wi == 2 ? vv.z : vv.w;
    out = bf16 ? ((e & 1) ? (w & 0xFFFF0000u) : (w << 16)) : w;
  }
  return __shfl_sync(0xffffffffu, out, owner);
}

// residual (or p) mass of a piece held in registers
__device__ __forceinline__ float piece_resid(const uint4 (&t)[4], const uint4 (&d)[4], int bf16,
                                             const StopInfo& st) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t tw[4] = {t[i].x, t[i].y, t[i].z, t[i].w};
    const uint32_t dw[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
    if (bf16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float tv = (e & 1) ? bf16_hi(tw[e >> 1]) : bf16_lo(tw[e >> 1]);
        const float dv = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
        acc += resid_val(tv, dv, st.ct, st.cd, st.invSt, st.invSd, st.mode);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc += resid_val(__uint_as_float(tw[e]), __uint_as_float(dw[e]), st.ct, st.cd, st.invSt,
                         st.invSd, st.mode);
    }
  }
  return warp_sum(acc);
}

__device__ __forceinline__ void combine_part(const UnitPart& u, float& Ct, ff& St, float& Cd,
                                             ff& Sd) {
  const ff ut{u.St_hi, u.St_lo}, ud{u.Sd_hi, u.Sd_lo};
  if (u.ct > Ct) {
    St = ff_add(ff_mul_f(St, part_scale(Ct, u.ct)), ut);
    Ct = u.ct;
  } else {
    St = ff_add(St, ff_mul_f(ut, part_scale(u.ct, Ct)));
  }
  if (u.cd > Cd) {
    Sd = ff_add(ff_mul_f(Sd, part_scale(Cd, u.cd)), ud);
    Cd = u.cd;
  } else {
    Sd = ff_add(Sd, ff_mul_f(ud, part_scale(u.cd, Cd)));
  }
}

// warp-wide combination of per-lane (C, S) pairs
__device__ __forceinline__ void warp_combine(float& C, ff& S) {
  const float Cw = warp_max(C);
  S = warp_sum_ff(ff_mul_f(S, part_scale(C, Cw)));
  C = Cw;
}

struct FinShared {
  float c[4][kMaxG];  // per position: Ct, St, Cd, Sd (the stop position's constants)
  int n;              // first rejected position (G + 1: none)
  int err;
};

// Row b's decisions, by the CTA that completed its statistics (all warps).
// Warp w combines the chunk partials of positions w, w + 16, ...; then the
// first rejection n, the stop record and the outputs other than token n.
__device__ void finalize_row(const DenseParams& P, int b, int warp, int lane, FinShared& F) {
  const int G = P.G, nc = P.g.nc;
  UnitPart* up_row = ws_at<UnitPart>(P, P.L.upart) + (size_t)b * (G + 1) * nc;
  if (threadIdx.x == 0) {
    F.n = G + 1;
    F.err = 0;
  }
  __syncthreads();
  for (int j = warp; j <= G; j += kWarps) {
    float Ct = -INFINITY, Cd = -INFINITY;
    ff St{0.f, 0.f}, Sd{0.f, 0.f};
    uint32_t txb = kNoTokenBits, dxb = kNoTokenBits;
    for (int k = lane; k < nc; k += 32) {
      UnitPart* q = up_row + (size_t)j * nc + k;
      const UnitPart u = ldcg32(q);
      zero32(q);  // consumed: leave the workspace zero
      combine_part(u, Ct, St, Cd, Sd);
      if (__float_as_uint(u.tx) != kNoTokenBits) {
        txb = __float_as_uint(u.tx);
        dxb = __float_as_uint(u.dx);
      }
    }
    warp_combine(Ct, St);
    warp_combine(Cd, Sd);
    const unsigned hx = __ballot_sync(0xffffffffu, txb != kNoTokenBits);
    if (hx) {
      txb = __shfl_sync(0xffffffffu, txb, __ffs(hx) - 1);
      dxb = __shfl_sync(0xffffffffu, dxb, __ffs(hx) - 1);
    }
    const float Stf = ff_to_f(St), Sdf = ff_to_f(Sd);
    int err = !(Ct > -INFINITY && Ct < INFINITY && Stf > 0.f && Stf < INFINITY);
    if (j < G) {
      err |= !(Cd > -INFINITY && Cd < INFINITY && Sdf > 0.f && Sdf < INFINITY);
      err |= !hx;  // no chunk held x_j: the draft id is out of range
    }
    int acc = 1;
    float a = 0.f;
    if (j < G && !err) {
      // p/q = 2^((tx L - Ct) - (dx L - Cd)) * (Sd / St); the exponent is formed
      // exactly (two-product) and rounded once
      const float tx = __uint_as_float(txb), dx = __uint_as_float(dxb);
      float ratio = 0.f;
      if (tx > -INFINITY && dx > -INFINITY) {
        const ff ea = ff_add_f(two_prod(tx, kLog2e), -Ct);
        const ff ed = ff_add_f(two_prod(dx, kLog2e), -Cd);
        ratio = exp2f(ff_to_f(ff_sub(ea, ed))) * __fdiv_rn(Sdf, Stf);
      }
      a = fminf(ratio, 1.f);
      acc = P.u_acc[(size_t)b * G + j] < a;
    }
    if (lane == 0) {
      if (j < G && P.acc_out) P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : a;
      F.c[0][j] = Ct;
      F.c[1][j] = Stf;
      F.c[2][j] = Cd;
      F.c[3][j] = Sdf;
      if (err) atomicOr(&F.err, 1);
      if (!acc) atomicMin(&F.n, j);
    }
  }
  __syncthreads();
  const int err = F.err;
  const int n = min(F.n, G);
  if (threadIdx.x == 0) {
    StopInfo st;
    st.n = n;
    st.T = 0.0;
    if (err) {
      st.mode = 2;
      st.ct = st.cd = st.invSt = st.invSd = 0.f;
      atomicOr(&hdr_of(P)->status, kStatusInputErr);
    } else if (n < G) {
      st.mode = 0;
      st.ct = F.c[0][n];
      st.cd = F.c[2][n];
      st.invSt = __fdiv_rn(1.f, F.c[1][n]);
      st.invSd = __fdiv_rn(1.f, F.c[3][n]);
    } else {
      st.mode = 1;
      st.ct = F.c[0][n];
      st.cd = 0.f;
      st.invSt = __fdiv_rn(1.f, F.c[1][n]);
      st.invSd = 0.f;
    }
    ws_at<StopInfo>(P, P.L.stop)[b] = st;
    ws_at<uint32_t>(P, P.L.cnt_row)[b] = 0;
    P.n_out[b] = err ? -1 : n;
  }
  // tokens: x_0..x_{n-1}, then (token n from the residual kernel), then -1
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  for (int j = threadIdx.x; j <= G; j += kThreads) {
    if (err)
      tok[j] = -1;
    else if (j < n)
      tok[j] = P.x[(size_t)b * G + j];
    else if (j > n)
      tok[j] = -1;
  }
}

// ---------------------------------------------------------------------------
// kernel 1: statistics of one 32 KB chunk of (row b, position j), target and
// draft; the CTA completing a row finalises it
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) dense_stats_kernel(const __grid_constant__ DenseParams P) {
  __shared__ float s_c[2][kWarps], s_s[2][kWarps];
  __shared__ uint32_t s_x[2];
  __shared__ int s_last;
  __shared__ FinShared F;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = P.G, nc = P.g.nc, pe = P.g.pe;
  const long long t = blockIdx.x;
  const long long r = t / nc;
  const int c = (int)(t - r * nc);
  const int b = (int)(r / (G + 1));
  const int j = (int)(r - (long long)b * (G + 1));
  const bool has_d = j < G;
  const int k = c * kWarps + warp;  // this warp's piece
  const int ne = (k < P.g.np) ? min(pe, P.V - k * pe) : 0;
  const int x = has_d ? __ldg(P.x + (size_t)b * G + j) : -1;
  if (threadIdx.x < 2) s_x[threadIdx.x] = kNoTokenBits;

  uint4 rt[4], rd[4];
  const size_t off = (size_t)k * kPieceBytes;
  load_piece(target_row(P, b, j) + off, ne, P.bf16, P.aligned, lane, rt);
  if (has_d) {
    load_piece(draft_row(P, b, j) + off, ne, P.bf16, P.aligned, lane, rd);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) rd[i] = make_uint4(0, 0, 0, 0);
  }
  float ct, st, cd = -INFINITY, sd = 0.f;
  piece_stats(rt, P.bf16, ct, st);
  if (has_d) piece_stats(rd, P.bf16, cd, sd);
  // the logits at the draft token, if this piece holds it
  const int xl = x - k * pe;
  if (has_d && xl >= 0 && xl < ne) {
    const uint32_t tb = piece_element(rt, xl, P.bf16, lane);
    const uint32_t db = piece_element(rd, xl, P.bf16, lane);
    if (lane == 0) {
      s_x[0] = tb;
      s_x[1] = db;
    }
  }
  if (lane == 0) {
    s_c[0][warp] = ct;
    s_s[0][warp] = st;
    s_c[1][warp] = cd;
    s_s[1][warp] = sd;
  }
  __syncthreads();
  if (warp == 0) {
    const bool on = lane < kWarps;
    float Ct = on ? s_c[0][lane] : -INFINITY, Cd = on ? s_c[1][lane] : -INFINITY;
    ff St{on ? s_s[0][lane] : 0.f, 0.f}, Sd{on ? s_s[1][lane] : 0.f, 0.f};
    warp_combine(Ct, St);
    warp_combine(Cd, Sd);
    if (lane == 0) {
      UnitPart u;
      u.St_hi = St.hi;
      u.St_lo = St.lo;
      u.Sd_hi = Sd.hi;
      u.Sd_lo = Sd.lo;
      u.ct = Ct;
      u.cd = Cd;
      u.tx = __uint_as_float(s_x[0]);
      u.dx = __uint_as_float(s_x[1]);
      ws_at<UnitPart>(P, P.L.upart)[((size_t)b * (G + 1) + j) * nc + c] = u;
      __threadfence();
      const unsigned old = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_row) + b, 1u);
      s_last = (old == (unsigned)((G + 1) * nc) - 1);
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // every chunk's partial is visible before it is read
  finalize_row(P, b, warp, lane, F);
}

// ---------------------------------------------------------------------------
// token draw of row b from its per-piece masses (one warp): a float-float
// prefix over the pieces picks the piece, a float-float prefix over its fp32
// element values picks the token.  Masses, then the piece's two slices, are
// staged in the shared scratch with cp.async.
// ---------------------------------------------------------------------------
template <int BF16>
__device__ __forceinline__ float piece_val(const float* tsm, const float* dsm, int e,
                                           const StopInfo& st) {
  float t, d;
  if (BF16) {
    t = bf16_to_f32(reinterpret_cast<const uint16_t*>(tsm)[e]);
    d = bf16_to_f32(reinterpret_cast<const uint16_t*>(dsm)[e]);
  } else {
    t = tsm[e];
    d = dsm[e];
  }
  return resid_val(t, d, st.ct, st.cd, st.invSt, st.invSd, st.mode);
}

constexpr int kScrFloats = 1024;  // 4 KB: the masses, or one piece's two slices

template <int BF16>
__device__ void final_select(const DenseParams& P, int b, int lane, float* scr) {
  const int G = P.G, V = P.V, np = P.g.np, pe = P.g.pe;
  float* rm = ws_at<float>(P, P.L.rmass) + (size_t)b * P.g.np4;
  const bool staged = np <= kScrFloats;
  // the mass copies and the stop-record load are in flight together
  if (staged)
    for (int k = lane * 4; k < np; k += 128) cp_async16(scr + k, rm + k);
  StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
  const float us = P.u_s[b];
  const int n = st.n;
  ff T{0.f, 0.f};
  cp_async_wait_all();
  __syncwarp();
  if (st.mode != 2) {
    const unsigned char* trow = target_row(P, b, n);
    const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, n) : nullptr;
    const float* mv = staged ? scr : rm;
    const int per = (np + 31) / 32;
    const int k0 = min(np, lane * per), k1 = min(np, k0 + per);
    ff ls{0.f, 0.f};
    for (int k = k0; k < k1; ++k) ls = ff_add_f(ls, staged ? mv[k] : __ldcg(mv + k));
    ff ex = warp_exclusive_scan_ff(ls, lane);
    T = ff_shfl(ff_add(ex, ls), 31);
    if (!(T.hi > 0.f) && st.mode == 0) {
      // zero residual after a rejection (only through rounding): draw from p_n
      st.mode = 1;
      drow = nullptr;
      for (int k = 0; k < np; ++k) {
        const int y0 = k * pe, ne = min(pe, V - y0);
        float sum = 0.f;
        for (int e = lane; e < ne; e += 32)
          sum += resid_val(load_logit(trow, y0 + e, BF16), 0.f, st.ct, st.cd, st.invSt, st.invSd, 1);
        sum = warp_sum(sum);
        if (lane == 0) {
          if (staged)
            scr[k] = sum;
          else
            rm[k] = sum;
        }
      }
      __threadfence();
      __syncwarp();
      ls = ff{0.f, 0.f};
      for (int k = k0; k < k1; ++k) ls = ff_add_f(ls, staged ? scr[k] : __ldcg(rm + k));
      ex = warp_exclusive_scan_ff(ls, lane);
      T = ff_shfl(ff_add(ex, ls), 31);
    }
    const ff target = ff_mul_f(T, us);
    // piece level
    const unsigned hit = __ballot_sync(0xffffffffu, (k1 > k0) && ff_gt(ff_add(ex, ls), target));
    int kstar = -1;
    ff base{0.f, 0.f};
    bool clamp = false;
    if (hit) {
      const int fl = __ffs(hit) - 1;
      if (lane == fl) {
        ff acc = ex;
        ff prev = ex;
        for (int k = k0; k < k1; ++k) {
          prev = acc;
          acc = ff_add_f(acc, staged ? scr[k] : __ldcg(rm + k));
          if (ff_gt(acc, target)) {
            kstar = k;
            base = prev;
            break;
          }
        }
        if (kstar < 0) {  // rounding between the two sums: last piece of the lane
          kstar = k1 - 1;
          base = prev;
        }
      }
      kstar = __shfl_sync(0xffffffffu, kstar, fl);
      base = ff_shfl(base, fl);
    } else {
      clamp = true;  // u*T at or past the total: last piece with mass
      int last = -1;
      for (int k = k0; k < k1; ++k)
        if ((staged ? scr[k] : __ldcg(rm + k)) > 0.f) last = k;
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      kstar = last < 0 ? 0 : last;
    }
    __syncwarp();
    // element level within piece kstar: stage its target and draft slices
    const int y0 = kstar * pe, ne = min(pe, V - y0);
    const float* tsm = scr;
    const float* dsm = scr + 512;  // 2 KB in
    if (P.aligned) {
      const int nchunk = (ne * (BF16 ? 2 : 4)) / 16;  // whole 16-byte chunks (rows are aligned)
      const unsigned char* ts = trow + (size_t)y0 * (BF16 ? 2 : 4);
      const unsigned char* ds = drow ? drow + (size_t)y0 * (BF16 ? 2 : 4) : nullptr;
      for (int c = lane; c < nchunk; c += 32) {
        cp_async16(reinterpret_cast<unsigned char*>(scr) + 16 * c, ts + 16 * c);
        if (ds) cp_async16(reinterpret_cast<unsigned char*>(scr + 512) + 16 * c, ds + 16 * c);
      }
      cp_async_wait_all();
    } else {
      for (int e = lane; e < ne; e += 32) {
        if (BF16) {
          reinterpret_cast<uint16_t*>(scr)[e] = reinterpret_cast<const uint16_t*>(trow)[y0 + e];
          if (drow) reinterpret_cast<uint16_t*>(scr + 512)[e] = reinterpret_cast<const uint16_t*>(drow)[y0 + e];
        } else {
          scr[e] = reinterpret_cast<const float*>(trow)[y0 + e];
          if (drow) scr[512 + e] = reinterpret_cast<const float*>(drow)[y0 + e];
        }
      }
    }
    if (!drow) {  // bonus / fallback: the draft slice is unused; keep it finite
      for (int e = lane; e < 512; e += 32) scr[512 + e] = 0.f;
    }
    __syncwarp();
    const int q = (ne + 31) / 32;
    const int e0 = min(ne, lane * q), e1 = min(ne, e0 + q);
    ff es{0.f, 0.f};
    int lastpos = -1;
    for (int e = e0; e < e1; ++e) {
      const float rv = piece_val<BF16>(tsm, dsm, e, st);
      es = ff_add_f(es, rv);
      if (rv > 0.f) lastpos = e;
    }
    const ff eex = warp_exclusive_scan_ff(es, lane);
    const ff tl = ff_sub(target, base);
    const unsigned ehit =
        clamp ? 0u : __ballot_sync(0xffffffffu, (e1 > e0) && ff_gt(ff_add(eex, es), tl));
    int y;
    if (ehit) {
      const int fl = __ffs(ehit) - 1;
      int yy = -1;
      if (lane == fl) {
        ff acc = ff_add(base, eex);
        for (int e = e0; e < e1; ++e) {
          acc = ff_add_f(acc, piece_val<BF16>(tsm, dsm, e, st));
          if (ff_gt(acc, target)) {
            yy = e;
            break;
          }
        }
        if (yy < 0) yy = lastpos >= 0 ? lastpos : e1 - 1;
      }
      y = y0 + __shfl_sync(0xffffffffu, yy, fl);
    } else {
      int lp = lastpos;
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      y = y0 + (lp < 0 ? 0 : lp);
    }
    if (lane == 0) P.tok_out[(size_t)b * (G + 1) + n] = y;
  }
  // the masses are consumed: leave the workspace zero
  for (int k = lane; k < np; k += 32) rm[k] = 0.f;
  if (lane == 0) {
    StopInfo* sp = ws_at<StopInfo>(P, P.L.stop) + b;
    if (P.keep_stop) {  // read (and cleared) by the residual-output kernel
      sp->mode = st.mode;
      sp->T = (double)T.hi + (double)T.lo;
    } else {
      zero32(sp);
    }
    ws_at<uint32_t>(P, P.L.cnt_res)[b] = 0;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// kernel 2: residual (or p) masses of one 32 KB chunk of the stop position's
// rows, one per piece; the CTA completing a row draws its token
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) dense_resid_kernel(const __grid_constant__ DenseParams P) {
  __shared__ __align__(16) float scr[kScrFloats];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = P.g.nc, pe = P.g.pe;
  const int b = (int)(blockIdx.x / nc);
  const int c = (int)(blockIdx.x - (long long)b * nc);
  const int k = c * kWarps + warp;
  const StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
  if (k < P.g.np) {
    float mass = 0.f;
    if (st.mode != 2) {
      const int ne = min(pe, P.V - k * pe);
      const size_t off = (size_t)k * kPieceBytes;
      uint4 rt[4], rd[4];
      load_piece(target_row(P, b, st.n) + off, ne, P.bf16, P.aligned, lane, rt);
      if (st.mode == 0) {
        load_piece(draft_row(P, b, st.n) + off, ne, P.bf16, P.aligned, lane, rd);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) rd[i] = rt[i];  // unused by mode 1
      }
      mass = piece_resid(rt, rd, P.bf16, st);
    }
    if (lane == 0) ws_at<float>(P, P.L.rmass)[(size_t)b * P.g.np4 + k] = mass;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_res) + b, 1u);
    s_last = (old == (unsigned)nc - 1);
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();  // every chunk's masses are visible before they are read
  if (P.bf16)
    final_select<1>(P, b, lane, scr);
  else
    final_select<0>(P, b, lane, scr);
}

// residual_out: the distribution the emitted token was drawn from.  One CTA
// per row; it clears the row's stop record once every thread has read it.
__global__ void dense_resid_out_kernel(const __grid_constant__ DenseParams P, float* out) {
  const int b = blockIdx.x;
  StopInfo* sp = ws_at<StopInfo>(P, P.L.stop) + b;
  const StopInfo st = ldcg32(sp);
  __syncthreads();
  if (threadIdx.x == 0) zero32(sp);
  float* o = out + (size_t)b * P.V;
  if (st.mode == 2 || !(st.T > 0.0)) {
    for (int y = threadIdx.x; y < P.V; y += blockDim.x) o[y] = 0.f;
    return;
  }
  const unsigned char* trow = target_row(P, b, st.n);
  const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, st.n) : nullptr;
  const float invT = __fdiv_rn(1.f, (float)st.T);
  for (int y = threadIdx.x; y < P.V; y += blockDim.x) {
    const float t = load_logit(trow, y, P.bf16);
    const float d = drow ? load_logit(drow, y, P.bf16) : 0.f;
    o[y] = resid_val(t, d, st.ct, st.cd, st.invSt, st.invSd, st.mode) * invT;
  }
}

}  // namespace

cudaError_t launch_dense(const DenseParams& p, cudaStream_t s) {
  const long long g1 = (long long)p.B * (p.G + 1) * p.g.nc;
  const long long g2 = (long long)p.B * p.g.nc;
  dense_stats_kernel<<<(unsigned)g1, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dense_resid_kernel<<<(unsigned)g2, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s) {
  dense_resid_out_kernel<<<p.B, 512, 0, s>>>(p, resid_out);
  return cudaGetLastError();
}

}  // namespace sv
