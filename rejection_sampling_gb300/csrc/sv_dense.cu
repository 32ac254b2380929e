// sv_dense.cu -- dense verification for large vocabularies.
//
// Computes, for every row b (DFlash/DFlash2 guide, 4.4; Uno article, "What
// 'lossless' actually has to mean"):
//   p_j = softmax(target[b, j]), q_j = softmax(draft[b, j]) for all positions,
//   a_j = min(1, p_j(x_j) / q_j(x_j))  (0 where q_j(x_j) = 0),
//   n   = first j with u_accept[b, j] >= a_j (gamma if none),
//   token n = inverse CDF of max(p_n - q_n, 0) (n < gamma) or of p_gamma
//   (bonus, DFlash/DFlash2 guide section 2) at u_sample[b].
//
// Design (two kernels per call, one HBM pass over every logit plus a second
// read of each row's stop position).
//  * A logit row is cut into 2 KB pieces; piece (b, j, k) pairs target piece
//    k of row-position (b, j) with the same draft piece.
//  * dense_stats_kernel: a persistent grid, one CTA of 24 warps per SM.
//    Every warp takes one contiguous range of pieces (in (b, j, k) order) and
//    streams it through a private two-stage ring of 4 KB shared-memory stages
//    filled by 16-byte cp.async.  Per piece it forms c = log2e * max
//    (max.bf16x2) and S = sum 2^(v log2e - c) (ex2.approx) for the target and
//    the draft piece and folds them into the running statistics of the
//    (b, j) segment it is in; the piece holding the draft token also gives
//    the two logits there.  Each segment of a range ends in one 32-byte record
//    at the segment's first piece; when the range leaves a row (or ends) the
//    warp adds its pieces of that row to the row's count (release).
//  * dense_row_kernel: one thread-block cluster of C CTAs per row, launched
//    as a programmatic dependent of the statistics kernel.  A CTA starts on
//    its row once the row's count is complete (acquire; a row's pieces come
//    from a few statistics CTAs, so most rows are decided while the grid
//    still streams others).  Every CTA finds
//    the row's records from the statistics warps' ranges, combines them per
//    position (float-float), forms p/q at the draft token, runs the accept
//    tests and takes the first rejection n and the draw constants.  Each CTA
//    then computes the residual (or p) mass of its share of the stop
//    position's pieces, with 32 run sums per piece, into the rank-0 CTA's
//    shared memory (st.shared::cluster).  After a cluster barrier one warp of
//    rank 0 draws the token -- float-float prefixes over the piece masses and
//    the chosen piece's run sums, then an fp32 prefix over the chosen run's
//    elements -- while the other CTAs clear the row's records.
//  * The statistics kernel is itself a programmatic dependent of whatever
//    precedes it and waits before it reads anything, so back-to-back calls do
//    not pay its launch latency.  The workspace is all zero again after every
//    call.
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kWarps = 16;  // warps per row-kernel CTA
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
// (the statistics records carry integer reference points, so this is an
// exact power of two formed on the integer pipe)
__device__ __forceinline__ float part_scale(float c, float C) { return scale_exact(c, C); }

// r(y) from fp32 logits; identical operations wherever it is evaluated so the
// masses and the final walk see bit-identical values.
__device__ __forceinline__ float resid_val(float t, float d, float ct, float cd, float invSt,
                                           float invSd, int mode) {
  const float p = __fmul_rn(ex2_ordered(__fmaf_rn(t, kLog2e, -ct)), invSt);
  if (mode != 0) return p;
  const float q = __fmul_rn(ex2_ordered(__fmaf_rn(d, kLog2e, -cd)), invSd);
  const float r = __fsub_rn(p, q);
  return r > 0.f ? r : 0.f;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
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

// Fold this lane's 32 elements of a piece (its four 16-byte vectors) into its
// running (C, S): the integer reference point C = ceil(log2e * max) grows
// when the piece holds a larger element (the sum is then rescaled exactly),
// then S += sum 2^(v log2e - C).  A NaN element makes S NaN, -inf elements
// add 0, and an all -inf lane keeps C = -inf, S = 0.  No cross-lane work:
// the lanes of a warp are combined once, when its range leaves the segment.
__device__ __forceinline__ void lane_fold(const uint4 (&r)[4], int bf16, float& C, ff& S) {
  float m;
  if (bf16) {
    uint32_t mx = bf16x2_max(bf16x2_max(r[0].x, r[0].y), bf16x2_max(r[0].z, r[0].w));
#pragma unroll
    for (int i = 1; i < 4; ++i)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(r[i].x, r[i].y), bf16x2_max(r[i].z, r[i].w)));
    m = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(r[i].x), __uint_as_float(r[i].y)),
                         fmaxf(__uint_as_float(r[i].z), __uint_as_float(r[i].w))));
  }
  const float c = ref_point(m);
  if (c > C) {
    S = ff_mul_f(S, scale_exact(C, c));
    C = c;
  }
  const float cc = (C == -INFINITY) ? 0.f : C;
  // four running sums a0..a3 as two packed pairs: (a0, a1) and (a2, a3)
  const f32x2 L2 = f2_pack(kLog2e, kLog2e), nc = f2_pack(-cc, -cc);
  f32x2 a01 = f2_pack(0.f, 0.f), a23 = a01;
  if (bf16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a01 = f2_add(a01, f2_exp2_shift_ordered(f2_bf16(r[i].x), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift_ordered(f2_bf16(r[i].y), L2, nc));
      a01 = f2_add(a01, f2_exp2_shift_ordered(f2_bf16(r[i].z), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift_ordered(f2_bf16(r[i].w), L2, nc));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a01 = f2_add(a01, f2_exp2_shift_ordered(f2_pack(__uint_as_float(r[i].x), __uint_as_float(r[i].y)), L2, nc));
      a23 = f2_add(a23, f2_exp2_shift_ordered(f2_pack(__uint_as_float(r[i].z), __uint_as_float(r[i].w)), L2, nc));
    }
  }
  float a0, a1, a2, a3;
  f2_unpack(a01, a0, a1);
  f2_unpack(a23, a2, a3);
  S = ff_add_f(S, __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3)));
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


// ---------------------------------------------------------------------------
// the residual pass: lane l loads vectors l + 32 i (coalesced) and sums each
// of its four 16-byte vectors; the warp then regroups the 128 vector sums into
// 32 run sums, run g = vectors 4 g .. 4 g + 3 (contiguous elements), the
// prefix steps the token draw uses
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_run(const unsigned char* base, int ne, int bf16, int aligned,
                                         int lane, uint4 (&r)[4]) {
  const int epv = bf16 ? 8 : 4;
  const uint32_t ninf = bf16 ? kNegInf2 : kNegInfF;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    if (aligned) {
      r[i] = (vi * epv < ne) ? ld_stream(base + 16 * (size_t)vi) : make_uint4(ninf, ninf, ninf, ninf);
    } else {
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
}
// this lane's run of a 16-byte aligned piece -> shared memory (cp.async)
__device__ __forceinline__ void stage_run(const unsigned char* base, int ne, int bf16, int lane,
                                          unsigned char* dst) {
  const int epv = bf16 ? 8 : 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    if (vi * epv < ne) cp_async16(dst + 16 * vi, base + 16 * (size_t)vi);
  }
}
__device__ __forceinline__ void read_run(const unsigned char* src, int ne, int bf16, int lane,
                                         uint4 (&r)[4]) {
  const int epv = bf16 ? 8 : 4;
  const uint32_t ninf = bf16 ? kNegInf2 : kNegInfF;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    r[i] = (vi * epv < ne) ? *reinterpret_cast<const uint4*>(src + 16 * vi) : make_uint4(ninf, ninf, ninf, ninf);
  }
}
// run sum g of r (or p) on lane g: each vector summed in element order, the
// vector sums regrouped through the warp's 512-byte scratch `vs`
__device__ __forceinline__ float run_resid(const uint4 (&t)[4], const uint4 (&d)[4], int bf16,
                                           const StopInfo& st, float* vs, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t tw[4] = {t[i].x, t[i].y, t[i].z, t[i].w};
    const uint32_t dw[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
    float acc = 0.f;
    if (bf16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float tv = (e & 1) ? bf16_hi(tw[e >> 1]) : bf16_lo(tw[e >> 1]);
        const float dv = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
        acc = __fadd_rn(acc, resid_val(tv, dv, st.ct, st.cd, st.invSt, st.invSd, st.mode));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc = __fadd_rn(acc, resid_val(__uint_as_float(tw[e]), __uint_as_float(dw[e]), st.ct,
                                       st.cd, st.invSt, st.invSd, st.mode));
    }
    vs[lane + 32 * i] = acc;
  }
  __syncwarp();
  const float4 g = reinterpret_cast<const float4*>(vs)[lane];
  __syncwarp();  // the scratch is reused by the next piece
  return __fadd_rn(__fadd_rn(__fadd_rn(g.x, g.y), g.z), g.w);
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


struct FinShared {
  float c[4][kMaxG];  // per position: Ct, St, Cd, Sd (the stop position's constants)
  float u[kMaxG];     // u_accept of the row (prefetched)
  int x[kMaxG];       // draft tokens of the row (prefetched)
  int n;              // first rejected position (G + 1: none)
  int err;
  int tmo;            // the wait for the row's statistics ran out
  float us;           // u_sample of the row (prefetched)
  StopInfo st;        // the result: stop position and its draw constants
};

// Row b's decisions (all warps of the CTA).  Warp w combines the segment
// records of positions w, w + 16, ...; then the first rejection n and the draw
// constants (F.st).  The owner also writes the accept probabilities, n and
// every token but token n.
__device__ void finalize_row(const DenseParams& P, int b, int warp, int lane, FinShared& F,
                             bool owner) {
  const int G = P.G, np = P.g.np;
  const UnitPart* rec = ws_at<UnitPart>(P, P.L.upart);
  // the statistics grid gave warp g the pieces [lo(g), lo(g + 1)), lo(g) =
  // g W / nwt; a segment record sits at the first piece of the segment
  const long long W = (long long)P.B * (G + 1) * np, nwt = P.stats_warps;
  // the range arithmetic in 32 bits when every product fits (a 64-bit
  // division is a long software sequence on the critical path of every row)
  const bool idx32 = (unsigned long long)(nwt + 1) * (unsigned long long)(W + 1) < (1ull << 32);
  const unsigned W32 = (unsigned)W, n32 = (unsigned)nwt;
  if (threadIdx.x == 0) {
    F.n = G + 1;
    F.err = F.tmo;  // a row whose statistics never arrived is failed like an input error
  }
  __syncthreads();
  for (int j = warp; j <= G; j += kWarps) {
    float Ct = -INFINITY, Cd = -INFINITY;
    ff St{0.f, 0.f}, Sd{0.f, 0.f};
    uint32_t txb = kNoTokenBits, dxb = kNoTokenBits;
    const long long P0 = ((long long)b * (G + 1) + j) * np, P1 = P0 + np;
    // warps whose ranges meet [P0, P1): lo(g) <= P0 for the first, lo(g) < P1 for the last
    const long long g0 = idx32 ? (long long)(((unsigned)(P0 + 1) * n32 + W32 - 1) / W32) - 1
                               : ((P0 + 1) * nwt + W - 1) / W - 1;
    const long long g1 = idx32 ? (long long)(((unsigned)P1 * n32 + W32 - 1) / W32) - 1
                               : (P1 * nwt + W - 1) / W - 1;
    for (long long g = g0 + lane; g <= g1; g += 32) {
      const long long lo = idx32 ? (long long)((unsigned)g * W32 / n32) : g * W / nwt;
      const long long lo1 = idx32 ? (long long)((unsigned)(g + 1) * W32 / n32) : (g + 1) * W / nwt;
      if (lo1 <= lo) continue;  // an empty range writes nothing
      const UnitPart u = ldcg32(rec + (lo > P0 ? lo : P0));
      combine_part(u, Ct, St, Cd, Sd);
      if (__float_as_uint(u.tx) != kNoTokenBits) {
        txb = __float_as_uint(u.tx);
        dxb = __float_as_uint(u.dx);
      }
    }
    warp_combine_pair(Ct, St, Cd, Sd);
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
      acc = F.u[j] < a;
    }
    if (lane == 0) {
      if (owner && j < G && P.acc_out)
        P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : a;
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
      if (owner) atomicOr(&hdr_of(P)->status, F.tmo ? kStatusTimeout : kStatusInputErr);
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
    F.st = st;
    if (owner) P.n_out[b] = err ? -1 : n;
  }
  __syncthreads();
  if (!owner) return;
  // tokens: x_0..x_{n-1}, then (token n, drawn later), then -1
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  for (int j = threadIdx.x; j <= G; j += kThreads) {
    if (err)
      tok[j] = -1;
    else if (j < n)
      tok[j] = F.x[j];
    else if (j > n)
      tok[j] = -1;
  }
}

// ---------------------------------------------------------------------------
// kernel 1: statistics of every piece.  Work items are the pieces (b, j, k)
// in row order; every warp of the persistent grid takes one contiguous range
// of them and streams it through a private kStages-deep ring of 4 KB shared
// stages (2 KB target piece + 2 KB draft piece), filled by cp.async 16-byte
// copies: while one item is reduced, the next kStages - 1 are in flight.
// Each lane copies, and later reads, only its own vectors, so the ring needs
// no synchronisation beyond the lane's own cp.async groups.
// ---------------------------------------------------------------------------
constexpr int kStatsWarps = 24;  // warps per statistics CTA
constexpr int kStatsCtas = 1;    // statistics CTAs per SM
constexpr int kStatsThreads = 32 * kStatsWarps;
constexpr int kStages = 2;
constexpr int kStageBytes = 2 * kPieceBytes;
constexpr size_t kStatsSmem = (size_t)kStatsWarps * kStages * kStageBytes;

struct Item {  // piece k of row-position (b, j)
  int b, j, k;
};
__device__ __forceinline__ Item item_at(long long w, int G, int np) {
  const long long r = w / np;
  Item it;
  it.k = (int)(w - r * np);
  it.b = (int)(r / (G + 1));
  it.j = (int)(r - (long long)it.b * (G + 1));
  return it;
}
__device__ __forceinline__ void item_next(Item& it, int G, int np) {
  if (++it.k == np) {
    it.k = 0;
    if (++it.j == G + 1) {
      it.j = 0;
      ++it.b;
    }
  }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// this lane's vectors of piece `it` (target, and draft for j < G) -> stage
__device__ __forceinline__ void issue_item(const DenseParams& P, const Item& it,
                                           unsigned char* stage, int lane) {
  const int pe = P.g.pe, epv = P.bf16 ? 8 : 4;
  const int ne = min(pe, P.V - it.k * pe);
  const size_t off = (size_t)it.k * kPieceBytes;
  const unsigned char* ts = target_row(P, it.b, it.j) + off;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    if (vi * epv < ne) cp_async16(stage + 16 * vi, ts + 16 * vi);
  }
  if (it.j < P.G) {
    const unsigned char* ds = draft_row(P, it.b, it.j) + off;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = lane + 32 * i;
      if (vi * epv < ne) cp_async16(stage + kPieceBytes + 16 * vi, ds + 16 * vi);
    }
  }
}

// Running statistics of the (row, position) segment a warp is streaming:
// each lane folds its elements of every piece of the segment into its own
// (C, S); when the warp's range leaves the segment the lanes are combined
// and written as one record, in the slot of the segment's first piece; the
// other slots of the segment stay zero ("empty": St = 0 and c = 0, which no
// real record has).
struct SegAcc {
  long long w0;  // record slot: the segment's first piece
  int b, j;
  int x;         // the segment's draft token (-1 at the bonus position)
  float Ct, Cd;  // this lane's reference points
  ff St, Sd;     // this lane's sums
  uint32_t tb, db;  // logits at the draft token, if a piece of the segment held it
};

__device__ __forceinline__ void seg_begin(SegAcc& a, const Item& it, long long w,
                                          const DenseParams& P) {
  a.w0 = w;
  a.b = it.b;
  a.j = it.j;
  a.x = (it.j < P.G) ? __ldg(P.x + (size_t)it.b * P.G + it.j) : -1;
  a.Ct = a.Cd = -INFINITY;
  a.St = a.Sd = ff{0.f, 0.f};
  a.tb = a.db = kNoTokenBits;
}

// every lane (the lanes are combined first)
__device__ __forceinline__ void seg_write(const DenseParams& P, SegAcc& a, int lane) {
  warp_combine_pair(a.Ct, a.St, a.Cd, a.Sd);
  if (lane == 0) {
    float4* q = reinterpret_cast<float4*>(ws_at<UnitPart>(P, P.L.upart) + a.w0);
    q[0] = make_float4(a.St.hi, a.St.lo, a.Sd.hi, a.Sd.lo);
    q[1] = make_float4(a.Ct, a.Cd, __uint_as_float(a.tb), __uint_as_float(a.db));
  }
}

// fold piece `it`, held in rt / rd, into this lane's segment statistics; the
// warp whose piece holds the draft token keeps the two logits there
__device__ __forceinline__ void piece_accumulate(const DenseParams& P, const Item& it,
                                                 const uint4 (&rt)[4], const uint4 (&rd)[4],
                                                 int lane, SegAcc& a) {
  const int pe = P.g.pe;
  lane_fold(rt, P.bf16, a.Ct, a.St);
  if (it.j < P.G) {
    lane_fold(rd, P.bf16, a.Cd, a.Sd);
    const int ne = min(pe, P.V - it.k * pe);
    const int xl = a.x - it.k * pe;
    if (a.x >= 0 && xl >= 0 && xl < ne) {
      a.tb = piece_element(rt, xl, P.bf16, lane);
      a.db = piece_element(rd, xl, P.bf16, lane);
    }
  }
}

__global__ void __launch_bounds__(kStatsThreads, kStatsCtas) dense_stats_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // Launched as a programmatic dependent of whatever precedes it on the
  // stream (often the previous call's row kernel): the CTAs may be resident
  // early, but nothing is read before that grid has completed and its
  // memory is visible -- it may have produced these logits.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = P.G, np = P.g.np, pe = P.g.pe, epv = P.bf16 ? 8 : 4;
  const long long W = (long long)P.B * (G + 1) * np;
  const long long nwt = (long long)gridDim.x * kStatsWarps;
  const long long gw = (long long)blockIdx.x * kStatsWarps + warp;
  const long long lo = gw * W / nwt, hi = (gw + 1) * W / nwt;
  // the dependent row kernel may be scheduled as soon as SMs free up; each of
  // its CTAs waits for its row's count before it reads the row's records
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lo >= hi) return;
  const uint32_t ninf = P.bf16 ? kNegInf2 : kNegInfF;

  if (!P.aligned) {  // rows not 16-byte aligned: plain loads, no ring
    Item it = item_at(lo, G, np);
    SegAcc acc;
    seg_begin(acc, it, lo, P);
    long long rstart = lo;  // this range's first piece in row acc.b
    for (long long w = lo; w < hi; ++w, item_next(it, G, np)) {
      if (it.b != acc.b || it.j != acc.j) {
        seg_write(P, acc, lane);
        if (it.b != acc.b) {
          row_signal(P, acc.b, w - rstart, lane);
          rstart = w;
        }
        seg_begin(acc, it, w, P);
      }
      const int ne = min(pe, P.V - it.k * pe);
      const size_t off = (size_t)it.k * kPieceBytes;
      uint4 rt[4], rd[4];
      load_piece(target_row(P, it.b, it.j) + off, ne, P.bf16, 0, lane, rt);
      if (it.j < G)
        load_piece(draft_row(P, it.b, it.j) + off, ne, P.bf16, 0, lane, rd);
      else
        for (int i = 0; i < 4; ++i) rd[i] = make_uint4(ninf, ninf, ninf, ninf);
      piece_accumulate(P, it, rt, rd, lane, acc);
    }
    seg_write(P, acc, lane);
    row_signal(P, acc.b, hi - rstart, lane);
    return;
  }

  unsigned char* ring = smem_raw + (size_t)warp * kStages * kStageBytes;
  Item in = item_at(lo, G, np), out = in;
  long long wi = lo;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (wi < hi) {
      issue_item(P, in, ring + s * kStageBytes, lane);
      item_next(in, G, np);
      ++wi;
    }
    cp_async_commit();
  }
  int slot = 0, islot = kStages - 1;
  SegAcc acc;
  seg_begin(acc, out, lo, P);
  long long rstart = lo;  // this range's first piece in row acc.b
  for (long long w = lo; w < hi; ++w) {
    if (out.b != acc.b || out.j != acc.j) {
      seg_write(P, acc, lane);
      if (out.b != acc.b) {  // the range has left row acc.b: its records are all stored
        row_signal(P, acc.b, w - rstart, lane);
        rstart = w;
      }
      seg_begin(acc, out, w, P);
    }
    if (wi < hi) {
      issue_item(P, in, ring + islot * kStageBytes, lane);
      item_next(in, G, np);
      ++wi;
    }
    cp_async_commit();
    cp_async_wait_group<kStages - 1>();
    const unsigned char* stage = ring + slot * kStageBytes;
    const int ne = min(pe, P.V - out.k * pe);
    const bool has_d = out.j < G;
    uint4 rt[4], rd[4];
    if (ne == pe) {  // a whole piece: every vector is valid
#pragma unroll
      for (int i = 0; i < 4; ++i) rt[i] = *reinterpret_cast<const uint4*>(stage + 16 * (lane + 32 * i));
      if (has_d) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          rd[i] = *reinterpret_cast<const uint4*>(stage + kPieceBytes + 16 * (lane + 32 * i));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int vi = lane + 32 * i;
        const bool v = vi * epv < ne;
        rt[i] = v ? *reinterpret_cast<const uint4*>(stage + 16 * vi) : make_uint4(ninf, ninf, ninf, ninf);
        rd[i] = (v && has_d) ? *reinterpret_cast<const uint4*>(stage + kPieceBytes + 16 * vi)
                             : make_uint4(ninf, ninf, ninf, ninf);
      }
    }
    piece_accumulate(P, out, rt, rd, lane, acc);
    item_next(out, G, np);
    slot = (slot + 1 == kStages) ? 0 : slot + 1;
    islot = (islot + 1 == kStages) ? 0 : islot + 1;
  }
  seg_write(P, acc, lane);
  row_signal(P, acc.b, hi - rstart, lane);
  cp_async_wait_group<0>();
}

// ---------------------------------------------------------------------------
// kernel 2: everything after the statistics, one thread-block cluster of C
// CTAs per row.  Every CTA of the cluster finalises the row from the piece
// records (the same arithmetic, so the same n and constants), then computes
// the residual (or p) mass of its share of the stop position's pieces.  After
// a cluster barrier the rank-0 CTA draws the token: a prefix over the row's
// piece masses picks the piece, a prefix over that piece's element values
// picks the token.  Both prefixes are block-wide scans in fp64 (a few hundred
// additions per row), so no thread walks more than a handful of values.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// all threads of every CTA of the cluster; orders their earlier memory
// operations before everything after the barrier, cluster-wide
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float logit_at(const unsigned char* row, int y, int bf16) {
  return bf16 ? bf16_to_f32(__ldg(reinterpret_cast<const uint16_t*>(row) + y))
              : __ldg(reinterpret_cast<const float*>(row) + y);
}

struct SelShared {
  float whi[kWarps], wlo[kWarps];
  ff base, T;
  int clamp;
  int wa[kWarps], wb[kWarps];
  int kstar, y;
};

// Block-wide exclusive prefix of v in float-float; `total` receives the sum.
// (float-float rather than fp64: GB300 runs fp64 at a small fraction of the
// fp32 rate, and here every thread of the block takes part.)
__device__ __forceinline__ ff block_exclusive_scan_ff(ff v, SelShared& S, ff& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ff x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y = ff_shfl_up(x, o);
    if (lane >= o) x = ff_add(x, y);
  }
  ff ex = ff_shfl_up(x, 1);
  if (lane == 0) ex = ff{0.f, 0.f};
  if (lane == 31) {
    S.whi[warp] = x.hi;
    S.wlo[warp] = x.lo;
  }
  __syncthreads();
  ff wbase{0.f, 0.f}, tot{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const ff t{S.whi[w], S.wlo[w]};
    if (w < warp) wbase = ff_add(wbase, t);
    tot = ff_add(tot, t);
  }
  __syncthreads();  // whi / wlo may be reused
  total = tot;
  return ff_add(wbase, ex);
}

// shared-memory address of `p` in the rank-0 CTA of the cluster, and a store there
__device__ __forceinline__ uint32_t map_rank0(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
constexpr int kMassSmem = 1024;  // pieces per row whose masses are kept on chip

// block-wide: the first thread with `cond` (kThreads if none) and the largest
// `v` (one ballot / reduction per warp, then one pass over the warps; no
// contended shared-memory atomics)
__device__ __forceinline__ void block_first_and_max(bool cond, int v, SelShared& S, int& first,
                                                    int& vmax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, cond);
  const int wm = (int)__reduce_max_sync(0xffffffffu, (unsigned)(v + 1)) - 1;  // v >= -1
  if (lane == 0) {
    S.wa[warp] = bal ? warp * 32 + __ffs(bal) - 1 : kThreads;
    S.wb[warp] = wm;
  }
  __syncthreads();
  int f = kThreads, m = -1;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    f = min(f, S.wa[w]);
    m = max(m, S.wb[w]);
  }
  __syncthreads();  // wa / wb may be reused
  first = f;
  vmax = m;
}

__device__ __forceinline__ float warp_inclusive_scan_f(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = __fadd_rn(v, y);
  }
  return v;
}

constexpr int kLanePieces = 160;  // pieces per row whose lane run sums are kept on chip

// The token draw from the piece masses `sm` and the lane run sums `sl` kept
// in shared memory, by one warp: a float-float prefix over the pieces picks
// the piece, one over its 32 run sums picks the run, an fp32 prefix over the
// run's elements (plus the float-float base) picks the token.  Returns T; a
// zero residual after a rejection (only through rounding) returns T = 0 and
// draws nothing: the caller then takes the general path.
__device__ double select_fast(const DenseParams& P, int b, const StopInfo& st, const float* sm,
                              const float* sl, float us, int lane) {
  const int V = P.V, np = P.g.np, pe = P.g.pe, run = pe / 32;
  const int per = (np + 31) / 32;
  const int k0 = min(np, lane * per), k1 = min(np, k0 + per);
  ff ls{0.f, 0.f};
  for (int k = k0; k < k1; ++k) ls = ff_add_f(ls, sm[k]);
  const ff ex = warp_exclusive_scan_ff(ls, lane);
  const ff T = ff_shfl(ff_add(ex, ls), 31);
  if (!(T.hi > 0.f) && st.mode == 0) return 0.0;
  const ff target = ff_mul_f(T, us);
  // piece level
  const unsigned hit = __ballot_sync(0xffffffffu, (k1 > k0) && ff_gt(ff_add(ex, ls), target));
  int kstar = 0;
  ff base{0.f, 0.f};
  if (hit) {
    const int fl = __ffs(hit) - 1;
    if (lane == fl) {
      ff acc = ex;
      for (int k = k0; k < k1; ++k) {
        base = acc;
        acc = ff_add_f(acc, sm[k]);
        kstar = k;
        if (ff_gt(acc, target)) break;
      }
    }
    kstar = __shfl_sync(0xffffffffu, kstar, fl);
    base = ff_shfl(base, fl);
  } else {  // u*T at or past the total: the last piece with mass
    int last = -1;
    for (int k = k0; k < k1; ++k)
      if (sm[k] > 0.f) last = k;
    last = (int)__reduce_max_sync(0xffffffffu, (unsigned)(last + 1)) - 1;
    kstar = last < 0 ? 0 : last;
  }
  // run level
  const float lv = sl[kstar * 32 + lane];
  const ff lbase = ff_add(base, warp_exclusive_scan_ff(ff{lv, 0.f}, lane));
  const unsigned hit2 = hit ? __ballot_sync(0xffffffffu, ff_gt(ff_add_f(lbase, lv), target)) : 0u;
  int fr;
  if (hit2) {
    fr = __ffs(hit2) - 1;
  } else {  // the last run with mass
    fr = (int)__reduce_max_sync(0xffffffffu, (unsigned)(lv > 0.f ? lane + 1 : 0)) - 1;
    if (fr < 0) fr = 0;
  }
  // element level: lane e takes element e of run fr
  const int y0 = kstar * pe, ne = min(pe, V - y0);
  const int e = fr * run + lane;
  const bool valid = lane < run && e < ne;
  const unsigned char* trow = target_row(P, b, st.n);
  float r = 0.f;
  if (valid)
    r = resid_val(logit_at(trow, y0 + e, P.bf16),
                  st.mode == 0 ? logit_at(draft_row(P, b, st.n), y0 + e, P.bf16) : 0.f, st.ct,
                  st.cd, st.invSt, st.invSd, st.mode);
  const float incl = warp_inclusive_scan_f(r, lane);
  const ff lb = ff_shfl(lbase, fr);
  const unsigned cross = hit2 ? __ballot_sync(0xffffffffu, valid && ff_gt(ff_add_f(lb, incl), target)) : 0u;
  int y;
  if (cross) {
    y = y0 + fr * run + __ffs(cross) - 1;
  } else {  // rounding between the sums, or past the total: the run's last element with mass
    const int lp = (int)__reduce_max_sync(0xffffffffu, (unsigned)(r > 0.f ? e + 1 : 0)) - 1;
    y = y0 + (lp >= 0 ? lp : fr * run);
  }
  if (lane == 0) P.tok_out[(size_t)b * (P.G + 1) + st.n] = y;
  return (double)T.hi + (double)T.lo;
}

// the token of row b from its piece masses `mv` (shared memory of this CTA,
// or the workspace); whole CTA; returns T
__device__ double select_row(const DenseParams& P, int b, StopInfo& st, float* mv, bool mv_shared,
                             SelShared& S) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // masses written by other CTAs: shared memory, or global memory read around L1
  auto mass = [&](int k) -> float { return mv_shared ? mv[k] : __ldcg(mv + k); };
  const int V = P.V, np = P.g.np, pe = P.g.pe;
  const float us = P.u_s[b];
  const unsigned char* trow = target_row(P, b, st.n);
  const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, st.n) : nullptr;
  // piece level, one warp: lane l sums its run of masses, a warp prefix
  // finds the first piece whose inclusive prefix exceeds u * T
  const int per = (np + 31) / 32;
  const int k0 = min(np, lane * per), k1 = min(np, k0 + per);
  ff T{0.f, 0.f};
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (warp == 0) {
      ff ls{0.f, 0.f};
      for (int k = k0; k < k1; ++k) ls = ff_add_f(ls, mass(k));
      const ff ex = warp_exclusive_scan_ff(ls, lane);
      const ff tot = ff_shfl(ff_add(ex, ls), 31);
      const ff target = ff_mul_f(tot, us);
      const unsigned hit = __ballot_sync(0xffffffffu, (k1 > k0) && ff_gt(ff_add(ex, ls), target));
      int kstar = 0;
      ff base{0.f, 0.f};
      if (hit) {
        const int fl = __ffs(hit) - 1;
        if (lane == fl) {
          ff acc = ex;
          for (int k = k0; k < k1; ++k) {
            base = acc;
            acc = ff_add_f(acc, mass(k));
            kstar = k;
            if (ff_gt(acc, target)) break;
          }
        }
        kstar = __shfl_sync(0xffffffffu, kstar, fl);
        base = ff_shfl(base, fl);
      } else {  // u*T at or past the total: the last piece with mass
        int last = -1;
        for (int k = k0; k < k1; ++k)
          if (mass(k) > 0.f) last = k;
        last = (int)__reduce_max_sync(0xffffffffu, (unsigned)(last + 1)) - 1;
        kstar = last < 0 ? 0 : last;
      }
      if (lane == 0) {
        S.kstar = kstar;
        S.base = base;
        S.T = tot;
        S.clamp = hit == 0u;
      }
    }
    __syncthreads();
    T = S.T;
    if (T.hi > 0.f || st.mode != 0 || attempt == 1) break;
    // zero residual after a rejection (only through rounding): draw from p_n
    st.mode = 1;
    drow = nullptr;
    for (int k = warp; k < np; k += kWarps) {
      const int y0 = k * pe, ne = min(pe, V - y0);
      float sum = 0.f;
      for (int e = lane; e < ne; e += 32)
        sum += resid_val(logit_at(trow, y0 + e, P.bf16), 0.f, st.ct, st.cd, st.invSt, st.invSd, 1);
      sum = warp_sum(sum);
      if (lane == 0) mv[k] = sum;
    }
    __threadfence_block();
    __syncthreads();
  }
  const ff target = ff_mul_f(T, us);
  const bool clamp = S.clamp;
  const int kstar = S.kstar;
  const ff base = S.base;
  // element level: thread t takes the contiguous run [t q, t q + q) of piece kstar
  constexpr int kMaxQ = kPieceBytes / 2 / kThreads;  // 2 (bf16); fp32 uses 1
  const int q = pe / kThreads;
  const int y0 = kstar * pe, ne = min(pe, V - y0);
  float rv[kMaxQ];
  float tot = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int i = 0; i < kMaxQ; ++i) {
    const int e = t * q + i;
    float r = 0.f;
    if (i < q && e < ne)
      r = resid_val(logit_at(trow, y0 + e, P.bf16), drow ? logit_at(drow, y0 + e, P.bf16) : 0.f,
                    st.ct, st.cd, st.invSt, st.invSd, st.mode);
    rv[i] = r;
    tot = __fadd_rn(tot, r);
    if (r > 0.f) lastpos = e;
  }
  ff ptot;
  const ff lbase = ff_add(base, block_exclusive_scan_ff(ff{tot, 0.f}, S, ptot));
  int ecross, elast;
  block_first_and_max(!clamp && ff_gt(ff_add_f(lbase, tot), target), lastpos, S, ecross, elast);
  if (t == ecross) {
    ff acc = lbase;
    int yy = -1, lp = -1;
#pragma unroll
    for (int i = 0; i < kMaxQ; ++i) {
      if (i < q && yy < 0) {
        acc = ff_add_f(acc, rv[i]);
        if (rv[i] > 0.f) lp = t * q + i;
        if (ff_gt(acc, target)) yy = t * q + i;
      }
    }
    // rounding between the two sums: the run's last element with mass
    if (yy < 0) yy = lp >= 0 ? lp : lastpos;
    S.y = yy < 0 ? 0 : yy;
  } else if (t == 0 && ecross == kThreads) {
    S.y = max(elast, 0);
  }
  __syncthreads();
  if (t == 0) P.tok_out[(size_t)b * (P.G + 1) + st.n] = y0 + S.y;
  return (double)T.hi + (double)T.lo;
}

constexpr size_t kRowWarpBuf = 2 * kPieceBytes + 512;  // a prefetched piece pair + vector sums
constexpr size_t kRowSmem = (size_t)kWarps * kRowWarpBuf + (size_t)kLanePieces * 32 * sizeof(float);

__global__ void __launch_bounds__(kThreads, 2) dense_row_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(16) unsigned char row_smem[];
  __shared__ FinShared F;
  __shared__ SelShared S;
  __shared__ float s_mass[kMassSmem];  // the row's piece masses (rank 0), when they fit
  __shared__ double s_T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = (int)cluster_size(), r = (int)cluster_rank();
  const int b = blockIdx.x / C;
  const bool owner = r == 0;
  const int G = P.G, np = P.g.np, pe = P.g.pe;
  const bool in_smem = np <= kMassSmem;   // masses on chip
  const bool fast = np <= kLanePieces;    // lane run sums on chip too: one-warp draw
  unsigned char* wbuf = row_smem + (size_t)warp * kRowWarpBuf;
  float* vs = reinterpret_cast<float*>(wbuf + 2 * kPieceBytes);
  float* s_lane = reinterpret_cast<float*>(row_smem + (size_t)kWarps * kRowWarpBuf);
  // the next call's statistics kernel may be scheduled as CTAs of this one
  // leave (it waits for this grid before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // inputs first (they do not come from the statistics kernel) ...
  // (read from L2: this grid does not wait for the grids before it)
  for (int j = threadIdx.x; j < G; j += kThreads) {
    F.u[j] = __ldcg(P.u_acc + (size_t)b * G + j);
    F.x[j] = __ldcg(P.x + (size_t)b * G + j);
  }
  if (threadIdx.x == 0) F.us = __ldcg(P.u_s + b);
  // ... then wait for the row's statistics alone: the count is complete once
  // every statistics warp whose range meets the row has stored its records
  // there (release by that warp, acquire here), often while the grid still
  // streams later rows.  A launch as a programmatic dependent makes every
  // statistics CTA resident before any CTA of this grid starts, so the wait
  // needs nothing from this grid to end.
  if (threadIdx.x == 0) F.tmo = wait_row_ready(P, b, (uint32_t)(G + 1) * (uint32_t)np) ? 0 : 1;
  __syncthreads();
  finalize_row(P, b, warp, lane, F, owner);
  StopInfo st = F.st;
  // residual (or p) masses of this CTA's share of the stop position's pieces,
  // two pieces per warp at a time: the second is staged by cp.async while
  // the first is loaded straight into registers and reduced
  if (st.mode != 2) {
    const int k_lo = (int)((long long)r * np / C), k_hi = (int)((long long)(r + 1) * np / C);
    const uint32_t ninf = P.bf16 ? kNegInf2 : kNegInfF;
    const unsigned char* trow = target_row(P, b, st.n);
    const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, st.n) : nullptr;
    auto publish = [&](int k, float lsum) {
      const float mass = warp_sum(lsum);
      if (fast) st_cluster_f32(map_rank0(&s_lane[k * 32 + lane]), lsum);
      if (lane == 0) {
        if (in_smem)  // into the rank-0 CTA's shared memory
          st_cluster_f32(map_rank0(&s_mass[k]), mass);
        else
          ws_at<float>(P, P.L.rmass)[(size_t)b * P.g.np4 + k] = mass;
      }
    };
    for (int k = k_lo + warp; k < k_hi; k += 2 * kWarps) {
      const int k2 = k + kWarps;
      const bool pre = k2 < k_hi && P.aligned;
      if (pre) {
        const int ne2 = min(pe, P.V - k2 * pe);
        stage_run(trow + (size_t)k2 * kPieceBytes, ne2, P.bf16, lane, wbuf);
        if (drow) stage_run(drow + (size_t)k2 * kPieceBytes, ne2, P.bf16, lane, wbuf + kPieceBytes);
      }
      cp_async_commit();
      uint4 rt[4], rd[4];
      {
        const int ne = min(pe, P.V - k * pe);
        load_run(trow + (size_t)k * kPieceBytes, ne, P.bf16, P.aligned, lane, rt);
        if (drow)
          load_run(drow + (size_t)k * kPieceBytes, ne, P.bf16, P.aligned, lane, rd);
        else
          for (int i = 0; i < 4; ++i) rd[i] = make_uint4(ninf, ninf, ninf, ninf);
        publish(k, run_resid(rt, rd, P.bf16, st, vs, lane));
      }
      if (k2 < k_hi) {
        const int ne2 = min(pe, P.V - k2 * pe);
        if (pre) {
          cp_async_wait_group<0>();
          read_run(wbuf, ne2, P.bf16, lane, rt);
          if (drow) read_run(wbuf + kPieceBytes, ne2, P.bf16, lane, rd);
        } else {
          load_run(trow + (size_t)k2 * kPieceBytes, ne2, P.bf16, P.aligned, lane, rt);
          if (drow) load_run(drow + (size_t)k2 * kPieceBytes, ne2, P.bf16, P.aligned, lane, rd);
        }
        if (!drow)
          for (int i = 0; i < 4; ++i) rd[i] = make_uint4(ninf, ninf, ninf, ninf);
        publish(k2, run_resid(rt, rd, P.bf16, st, vs, lane));
      }
    }
  }
  cluster_barrier();  // every CTA's masses are written; every record was read
  UnitPart* up_row = ws_at<UnitPart>(P, P.L.upart) + (size_t)b * (G + 1) * np;
  const int nrec = (G + 1) * np;
  if (!owner) {
    // ranks 1 .. C-1 leave the row's records zero while rank 0 draws (its
    // warps' loads would otherwise queue behind these stores)
    const int lo = (int)((long long)(r - 1) * nrec / (C - 1));
    const int hi = (int)((long long)r * nrec / (C - 1));
    for (int i = lo + (int)threadIdx.x; i < hi; i += kThreads) zero32(up_row + i);
    // this grid completes only after the statistics grid (whatever follows
    // on the stream may rely on both)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  if (threadIdx.x == 0) *row_count(P, b) = 0u;  // every CTA of the cluster has passed its wait
  // the draw; the masses kept off chip are consumed
  float* rm = ws_at<float>(P, P.L.rmass) + (size_t)b * P.g.np4;
  double T = 0.0;
  if (fast && st.mode != 2) {
    if (warp == 0) {
      T = select_fast(P, b, st, s_mass, s_lane, F.us, lane);
      if (lane == 0) s_T = T;
    }
    __syncthreads();
    T = s_T;
    if (!(T > 0.0) && st.mode == 0) T = select_row(P, b, st, s_mass, true, S);  // zero residual
  } else if (st.mode != 2) {
    T = select_row(P, b, st, in_smem ? s_mass : rm, in_smem, S);
  }
  if (C == 1)
    for (int i = threadIdx.x; i < nrec; i += kThreads) zero32(up_row + i);
  if (!in_smem)
    for (int k = threadIdx.x; k < np; k += kThreads) rm[k] = 0.f;
  if (threadIdx.x == 0 && P.keep_stop) {  // read (and cleared) by the residual-output kernel
    st.T = T;
    ws_at<StopInfo>(P, P.L.stop)[b] = st;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {  // once per device: SM count and the ring's shared memory
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dense_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStatsSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dense_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kRowSmem);
    if (e != cudaSuccess) return e;
    sms[dev] = n;
  }
  const long long pieces = (long long)p.B * (p.G + 1) * p.g.np;
  long long grid = (long long)sms[dev] * kStatsCtas;
  if (grid * kStatsWarps > pieces) grid = (pieces + kStatsWarps - 1) / kStatsWarps;
  DenseParams q = p;
  q.stats_warps = grid * kStatsWarps;
  {
    cudaLaunchConfig_t k1 = {};
    k1.gridDim = dim3((unsigned)grid, 1, 1);
    k1.blockDim = dim3(kStatsThreads, 1, 1);
    k1.dynamicSmemBytes = kStatsSmem;
    k1.stream = s;
    cudaLaunchAttribute a1[1];
    a1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a1[0].val.programmaticStreamSerializationAllowed = 1;
    k1.attrs = a1;
    k1.numAttrs = 1;
    e = cudaLaunchKernelEx(&k1, dense_stats_kernel, q);
    if (e != cudaSuccess) return e;
  }
  // clusters of C CTAs per row: about two CTAs per SM in all, at most 8
  int C = (int)((2ll * sms[dev]) / p.B);
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  if (C > p.g.np) C = p.g.np;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)p.B * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kRowSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, dense_row_kernel, q);
}

cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s) {
  dense_resid_out_kernel<<<p.B, 512, 0, s>>>(p, resid_out);
  return cudaGetLastError();
}

}  // namespace sv
