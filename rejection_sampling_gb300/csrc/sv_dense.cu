// sv_dense.cu -- fused single-HBM-pass dense verification for large vocabularies.
//
// Computes, for every row b (DFlash/DFlash2 guide, 4.4; Uno article, "What
// 'lossless' actually has to mean"):
//   p_j = softmax(target[b, j]), q_j = softmax(draft[b, j]) for all positions,
//   a_j = min(1, p_j(x_j) / q_j(x_j))  (0 where q_j(x_j) = 0),
//   n   = first j with u_accept[b, j] >= a_j (gamma if none),
//   token n = inverse CDF of max(p_n - q_n, 0) (n < gamma) or of p_gamma
//   (bonus, DFlash/DFlash2 guide section 2) at u_sample[b].
//
// Design (one persistent kernel, one launch per call):
//  * Work is a stream of tickets taken with one atomicAdd each.  Tickets are
//    ordered row by row: the statistics units of row r, then the residual
//    units of row r - lag.  A statistics unit is up to 8 x 4 KB pieces of the
//    target row (b, j) plus the same pieces of the draft row (b, j); a
//    residual unit is up to 8 pieces of 2 KB target + 2 KB draft of the stop
//    position (b, n).
//  * Each CTA = 1 producer warp + 16 consumer warps around a 32-stage ring of
//    4 KB shared-memory stages.  The producer moves pieces with 1-D bulk
//    copies (cp.async.bulk, TMA) completing on per-stage mbarriers; every
//    consumer warp takes every 16th stage.
//  * A consumer warp reduces a 4 KB piece to (c, s): c = log2e * max, s =
//    sum 2^(v*log2e - c) (MUFU ex2).  The last warp of a unit combines the
//    unit's pieces and publishes one partial; the last unit of a (row,
//    position) finalises its accept test in fp64; the last position of a row
//    finds the first rejection n and publishes the stop constants.  These
//    hand-offs are last-arriver atomics: no warp ever waits for another CTA
//    except the producer of a residual unit, which waits (bounded) for its
//    row's stop constants.  Every ticket it could wait on was taken earlier by
//    a running CTA, so the wait always ends.
//  * Residual units recompute r(y) = max(p(y) - q(y), 0) for the stop
//    position only (the rows are still in L2: they were read a few rows of
//    work earlier) and publish per-piece masses; the last one selects the
//    piece and then the token by an fp64 prefix over fp32 element values.
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kNS = 32;  // ring stages
constexpr int kNW = 16;  // consumer warps
constexpr int kThreads = 32 * (kNW + 1);

enum StageKind : int { kStatsT = 0, kStatsD = 1, kResid = 2, kResidSkip = 3, kEnd = 4 };

struct StageMeta {
  int kind, b, j, kp, ne, uslot, upieces, pidx, unit_c, npc, mode, pad;
  float ct, cd, invSt, invSd;
};

struct UnitSlot {
  unsigned int count;
  unsigned int pad[3];
  float c[2 * kUnitPieces];
  float s[2 * kUnitPieces];
};

struct Smem {
  alignas(128) unsigned char ring[kNS][kPieceBytes];
  uint64_t full[kNS];
  uint64_t empty[kNS];
  StageMeta meta[kNS];
  UnitSlot unit[kNS];
};

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

// ---------------------------------------------------------------------------
// bounded waits (every spin has a limit; on expiry: timeout + abort flags)
// ---------------------------------------------------------------------------
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, const DenseParams& P) {
  if (mbar_try_wait(bar, parity)) return true;
  WsHeader* h = hdr_of(P);
  const long long t0 = clock64();
  unsigned it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) return false;
      if (clock64() - t0 > P.wait_bound) {
        atomicOr(&h->status, kStatusTimeout);
        atomicExch(&h->abort, 1u);
        return false;
      }
    }
  }
  return true;
}

// producer lane 0: wait until row b's stop constants are published
__device__ bool wait_ready(const DenseParams& P, int b) {
  const uint32_t* rdy = ws_at<uint32_t>(P, P.L.ready) + b;
  if (ld_acquire_u32(rdy)) return true;
  WsHeader* h = hdr_of(P);
  const long long t0 = clock64();
  while (!ld_acquire_u32(rdy)) {
    if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) return false;
    if (clock64() - t0 > P.wait_bound) {
      atomicOr(&h->status, kStatusTimeout);
      atomicExch(&h->abort, 1u);
      return false;
    }
    nanosleep_ns(128);
  }
  return true;
}

// ---------------------------------------------------------------------------
// ticket -> work unit
// ---------------------------------------------------------------------------
struct Unit {
  int resid, b, j, c;
};

__device__ __forceinline__ Unit decode_ticket(long long t, const DenseParams& P) {
  long long rem;
  int b, resid;
  dense_ticket_row(t, P.B, P.G, P.g.nc_s, P.g.nc_r, P.lag, &resid, &b, &rem);
  Unit u;
  u.resid = resid;
  u.b = b;
  if (!resid) {
    u.j = (int)(rem / P.g.nc_s);
    u.c = (int)(rem % P.g.nc_s);
  } else {
    u.j = 0;
    u.c = (int)rem;
  }
  return u;
}

// ---------------------------------------------------------------------------
// producer
// ---------------------------------------------------------------------------
__device__ __forceinline__ void copy_plain(unsigned char* dst, const unsigned char* src, int bytes,
                                           int es, int lane) {
  if (es == 2) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
    for (int i = lane; i < bytes / 2; i += 32) d[i] = s[i];
  } else {
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d = reinterpret_cast<uint32_t*>(dst);
    for (int i = lane; i < bytes / 4; i += 32) d[i] = s[i];
  }
}

// fill stage `slot` with up to two row slices; completes full[slot]
__device__ __forceinline__ void issue_stage(const DenseParams& P, Smem& S, int slot,
                                            const unsigned char* src0, int bytes0,
                                            const unsigned char* src1, int bytes1, int lane) {
  if (P.aligned) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(bytes0 + bytes1));
      if (bytes0) bulk_g2s(S.ring[slot], src0, (uint32_t)bytes0, &S.full[slot]);
      if (bytes1) bulk_g2s(S.ring[slot] + kResidRowBytes, src1, (uint32_t)bytes1, &S.full[slot]);
    }
  } else {
    if (bytes0) copy_plain(S.ring[slot], src0, bytes0, P.g.es, lane);
    if (bytes1) copy_plain(S.ring[slot] + kResidRowBytes, src1, bytes1, P.g.es, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.full[slot]);
  }
}

__device__ void producer(const DenseParams& P, Smem& S, int lane) {
  WsHeader* h = hdr_of(P);
  const int G = P.G, V = P.V, es = P.g.es;
  uint32_t seq = 0, useq = 0;
  bool ok = true;

  auto acquire = [&](uint32_t s) -> bool {
    if (s < (uint32_t)kNS) return true;
    return wait_phase(&S.empty[s % kNS], ((s / kNS) - 1) & 1, P);
  };

  while (ok) {
    unsigned long long t = 0;
    if (lane == 0) t = atomicAdd(&h->ticket, 1ull);
    t = __shfl_sync(0xffffffffu, t, 0);
    if ((long long)t >= P.tickets) break;
    if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) break;
    const Unit u = decode_ticket((long long)t, P);
    if (!u.resid) {
      const int npc = min(kUnitPieces, P.g.np_s - u.c * kUnitPieces);
      const int up = (u.j < G) ? 2 * npc : npc;
      const int uslot = useq % kNS;
      ++useq;
      for (int pi = 0; pi < up; ++pi) {
        const int isd = pi >= npc;
        const int kp = u.c * kUnitPieces + (isd ? pi - npc : pi);
        const int ne = min(P.g.pe, V - kp * P.g.pe);
        const unsigned char* row = isd ? draft_row(P, u.b, u.j) : target_row(P, u.b, u.j);
        if (!(ok = acquire(seq))) break;
        const int slot = seq % kNS;
        if (lane == 0) {
          StageMeta& m = S.meta[slot];
          m.kind = isd ? kStatsD : kStatsT;
          m.b = u.b;
          m.j = u.j;
          m.kp = kp;
          m.ne = ne;
          m.uslot = uslot;
          m.upieces = up;
          m.pidx = pi;
          m.unit_c = u.c;
          m.npc = npc;
        }
        issue_stage(P, S, slot, row + (size_t)kp * kPieceBytes, ne * es, nullptr, 0, lane);
        ++seq;
      }
    } else {
      uint32_t rdy = 1;
      if (lane == 0) rdy = wait_ready(P, u.b) ? 1u : 0u;
      rdy = __shfl_sync(0xffffffffu, rdy, 0);
      __syncwarp();
      if (!rdy) {
        ok = false;
        break;
      }
      const StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + u.b);
      const int npc = min(kUnitPieces, P.g.np_r - u.c * kUnitPieces);
      const int uslot = useq % kNS;
      ++useq;
      const unsigned char* trow = target_row(P, u.b, st.n);
      const unsigned char* drow = (st.mode == 0) ? draft_row(P, u.b, st.n) : nullptr;
      for (int pi = 0; pi < npc; ++pi) {
        const int kp = u.c * kUnitPieces + pi;
        const int ne = min(P.g.re, V - kp * P.g.re);
        if (!(ok = acquire(seq))) break;
        const int slot = seq % kNS;
        if (lane == 0) {
          StageMeta& m = S.meta[slot];
          m.kind = (st.mode == 2) ? kResidSkip : kResid;
          m.b = u.b;
          m.j = st.n;
          m.kp = kp;
          m.ne = ne;
          m.uslot = uslot;
          m.upieces = npc;
          m.pidx = pi;
          m.unit_c = u.c;
          m.npc = npc;
          m.mode = st.mode;
          m.ct = st.ct;
          m.cd = st.cd;
          m.invSt = st.invSt;
          m.invSd = st.invSd;
        }
        if (st.mode == 2) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.full[slot]);
        } else {
          const size_t off = (size_t)kp * kResidRowBytes;
          issue_stage(P, S, slot, trow + off, ne * es, drow ? drow + off : nullptr,
                      drow ? ne * es : 0, lane);
        }
        ++seq;
      }
    }
  }
  // one end marker per consumer warp
  for (int w = 0; w < kNW && ok; ++w) {
    if (!(ok = acquire(seq))) break;
    const int slot = seq % kNS;
    if (lane == 0) {
      S.meta[slot].kind = kEnd;
      mbar_arrive(&S.full[slot]);
    }
    ++seq;
  }
  // never leave the CTA with bulk copies in flight
  if (lane == 0) {
    const uint32_t first = seq > (uint32_t)kNS ? seq - kNS : 0u;
    for (uint32_t s = first; s < seq; ++s) {
      const int slot = s % kNS;
      if (!mbar_try_wait(&S.full[slot], (s / kNS) & 1)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&S.full[slot], (s / kNS) & 1) && clock64() - t0 < P.wait_bound) {
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// consumer: statistics of one 4 KB piece
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stats_piece(const unsigned char* slot, int ne, int bf16, int lane,
                                            float& c_out, float& s_out) {
  const uint4* v = reinterpret_cast<const uint4*>(slot);
  constexpr uint32_t kNegInf2 = 0xFF80FF80u;  // two bf16 -inf
  uint4 r[8];
  const int epv = bf16 ? 8 : 4;  // elements per 16-byte vector
  const int nv = (ne + epv - 1) / epv;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int vi = lane + 32 * i;
    if (vi < nv) {
      r[i] = v[vi];
      const int rem = ne - vi * epv;  // valid elements in this vector
      if (rem < epv) {                // ragged tail: mask to -inf
        uint32_t* w = reinterpret_cast<uint32_t*>(&r[i]);
        if (bf16) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e >= rem) {
              uint32_t& ww = w[e >> 1];
              ww = (e & 1) ? ((ww & 0x0000FFFFu) | 0xFF800000u) : ((ww & 0xFFFF0000u) | 0xFF80u);
            }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (e >= rem) w[e] = 0xFF800000u;
        }
      }
    } else {
      r[i] = bf16 ? make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2)
                  : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    }
  }
  float m;
  if (bf16) {
    uint32_t mx = kNegInf2;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(r[i].x, r[i].y), bf16x2_max(r[i].z, r[i].w)));
    m = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(r[i].x), __uint_as_float(r[i].y)),
                         fmaxf(__uint_as_float(r[i].z), __uint_as_float(r[i].w))));
  }
  m = warp_max(m);
  // c = log2e * max; an all -inf piece keeps c = 0 so NaN inputs still poison s
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (bf16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
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
    for (int i = 0; i < 8; ++i) {
      a0 += ex2(fmaf(__uint_as_float(r[i].x), kLog2e, -c));
      a1 += ex2(fmaf(__uint_as_float(r[i].y), kLog2e, -c));
      a2 += ex2(fmaf(__uint_as_float(r[i].z), kLog2e, -c));
      a3 += ex2(fmaf(__uint_as_float(r[i].w), kLog2e, -c));
    }
  }
  s_out = warp_sum((a0 + a1) + (a2 + a3));
  c_out = (m == -INFINITY) ? -INFINITY : c;
}

// residual (or p) mass of one residual piece: target at slot[0..], draft at slot[2048..]
__device__ __forceinline__ float resid_piece(const unsigned char* slot, const StageMeta& m,
                                             int bf16, int lane) {
  float acc = 0.f;
  const int epv = bf16 ? 8 : 4;
  const int nv = (m.ne + epv - 1) / epv;
  const uint4* tv = reinterpret_cast<const uint4*>(slot);
  const uint4* dv = reinterpret_cast<const uint4*>(slot + kResidRowBytes);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vi = lane + 32 * i;
    if (vi >= nv) continue;
    const uint4 t4 = tv[vi];
    const uint4 d4 = (m.mode == 0) ? dv[vi] : make_uint4(0, 0, 0, 0);
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(&t4);
    const uint32_t* dw = reinterpret_cast<const uint32_t*>(&d4);
    const int rem = m.ne - vi * epv;
    if (bf16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e < rem) {
          const float t = (e & 1) ? bf16_hi(tw[e >> 1]) : bf16_lo(tw[e >> 1]);
          const float d = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
          acc += resid_val(t, d, m.ct, m.cd, m.invSt, m.invSd, m.mode);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < rem)
          acc += resid_val(__uint_as_float(tw[e]), __uint_as_float(dw[e]), m.ct, m.cd, m.invSt,
                           m.invSd, m.mode);
      }
    }
  }
  return warp_sum(acc);
}

// ---------------------------------------------------------------------------
// hand-offs: position -> row -> residual -> token
// ---------------------------------------------------------------------------
__device__ void final_select(const DenseParams& P, int b, int lane);

__device__ void finalize_row(const DenseParams& P, int b, int lane) {
  __threadfence();
  const int G = P.G;
  const PosInfo* pp = ws_at<PosInfo>(P, P.L.pos) + (size_t)b * (G + 1);
  int n = G, err = 0;
  for (int j0 = 0; j0 <= G; j0 += 32) {
    const int j = j0 + lane;
    int e = 0, rej = 0;
    if (j <= G) {
      const PosInfo q = ldcg32(pp + j);
      e = q.err;
      rej = (j < G) && !q.accept;
    }
    err |= __any_sync(0xffffffffu, e);
    const unsigned bal = __ballot_sync(0xffffffffu, rej);
    if (bal && n == G) n = j0 + __ffs(bal) - 1;
  }
  if (lane == 0) {
    StopInfo st;
    st.n = n;
    st.T = 0.0;
    if (err) {
      st.mode = 2;
      st.ct = st.cd = st.invSt = st.invSd = 0.f;
    } else if (n < G) {
      const PosInfo q = ldcg32(pp + n);
      st.mode = 0;
      st.ct = q.ct;
      st.cd = q.cd;
      st.invSt = (float)(1.0 / q.St);
      st.invSd = (float)(1.0 / q.Sd);
    } else {
      const PosInfo q = ldcg32(pp + G);
      st.mode = 1;
      st.ct = q.ct;
      st.cd = 0.f;
      st.invSt = (float)(1.0 / q.St);
      st.invSd = 0.f;
    }
    ws_at<StopInfo>(P, P.L.stop)[b] = st;
    ws_at<uint32_t>(P, P.L.cnt_row)[b] = 0;
    __threadfence();
    st_release_u32(ws_at<uint32_t>(P, P.L.ready) + b, 1u);
  }
  __syncwarp();
}

__device__ void finalize_position(const DenseParams& P, int b, int j, int lane) {
  __threadfence();
  const int G = P.G, nc = P.g.nc_s;
  const UnitPart* up = ws_at<UnitPart>(P, P.L.upart) + ((size_t)b * (G + 1) + j) * nc;
  float Ct = -INFINITY, Cd = -INFINITY;
  for (int k = lane; k < nc; k += 32) {
    const UnitPart u = ldcg32(up + k);
    Ct = fmaxf(Ct, u.ct);
    Cd = fmaxf(Cd, u.cd);
  }
  Ct = warp_max(Ct);
  Cd = warp_max(Cd);
  double St = 0.0, Sd = 0.0;
  for (int k = lane; k < nc; k += 32) {
    const UnitPart u = ldcg32(up + k);
    St += u.St * (double)part_scale(u.ct, Ct);
    Sd += u.Sd * (double)part_scale(u.cd, Cd);
  }
  St = warp_sum_d(St);
  Sd = warp_sum_d(Sd);
  int err = !(Ct > -INFINITY && Ct < INFINITY && St > 0.0 && St < INFINITY);
  if (j < G) err |= !(Cd > -INFINITY && Cd < INFINITY && Sd > 0.0 && Sd < INFINITY);
  int acc = 0;
  double a = 0.0;
  if (j < G) {
    const int x = P.x[(size_t)b * G + j];
    if (x < 0 || x >= P.V) err = 1;
    if (!err) {
      const float tx = load_logit(target_row(P, b, j), x, P.bf16);
      const float dx = load_logit(draft_row(P, b, j), x, P.bf16);
      const double L = (double)kLog2e;
      const double p = (tx == -INFINITY) ? 0.0 : exp2((double)tx * L - (double)Ct) / St;
      const double q = (dx == -INFINITY) ? 0.0 : exp2((double)dx * L - (double)Cd) / Sd;
      const double ratio = (q > 0.0) ? p / q : 0.0;
      a = ratio < 1.0 ? ratio : 1.0;
      acc = (double)P.u_acc[(size_t)b * G + j] < a;
    }
  }
  int row_done = 0;
  if (lane == 0) {
    PosInfo pi;
    pi.St = St;
    pi.Sd = Sd;
    pi.ct = Ct;
    pi.cd = Cd;
    pi.accept = acc;
    pi.err = err;
    ws_at<PosInfo>(P, P.L.pos)[(size_t)b * (G + 1) + j] = pi;
    if (P.acc_out && j < G) P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : (float)a;
    if (err) atomicOr(&hdr_of(P)->status, kStatusInputErr);
    ws_at<uint32_t>(P, P.L.cnt_pos)[(size_t)b * (G + 1) + j] = 0;
    __threadfence();
    const unsigned o = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_row) + b, 1u);
    row_done = (o == (unsigned)G);
  }
  row_done = __shfl_sync(0xffffffffu, row_done, 0);
  if (row_done) finalize_row(P, b, lane);
}

// Select the token of row b from its per-piece masses (fp64 prefix over
// pieces, then over the fp32 element values of the chosen piece).
__device__ void final_select(const DenseParams& P, int b, int lane) {
  __threadfence();
  const int G = P.G, V = P.V, np = P.g.np_r, re = P.g.re;
  StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  float* rm = ws_at<float>(P, P.L.rmass) + (size_t)b * np;
  const int n = st.n;
  int y = -1;
  double T = 0.0;
  if (st.mode != 2) {
    const unsigned char* trow = target_row(P, b, n);
    const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, n) : nullptr;
    const int per = (np + 31) / 32;
    for (int attempt = 0; attempt < 2; ++attempt) {
      const int k0 = min(np, lane * per), k1 = min(np, k0 + per);
      double ls = 0.0;
      for (int k = k0; k < k1; ++k) ls += (double)__ldcg(rm + k);
      const double ex = warp_exclusive_scan_d(ls, lane);
      T = __shfl_sync(0xffffffffu, ex + ls, 31);
      if (!(T > 0.0) && st.mode == 0 && attempt == 0) {
        // zero residual after a rejection (only through rounding): draw from p_n
        st.mode = 1;
        drow = nullptr;
        for (int k = 0; k < np; ++k) {
          const int y0 = k * re, ne = min(re, V - y0);
          float s = 0.f;
          for (int e = lane; e < ne; e += 32)
            s += resid_val(load_logit(trow, y0 + e, P.bf16), 0.f, st.ct, st.cd, st.invSt,
                           st.invSd, 1);
          s = warp_sum(s);
          if (lane == 0) rm[k] = s;
        }
        __threadfence();
        __syncwarp();
        continue;
      }
      break;
    }
    const double target = (double)P.u_s[b] * T;
    // piece level
    const int k0 = min(np, lane * per), k1 = min(np, k0 + per);
    double ls = 0.0;
    for (int k = k0; k < k1; ++k) ls += (double)__ldcg(rm + k);
    const double ex = warp_exclusive_scan_d(ls, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, (k1 > k0) && (ex + ls > target));
    int kstar = -1;
    double base = 0.0;
    bool clamp = false;
    if (hit) {
      const int fl = __ffs(hit) - 1;
      if (lane == fl) {
        double acc = ex;
        for (int k = k0; k < k1; ++k) {
          const double mk = (double)__ldcg(rm + k);
          if (acc + mk > target) {
            kstar = k;
            base = acc;
            break;
          }
          acc += mk;
        }
        if (kstar < 0) {  // rounding between the two sums: last piece of the lane
          kstar = k1 - 1;
          base = acc - (double)__ldcg(rm + kstar);
        }
      }
      kstar = __shfl_sync(0xffffffffu, kstar, fl);
      base = __shfl_sync(0xffffffffu, base, fl);
    } else {
      clamp = true;  // u*T at or past the total: last piece with mass
      int last = -1;
      for (int k = k0; k < k1; ++k)
        if (__ldcg(rm + k) > 0.f) last = k;
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      kstar = last < 0 ? 0 : last;
    }
    // element level within piece kstar
    const int y0 = kstar * re, ne = min(re, V - y0);
    const int q = (ne + 31) / 32;
    const int e0 = min(ne, lane * q), e1 = min(ne, e0 + q);
    double es = 0.0;
    int lastpos = -1;
    for (int e = e0; e < e1; ++e) {
      const float t = load_logit(trow, y0 + e, P.bf16);
      const float d = drow ? load_logit(drow, y0 + e, P.bf16) : 0.f;
      const float r = resid_val(t, d, st.ct, st.cd, st.invSt, st.invSd, st.mode);
      es += (double)r;
      if (r > 0.f) lastpos = e;
    }
    const double eex = warp_exclusive_scan_d(es, lane);
    const double tl = target - base;
    const unsigned ehit = clamp ? 0u : __ballot_sync(0xffffffffu, (e1 > e0) && (eex + es > tl));
    if (ehit) {
      const int fl = __ffs(ehit) - 1;
      if (lane == fl) {
        double acc = base + eex;
        for (int e = e0; e < e1; ++e) {
          const float t = load_logit(trow, y0 + e, P.bf16);
          const float d = drow ? load_logit(drow, y0 + e, P.bf16) : 0.f;
          acc += (double)resid_val(t, d, st.ct, st.cd, st.invSt, st.invSd, st.mode);
          if (acc > target) {
            y = y0 + e;
            break;
          }
        }
        if (y < 0) y = y0 + (lastpos >= 0 ? lastpos : e1 - 1);
      }
      y = __shfl_sync(0xffffffffu, y, fl);
    } else {
      int lp = lastpos;
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      y = y0 + (lp < 0 ? 0 : lp);
    }
  }
  // outputs
  const int nn = (st.mode == 2) ? -1 : n;
  for (int j = lane; j <= G; j += 32) {
    int v = -1;
    if (nn >= 0) v = (j < nn) ? P.x[(size_t)b * G + j] : (j == nn ? y : -1);
    tok[j] = v;
  }
  if (lane == 0) {
    P.n_out[b] = nn;
    StopInfo* sp = ws_at<StopInfo>(P, P.L.stop) + b;
    sp->mode = st.mode;
    sp->T = T;
    ws_at<uint32_t>(P, P.L.cnt_res)[b] = 0;
    ws_at<uint32_t>(P, P.L.ready)[b] = 0;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// consumer loop
// ---------------------------------------------------------------------------
__device__ void consumer(const DenseParams& P, Smem& S, int cw, int lane) {
  const int G = P.G;
  for (uint32_t s = cw;; s += kNW) {
    const int slot = s % kNS;
    if (!wait_phase(&S.full[slot], (s / kNS) & 1, P)) break;
    const StageMeta m = S.meta[slot];
    if (m.kind == kEnd) break;
    UnitSlot& U = S.unit[m.uslot];
    if (m.kind == kStatsT || m.kind == kStatsD) {
      float c, sm;
      stats_piece(S.ring[slot], m.ne, P.bf16, lane, c, sm);
      unsigned old = 0;
      if (lane == 0) {
        U.c[m.pidx] = c;
        U.s[m.pidx] = sm;
        __threadfence_block();
        old = atomicAdd(&U.count, 1u);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      int pos_done = 0;
      if (old == (unsigned)m.upieces - 1) {
        __threadfence_block();
        __syncwarp();
        const bool have = lane < m.upieces;
        const bool isd = lane >= m.npc;
        const float cl = have ? U.c[lane] : -INFINITY;
        const float sl = have ? U.s[lane] : 0.f;
        const float Ct = warp_max((have && !isd) ? cl : -INFINITY);
        const float Cd = warp_max((have && isd) ? cl : -INFINITY);
        const double wt = (have && !isd) ? (double)sl * (double)part_scale(cl, Ct) : 0.0;
        const double wd = (have && isd) ? (double)sl * (double)part_scale(cl, Cd) : 0.0;
        const double St = warp_sum_d(wt), Sd = warp_sum_d(wd);
        if (lane == 0) {
          UnitPart u;
          u.St = St;
          u.Sd = Sd;
          u.ct = Ct;
          u.cd = Cd;
          u.pad[0] = u.pad[1] = 0.f;
          ws_at<UnitPart>(P, P.L.upart)[((size_t)m.b * (G + 1) + m.j) * P.g.nc_s + m.unit_c] = u;
          U.count = 0;
          __threadfence();
          const unsigned o2 =
              atomicAdd(ws_at<uint32_t>(P, P.L.cnt_pos) + (size_t)m.b * (G + 1) + m.j, 1u);
          pos_done = (o2 == (unsigned)P.g.nc_s - 1);
        }
        pos_done = __shfl_sync(0xffffffffu, pos_done, 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (pos_done) finalize_position(P, m.b, m.j, lane);
    } else {
      const float mass = (m.kind == kResid) ? resid_piece(S.ring[slot], m, P.bf16, lane) : 0.f;
      unsigned old = 0;
      if (lane == 0) {
        U.s[m.pidx] = mass;
        __threadfence_block();
        old = atomicAdd(&U.count, 1u);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      int row_done = 0;
      if (lane == 0 && old == (unsigned)m.upieces - 1) {
        __threadfence_block();
        float* rm = ws_at<float>(P, P.L.rmass) + (size_t)m.b * P.g.np_r + m.unit_c * kUnitPieces;
        for (int k = 0; k < m.upieces; ++k) rm[k] = U.s[k];
        U.count = 0;
        __threadfence();
        const unsigned o2 = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_res) + m.b, 1u);
        row_done = (o2 == (unsigned)P.g.nc_r - 1);
      }
      row_done = __shfl_sync(0xffffffffu, row_done, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (row_done) final_select(P, m.b, lane);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) dense_verify_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
      S.unit[i].count = 0;
    }
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0)
    producer(P, S, lane);
  else
    consumer(P, S, warp - 1, lane);
  __syncthreads();
  if (threadIdx.x == 0) {
    WsHeader* h = hdr_of(P);
    __threadfence();
    const unsigned prev = atomicAdd(&h->exit_cnt, 1u);
    if (prev == gridDim.x - 1) {
      h->ticket = 0ull;
      h->exit_cnt = 0u;
      __threadfence();
    }
  }
}

// residual_out: the distribution the emitted token was drawn from
__global__ void dense_resid_out_kernel(const __grid_constant__ DenseParams P, float* out) {
  const int b = blockIdx.x;
  const StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
  float* o = out + (size_t)b * P.V;
  const int stride = gridDim.y * blockDim.x;
  const int first = blockIdx.y * blockDim.x + threadIdx.x;
  if (st.mode == 2 || !(st.T > 0.0)) {
    for (int y = first; y < P.V; y += stride) o[y] = 0.f;
    return;
  }
  const unsigned char* trow = target_row(P, b, st.n);
  const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, st.n) : nullptr;
  const double invT = 1.0 / st.T;
  for (int y = first; y < P.V; y += stride) {
    const float t = load_logit(trow, y, P.bf16);
    const float d = drow ? load_logit(drow, y, P.bf16) : 0.f;
    o[y] = (float)((double)resid_val(t, d, st.ct, st.cd, st.invSt, st.invSd, st.mode) * invT);
  }
}

}  // namespace

size_t dense_smem_bytes() { return sizeof(Smem); }
int dense_ctas_per_sm() { return 1; }

cudaError_t launch_dense(const DenseParams& p, int grid, cudaStream_t s) {
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(dense_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  dense_verify_kernel<<<grid, kThreads, sizeof(Smem), s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s) {
  const int threads = 256;
  int gy = (p.V + threads * 4 - 1) / (threads * 4);
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  dim3 grid(p.B, gy);
  dense_resid_out_kernel<<<grid, threads, 0, s>>>(p, resid_out);
  return cudaGetLastError();
}

}  // namespace sv
