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
//  * Statistics work is a stream of tickets in row order, taken with one
//    atomicAdd each (prefetched one ahead).  A statistics unit is up to
//    8 x 4 KB pieces of the target row (b, j) plus the same pieces of the
//    draft row (b, j).  When a row's statistics are complete its finaliser
//    publishes the row's residual units -- up to 8 pieces of 2 KB target +
//    2 KB draft of the stop position (b, n) -- to a queue that producers
//    drain before taking new tickets.
//  * Each CTA = 1 producer warp + NW consumer warps + 1 finaliser warp around
//    an NS-stage ring of 4 KB shared-memory stages.  The producer moves pieces with 1-D bulk
//    copies (cp.async.bulk, TMA) completing on per-stage mbarriers; consumer
//    warp w takes stages w, w + NW, ...  A consumer releases its stage as soon
//    as the data is in registers, so slow bookkeeping never holds the ring.
//  * A consumer warp reduces a 4 KB piece to (c, s): c = log2e * max, s =
//    sum 2^(v*log2e - c) (MUFU ex2).  The last warp of a unit combines the
//    unit's pieces and publishes one partial; the last unit of a row runs all
//    of the row's accept tests (one lane per position), finds the first
//    rejection n and publishes the stop constants.  These
//    hand-offs are last-arriver atomics; the consumer that completes a row
//    queues the row for its CTA's finaliser warp, so the latency of the
//    row-level work never stalls the data pipeline.  No warp ever waits for
//    another CTA
//    while it holds statistics work.  A producer waits (bounded) for a queue
//    entry only once every statistics ticket is taken; every such entry is
//    published by a row whose statistics units are all held by running CTAs
//    that never wait, so the wait always ends.
//  * Residual units recompute r(y) = max(p(y) - q(y), 0) for the stop
//    position only (the rows are still in L2: they were read a few rows of
//    work earlier) and publish per-piece masses; the last one selects the
//    piece and then the token by a float-float prefix over fp32 element values.
#include "sv_common.cuh"

namespace sv {
namespace {

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

constexpr int kFinQ = 64;  // finaliser queue entries

template <int NS, int NW>
struct Smem {
  // Stage s lives in slot s % NS and is consumed by warp s % NW.  With NS a
  // multiple of NW the stage that last used a slot (s - NS) belongs to the
  // same warp, which consumed it first; a warp can therefore never wait on a
  // slot two phases ahead, where an mbarrier parity wait would alias.
  static_assert(NS % NW == 0, "ring depth must be a multiple of the consumer warps");
  static constexpr int NU = 2 * NS;  // unit slots
  alignas(128) unsigned char ring[NS][kPieceBytes];
  uint64_t full[NS];
  uint64_t empty[NS];
  uint64_t ufree[NU];
  StageMeta meta[NS];
  UnitSlot unit[NU];
  // consumer -> finaliser hand-off: +(b+1) finalise row b, -(b+1) select its token
  UnitPart fin_scratch[128];  // finaliser staging (4 KB)
  int fin_item[kFinQ];
  unsigned fin_seq[kFinQ];
  unsigned fin_tail;
  unsigned fin_head;
  unsigned cons_done;
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
// bounded waits (every spin has a limit; on expiry: timeout + abort flags and
// the first expired site recorded in the header for diagnosis)
// ---------------------------------------------------------------------------
enum WaitSite : unsigned {
  kSiteProdEmpty = 1, kSiteProdUnit = 2, kSiteEntry = 4, kSiteConsFull = 5, kSiteFinPush = 6,
  kSiteFinIdle = 7
};

__device__ void record_timeout(const DenseParams& P, unsigned site, unsigned info) {
  WsHeader* h = hdr_of(P);
  if (atomicCAS(&h->timeout_site, 0u, site) == 0u) h->timeout_info = info;
  atomicOr(&h->status, kStatusTimeout);
  atomicExch(&h->abort, 1u);
}

__device__ bool wait_phase(uint64_t* bar, uint32_t parity, const DenseParams& P, unsigned site,
                           unsigned info) {
  if (mbar_try_wait(bar, parity)) return true;
  WsHeader* h = hdr_of(P);
  const long long t0 = clock64();
  unsigned it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) return false;
      if (clock64() - t0 > P.wait_bound) {
        record_timeout(P, site, info);
        return false;
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// ticket -> work unit
// ---------------------------------------------------------------------------
struct Unit {
  int b, j, c;
};

__device__ __forceinline__ Unit decode_ticket(long long t, const DenseParams& P) {
  Unit u;
  if (P.small_tickets)
    dense_ticket_fast((unsigned)t, P.tk, &u.b, &u.j, &u.c);
  else
    dense_ticket(t, P.G, P.g.nc_s, &u.b, &u.j, &u.c);
  return u;
}

// residual queue entry: (row + 1) << 32 | unit, 0 while unpublished
__device__ __forceinline__ unsigned long long* rq_of(const DenseParams& P) {
  return ws_at<unsigned long long>(P, P.L.rq);
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// producer lane 0: wait until residual queue entry i is published (bounded)
__device__ unsigned long long wait_entry(const DenseParams& P, unsigned i) {
  const unsigned long long* e = rq_of(P) + i;
  unsigned long long v = ld_acquire_u64(e);
  if (v) return v;
  WsHeader* h = hdr_of(P);
  const long long t0 = clock64();
  while (!(v = ld_acquire_u64(e))) {
    if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) return 0;
    if (clock64() - t0 > P.wait_bound) {
      record_timeout(P, kSiteEntry, i);
      return 0;
    }
    nanosleep_ns(64);
  }
  return v;
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
template <int NS, int NW>
__device__ __forceinline__ void issue_stage(const DenseParams& P, Smem<NS, NW>& S, int slot,
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

template <int NS, int NW>
__device__ void producer(const DenseParams& P, Smem<NS, NW>& S, int lane) {
  constexpr int NU = Smem<NS, NW>::NU;
  WsHeader* h = hdr_of(P);
  const int G = P.G, V = P.V, es = P.g.es;
  uint32_t seq = 0, useq = 0;
  bool ok = true;

  auto acquire = [&](uint32_t s) -> bool {
    if (s < (uint32_t)NS) return true;
    return wait_phase(&S.empty[s % NS], ((s / NS) - 1) & 1, P, kSiteProdEmpty, s);
  };
  auto acquire_unit = [&](uint32_t u) -> bool {
    if (u < (uint32_t)NU) return true;
    return wait_phase(&S.ufree[u % NU], ((u / NU) - 1) & 1, P, kSiteProdUnit, u);
  };
  // Stage i of a unit is issued by lane i: its own ring-slot wait, metadata,
  // expect-tx and bulk copy.  A lane issues as soon as its slot is free, so the
  // ring refills stage by stage rather than a whole unit at a time.  (Rows
  // that are not 16-byte aligned take the warp-wide plain-copy path.)
  auto lane_acquire = [&](bool mine, uint32_t s) -> bool {
    bool ok_l = true;
    if (mine && s >= (uint32_t)NS)
      ok_l = wait_phase(&S.empty[s % NS], ((s / NS) - 1) & 1, P, kSiteProdEmpty, s);
    return __all_sync(0xffffffffu, ok_l);
  };
  // run issue(lane) on every lane with `mine` as soon as its stage's slot is free
  auto lane_issue = [&](bool mine, uint32_t s, auto&& issue) -> bool {
    bool pending = mine;
    if (pending && s < (uint32_t)NS) {
      issue();
      pending = false;
    }
    const long long t0 = clock64();
    unsigned it = 0;
    while (__any_sync(0xffffffffu, pending)) {
      if (pending && mbar_test_wait(&S.empty[s % NS], ((s / NS) - 1) & 1)) {
        issue();
        pending = false;
      }
      if ((++it & 63u) == 0) {
        bool stop = *reinterpret_cast<volatile uint32_t*>(&h->abort) != 0;
        if (!stop && clock64() - t0 > P.wait_bound) {
          if (pending) record_timeout(P, kSiteProdEmpty, s);
          stop = true;
        }
        if (__any_sync(0xffffffffu, stop)) return false;
      }
    }
    return true;
  };

  auto issue_stats = [&](const Unit& u) -> bool {
    if (!acquire_unit(useq)) return false;
    const int uslot = useq % NU;
    ++useq;
    const int npc = min(kUnitPieces, P.g.np_s - u.c * kUnitPieces);
    const int up = (u.j < G) ? 2 * npc : npc;
    if (P.aligned) {
      const int pi = lane;
      const bool mine = pi < up;
      const uint32_t sq = seq + (uint32_t)pi;
      const bool ok_i = lane_issue(mine, sq, [&]() {
        const int isd = pi >= npc;
        const int kp = u.c * kUnitPieces + (isd ? pi - npc : pi);
        const int ne = min(P.g.pe, V - kp * P.g.pe);
        const unsigned char* row = isd ? draft_row(P, u.b, u.j) : target_row(P, u.b, u.j);
        const int slot = sq % NS;
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
        mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(ne * es));
        bulk_g2s(S.ring[slot], row + (size_t)kp * kPieceBytes, (uint32_t)(ne * es), &S.full[slot]);
      });
      seq += (uint32_t)up;
      return ok_i;
    }
    for (int pi = 0; pi < up; ++pi) {
      const int isd = pi >= npc;
      const int kp = u.c * kUnitPieces + (isd ? pi - npc : pi);
      const int ne = min(P.g.pe, V - kp * P.g.pe);
      const unsigned char* row = isd ? draft_row(P, u.b, u.j) : target_row(P, u.b, u.j);
      if (!acquire(seq)) return false;
      const int slot = seq % NS;
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
    return true;
  };

  // residual unit (b, c) of a row whose stop constants are published
  auto issue_resid = [&](int b, int c) -> bool {
    if (!acquire_unit(useq)) return false;
    const int uslot = useq % NU;
    ++useq;
    const StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
    const int npc = min(kUnitPieces, P.g.np_r - c * kUnitPieces);
    const unsigned char* trow = target_row(P, b, st.n);
    const unsigned char* drow = (st.mode == 0) ? draft_row(P, b, st.n) : nullptr;
    auto fill_meta = [&](StageMeta& m, int kp, int ne, int pi) {
      m.kind = (st.mode == 2) ? kResidSkip : kResid;
      m.b = b;
      m.j = st.n;
      m.kp = kp;
      m.ne = ne;
      m.uslot = uslot;
      m.upieces = npc;
      m.pidx = pi;
      m.unit_c = c;
      m.npc = npc;
      m.mode = st.mode;
      m.ct = st.ct;
      m.cd = st.cd;
      m.invSt = st.invSt;
      m.invSd = st.invSd;
    };
    if (P.aligned || st.mode == 2) {
      const int pi = lane;
      const bool mine = pi < npc;
      const uint32_t sq = seq + (uint32_t)pi;
      const bool ok_i = lane_issue(mine, sq, [&]() {
        const int kp = c * kUnitPieces + pi;
        const int ne = min(P.g.re, V - kp * P.g.re);
        const int slot = sq % NS;
        fill_meta(S.meta[slot], kp, ne, pi);
        if (st.mode == 2) {
          mbar_arrive(&S.full[slot]);
        } else {
          const size_t off = (size_t)kp * kResidRowBytes;
          const uint32_t bytes = (uint32_t)(ne * es);
          mbar_arrive_expect_tx(&S.full[slot], drow ? 2 * bytes : bytes);
          bulk_g2s(S.ring[slot], trow + off, bytes, &S.full[slot]);
          if (drow) bulk_g2s(S.ring[slot] + kResidRowBytes, drow + off, bytes, &S.full[slot]);
        }
      });
      seq += (uint32_t)npc;
      return ok_i;
    }
    for (int pi = 0; pi < npc; ++pi) {
      const int kp = c * kUnitPieces + pi;
      const int ne = min(P.g.re, V - kp * P.g.re);
      if (!acquire(seq)) return false;
      const int slot = seq % NS;
      if (lane == 0) fill_meta(S.meta[slot], kp, ne, pi);
      const size_t off = (size_t)kp * kResidRowBytes;
      issue_stage(P, S, slot, trow + off, ne * es, drow ? drow + off : nullptr,
                  drow ? ne * es : 0, lane);
      ++seq;
    }
    return true;
  };

  // Work loop.  Ready residual work (published by row finalisers) is taken
  // first -- its rows were just read and are still in L2 -- otherwise the next
  // statistics ticket.  Every global round trip of the loop (the next ticket,
  // the queue counters, a queue claim, the value of a claimed entry) is issued
  // by lane 0 one iteration ahead and consumed in the next, so while
  // statistics work remains the producer never stalls on a round trip.  A
  // claimed entry that is not yet published is waited for only when no
  // statistics ticket is left.
  enum : int { kActStats = 0, kActResid = 1, kActWait = 2, kActClaim = 3, kActDone = 4 };
  constexpr uint32_t kNone = 0xffffffffu;
  WsHeader* hq = h;
  unsigned long long next = 0;     // prefetched statistics ticket
  uint32_t v_head = 0, v_res = 0;  // queue counters seen one iteration ago
  uint32_t claim = kNone;          // queue claim issued last iteration
  unsigned long long ev = 0;       // entry[held] as loaded last iteration
  long long held = -1;             // claimed queue entry not yet issued
  if (lane == 0) {
    next = atomicAdd(&h->ticket, 1ull);
    v_head = ld_relaxed_u32(&hq->rq_head);
    v_res = ld_relaxed_u32(&hq->rq_reserve);
  }
  while (ok) {
    if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) {
      ok = false;
      break;
    }
    int act = kActStats;
    if (lane == 0) {
      const bool stats_left = (long long)next < P.tickets;
      if (claim != kNone) {  // resolve last iteration's claim
        if (claim < P.resid_units) {
          held = claim;
          ev = 0;  // its value is loaded below, for the next iteration
        } else if (!stats_left) {
          act = kActDone;  // every residual unit is claimed
        }
        claim = kNone;
      }
      if (act != kActDone) {
        if (held >= 0 && ev != 0)
          act = kActResid;
        else if (held >= 0 && !stats_left)
          act = kActWait;
        else if (stats_left)
          act = kActStats;
        else
          act = kActClaim;
      }
    }
    act = __shfl_sync(0xffffffffu, act, 0);
    if (act == kActDone) break;
    if (act == kActResid || act == kActWait) {
      unsigned long long e = 0;
      if (lane == 0) {
        // acquire: the row's stop record was written before the entry
        e = (act == kActWait) ? wait_entry(P, (unsigned)held) : ld_acquire_u64(rq_of(P) + held);
        if (e) rq_of(P)[held] = 0ull;  // self-reset for the next call
        held = -1;
      }
      e = __shfl_sync(0xffffffffu, e, 0);
      __syncwarp();
      if (!e) {  // the bounded wait ran out
        ok = false;
        break;
      }
      ok = issue_resid((int)(e >> 32) - 1, (int)(e & 0xffffffffu));
    } else if (act == kActStats) {
      const unsigned long long t = __shfl_sync(0xffffffffu, next, 0);
      if (lane == 0) next = atomicAdd(&h->ticket, 1ull);  // next ticket, used next iteration
      ok = issue_stats(decode_ticket((long long)t, P));
    } else {  // kActClaim: no statistics left; the claim resolves next iteration
      if (lane == 0) claim = atomicAdd(&hq->rq_head, 1u);
    }
    // round trips for the next iteration
    if (lane == 0) {
      if (held >= 0) {
        ev = ld_relaxed_u64(rq_of(P) + held);
      } else if (claim == kNone && v_head < v_res && (long long)next < P.tickets) {
        claim = atomicAdd(&hq->rq_head, 1u);  // published work is waiting: claim one
      }
      v_head = ld_relaxed_u32(&hq->rq_head);
      v_res = ld_relaxed_u32(&hq->rq_reserve);
    }
  }
  // one end marker per consumer warp (lane w marks the stage consumer w takes next)
  static_assert(NW <= 32, "one lane per consumer warp");
  if (ok) {
    const bool mine = lane < NW;
    const uint32_t sq = seq + (uint32_t)lane;
    ok = lane_acquire(mine, sq);
    if (ok && mine) {
      const int slot = sq % NS;
      S.meta[slot].kind = kEnd;
      mbar_arrive(&S.full[slot]);
    }
    seq += NW;
  }
  // never leave the CTA with bulk copies in flight
  if (lane == 0) {
    const uint32_t first = seq > (uint32_t)NS ? seq - NS : 0u;
    for (uint32_t s = first; s < seq; ++s) {
      const int slot = s % NS;
      if (!mbar_try_wait(&S.full[slot], (s / NS) & 1)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&S.full[slot], (s / NS) & 1) && clock64() - t0 < P.wait_bound) {
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// consumer: statistics of one 4 KB piece.  Releases the stage (`release`)
// as soon as every loaded register has been consumed.
// ---------------------------------------------------------------------------
template <class Release>
__device__ __forceinline__ void stats_piece(const unsigned char* slot, int ne, int bf16, int lane,
                                            float& c_out, float& s_out, Release release) {
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
  // every loaded register has been read by the max: hand the stage back
  release();
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
// Last statistics unit of row b: combine every position's unit partials, run
// all accept tests (lane j = position j), find the first rejection n
// and publish the stop constants.  The row's partials are staged through a
// 4 KB shared-memory scratch with one cooperative load per round, so the
// whole hand-off costs a few global round trips.
constexpr int kFinScratch = 128;  // unit partials (4 KB)

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
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

__device__ void finalize_row(const DenseParams& P, int b, int lane, UnitPart* scr) {
  fence_acq_rel_gpu();
  const int G = P.G, nc = P.g.nc_s;
  UnitPart* up_row = ws_at<UnitPart>(P, P.L.upart) + (size_t)b * (G + 1) * nc;
  // reserve the row's queue entries now; the result is needed only at the end
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(&hdr_of(P)->rq_reserve, (unsigned)P.g.nc_r);
  int n = G, err_any = 0, have_stop = 0;
  float s_ct = 0.f, s_cd = 0.f, s_St = 1.f, s_Sd = 1.f;
  for (int j0 = 0; j0 <= G; j0 += 32) {
    const int j = j0 + lane;
    const bool on = j <= G;
    const int npos = min(32, G + 1 - j0);
    int err = 0, x = 0;
    float uacc = 0.f;
    if (on && j < G) {
      x = P.x[(size_t)b * G + j];
      uacc = P.u_acc[(size_t)b * G + j];
    }
    float Ct = -INFINITY, Cd = -INFINITY;
    ff St{0.f, 0.f}, Sd{0.f, 0.f};
    const int kstep = max(1, kFinScratch / npos);
    bool gathered = false;
    float tx = 0.f, dx = 0.f;
    for (int k0 = 0; k0 < nc; k0 += kstep) {
      const int kn = min(kstep, nc - k0);
      const int total = npos * kn;  // <= kFinScratch
      // cooperative copy of this round's partials into the scratch: every
      // copy in flight at once (cp.async, no registers), then zero the source
      __syncwarp();  // the previous round's reads of the scratch are done
      for (int f = lane; f < total; f += 32) {
        const int pp = f / kn, kk = f - pp * kn;
        const unsigned char* q =
            reinterpret_cast<const unsigned char*>(up_row + (size_t)(j0 + pp) * nc + k0 + kk);
        cp_async16(scr + f, q);
        cp_async16(reinterpret_cast<unsigned char*>(scr + f) + 16, q + 16);
      }
      if (!gathered) {  // the gather at the draft token, overlapping the copies
        gathered = true;
        if (on && j < G) {
          if (x < 0 || x >= P.V) {
            err = 1;
          } else {
            tx = load_logit(target_row(P, b, j), x, P.bf16);
            dx = load_logit(draft_row(P, b, j), x, P.bf16);
          }
        }
      }
      cp_async_wait_all();
      for (int f = lane; f < total; f += 32) {  // consumed: leave the workspace zero
        const int pp = f / kn, kk = f - pp * kn;
        int4* q = reinterpret_cast<int4*>(up_row + (size_t)(j0 + pp) * nc + k0 + kk);
        q[0] = make_int4(0, 0, 0, 0);
        q[1] = make_int4(0, 0, 0, 0);
      }
      __syncwarp();
      if (on)
        for (int k = 0; k < kn; ++k) combine_part(scr[lane * kn + k], Ct, St, Cd, Sd);
    }
    const float Stf = ff_to_f(St), Sdf = ff_to_f(Sd);
    if (on) {
      err |= !(Ct > -INFINITY && Ct < INFINITY && Stf > 0.f && Stf < INFINITY);
      if (j < G) err |= !(Cd > -INFINITY && Cd < INFINITY && Sdf > 0.f && Sdf < INFINITY);
    }
    int acc = 1;
    float a = 0.f;
    if (on && j < G && !err) {
      // p/q = 2^((tx L - Ct) - (dx L - Cd)) * (Sd / St); the exponent is formed
      // exactly (two-product) and rounded once
      float ratio = 0.f;
      if (tx > -INFINITY && dx > -INFINITY) {
        const ff ea = ff_add_f(two_prod(tx, kLog2e), -Ct);
        const ff ed = ff_add_f(two_prod(dx, kLog2e), -Cd);
        ratio = exp2f(ff_to_f(ff_sub(ea, ed))) * __fdiv_rn(Sdf, Stf);
      }
      a = fminf(ratio, 1.f);
      acc = uacc < a;
    }
    if (on && j < G && P.acc_out) P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : a;
    err_any |= __any_sync(0xffffffffu, on && err);
    const unsigned rej = __ballot_sync(0xffffffffu, on && j < G && !acc);
    int src = -1;
    if (!have_stop && rej) {
      n = j0 + __ffs(rej) - 1;
      src = n - j0;
    } else if (!have_stop && G <= j0 + 31) {
      src = G - j0;  // no rejection anywhere: the bonus position
    }
    if (src >= 0) {
      have_stop = 1;
      s_ct = __shfl_sync(0xffffffffu, Ct, src);
      s_cd = __shfl_sync(0xffffffffu, Cd, src);
      s_St = __shfl_sync(0xffffffffu, Stf, src);
      s_Sd = __shfl_sync(0xffffffffu, Sdf, src);
    }
  }
  if (lane == 0) {
    StopInfo st;
    st.n = n;
    st.T = 0.0;
    if (err_any) {
      st.mode = 2;
      st.ct = st.cd = st.invSt = st.invSd = 0.f;
      atomicOr(&hdr_of(P)->status, kStatusInputErr);
    } else if (n < G) {
      st.mode = 0;
      st.ct = s_ct;
      st.cd = s_cd;
      st.invSt = __fdiv_rn(1.f, s_St);
      st.invSd = __fdiv_rn(1.f, s_Sd);
    } else {
      st.mode = 1;
      st.ct = s_ct;
      st.cd = 0.f;
      st.invSt = __fdiv_rn(1.f, s_St);
      st.invSd = 0.f;
    }
    ws_at<StopInfo>(P, P.L.stop)[b] = st;
    ws_at<uint32_t>(P, P.L.cnt_row)[b] = 0;
    fence_acq_rel_gpu();
  }
  // publish the row's residual units to the queue
  base = __shfl_sync(0xffffffffu, base, 0);
  __syncwarp();
  for (int c = lane; c < P.g.nc_r; c += 32)
    st_release_u64(rq_of(P) + base + c, ((unsigned long long)(b + 1) << 32) | (unsigned)c);
  __syncwarp();
}

// Select the token of row b from its per-piece masses (float-float prefix over
// pieces, then over the fp32 element values of the chosen piece).  The
// masses, then the chosen piece's logits, are staged in the shared scratch
// with cp.async: two global round trips.
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

template <int BF16>
__device__ void final_select(const DenseParams& P, int b, int lane, float* scr) {
  fence_acq_rel_gpu();
  const int G = P.G, V = P.V, np = P.g.np_r, re = P.g.re;
  float* rm = ws_at<float>(P, P.L.rmass) + (size_t)b * P.g.np_r4;
  constexpr int kScrFloats = 1024;  // 4 KB
  const bool staged = np <= kScrFloats;
  // the mass copies and the stop-record load are in flight together
  if (staged)
    for (int k = lane * 4; k < np; k += 128) cp_async16(scr + k, rm + k);
  StopInfo st = ldcg32(ws_at<StopInfo>(P, P.L.stop) + b);
  const float us = P.u_s[b];
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  const int n = st.n;
  int y = -1;
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
    for (int k = k0; k < k1; ++k) ls = ff_add_f(ls, mv[k]);
    ff ex = warp_exclusive_scan_ff(ls, lane);
    T = ff_shfl(ff_add(ex, ls), 31);
    if (!(T.hi > 0.f) && st.mode == 0) {
      // zero residual after a rejection (only through rounding): draw from p_n
      st.mode = 1;
      drow = nullptr;
      for (int k = 0; k < np; ++k) {
        const int y0 = k * re, ne = min(re, V - y0);
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
      fence_acq_rel_gpu();
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
    // the masses are consumed: leave the workspace zero for the next call
    for (int k = lane; k < np; k += 32) rm[k] = 0.f;
    __syncwarp();
    // element level within piece kstar: stage its target and draft slices
    const int y0 = kstar * re, ne = min(re, V - y0);
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
      const float r = piece_val<BF16>(tsm, dsm, e, st);
      es = ff_add_f(es, r);
      if (r > 0.f) lastpos = e;
    }
    const ff eex = warp_exclusive_scan_ff(es, lane);
    const ff tl = ff_sub(target, base);
    const unsigned ehit =
        clamp ? 0u : __ballot_sync(0xffffffffu, (e1 > e0) && ff_gt(ff_add(eex, es), tl));
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
  }
  if (st.mode == 2)  // an error row never reached the piece-level search
    for (int k = lane; k < np; k += 32) rm[k] = 0.f;
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
    if (P.keep_stop) {  // read (and cleared) by the residual-output kernel
      sp->mode = st.mode;
      sp->T = (double)T.hi + (double)T.lo;
    } else {
      int4* qq = reinterpret_cast<int4*>(sp);
      qq[0] = make_int4(0, 0, 0, 0);
      qq[1] = make_int4(0, 0, 0, 0);
    }
    ws_at<uint32_t>(P, P.L.cnt_res)[b] = 0;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// consumer loop
// ---------------------------------------------------------------------------
// queue a row hand-off for this CTA's finaliser warp (lane 0 of a consumer)
template <int NS, int NW>
__device__ __forceinline__ void fin_push(const DenseParams& P, Smem<NS, NW>& S, int item, int lane) {
  if (lane == 0) {
    const unsigned pos = atomicAdd(&S.fin_tail, 1u);
    // the queue has kFinQ entries; wait (bounded) while it is full
    const long long t0 = clock64();
    while (pos - *reinterpret_cast<volatile unsigned*>(&S.fin_head) >= (unsigned)kFinQ) {
      if (clock64() - t0 > P.wait_bound) {
        record_timeout(P, kSiteFinPush, pos);
        break;
      }
      nanosleep_ns(32);
    }
    S.fin_item[pos % kFinQ] = item;
    __threadfence_block();
    *reinterpret_cast<volatile unsigned*>(&S.fin_seq[pos % kFinQ]) = pos + 1;
  }
  __syncwarp();
}
template <int NS, int NW>
__device__ void consumer(const DenseParams& P, Smem<NS, NW>& S, int cw, int lane) {
  const int G = P.G;
  for (uint32_t s = cw;; s += NW) {
    const int slot = s % NS;
    if (!wait_phase(&S.full[slot], (s / NS) & 1, P, kSiteConsFull, s)) break;
    const StageMeta m = S.meta[slot];
    if (m.kind == kEnd) break;
    UnitSlot& U = S.unit[m.uslot];
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
    };
    if (m.kind == kStatsT || m.kind == kStatsD) {
      float c, sm;
      stats_piece(S.ring[slot], m.ne, P.bf16, lane, c, sm, release);
      unsigned old = 0;
      if (lane == 0) {
        U.c[m.pidx] = c;
        U.s[m.pidx] = sm;
        __threadfence_block();
        old = atomicAdd(&U.count, 1u);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      int row_done = 0;
      if (old == (unsigned)m.upieces - 1) {
        __threadfence_block();
        __syncwarp();
        const bool have = lane < m.upieces;
        const bool isd = lane >= m.npc;
        const float cl = have ? U.c[lane] : -INFINITY;
        const float sl = have ? U.s[lane] : 0.f;
        const float Ct = warp_max((have && !isd) ? cl : -INFINITY);
        const float Cd = warp_max((have && isd) ? cl : -INFINITY);
        const ff wt = (have && !isd) ? two_prod(sl, part_scale(cl, Ct)) : ff{0.f, 0.f};
        const ff wd = (have && isd) ? two_prod(sl, part_scale(cl, Cd)) : ff{0.f, 0.f};
        const ff St = warp_sum_ff(wt), Sd = warp_sum_ff(wd);
        if (lane == 0) {
          U.count = 0;
          mbar_arrive(&S.ufree[m.uslot]);
          UnitPart u;
          u.St_hi = St.hi;
          u.St_lo = St.lo;
          u.Sd_hi = Sd.hi;
          u.Sd_lo = Sd.lo;
          u.ct = Ct;
          u.cd = Cd;
          u.pad[0] = u.pad[1] = 0.f;
          ws_at<UnitPart>(P, P.L.upart)[((size_t)m.b * (G + 1) + m.j) * P.g.nc_s + m.unit_c] = u;
          fence_acq_rel_gpu();
          const unsigned o2 = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_row) + m.b, 1u);
          row_done = (o2 == (unsigned)((G + 1) * P.g.nc_s) - 1);
        }
        row_done = __shfl_sync(0xffffffffu, row_done, 0);
      }
      if (row_done) fin_push(P, S, m.b + 1, lane);
    } else {
      const float mass = (m.kind == kResid) ? resid_piece(S.ring[slot], m, P.bf16, lane) : 0.f;
      release();
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
        float* rm = ws_at<float>(P, P.L.rmass) + (size_t)m.b * P.g.np_r4 + m.unit_c * kUnitPieces;
        for (int k = 0; k < m.upieces; ++k) rm[k] = U.s[k];
        U.count = 0;
        mbar_arrive(&S.ufree[m.uslot]);
        fence_acq_rel_gpu();
        const unsigned o2 = atomicAdd(ws_at<uint32_t>(P, P.L.cnt_res) + m.b, 1u);
        row_done = (o2 == (unsigned)P.g.nc_r - 1);
      }
      row_done = __shfl_sync(0xffffffffu, row_done, 0);
      if (row_done) fin_push(P, S, -(m.b + 1), lane);
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    atomicAdd(&S.cons_done, 1u);
  }
}

// finaliser warp: runs the row hand-offs the consumers queue, in order
template <int NS, int NW>
__device__ void finaliser(const DenseParams& P, Smem<NS, NW>& S, int lane) {
  WsHeader* h = hdr_of(P);
  unsigned head = 0;
  long long t0 = clock64();
  for (;;) {
    int item = 0, state = 0;  // state 1: item, 2: done, 3: timeout/abort
    if (lane == 0) {
      const volatile unsigned* seq = S.fin_seq;
      if (seq[head % kFinQ] == head + 1) {
        __threadfence_block();
        item = S.fin_item[head % kFinQ];
        state = 1;
      } else if (*reinterpret_cast<volatile unsigned*>(&S.cons_done) == (unsigned)NW &&
                 *reinterpret_cast<volatile unsigned*>(&S.fin_tail) == head) {
        state = 2;
      } else if (*reinterpret_cast<volatile uint32_t*>(&h->abort)) {
        state = 3;
      } else if (clock64() - t0 > 4 * P.wait_bound) {
        // the finaliser only waits on its own CTA, whose waits have the
        // shorter bound: a longer one here lets the root cause report first
        record_timeout(P, kSiteFinIdle, head);
        state = 3;
      } else {
        nanosleep_ns(256);
      }
    }
    state = __shfl_sync(0xffffffffu, state, 0);
    if (state >= 2) break;
    if (state == 0) continue;
    item = __shfl_sync(0xffffffffu, item, 0);
    __syncwarp();
    if (item > 0) {
      finalize_row(P, item - 1, lane, S.fin_scratch);
    } else if (P.bf16) {
      final_select<1>(P, -item - 1, lane, reinterpret_cast<float*>(S.fin_scratch));
    } else {
      final_select<0>(P, -item - 1, lane, reinterpret_cast<float*>(S.fin_scratch));
    }
    ++head;
    if (lane == 0) *reinterpret_cast<volatile unsigned*>(&S.fin_head) = head;
    t0 = clock64();
  }
}

// register budget: each of the SM's four sub-partitions has 16K registers and
// holds ceil(warps / 4) of the resident warps
template <int NW, int CTAS>
constexpr int dense_regs() {
  constexpr int per_part = ((NW + 2) * CTAS + 3) / 4;
  constexpr int r = 16384 / (32 * per_part) / 8 * 8;
  return r > 255 ? 255 : r;
}

template <int NS, int NW, int CTAS>
__global__ void __maxnreg__((dense_regs<NW, CTAS>()))
    dense_verify_kernel(const __grid_constant__ DenseParams P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  using SM = Smem<NS, NW>;
  SM& S = *reinterpret_cast<SM*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < SM::NU; ++i) {
      mbar_init(&S.ufree[i], 1);
      S.unit[i].count = 0;
    }
    for (int i = 0; i < kFinQ; ++i) S.fin_seq[i] = 0u;
    S.fin_tail = S.fin_head = S.cons_done = 0u;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0)
    producer(P, S, lane);
  else if (warp <= NW)
    consumer(P, S, warp - 1, lane);
  else
    finaliser(P, S, lane);
  __syncthreads();
  if (threadIdx.x == 0) {
    WsHeader* h = hdr_of(P);
    fence_acq_rel_gpu();
    const unsigned prev = atomicAdd(&h->exit_cnt, 1u);
    // after a timeout the counters are left as they are, for diagnosis
    if (prev == gridDim.x - 1 && !*reinterpret_cast<volatile uint32_t*>(&h->abort)) {
      h->ticket = 0ull;
      h->rq_head = 0u;
      h->rq_reserve = 0u;
      h->exit_cnt = 0u;
      fence_acq_rel_gpu();
    }
  }
}

// residual_out: the distribution the emitted token was drawn from.  One CTA
// per row; it clears the row's stop record once every thread has read it.
__global__ void dense_resid_out_kernel(const __grid_constant__ DenseParams P, float* out) {
  const int b = blockIdx.x;
  StopInfo* sp = ws_at<StopInfo>(P, P.L.stop) + b;
  const StopInfo st = ldcg32(sp);
  __syncthreads();
  if (threadIdx.x == 0) {
    int4* q = reinterpret_cast<int4*>(sp);
    q[0] = make_int4(0, 0, 0, 0);
    q[1] = make_int4(0, 0, 0, 0);
  }
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

// kernel configurations: ring stages, consumer warps, CTAs per SM
struct DenseConfig {
  void (*fn)(DenseParams);
  size_t smem;
  int threads;
  int ctas_per_sm;
};

template <int NS, int NW, int CTAS>
DenseConfig make_config() {
  DenseConfig c;
  c.fn = dense_verify_kernel<NS, NW, CTAS>;
  c.smem = sizeof(Smem<NS, NW>);
  c.threads = 32 * (NW + 2);
  c.ctas_per_sm = CTAS;
  return c;
}

const DenseConfig& active_config() {
  // 2 CTAs per SM, 24-stage rings, 8 consumer warps each (measured fastest of
  // the configurations whose ring depth is a multiple of the consumer warps)
  static const DenseConfig cfg = make_config<24, 8, 2>();
  return cfg;
}

}  // namespace

size_t dense_smem_bytes() { return active_config().smem; }
int dense_ctas_per_sm() { return active_config().ctas_per_sm; }

cudaError_t launch_dense(const DenseParams& p, int grid, cudaStream_t s) {
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const DenseConfig& c = active_config();
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(c.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  c.fn<<<grid, c.threads, c.smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dense_resid_out(const DenseParams& p, float* resid_out, cudaStream_t s) {
  dense_resid_out_kernel<<<p.B, 512, 0, s>>>(p, resid_out);
  return cudaGetLastError();
}

}  // namespace sv
