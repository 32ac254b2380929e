// sv_support.cu -- sparse support lists from dense logits: temperature,
// top-k, top-p.
//
// The pages name this preprocessing without spelling it out (the Uno
// article's test setting: temperature 1, top-k 50, top-p 0.95; DFlash/DFlash2
// guide, Q3: both logit sets are temperature scaled before the acceptance
// ratio).  Per row of V logits:
//   S   = the K largest logits (the smaller id first on ties; the same set for
//         every temperature T > 0),
//   p_i = softmax(l_i / T) renormalised over S,
//   keep the shortest prefix of S in decreasing p (ties: smaller id) whose
//   cumulative mass reaches top_p (at least one entry), renormalise it, give
//   the rest of S probability 0,
// and write S as a K-entry list in ascending id order -- the lists
// spec_verify_sparse takes.
//
// Design: one CTA of 8 warps per row, one HBM pass (3 rows per SM).  Warps
// stream interleaved 2 KB chunks of the row through a per-warp cp.async ring
// and only compare each 16-byte vector's largest element with a threshold --
// a value that at least K elements of the row reach, so it never exceeds the
// K-th largest logit.  It starts as the K-th largest of the CTA's 256 lane
// maxima over the first two chunk rounds.  A vector that reaches it is parked
// (its index only); parked vectors are expanded into 64-bit keys -- the logit's
// order-preserving bits above the complemented id, so one unsigned comparison
// orders by value, then by the smaller id -- only when the parking buffer
// fills (then a warp's keys may be cut back to its top K, raising its
// threshold) and at the end.  At the end the K-th largest of the lanes'
// maxima over the whole row is a far tighter threshold: the keys that reach
// it (a few more than K) are gathered into one list, which warp 0 sorts with
// a warp-wide bitonic network before forming the probabilities, the top-p cut
// and the id-sorted output.  With heavy ties the list may overflow; each warp
// then selects its own top K and warp 0 merges them.
#include <climits>

#include "sv_common.cuh"

namespace sv {
namespace {


__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// value in the high half, complemented id in the low half: larger key =
// larger value, or the same value and a smaller id
__device__ __forceinline__ uint64_t make_key(float v, int id) {
  return ((uint64_t)ordered_bits(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ float key_value(uint64_t k) { return from_ordered((uint32_t)(k >> 32)); }
__device__ __forceinline__ int key_id(uint64_t k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

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
// largest of a vector's elements (NaN if one is NaN)
__device__ __forceinline__ float vec_max(const uint32_t (&w)[4], int bf16) {
  if (bf16) {
    const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(w[0], w[1]), bf16x2_max_nan(w[2], w[3]));
    return fmax_nan(bf16_lo(m), bf16_hi(m));
  }
  return fmax_nan(fmax_nan(__uint_as_float(w[0]), __uint_as_float(w[1])),
                  fmax_nan(__uint_as_float(w[2]), __uint_as_float(w[3])));
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}

// Warp-wide bitonic network over M = 32 NPL elements, element p = r * 32 +
// lane in x[r].  sort_desc sorts in decreasing order; merge_desc sorts a
// bitonic sequence in decreasing order.
template <int NPL>
__device__ __forceinline__ void cmpx(uint64_t (&x)[NPL], int k, int j, int lane) {
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int p = r * 32 + lane;
    const bool desc_block = (p & k) == 0;
    if (j >= 32) {
      const int r2 = r ^ (j >> 5);
      if (r < r2) {
        const uint64_t a = x[r], b = x[r2];
        const bool swap = desc_block ? (a < b) : (a > b);
        if (swap) {
          x[r] = b;
          x[r2] = a;
        }
      }
    } else {
      const uint64_t o = shfl_xor64(x[r], j);
      const bool lower = (lane & j) == 0;
      const bool take_max = (lower == desc_block);
      x[r] = take_max ? (x[r] > o ? x[r] : o) : (x[r] < o ? x[r] : o);
    }
  }
}
template <int NPL>
__device__ __forceinline__ void sort_desc(uint64_t (&x)[NPL], int lane) {
  constexpr int M = 32 * NPL;
#pragma unroll
  for (int k = 2; k <= M; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) cmpx<NPL>(x, k, j, lane);
}
template <int NPL>
__device__ __forceinline__ void merge_desc(uint64_t (&x)[NPL], int lane) {
  constexpr int M = 32 * NPL;
#pragma unroll
  for (int j = M >> 1; j > 0; j >>= 1) cmpx<NPL>(x, 2 * M, j, lane);  // (p & 2M) == 0: all decreasing
}
// list <- the top M of list (sorted decreasing) and b (sorted decreasing)
template <int NPL>
__device__ __forceinline__ void merge_into(uint64_t (&list)[NPL], const uint64_t (&b)[NPL], int lane) {
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const uint64_t rev = shfl64(b[NPL - 1 - r], 31 - lane);  // element M-1-p of b
    list[r] = list[r] > rev ? list[r] : rev;
  }
  merge_desc<NPL>(list, lane);
}

// vector vi of a row (16-byte load when the row allows it; elements past V
// left as they are, i.e. -inf)
__device__ __forceinline__ void load_vector(const unsigned char* base, int vi, int V, int bf16,
                                            int aligned, uint32_t (&w)[4]) {
  const int epv = bf16 ? 8 : 4;
  if (aligned && (vi + 1) * epv <= V) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(base) + vi);
    w[0] = u.x;
    w[1] = u.y;
    w[2] = u.z;
    w[3] = u.w;
    return;
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if (bf16) {
      const int e0 = vi * 8 + 2 * t;
      const uint16_t* h = reinterpret_cast<const uint16_t*>(base);
      const uint32_t lo = (e0 < V) ? h[e0] : 0xFF80u;
      const uint32_t hi = (e0 + 1 < V) ? h[e0 + 1] : 0xFF80u;
      w[t] = lo | (hi << 16);
    } else {
      const int e = vi * 4 + t;
      w[t] = (e < V) ? reinterpret_cast<const uint32_t*>(base)[e] : 0xFF800000u;
    }
  }
}

struct SupportParams {
  const unsigned char* lt;  // [N, V]
  int N, V, K, bf16, aligned;
  float invT;               // 1 / temperature
  float top_p;
  int32_t* ids;             // [N, K]
  float* probs;             // [N, K]
  uint32_t* status;
};

// this warp's top M keys of wbuf[0, cnt) into `list` (batches of M keys,
// each sorted and merged in)
template <int NPL>
__device__ __forceinline__ void warp_select(const uint64_t* wbuf, int cnt, uint64_t (&list)[NPL],
                                            int lane) {
  constexpr int M = 32 * NPL;
#pragma unroll
  for (int r = 0; r < NPL; ++r) list[r] = 0ull;
  for (int base = 0; base < cnt; base += M) {
    uint64_t batch[NPL];
#pragma unroll
    for (int r = 0; r < NPL; ++r) {
      const int i = base + r * 32 + lane;
      batch[r] = (i < cnt) ? wbuf[i] : 0ull;
    }
    sort_desc<NPL>(batch, lane);
    merge_into<NPL>(list, batch, lane);
  }
}

// Out of line (rare): this warp's top K of wbuf[0, cnt) back into wbuf[0, K);
// returns the K-th largest value, which K of this warp's elements reach.
template <int NPL>
__device__ __noinline__ float warp_compact(uint64_t* wbuf, int cnt, int K, int lane) {
  uint64_t list[NPL];
  __syncwarp();
  warp_select<NPL>(wbuf, cnt, list, lane);
  __syncwarp();
#pragma unroll
  for (int r = 0; r < NPL; ++r)
    if (r * 32 + lane < K) wbuf[r * 32 + lane] = list[r];
  uint64_t kk = list[0];
#pragma unroll
  for (int r = 1; r < NPL; ++r)
    if (r == ((K - 1) >> 5)) kk = list[r];
  kk = shfl64(kk, (K - 1) & 31);
  __syncwarp();
  return key_value(kk);
}

// element e (0..7 bf16, 0..3 f32) of a 16-byte vector, as fp32
__device__ __forceinline__ float vec_elem(const uint32_t (&w)[4], int e, int bf16) {
  const int q = bf16 ? (e >> 1) : e;
  const uint32_t x = (q & 2) ? ((q & 1) ? w[3] : w[2]) : ((q & 1) ? w[1] : w[0]);
  if (!bf16) return __uint_as_float(x);
  return __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));
}

constexpr int kU = 4;             // 16-byte vectors per lane per chunk: a chunk is 2 KB of a row
constexpr int kChunkVec = 32 * kU;
constexpr int kChunkB = 16 * kChunkVec;
constexpr int kRStages = 2;       // per-warp ring of chunk stages (cp.async)
constexpr int kVCap = 384;        // parked vector indices per warp

template <int NPL>
__host__ __device__ constexpr int key_cap() {  // candidate keys per warp: a cut to K + one flush round
  return 32 * NPL + 256;
}
template <int NPL>
__host__ __device__ constexpr int gather_cap() {  // keys the final filter may gather
  return 64 * NPL + 128;
}

struct FlushOut {
  float thr;
  int wcnt;
};

// Expand this warp's parked vectors (row vector indices vbuf[0,
// vcnt), one per lane per round, re-read from the row) into keys of their
// elements at or above thr, appended to wbuf; when a round's keys do not fit,
// the buffer is first cut back to its top K, which raises thr.
template <int NPL>
__device__ __forceinline__ FlushOut warp_flush(const unsigned char* base, const int* vbuf, int vcnt,
                                            uint64_t* wbuf, int wcnt, float thr, int K, int V,
                                            int bf16, int aligned, int lane) {
  constexpr int kCap = key_cap<NPL>();
  const int epv = bf16 ? 8 : 4;
  __syncwarp();
  for (int b0 = 0; b0 < vcnt; b0 += 4 * 32) {
    uint32_t w[4][4];  // up to 4 vectors per lane, all loads issued first
    int id0[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = b0 + q * 32 + lane;
      id0[q] = -1;
      if (i < vcnt) {
        const int vi = vbuf[i];
        load_vector(base, vi, V, bf16, aligned, w[q]);
        id0[q] = vi * epv;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (b0 + q * 32 >= vcnt) break;
      unsigned em = 0;
      if (id0[q] >= 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e < epv && id0[q] + e < V && vec_elem(w[q], e, bf16) >= thr) em |= 1u << e;
      }
      const int cnt = __popc(em);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);  // <= 32 epv
      if (wcnt + total > kCap) {  // cut back to the top K first (K + 32 epv <= kCap)
        thr = fmaxf(thr, warp_compact<NPL>(wbuf, wcnt, K, lane));
        wcnt = K;
      }
      int pos = wcnt + incl - cnt;
      while (em) {
        const int e = __ffs(em) - 1;
        wbuf[pos++] = make_key(vec_elem(w[q], e, bf16), id0[q] + e);
        em &= em - 1;
      }
      wcnt += total;
    }
  }
  __syncwarp();
  return FlushOut{thr, wcnt};
}

// The keys at or above t among this warp's buffered keys and
// parked vectors, appended to the CTA's gather list (slots reserved with one
// shared atomic per round; *gcnt counts them all, slots past cap are not
// written).
template <int NPL>
__device__ __forceinline__ void warp_gather(const unsigned char* base, const int* vbuf, int vcnt,
                                         const uint64_t* wbuf, int wcnt, float t, int V, int bf16,
                                         int aligned, uint64_t* gather, int* gcnt, int lane) {
  constexpr int kGCap = gather_cap<NPL>();
  const unsigned ltm = (1u << lane) - 1u;
  for (int b0 = 0; b0 < wcnt; b0 += 32) {
    const int i = b0 + lane;
    const uint64_t k = (i < wcnt) ? wbuf[i] : 0ull;
    const bool pred = (i < wcnt) && key_value(k) >= t;
    const unsigned m = __ballot_sync(0xffffffffu, pred);
    if (!m) continue;
    int g = 0;
    if (lane == 0) g = atomicAdd(gcnt, __popc(m));
    g = __shfl_sync(0xffffffffu, g, 0);
    const int pos = g + __popc(m & ltm);
    if (pred && pos < kGCap) gather[pos] = k;
  }
  const int epv = bf16 ? 8 : 4;
  for (int b0 = 0; b0 < vcnt; b0 += 4 * 32) {
    uint32_t w[4][4];  // up to 4 vectors per lane, all loads issued first
    int id0[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = b0 + q * 32 + lane;
      id0[q] = -1;
      if (i < vcnt) {
        const int vi = vbuf[i];
        load_vector(base, vi, V, bf16, aligned, w[q]);
        id0[q] = vi * epv;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (b0 + q * 32 >= vcnt) break;
      unsigned em = 0;
      if (id0[q] >= 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e < epv && id0[q] + e < V && vec_elem(w[q], e, bf16) >= t) em |= 1u << e;
      }
      const int cnt = __popc(em);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (total == 0) continue;
      int g = 0;
      if (lane == 0) g = atomicAdd(gcnt, total);
      g = __shfl_sync(0xffffffffu, g, 0);
      int pos = g + incl - cnt;
      while (em) {
        const int e = __ffs(em) - 1;
        if (pos < kGCap) gather[pos] = make_key(vec_elem(w[q], e, bf16), id0[q] + e);
        ++pos;
        em &= em - 1;
      }
    }
  }
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

// the K-th largest of the CTA's 32 W lane values x (each a distinct element of
// the row, or -inf): each warp sorts its 32, then every thread finds its
// value's rank among all 256 (value, then warp, then position); the thread of
// rank K-1 writes it to *out.  Ends with a barrier; x must not be NaN.
template <int W>
__device__ __forceinline__ void cta_kth_of_lanes(float x, int K, float (*s_lv)[32], float* out,
                                                 int warp, int lane) {
  uint32_t k = ordered_bits(x);  // bitonic sort of the warp's 32 keys, decreasing
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, k, j);
      const bool take_max = (((lane & j) == 0) == ((lane & kk) == 0));
      k = take_max ? max(k, o) : min(k, o);
    }
  const float xs = from_ordered(k);
  s_lv[warp][lane] = xs;
  __syncthreads();
  int rank = lane;
#pragma unroll
  for (int w2 = 0; w2 < W; ++w2) {  // the searches are independent
    const bool ge = w2 < warp;  // equal values in lower warps come first
    int cnt = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
      const float y = s_lv[w2][cnt + step - 1];
      if (ge ? (y >= xs) : (y > xs)) cnt += step;
    }
    const float y = s_lv[w2][31];
    if (cnt == 31 && (ge ? (y >= xs) : (y > xs))) cnt = 32;
    if (w2 != warp) rank += cnt;
  }
  if (rank == K - 1) *out = xs;
  __syncthreads();
}

// Chunk c of a row (this lane's kU vectors) into stage memory d (this lane's
// slots): cp.async, no bounds checks for the full chunks c < nfull.
__device__ __forceinline__ void stage_chunk(unsigned char* d, const unsigned char* src, int c,
                                            int nfull, int nvec, int lane) {
  const unsigned char* g = src + (size_t)c * kChunkB;
  if (c < nfull) {
#pragma unroll
    for (int u = 0; u < kU; ++u) cp_async16(d + u * 512, g + u * 512);
  } else {
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (c * kChunkVec + u * 32 + lane < nvec) cp_async16(d + u * 512, g + u * 512);
  }
}

// This lane's kU vectors of chunk c: from stage memory d (aligned rows) or
// straight from the row (element loads); -inf past the row.
__device__ __forceinline__ void read_chunk(const unsigned char* d, const unsigned char* base, int c,
                                           int nfull, int nvec, int V, int bf16, int aligned,
                                           int lane, uint32_t (&w)[kU][4]) {
  if (c < nfull) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint4 x = *reinterpret_cast<const uint4*>(d + u * 512);
      w[u][0] = x.x;
      w[u][1] = x.y;
      w[u][2] = x.z;
      w[u][3] = x.w;
    }
    return;
  }
  const uint32_t ninf = bf16 ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int vi = c * kChunkVec + u * 32 + lane;
#pragma unroll
    for (int t = 0; t < 4; ++t) w[u][t] = ninf;
    if (vi >= nvec) continue;
    if (aligned) {
      const uint4 x = *reinterpret_cast<const uint4*>(d + u * 512);
      w[u][0] = x.x;
      w[u][1] = x.y;
      w[u][2] = x.z;
      w[u][3] = x.w;
    } else {
      load_vector(base, vi, V, bf16, 0, w[u]);
    }
  }
}

template <int NPL, int W>
__global__ void __launch_bounds__(32 * W, (W <= 3) ? 8 : ((W <= 6) ? 4 : 3))
    support_kernel(const __grid_constant__ SupportParams P) {
  constexpr int kCap = key_cap<NPL>();
  constexpr int kGCap = gather_cap<NPL>();
  extern __shared__ __align__(16) unsigned char s_ring_raw[];
  static_assert(32 * W >= 32 * NPL, "the lane-maxima thresholds need K <= 32 W lanes");
  __shared__ uint64_t s_wbuf[W][kCap];
  __shared__ int s_vbuf[W][kVCap];
  __shared__ uint64_t s_gather[kGCap];
  __shared__ float s_lv[W][32];
  __shared__ float s_thr;
  __shared__ int s_bad, s_gcnt;
  // a programmatic dependent of whatever precedes it on the stream: nothing is
  // read before that grid has completed; the next call may launch at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x, V = P.V, K = P.K;
  const size_t es = P.bf16 ? 2 : 4;
  const unsigned char* base = P.lt + (size_t)row * V * es;
  const int epv = P.bf16 ? 8 : 4;
  const int nvec = (V + epv - 1) / epv;
  const int nch = (nvec + kChunkVec - 1) / kChunkVec;
  const int nfull = P.aligned ? nvec / kChunkVec : 0;  // chunks read with no bounds checks
  if (tid == 0) {
    s_bad = 0;
    s_gcnt = 0;
  }
  uint64_t* wbuf = s_wbuf[warp];
  int* vbuf = s_vbuf[warp];
  // this lane's 16 bytes of each stage; chunk c's vector u of this lane is
  // row vector c * kChunkVec + u * 32 + lane
  unsigned char* const ring = s_ring_raw + (size_t)warp * kRStages * kChunkB + lane * 16;
  const unsigned char* const src = base + (size_t)lane * 16;

  // Warp w streams chunks w, w + W, w + 2 W, ...; chunk round i (chunk w + W i)
  // lands in stage i % kRStages (aligned rows), all stages filled ahead.
  if (P.aligned) {
#pragma unroll
    for (int st = 0; st < kRStages; ++st) {
      const int c = warp + st * W;
      if (c < nch) stage_chunk(ring + st * kChunkB, src, c, nfull, nvec, lane);
      cp_async_commit();
    }
  }

  // The starting threshold: the K-th largest of the CTA's 32 W lane maxima
  // over its first kRStages chunk rounds (the filled stages).  Those maxima
  // are distinct elements of the row, so at least K elements reach it: it
  // never exceeds the row's K-th largest logit.
  uint32_t w[kU][4];
  float thr;
  {
    if (P.aligned) cp_async_wait_group<0>();
    float tm = -INFINITY;
#pragma unroll
    for (int st = kRStages - 1; st >= 0; --st) {  // ends with chunk `warp` (stage 0) in w
      read_chunk(ring + st * kChunkB, base, warp + st * W, nfull, nvec, V, P.bf16, P.aligned, lane, w);
#pragma unroll
      for (int u = 0; u < kU; ++u) tm = fmaxf(tm, vec_max(w[u], P.bf16));  // NaN ignored here
    }
    cta_kth_of_lanes<W>(tm, K, s_lv, &s_thr, warp, lane);
    thr = s_thr;
  }
  float runmax = -INFINITY;  // this lane's largest element so far (NaN if one is NaN)
  int wcnt = 0;              // keys in this warp's buffer (warp-uniform)
  int vcnt = 0;              // parked vectors (warp-uniform)
  int slot = 0;              // stage of the chunk in w
  const unsigned lt_mask = (1u << lane) - 1u;

  // No barriers from here to the end of the stream: warps go at their own
  // pace.  The inner loop streams while the parking buffer has room for a
  // chunk; the outer one expands the parked vectors into keys between chunks.
  int c = warp;
  while (c < nch) {
    while (true) {
      if (P.aligned) {  // w holds chunk c: its stage takes the chunk kRStages rounds ahead
        const int cn = c + kRStages * W;
        if (cn < nch) stage_chunk(ring + slot * kChunkB, src, cn, nfull, nvec, lane);
        cp_async_commit();
        slot = (slot + 1 == kRStages) ? 0 : slot + 1;
      }
      // park the vectors whose largest element reaches the threshold (their
      // row index only; rare once the threshold has settled)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float vm = vec_max(w[u], P.bf16);
        runmax = fmax_nan(runmax, vm);
        const bool need = vm >= thr;
        const unsigned m = __ballot_sync(0xffffffffu, need);
        if (m) {
          if (need) vbuf[vcnt + __popc(m & lt_mask)] = c * kChunkVec + u * 32 + lane;
          vcnt += __popc(m);
        }
      }
      c += W;
      if (c >= nch || vcnt > kVCap - kChunkVec) break;
      if (P.aligned) cp_async_wait_group<kRStages - 1>();
      read_chunk(ring + slot * kChunkB, base, c, nfull, nvec, V, P.bf16, P.aligned, lane, w);
    }
    if (c >= nch) break;
    // the next chunk might not fit: expand the parked vectors into keys
    const FlushOut f = warp_flush<NPL>(base, vbuf, vcnt, wbuf, wcnt, thr, K, V, P.bf16, P.aligned, lane);
    thr = f.thr;
    wcnt = f.wcnt;
    vcnt = 0;
    if (P.aligned) cp_async_wait_group<kRStages - 1>();
    read_chunk(ring + slot * kChunkB, base, c, nfull, nvec, V, P.bf16, P.aligned, lane, w);
  }
  if (P.aligned) cp_async_wait_group<0>();

  // A NaN or +inf logit makes the row an input error.
  const int bad = (runmax != runmax) || (runmax == INFINITY);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&s_bad, 1);
  __syncthreads();
  int32_t* oid = P.ids + (size_t)row * K;
  float* op = P.probs + (size_t)row * K;
  if (s_bad) {
    if (warp == 0) {
      for (int i = lane; i < K; i += 32) {
        oid[i] = -1;
        op[i] = __int_as_float(0x7fc00000);
      }
      if (lane == 0) atomicOr(P.status, kStatusInputErr);
    }
    return;
  }
  // The final filter: the K-th largest of the lanes' maxima over the whole row
  // (again K distinct elements reach it), so only a few keys beyond the top K
  // pass.  They are gathered into one list; with heavy ties the list may
  // overflow, and then each warp selects its own top M and warp 0 merges.
  cta_kth_of_lanes<W>(runmax, K, s_lv, &s_thr, warp, lane);
  const float tf = fmaxf(thr, s_thr);
  warp_gather<NPL>(base, vbuf, vcnt, wbuf, wcnt, tf, V, P.bf16, P.aligned, s_gather, &s_gcnt, lane);
  __syncthreads();
  const int gcnt = s_gcnt;
  uint64_t list[NPL];
  if (gcnt <= kGCap) {
    if (warp != 0) return;
    warp_select<NPL>(s_gather, gcnt, list, lane);
  } else {
    if (vcnt > 0) {
      const FlushOut f = warp_flush<NPL>(base, vbuf, vcnt, wbuf, wcnt, thr, K, V, P.bf16, P.aligned, lane);
      wcnt = f.wcnt;
    }
    __syncwarp();
    warp_select<NPL>(wbuf, wcnt, list, lane);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < NPL; ++r) wbuf[r * 32 + lane] = list[r];
    __syncthreads();
    if (warp != 0) return;
    for (int w2 = 1; w2 < W; ++w2) {
      uint64_t b2[NPL];
#pragma unroll
      for (int r = 0; r < NPL; ++r) b2[r] = s_wbuf[w2][r * 32 + lane];
      merge_into<NPL>(list, b2, lane);
    }
  }
  // list[0..K) is the top-k set, decreasing
  const float vmax = key_value(shfl64(list[0], 0));
  if (!(vmax > -INFINITY)) {  // every logit -inf: no distribution
    for (int i = lane; i < K; i += 32) {
      oid[i] = -1;
      op[i] = __int_as_float(0x7fc00000);
    }
    if (lane == 0) atomicOr(P.status, kStatusInputErr);
    return;
  }
  // probabilities over the set (decreasing order p = r * 32 + lane)
  float pr[NPL];
  ff zs{0.f, 0.f};
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int p = r * 32 + lane;
    const float v = key_value(list[r]);
    pr[r] = (p < K && v > -INFINITY) ? exp2f((v - vmax) * P.invT * kLog2e) : 0.f;
    zs = ff_add_f(zs, pr[r]);
  }
  zs = warp_sum_ff(zs);
  // top-p: the shortest prefix (decreasing p) whose mass reaches top_p * Z
  int keep = K;
  if (P.top_p < 1.f) {
    const ff target = ff_mul_f(zs, P.top_p);
    ff carry{0.f, 0.f};
    keep = -1;
#pragma unroll
    for (int r = 0; r < NPL; ++r) {
      // inclusive prefix over the lanes of register r, plus the carry
      ff x{pr[r], 0.f};
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const ff y = ff_shfl_up(x, o);
        if (lane >= o) x = ff_add(x, y);
      }
      const ff incl = ff_add(carry, x);
      const unsigned hit = __ballot_sync(0xffffffffu, !ff_gt(target, incl) && (r * 32 + lane) < K);
      if (keep < 0 && hit) keep = r * 32 + __ffs(hit);
      carry = ff_shfl(incl, 31);
    }
    if (keep < 0 || keep > K) keep = K;
  }
  ff zk{0.f, 0.f};
#pragma unroll
  for (int r = 0; r < NPL; ++r)
    if (r * 32 + lane < keep) zk = ff_add_f(zk, pr[r]);
  zk = warp_sum_ff(zk);
  const float inv = __fdiv_rn(1.f, ff_to_f(zk));
  // re-key by id (ascending) for the output: entries past K sort last
  uint64_t bid[NPL];
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int p = r * 32 + lane;
    const float prob = (p < keep) ? pr[r] * inv : 0.f;
    const uint32_t idk = (p < K) ? (uint32_t)key_id(list[r]) : 0xFFFFFFFFu;
    // decreasing sort on (~id): ascending id
    bid[r] = ((uint64_t)(0xFFFFFFFFu - idk) << 32) | __float_as_uint(prob);
  }
  sort_desc<NPL>(bid, lane);
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int p = r * 32 + lane;
    if (p < K) {
      oid[p] = (int)(0xFFFFFFFFu - (uint32_t)(bid[r] >> 32));
      op[p] = __uint_as_float((uint32_t)bid[r]);
    }
  }
}

}  // namespace

cudaError_t launch_support(const unsigned char* lt, int N, int V, int K, int bf16, int aligned,
                           float temperature, float top_p, int32_t* ids, float* probs,
                           uint32_t* status, cudaStream_t s) {
  SupportParams p;
  p.lt = lt;
  p.N = N;
  p.V = V;
  p.K = K;
  p.bf16 = bf16;
  p.aligned = aligned;
  p.invT = 1.f / temperature;
  p.top_p = top_p;
  p.ids = ids;
  p.probs = probs;
  p.status = status;
  // K <= 64: 6 warps and about 51 KB of shared memory per row, 4 rows per SM
  // (measured 66.3 us against 68.2 us with 8 warps and 3 rows per SM for 960
  // rows of 128256 bf16 logits; 3 warps and 8 rows per SM took 98.7 us: the
  // per-row phases outside the stream lengthen); larger K: 8 warps
  const size_t ring = (size_t)8 * kRStages * kChunkB;
  const size_t ring6 = (size_t)6 * kRStages * kChunkB;
  static bool attr[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    const int carve = cudaSharedmemCarveoutMaxShared;
    e = cudaFuncSetAttribute(support_kernel<1, 6>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<2, 6>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<1, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring6);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<2, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring6);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<4, 8>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<8, 8>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<4, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(support_kernel<8, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  cudaLaunchAttribute pdl[1];  // launched as a programmatic dependent (see the kernel)
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)N, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = ring;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (K <= 64) {
    cfg.blockDim = dim3(6 * 32, 1, 1);
    cfg.dynamicSmemBytes = ring6;
    if (K <= 32) return cudaLaunchKernelEx(&cfg, support_kernel<1, 6>, p);
    return cudaLaunchKernelEx(&cfg, support_kernel<2, 6>, p);
  }
  if (K <= 128) return cudaLaunchKernelEx(&cfg, support_kernel<4, 8>, p);
  return cudaLaunchKernelEx(&cfg, support_kernel<8, 8>, p);
}

}  // namespace sv
