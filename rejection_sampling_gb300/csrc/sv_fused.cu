// sv_fused.cu -- dense verification in one pass over the logits: one
// thread-block cluster per (row, position).
//
// Computes, for every row b (DFlash/DFlash2 guide, 4.4; Uno article, "What
// 'lossless' actually has to mean"):
//   p_j = softmax(target[b, j]), q_j = softmax(draft[b, j]),
//   a_j = min(1, p_j(x_j) / q_j(x_j))  (0 where q_j(x_j) = 0),
//   n   = first j with u_accept[b, j] >= a_j (gamma if none),
//   token n = inverse CDF of max(p_n - q_n, 0) (n < gamma) or of p_gamma
//   (bonus, DFlash/DFlash2 guide section 2) at u_sample[b].
//
// Design.  A unit is one (row, position): the target row and, below gamma,
// the draft row.  One cluster of C CTAs takes a unit; rank r holds elements
// [r L, r L + L) of both rows in its shared memory, fetched by 1-D bulk copies
// (cp.async.bulk, one mbarrier per 8 KB chunk) that are all issued at once,
// so every logit crosses HBM exactly once and each CTA keeps 16-64 KB in
// flight.
//  1. Per chunk, as it lands, every thread folds its vectors into running
//     (c, S) (c = log2e * max, S = sum 2^(v log2e - c)) for both rows.
//  2. The CTA combines its threads, the cluster exchanges the CTA parts
//     through distributed shared memory, and every CTA combines them in rank
//     order -- the same arithmetic on the same values, so all ranks hold the
//     same statistics and take the same decision: the accept test at x_j (the
//     rank holding x_j publishes the two logits there).
//  3. A rejected position, or the bonus position, draws speculatively from
//     the slices still in shared memory: each rank forms the residual (or p)
//     mass of every 16-byte vector, the cluster exchanges the rank totals,
//     the rank whose prefix crosses u_sample * T walks its vector masses and
//     then the elements of one vector.  A position skips the draw when an
//     earlier position of its row is already known to be rejected (a per-row
//     word raised atomically; a hint only -- the first rejection always
//     draws).  Units are numbered position-major, so earlier positions are
//     normally decided before later ones start.
//  4. The CTA that finishes a unit writes its 32-byte record, and the last
//     unit of a row to finish (a per-row arrival counter, no waiting) takes
//     the first rejection n, writes n and the tokens, and returns the row's
//     workspace words to zero.
// The kernel is a programmatic dependent of whatever precedes it on the
// stream and reads nothing before that grid has completed; its own waits are
// on its own bulk copies and are bounded in time (a copy that never lands
// marks its row with a timeout instead of hanging).
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkVec = 2 * kThreads;  // 16-byte vectors per chunk of one row (8 KB)
constexpr int kMaxChunks = 8;
constexpr int kSliceBytes = 32 * 1024;     // preferred per-rank slice of one row (3 CTAs per SM)
constexpr int kSliceCapBytes = 48 * 1024;  // largest slice (6 chunks)
constexpr int kMaxCluster = 16;
constexpr int kMaxPos = 256;  // positions per row (gamma + 1 <= 256)
constexpr size_t kMaxDynSmem = 2 * (size_t)kSliceCapBytes + kSliceCapBytes / 4;  // rows + masses
constexpr unsigned long long kWaitNs = 1000000000ull;  // bounded copy wait: one second

constexpr uint32_t kNegInf2 = 0xFF80FF80u;  // two bf16 -inf
constexpr uint32_t kNegInfF = 0xFF800000u;  // fp32 -inf

// ---------------------------------------------------------------------------
// PTX helpers: mbarriers, bulk copies, clusters
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
// every thread of every CTA of the cluster; orders earlier memory operations
// before everything after it, cluster-wide
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}
// workspace words written by other CTAs: read around L1
__device__ __forceinline__ uint32_t ldcg_u32(const uint32_t* p) { return __ldcg(p); }

// ---------------------------------------------------------------------------
// arithmetic shared by every step
// ---------------------------------------------------------------------------
// partial sums carry integer reference points (sv_common.cuh): rescales are
// exact powers of two
__device__ __forceinline__ float part_scale(float c, float C) { return scale_exact(c, C); }
// r(y) (mode 0: max(p - q, 0); mode 1: p) from fp32 logits.  The masses and
// the final walk evaluate it with identical operations, so they see
// bit-identical values.
__device__ __forceinline__ float resid_val(float t, float d, float ct, float cd, float invSt,
                                           float invSd, int mode) {
  const float p = __fmul_rn(ex2(__fmaf_rn(t, kLog2e, -ct)), invSt);
  if (mode != 0) return p;
  const float q = __fmul_rn(ex2(__fmaf_rn(d, kLog2e, -cd)), invSd);
  const float r = __fsub_rn(p, q);
  return r > 0.f ? r : 0.f;
}

template <bool BF>
__device__ __forceinline__ uint4 neg_inf_vec() {
  const uint32_t n = BF ? kNegInf2 : kNegInfF;
  return make_uint4(n, n, n, n);
}
// element e of a 16-byte vector, widened to fp32 (bf16: a 16-bit shift, exact)
template <bool BF>
__device__ __forceinline__ float vec_elem(const uint4& v, int e) {
  if (BF) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
  const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  return __uint_as_float(w);
}

// Fold this thread's vectors of one chunk (v0 + i kThreads + tid, i < 2) into
// its running (C, S).  The chunk's maximum is taken first (bf16 pairs:
// max.bf16x2, NaN ignored), the running sum rescaled (exactly) when the
// reference point C = ceil(log2e * max) grows, then S += sum 2^(v log2e - C).  A NaN or +inf element makes S NaN (the row
// is then an input error); an all -inf side keeps C = -inf, S = 0.
template <bool BF>
__device__ __forceinline__ void fold_chunk(const unsigned char* s, int v0, int nv, int tid, float& C,
                                           ff& S) {
  uint4 a[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = v0 + i * kThreads + tid;
    a[i] = (v < nv) ? lds128(s + 16 * (size_t)v) : neg_inf_vec<BF>();
  }
  float m;
  if (BF) {
    const uint32_t m0 = bf16x2_max(bf16x2_max(a[0].x, a[0].y), bf16x2_max(a[0].z, a[0].w));
    const uint32_t m1 = bf16x2_max(bf16x2_max(a[1].x, a[1].y), bf16x2_max(a[1].z, a[1].w));
    const uint32_t mx = bf16x2_max(m0, m1);
    m = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(a[i].x), __uint_as_float(a[i].y)),
                         fmaxf(__uint_as_float(a[i].z), __uint_as_float(a[i].w))));
  }
  const float c = ref_point(m);
  if (c > C) {
    S = ff_mul_f(S, part_scale(C, c));
    C = c;
  }
  const float cc = (C == -INFINITY) ? 0.f : C;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (BF) {
      s0 += ex2(fmaf(bf16_lo(a[i].x), kLog2e, -cc));
      s1 += ex2(fmaf(bf16_hi(a[i].x), kLog2e, -cc));
      s2 += ex2(fmaf(bf16_lo(a[i].y), kLog2e, -cc));
      s3 += ex2(fmaf(bf16_hi(a[i].y), kLog2e, -cc));
      s0 += ex2(fmaf(bf16_lo(a[i].z), kLog2e, -cc));
      s1 += ex2(fmaf(bf16_hi(a[i].z), kLog2e, -cc));
      s2 += ex2(fmaf(bf16_lo(a[i].w), kLog2e, -cc));
      s3 += ex2(fmaf(bf16_hi(a[i].w), kLog2e, -cc));
    } else {
      s0 += ex2(fmaf(__uint_as_float(a[i].x), kLog2e, -cc));
      s1 += ex2(fmaf(__uint_as_float(a[i].y), kLog2e, -cc));
      s2 += ex2(fmaf(__uint_as_float(a[i].z), kLog2e, -cc));
      s3 += ex2(fmaf(__uint_as_float(a[i].w), kLog2e, -cc));
    }
  }
  S = ff_add_f(S, (s0 + s1) + (s2 + s3));
}

// ---------------------------------------------------------------------------
// block-wide helpers (kWarps warps)
// ---------------------------------------------------------------------------
struct BlockScratch {
  float hi[kWarps], lo[kWarps];
  int wa[kWarps], wb[kWarps];
};

// float-float sum over the block, valid in every thread
__device__ __forceinline__ ff block_sum_ff(ff v, BlockScratch& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_ff(v);
  if (lane == 0) {
    S.hi[warp] = v.hi;
    S.lo[warp] = v.lo;
  }
  __syncthreads();
  ff t{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t = ff_add(t, ff{S.hi[w], S.lo[w]});
  __syncthreads();
  return t;
}

// exclusive prefix of v over the threads in order (float-float)
__device__ __forceinline__ ff block_exclusive_scan_ff(ff v, BlockScratch& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ff x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y = ff_shfl_up(x, o);
    if (lane >= o) x = ff_add(x, y);
  }
  if (lane == 31) {
    S.hi[warp] = x.hi;
    S.lo[warp] = x.lo;
  }
  __syncthreads();
  ff base{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (w < warp) base = ff_add(base, ff{S.hi[w], S.lo[w]});
  __syncthreads();
  return ff_add(base, ff_sub(x, v));
}

// the first thread with `cond` (kThreads if none) and the largest `v` (>= -1)
__device__ __forceinline__ void block_first_and_max(bool cond, int v, BlockScratch& S, int& first,
                                                    int& vmax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, cond);
  const int wm = (int)__reduce_max_sync(0xffffffffu, (unsigned)(v + 1)) - 1;
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
  __syncthreads();
  first = f;
  vmax = m;
}

// ---------------------------------------------------------------------------
// the unit's decision, identical in every rank of the cluster
// ---------------------------------------------------------------------------
struct Decision {
  float ct, cd, invSt, invSd;  // draw constants
  float a;                     // min(1, p/q) at the draft token
  float us;                    // u_sample of the row
  int err, tmo, acc, draw, mode;
};

// Part of a unit's statistics exchanged between ranks (12 words):
//   0 Ct, 1-2 St, 3 Cd, 4-5 Sd, 6 target logit at x_j, 7 draft logit at x_j
//   (kNoTokenBits where the slice does not hold x_j), 8 timeout, 9 the row's
//   rejection word (rank 0's copy), 10-11 unused.  Each warp forms one, the
//   CTA combines its warps' parts, and the CTA's part is written into every
//   rank's shared memory (st.shared::cluster): after one cluster barrier each
//   rank reads only its own shared memory, so no rank waits for another to
//   finish reading before it leaves.
constexpr int kPartWords = 12;

__device__ __forceinline__ void st_cluster_f4(const void* p, unsigned rank, float4 v) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Sequential merge of K parts held in shared memory (every lane of the warp
// reads every part -- broadcast loads -- and merges them in index order, so
// all lanes, and all ranks merging the same parts, get bit-identical
// results): maxima first, then each sum scaled once (exactly) and added in
// float-float; the gathered logits from the part that has them, timeouts
// OR-ed, the hint from part 0.
struct Combined {
  float Ct, Cd;
  ff St, Sd;
  uint32_t txb, dxb, hint;
  int tmo, hx;
};
__device__ __forceinline__ Combined merge_parts(const float (*parts)[kPartWords], int K) {
  Combined c;
  c.Ct = c.Cd = -INFINITY;
  for (int k = 0; k < K; ++k) {
    c.Ct = fmaxf(c.Ct, parts[k][0]);
    c.Cd = fmaxf(c.Cd, parts[k][3]);
  }
  c.St = c.Sd = ff{0.f, 0.f};
  c.txb = c.dxb = kNoTokenBits;
  c.tmo = 0;
  c.hint = __float_as_uint(parts[0][9]);
  for (int k = 0; k < K; ++k) {
    const float4 a0 = *reinterpret_cast<const float4*>(&parts[k][0]);
    const float4 a1 = *reinterpret_cast<const float4*>(&parts[k][4]);
    const float4 a2 = *reinterpret_cast<const float4*>(&parts[k][8]);
    c.St = ff_add(c.St, ff_mul_f(ff{a0.y, a0.z}, part_scale(a0.x, c.Ct)));
    c.Sd = ff_add(c.Sd, ff_mul_f(ff{a1.x, a1.y}, part_scale(a0.w, c.Cd)));
    if (c.txb == kNoTokenBits && __float_as_uint(a1.z) != kNoTokenBits) {
      c.txb = __float_as_uint(a1.z);
      c.dxb = __float_as_uint(a1.w);
    }
    c.tmo |= __float_as_int(a2.x) != 0;
  }
  c.hx = c.txb != kNoTokenBits;
  return c;
}

// Record of a finished unit, then the row's arrival; the last unit of the
// row to arrive finalises it.  Warp 0 of the CTA that wrote the record.
__device__ void arrive_and_finalize(const FusedParams& P, int b, int lane) {
  const int G = P.G;
  // the row's draft tokens, read while the count is in flight (inputs: no
  // ordering needed); lane l holds x_{l + 32 i} in xs[i]
  int xs[(kMaxPos + 31) / 32];
#pragma unroll
  for (int i = 0; i < (kMaxPos + 31) / 32; ++i) {
    const int jj = lane + 32 * i;
    xs[i] = (jj < G) ? __ldg(P.x + (size_t)b * G + jj) : -1;
  }
  unsigned old = 0;
  if (lane == 0) {
    // the record (written by this thread) released with the count; the last
    // unit's count acquires every other unit's record
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(P.cnt + b) : "memory");
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != (unsigned)G) return;
  __syncwarp();
  UnitRec* R = P.rec + (size_t)b * (G + 1);
  int n = G, err = 0, tmo = 0;
  for (int jj = lane; jj <= G; jj += 32) {
    const uint32_t f = ldcg_u32(&R[jj].flags);
    err |= (f & kRecErr) != 0;
    tmo |= (f & kRecTimeout) != 0;
    if (jj < G && !(f & kRecAccept)) n = min(n, jj);
  }
  n = __reduce_min_sync(0xffffffffu, n);
  err = __any_sync(0xffffffffu, err);
  tmo = __any_sync(0xffffffffu, tmo);
  const bool bad = err || tmo;
  const int32_t tn = bad ? -1 : (int32_t)__ldcg(reinterpret_cast<const int*>(&R[n].token));
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
#pragma unroll
  for (int i = 0; i < (kMaxPos + 31) / 32; ++i) {
    const int jj = lane + 32 * i;
    if (jj <= G) tok[jj] = bad ? -1 : (jj < n ? xs[i] : (jj == n ? tn : -1));
  }
  // the records go back to zero, except the stop record that the
  // residual-output kernel reads (and clears) next
  for (int jj = lane; jj <= G; jj += 32)
    if (bad || !P.keep_stop || jj != n) {
      int4* q = reinterpret_cast<int4*>(R + jj);
      q[0] = make_int4(0, 0, 0, 0);
      q[1] = make_int4(0, 0, 0, 0);
    }
  if (lane == 0) {
    P.n_out[b] = bad ? -1 : n;
    if (err) atomicOr(P.status, kStatusInputErr);
    if (tmo) atomicOr(P.status, kStatusTimeout);
    P.cnt[b] = 0u;
    P.rej[b] = 0u;
  }
}

__device__ __forceinline__ void write_record(const FusedParams& P, int b, int j, uint32_t flags,
                                             int32_t token, const Decision& D, ff T) {
  float4* q = reinterpret_cast<float4*>(P.rec + (size_t)b * (P.G + 1) + j);
  q[0] = make_float4(__uint_as_float(flags), __int_as_float(token), D.ct, D.cd);
  q[1] = make_float4(D.invSt, D.invSd, T.hi, T.lo);
}

// the element of vector vs that the draw picks: the first whose running sum
// (from `acc`) exceeds `tgt`; else (rounding between the sums, or a clamped
// draw) the vector's last element with mass
template <bool BF>
__device__ __forceinline__ int walk_vector(const unsigned char* s_t, const unsigned char* s_d,
                                           int vs, const Decision& D, int mode, ff acc, ff tgt,
                                           bool clamp) {
  constexpr int epv = BF ? 8 : 4;
  const uint4 tv = lds128(s_t + 16 * (size_t)vs);
  const uint4 dv = (mode == 0) ? lds128(s_d + 16 * (size_t)vs) : make_uint4(0, 0, 0, 0);
  int hit = -1, last = -1;
#pragma unroll
  for (int e = 0; e < epv; ++e) {
    const float r = resid_val(vec_elem<BF>(tv, e), vec_elem<BF>(dv, e), D.ct, D.cd, D.invSt,
                              D.invSd, mode);
    if (r > 0.f) last = e;
    acc = ff_add_f(acc, r);
    if (hit < 0 && !clamp && ff_gt(acc, tgt)) hit = e;
  }
  return hit >= 0 ? hit : (last >= 0 ? last : 0);
}

template <bool BF>
__global__ void __launch_bounds__(kThreads, 3) dense_fused_kernel(const __grid_constant__ FusedParams P) {
  constexpr int es = BF ? 2 : 4, epv = 16 / es;
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ __align__(8) uint64_t bars[kMaxChunks];
  __shared__ __align__(16) float wpart[kWarps][kPartWords];      // this CTA's warps
  __shared__ __align__(16) float cpart[kMaxCluster][kPartWords];  // every rank's CTA part
  __shared__ __align__(16) float cmass[2][kMaxCluster][4];        // every rank's draw mass, per attempt
  __shared__ BlockScratch bs;
  __shared__ Decision D;
  __shared__ int s_redo, s_cstar, s_clamp, s_tok;
  __shared__ float s_tgt_hi, s_tgt_lo, s_T_hi, s_T_lo;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = (int)cluster_size(), rank = (int)cluster_rank();
  const int q = blockIdx.x / C;
  const int G = P.G;
  const int b = q % P.B, j = q / P.B;  // position-major unit order
  const bool has_d = j < G;
  const int y0 = rank * P.L;
  const int nel = max(0, min(P.L, P.V - y0));
  const int nv = nel / epv;  // the host keeps L and V multiples of epv
  const int nch = (nv + kChunkVec - 1) / kChunkVec;
  unsigned char* s_t = sm;
  unsigned char* s_d = sm + (size_t)P.L * es;
  float* mass = reinterpret_cast<float*>(sm + 2 * (size_t)P.L * es);

  // the next grid on the stream may be scheduled once every CTA of this one
  // has started; it waits for this grid to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // this grid may itself have been scheduled early: nothing is read before
  // the preceding grid (which may have produced the logits) has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every rank has started before any rank writes into another's shared
  // memory: arrive now, wait just before the first such write
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  const unsigned char* trow = P.lt + ((size_t)b * (G + 1) + j) * (size_t)P.V * es + (size_t)y0 * es;
  const unsigned char* drow =
      has_d ? P.ld + ((size_t)b * G + j) * (size_t)P.V * es + (size_t)y0 * es : nullptr;

  if (tid == 0) {  // the copy barriers, then every copy of the slice, issued at once
    for (int k = 0; k < nch; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
    s_redo = 0;
    for (int k = 0; k < nch; ++k) {
      const int v0 = k * kChunkVec;
      const unsigned bytes = 16u * (unsigned)min(kChunkVec, nv - v0);
      mbar_expect_tx(&bars[k], has_d ? 2u * bytes : bytes);
      bulk_g2s(s_t + 16 * (size_t)v0, trow + 16 * (size_t)v0, bytes, &bars[k]);
      if (has_d) bulk_g2s(s_d + 16 * (size_t)v0, drow + 16 * (size_t)v0, bytes, &bars[k]);
    }
  }
  __syncthreads();  // the barriers are initialised before anyone waits on them
  // the unit's small inputs, while the copies fly
  int xj = -1;
  float uj = 0.f, us = 0.f;
  uint32_t hint = 0u;
  if (warp == 0) {
    if (has_d) {
      xj = P.x[(size_t)b * G + j];
      uj = P.u_acc[(size_t)b * G + j];
    }
    us = P.u_s[b];
  }

  // 1. statistics of this rank's slices, chunk by chunk as they land
  float Ct = -INFINITY, Cd = -INFINITY;
  ff St{0.f, 0.f}, Sd{0.f, 0.f};
  bool ok = true;
  for (int k = 0; k < nch; ++k) {
    if (ok) ok = mbar_try_wait(&bars[k], 0) || mbar_wait_until(&bars[k], 0, globaltimer() + kWaitNs);
    const int v0 = k * kChunkVec;
    fold_chunk<BF>(s_t, v0, nv, tid, Ct, St);
    if (has_d) fold_chunk<BF>(s_d, v0, nv, tid, Cd, Sd);
  }
  const int wtmo = __any_sync(0xffffffffu, !ok);
  // the latest word on earlier rejections of this row (a hint; rank 0's copy
  // is the one every rank uses), read as late as possible
  if (tid == 0 && rank == 0) hint = ldcg_u32(P.rej + b);
  warp_combine_pair(Ct, St, Cd, Sd);
  if (lane == 0) {
    uint32_t txb = kNoTokenBits, dxb = kNoTokenBits;
    const int xl = xj - y0;
    if (warp == 0 && has_d && xj >= 0 && xj < P.V && xl >= 0 && xl < nel) {
      if (BF) {
        txb = (uint32_t)reinterpret_cast<const uint16_t*>(s_t)[xl] << 16;
        dxb = (uint32_t)reinterpret_cast<const uint16_t*>(s_d)[xl] << 16;
      } else {
        txb = reinterpret_cast<const uint32_t*>(s_t)[xl];
        dxb = reinterpret_cast<const uint32_t*>(s_d)[xl];
      }
    }
    float* w = wpart[warp];
    w[0] = Ct;
    w[1] = St.hi;
    w[2] = St.lo;
    w[3] = Cd;
    w[4] = Sd.hi;
    w[5] = Sd.lo;
    w[6] = __uint_as_float(txb);
    w[7] = __uint_as_float(dxb);
    w[8] = __int_as_float(wtmo);
    w[9] = __uint_as_float(hint);
    w[10] = w[11] = 0.f;
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every rank has started
  if (warp == 0) {  // the CTA's part, written into every rank's cpart[rank]
    const Combined c = merge_parts(wpart, kWarps);
    if (lane < C) {
      const float4 a0 = make_float4(c.Ct, c.St.hi, c.St.lo, c.Cd);
      const float4 a1 = make_float4(c.Sd.hi, c.Sd.lo, __uint_as_float(c.txb), __uint_as_float(c.dxb));
      const float4 a2 = make_float4(__int_as_float(c.tmo), __uint_as_float(c.hint), 0.f, 0.f);
      st_cluster_f4(&cpart[rank][0], (unsigned)lane, a0);
      st_cluster_f4(&cpart[rank][4], (unsigned)lane, a1);
      st_cluster_f4(&cpart[rank][8], (unsigned)lane, a2);
    }
  }
  cluster_sync();  // every rank's part is in every rank's shared memory

  // 2. the unit's statistics and decision (warp 0 of every rank, rank order)
  if (warp == 0) {
    const Combined c = merge_parts(cpart, C);
    const float Stf = ff_to_f(c.St), Sdf = ff_to_f(c.Sd);
    int err = !(c.Ct > -INFINITY && c.Ct < INFINITY && Stf > 0.f && Stf < INFINITY);
    if (has_d) {
      err |= !(c.Cd > -INFINITY && c.Cd < INFINITY && Sdf > 0.f && Sdf < INFINITY);
      err |= !c.hx;  // no rank held x_j: the draft id is out of range
    }
    int acc = 1;
    float a = 0.f;
    if (has_d && !err) {
      // p/q = 2^((tx L - Ct) - (dx L - Cd)) * (Sd / St); the exponent is formed
      // exactly (two-product) and rounded once
      const float tx = __uint_as_float(c.txb), dx = __uint_as_float(c.dxb);
      float ratio = 0.f;
      if (tx > -INFINITY && dx > -INFINITY) {
        const ff ea = ff_add_f(two_prod(tx, kLog2e), -c.Ct);
        const ff ed = ff_add_f(two_prod(dx, kLog2e), -c.Cd);
        ratio = exp2f(ff_to_f(ff_sub(ea, ed))) * __fdiv_rn(Sdf, Stf);
      }
      a = fminf(ratio, 1.f);
      acc = uj < a;
    }
    // an earlier position of the row already rejected: this draw is not needed
    const bool earlier = c.hint > (uint32_t)(G + 1 - j);
    const int draw = !err && !c.tmo && (j == G || !acc) && !earlier;
    if (lane == 0) {
      D.ct = c.Ct;
      D.cd = has_d ? c.Cd : 0.f;
      D.invSt = __fdiv_rn(1.f, Stf);
      D.invSd = has_d ? __fdiv_rn(1.f, Sdf) : 0.f;
      D.a = a;
      D.us = us;
      D.err = err;
      D.tmo = c.tmo;
      D.acc = acc;
      D.draw = draw;
      D.mode = has_d ? 0 : 1;
      if (rank == 0) {
        if (has_d && P.acc_out) P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : a;
        if (has_d && !err && !acc) atomicMax(P.rej + b, (uint32_t)(G + 1 - j));
      }
    }
  }
  __syncthreads();

  if (!D.draw) {
    if (rank == 0) {
      if (tid == 0) {
        const uint32_t f = (D.acc ? kRecAccept : 0u) | (D.err ? kRecErr : 0u) |
                           (D.tmo ? kRecTimeout : 0u) | (D.mode ? kRecPDraw : 0u);
        write_record(P, b, j, f, -1, D, ff{0.f, 0.f});
      }
      if (warp == 0) arrive_and_finalize(P, b, lane);
    }
  } else {
    // 3. the draw: residual (or p) mass of every vector of this rank's slice
    int mode = D.mode;
    for (int attempt = 0; attempt < 2; ++attempt) {
      ff ts{0.f, 0.f};
      for (int v = tid; v < nv; v += kThreads) {
        const uint4 tv = lds128(s_t + 16 * (size_t)v);
        const uint4 dv = (mode == 0) ? lds128(s_d + 16 * (size_t)v) : make_uint4(0, 0, 0, 0);
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < epv; ++e)
          m = __fadd_rn(m, resid_val(vec_elem<BF>(tv, e), vec_elem<BF>(dv, e), D.ct, D.cd, D.invSt,
                                     D.invSd, mode));
        mass[v] = m;
        ts = ff_add_f(ts, m);
      }
      const ff Tc = block_sum_ff(ts, bs);
      if (warp == 0 && lane < C)
        st_cluster_f4(&cmass[attempt][rank][0], (unsigned)lane, make_float4(Tc.hi, Tc.lo, 0.f, 0.f));
      cluster_sync();  // every rank's mass is in every rank's shared memory
      if (warp == 0) {
        const ff tl = (lane < C) ? ff{cmass[attempt][lane][0], cmass[attempt][lane][1]} : ff{0.f, 0.f};
        // inclusive prefix over the ranks
        ff incl = tl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff y = ff_shfl_up(incl, o);
          if (lane >= o) incl = ff_add(incl, y);
        }
        const ff T = ff_shfl(incl, 31);
        if (!(T.hi > 0.f) && mode == 0 && attempt == 0) {
          if (lane == 0) s_redo = 1;  // zero residual (rounding only): draw from p_n
        } else {
          const ff target = ff_mul_f(T, D.us);
          const unsigned hit = __ballot_sync(0xffffffffu, lane < C && ff_gt(incl, target));
          int cs;
          if (hit) {
            cs = __ffs(hit) - 1;
          } else {  // u T at or past the total: the last rank with mass
            cs = (int)__reduce_max_sync(0xffffffffu, (unsigned)((lane < C && tl.hi > 0.f) ? lane + 1 : 0)) - 1;
            if (cs < 0) cs = 0;
          }
          const ff base = ff_sub(ff_shfl(incl, cs), ff_shfl(tl, cs));
          if (lane == 0) {
            s_redo = 0;
            s_cstar = cs;
            s_clamp = hit == 0u;
            const ff tg = ff_sub(target, base);
            s_tgt_hi = tg.hi;
            s_tgt_lo = tg.lo;
            s_T_hi = T.hi;
            s_T_lo = T.lo;
          }
        }
      }
      __syncthreads();
      if (!s_redo) break;
      mode = 1;
    }
    if (rank == s_cstar) {
      // 4. this rank holds the draw: a prefix over its vector masses (thread
      // t takes the contiguous run [t k, t k + k)), then one vector's elements
      const bool clamp = s_clamp != 0;
      const ff tgt{s_tgt_hi, s_tgt_lo};
      const int kk = (nv + kThreads - 1) / kThreads;
      const int v0 = min(nv, tid * kk), v1 = min(nv, v0 + kk);
      ff tsum{0.f, 0.f};
      int lastm = -1;
      for (int v = v0; v < v1; ++v) {
        tsum = ff_add_f(tsum, mass[v]);
        if (mass[v] > 0.f) lastm = v;
      }
      const ff ex = block_exclusive_scan_ff(tsum, bs);
      const bool cross = !clamp && v1 > v0 && ff_gt(ff_add(ex, tsum), tgt);
      int first, vlast;
      block_first_and_max(cross, lastm, bs, first, vlast);
      if (first < kThreads) {
        if (tid == first) {
          ff acc = ex;
          int vs = -1;
          for (int v = v0; v < v1; ++v) {
            const ff nx = ff_add_f(acc, mass[v]);
            if (ff_gt(nx, tgt)) {
              vs = v;
              break;
            }
            acc = nx;
          }
          const bool rounding = vs < 0;  // the thread's sum crossed, its steps did not
          if (rounding) vs = lastm >= 0 ? lastm : v0;
          s_tok = y0 + vs * epv + walk_vector<BF>(s_t, s_d, vs, D, mode, acc, tgt, rounding);
        }
      } else if (tid == 0) {  // clamped draw: the last vector with mass, its last element with mass
        const int vs = vlast >= 0 ? vlast : 0;
        s_tok = y0 + vs * epv + walk_vector<BF>(s_t, s_d, vs, D, mode, ff{0.f, 0.f}, tgt, true);
      }
      __syncthreads();
      if (tid == 0) {
        const uint32_t f = (D.acc ? kRecAccept : 0u) | (mode ? kRecPDraw : 0u) | kRecDrawn;
        write_record(P, b, j, f, s_tok, D, ff{s_T_hi, s_T_lo});
      }
      if (warp == 0) arrive_and_finalize(P, b, lane);
    }
  }
  // every copy has landed (each barrier was waited on), unless a wait ran out:
  // then wait once more, bounded, before the shared memory is released
  if (D.tmo) {
    const unsigned long long deadline = globaltimer() + kWaitNs;
    for (int k = 0; k < nch; ++k) mbar_wait_until(&bars[k], 0, deadline);
  }
}

// residual_out: the distribution the emitted token was drawn from, from the
// stop record the finalising unit kept.  One CTA per row; the record is
// cleared once every thread has read it.
template <bool BF>
__global__ void fused_resid_out_kernel(const __grid_constant__ FusedParams P, float* out) {
  constexpr int es = BF ? 2 : 4;
  const int b = blockIdx.x, G = P.G;
  float* o = out + (size_t)b * P.V;
  const int n = P.n_out[b];
  if (n < 0) {
    for (int y = threadIdx.x; y < P.V; y += blockDim.x) o[y] = 0.f;
    return;
  }
  UnitRec* rp = P.rec + (size_t)b * (G + 1) + n;
  const float4 r0 = __ldcg(reinterpret_cast<const float4*>(rp));
  const float4 r1 = __ldcg(reinterpret_cast<const float4*>(rp) + 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int4* q = reinterpret_cast<int4*>(rp);
    q[0] = make_int4(0, 0, 0, 0);
    q[1] = make_int4(0, 0, 0, 0);
  }
  const uint32_t flags = __float_as_uint(r0.x);
  const int mode = (flags & kRecPDraw) ? 1 : 0;
  const double T = (double)r1.z + (double)r1.w;
  if (!(T > 0.0)) {
    for (int y = threadIdx.x; y < P.V; y += blockDim.x) o[y] = 0.f;
    return;
  }
  const unsigned char* trow = P.lt + ((size_t)b * (G + 1) + n) * (size_t)P.V * es;
  const unsigned char* drow = mode == 0 ? P.ld + ((size_t)b * G + n) * (size_t)P.V * es : nullptr;
  const float invT = __fdiv_rn(1.f, (float)T);
  for (int y = threadIdx.x; y < P.V; y += blockDim.x) {
    const float t = BF ? bf16_to_f32(reinterpret_cast<const uint16_t*>(trow)[y])
                       : reinterpret_cast<const float*>(trow)[y];
    const float d = drow ? (BF ? bf16_to_f32(reinterpret_cast<const uint16_t*>(drow)[y])
                               : reinterpret_cast<const float*>(drow)[y])
                         : 0.f;
    o[y] = resid_val(t, d, r0.z, r0.w, r1.x, r1.y, mode) * invT;
  }
}

// per device: SM count, and which cluster sizes can be resident at all
struct DevInfo {
  int sms;
  unsigned char fits[kMaxCluster + 1];
};
DevInfo g_info[64];
bool g_ready[64] = {false};

cudaError_t device_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_ready[dev]) {
    DevInfo d{};
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const void* kern[2] = {(const void*)dense_fused_kernel<true>, (const void*)dense_fused_kernel<false>};
    for (const void* k : kern) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    for (int c = 1; c <= kMaxCluster; ++c) {
      // resident clusters of c CTAs at the largest shared-memory request
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(c * 64), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = kMaxDynSmem;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = (unsigned)c;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      cfg.attrs = a;
      cfg.numAttrs = 1;
      int n = 0;
      const int ok = cudaOccupancyMaxActiveClusters(&n, dense_fused_kernel<true>, &cfg) == cudaSuccess &&
                     cudaOccupancyMaxActiveClusters(&n, dense_fused_kernel<false>, &cfg) == cudaSuccess;
      d.fits[c] = (ok && n > 0) ? 1 : 0;
      (void)cudaGetLastError();  // a refused size is an answer, not an error
    }
    g_info[dev] = d;
    g_ready[dev] = true;
  }
  *out = &g_info[dev];
  return cudaSuccess;
}




// dynamic shared memory of a CTA: both slices, then the vector masses
size_t fused_smem(int L, int es) { return 2 * (size_t)L * es + (size_t)(L / (16 / es)) * sizeof(float); }

// resident CTAs of the fused kernel for a cluster size and shared-memory size
// (cached per device for the last few shapes)
struct ResidentCache {
  int C[8];
  size_t smem[8];
  int ctas[8];
  int next;
};
ResidentCache g_res[64];

int resident_ctas(int C, size_t smem, int bf16) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  ResidentCache& rc = g_res[dev];
  for (int i = 0; i < 8; ++i)
    if (rc.C[i] == C && rc.smem[i] == smem) return rc.ctas[i];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(C * 64), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = (unsigned)C;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = bf16 ? cudaOccupancyMaxActiveClusters(&n, dense_fused_kernel<true>, &cfg)
                             : cudaOccupancyMaxActiveClusters(&n, dense_fused_kernel<false>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  const int i = rc.next;
  rc.next = (rc.next + 1) % 8;
  rc.C[i] = C;
  rc.smem[i] = smem;
  rc.ctas[i] = n * C;
  return n * C;
}

}  // namespace

int fused_plan(long long B, int G, int V, int es, bool single_wave, int* L_out) {
  DevInfo* d = nullptr;
  if (device_info(&d) != cudaSuccess) return -1;
  const long long rowb = (long long)V * es;
  if (rowb % 16 != 0) return 0;
  const int epv = 16 / es;
  long long C = (rowb + kSliceBytes - 1) / kSliceBytes;
  // few units: spread each over more SMs (about two CTAs per SM in all)
  const long long units = B * (G + 1);
  const long long want = (2LL * d->sms + units - 1) / units;
  if (C < want) C = want;
  if (C > kMaxCluster) C = kMaxCluster;
  for (; C <= kMaxCluster; ++C) {
    const long long per = (V + C - 1) / C;
    const long long L = (per + epv - 1) / epv * epv;
    if (L * es > kSliceCapBytes || !d->fits[C]) continue;
    if (units * C > 0x7fffffffLL) return 0;
    // Measured on GB300: while the whole grid is resident at once the single
    // pass wins (no second launch, no second read); with several waves each
    // CTA's serial tail (exchange, decision, draw) holds its shared memory
    // idle and the two-kernel path is faster.
    if (single_wave && units * C > resident_ctas((int)C, fused_smem((int)L, es), es == 2)) return 0;
    *L_out = (int)L;
    return (int)C;
  }
  return 0;
}

cudaError_t launch_dense_fused(const FusedParams& p, int C, cudaStream_t s) {
  const int es = p.bf16 ? 2 : 4;
  const size_t smem = fused_smem(p.L, es);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)p.B * (p.G + 1) * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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
  return p.bf16 ? cudaLaunchKernelEx(&cfg, dense_fused_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, dense_fused_kernel<false>, p);
}

cudaError_t launch_dense_fused_resid_out(const FusedParams& p, float* resid_out, cudaStream_t s) {
  if (p.bf16)
    fused_resid_out_kernel<true><<<p.B, 512, 0, s>>>(p, resid_out);
  else
    fused_resid_out_kernel<false><<<p.B, 512, 0, s>>>(p, resid_out);
  return cudaGetLastError();
}

}  // namespace sv
