// sv_rounds.cu -- windowed multi-round any-order verification.
//
// Self-Speculative Masked Diffusions, key design 4: one non-causal pass gives
// the draft distributions of a window of positions, and several causal
// verification rounds run on them.  Round r verifies the still-masked window
// positions in sigma order against round r's target logits (the causal layer's
// recompute) with round r's draft tokens (after a resample the later drafts
// change); it ends at its first rejection, whose position is resampled from
// max(p - q, 0) renormalised (the any-order rule, key design 2) and revealed,
// and the next round starts after it.  A round that accepts every remaining
// draft closes the window; there is no bonus token.
//
// Design, vocabularies up to 512 (rounds_lane_kernel): one warp per sequence,
// every round in one launch; lane j takes window slot j of the current group
// of 32, forms its rows' statistics alone and keeps its draft statistics in
// registers; a ballot finds the round's first position that is not accepted,
// so nothing synchronises the block.  fp32 rows of at most 32 logits in a
// window of at most 32 positions (and at most kXC rounds) take a shorter
// chain: each lane loads every round's draft token and uniform for its slot
// at once and reads the draft logits at those tokens from its staged draft
// row, so a round is one staging of its target rows, the ballot and the draw.
//
// Design, larger vocabularies (rounds_kernel): one CTA of 8 warps per
// sequence, every round in one launch.  A round takes its positions eight at
// a time, one warp per position: the warp reads
// the target row, forms its softmax statistics (c = log2e * max, S in
// float-float) and the accept probability at its draft token (the same
// arithmetic as the single-round kernels); the draft row's statistics are
// computed once per window position and kept in shared memory for the later
// rounds.  After each group a barrier finds the group's first non-accepted
// position; positions after it are never used (their errors do not count).
// Warp 0 then draws the replacement by a float-float prefix over the fp32
// residual in ascending id order.
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kRWarps = 8;
constexpr int kRThreads = 32 * kRWarps;
constexpr int kLWarps = 4;  // sequences (warps) per CTA of the lane-per-position kernel
constexpr int kLThreads = 32 * kLWarps;
constexpr int kDraftCache = 1024;  // window positions whose draft statistics are kept
constexpr int kLaneMaxV = 512;     // vocabularies a lane reduces alone
constexpr int kXC = 4;             // rounds whose inputs a lane keeps (the one-group fast path)

__device__ __forceinline__ float logit_at(const unsigned char* row, int y, int bf16) {
  if (bf16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[y]);
  return reinterpret_cast<const float*>(row)[y];
}

struct Stats {
  float c, S;  // c = log2e * max (-inf for no finite entry), S = sum 2^(v log2e - c)
  int bad;     // NaN, +inf or no finite entry
};

// softmax statistics of one logit row, the whole warp (lane-strided reads);
// every lane returns them
__device__ __forceinline__ Stats row_stats_global(const unsigned char* row, int V, int bf16, int lane) {
  float m = -INFINITY;
  int odd = 0;
  for (int y = lane; y < V; y += 32) {
    const float v = logit_at(row, y, bf16);
    odd |= (v != v) || (v == INFINITY);
    m = fmaxf(m, v);
  }
  m = warp_max(m);
  odd = __any_sync(0xffffffffu, odd);
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  ff a{0.f, 0.f};
  for (int y = lane; y < V; y += 32) a = ff_add_f(a, ex2(fmaf(logit_at(row, y, bf16), kLog2e, -c)));
  Stats s;
  s.S = ff_to_f(warp_sum_ff(a));
  s.c = (m == -INFINITY) ? -INFINITY : c;
  s.bad = odd || !(m > -INFINITY) || !(s.S > 0.f) || !(s.S < INFINITY);
  return s;
}

// min(1, p(x) / q(x)) from the two logits at x and the rows' statistics:
// log2 p(x) - log2 q(x) formed exactly (two-product), rounded once
__device__ __forceinline__ float accept_prob(float tx, float dx, const Stats& t, const Stats& d) {
  float ratio = 0.f;
  if (tx > -INFINITY && dx > -INFINITY) {
    const ff ea = ff_add_f(two_prod(tx, kLog2e), -t.c);
    const ff ed = ff_add_f(two_prod(dx, kLog2e), -d.c);
    ratio = exp2f(ff_to_f(ff_sub(ea, ed))) * __fdiv_rn(d.S, t.S);
  }
  return fminf(ratio, 1.f);
}

// residual (mode 0: max(p - q, 0)) or target (mode 1: p) mass of id y
__device__ __forceinline__ float draw_mass(const unsigned char* trow, const unsigned char* drow, int y,
                                           int bf16, float tc, float tinv, float dc, float dinv,
                                           int mode) {
  const float p = __fmul_rn(ex2(__fmaf_rn(logit_at(trow, y, bf16), kLog2e, -tc)), tinv);
  if (mode != 0) return p;
  const float q = __fmul_rn(ex2(__fmaf_rn(logit_at(drow, y, bf16), kLog2e, -dc)), dinv);
  const float r = __fsub_rn(p, q);
  return r > 0.f ? r : 0.f;
}

// Inverse CDF at one position, the whole warp: the smallest id whose
// inclusive prefix of the residual exceeds u T (T its total), ids ascending;
// a zero residual (possible only through rounding) draws from p instead, and
// u T at or past the total through rounding takes the last id with mass.
__device__ int warp_draw(const unsigned char* trow, const unsigned char* drow, int V, int bf16,
                         float tc, float tS, float dc, float dS, float u, int lane) {
  const float tinv = 1.f / tS, dinv = 1.f / dS;
  for (int mode = 0; mode < 2; ++mode) {
    ff tot{0.f, 0.f};
    for (int y = lane; y < V; y += 32) tot = ff_add_f(tot, draw_mass(trow, drow, y, bf16, tc, tinv, dc, dinv, mode));
    tot = warp_sum_ff(tot);
    if (!(tot.hi > 0.f)) continue;  // (mode 1 always has mass: the target row is valid)
    const ff target = ff_mul_f(tot, u);
    ff carry{0.f, 0.f};
    int last = -1;
    for (int y0 = 0; y0 < V; y0 += 32) {
      const int y = y0 + lane;
      const float m = (y < V) ? draw_mass(trow, drow, y, bf16, tc, tinv, dc, dinv, mode) : 0.f;
      const ff ex = warp_exclusive_scan_ff(ff{m, 0.f}, lane);
      const ff incl = ff_add(carry, ff_add_f(ex, m));
      const unsigned hit = __ballot_sync(0xffffffffu, y < V && ff_gt(incl, target));
      if (hit) return y0 + __ffs(hit) - 1;
      const unsigned pos = __ballot_sync(0xffffffffu, m > 0.f);
      if (pos) last = y0 + 31 - __clz(pos);
      carry = ff_shfl(incl, 31);
    }
    return last >= 0 ? last : V - 1;
  }
  return V - 1;
}

__global__ void __launch_bounds__(kRThreads) rounds_kernel(const __grid_constant__ RoundsParams P) {
  __shared__ float s_dc[kDraftCache], s_dS[kDraftCache];
  __shared__ unsigned char s_dstate[kDraftCache];  // 0 not yet, 1 computed, 2 bad row
  __shared__ int s_res[kRWarps];                   // 0 accepted, 1 rejected, 2 input error, 3 past the window
  __shared__ float s_st[kRWarps][4];               // target c, S and draft c, S of the warp's position
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, R = P.R, D = P.D, V = P.V;
  const size_t es = P.bf16 ? 2 : 4;
  const int32_t* sig = P.order + (size_t)b * D;
  int32_t* out = P.tok_out + (size_t)b * D;
  int32_t* racc = P.racc_out + (size_t)b * R;
  const int i0 = P.i0[b], W = P.win[b];
  int bad = (i0 < 0 || i0 > D || W < 1);
  const int e = bad ? 0 : ((W > D - i0) ? D : i0 + W);  // the window is sigma[i0, e)

  // sigma inside the window: in range and without repeats
  int odd = 0;
  for (int k = i0 + tid; k < e; k += kRThreads) {
    const int s = sig[k];
    odd |= (s < 0 || s >= D);
    for (int k2 = i0; k2 < k && !odd; ++k2) odd |= (sig[k2] == s);
  }
  for (int k = tid; k < kDraftCache; k += kRThreads) s_dstate[k] = 0;
  for (int r = tid; r < R; r += kRThreads) racc[r] = -1;  // rounds that do not run stay -1
  bad |= __syncthreads_or(odd);

  int i = i0;  // sigma index of the first still-masked window position
  for (int r = 0; r < R; ++r) {
    if (bad || i >= e) break;  // uniform
    const size_t rr = ((size_t)b * R + r) * (size_t)D;  // round r's [D] slice
    int stop = e, stop_w = 0, err = 0;
    for (int kb = i; kb < e; kb += kRWarps) {
      const int k = kb + warp;
      if (k < e) {
        const int s = sig[k];
        const int x = P.x[rr + s];
        const unsigned char* trow = P.lt + (rr + s) * (size_t)V * es;
        const unsigned char* drow = P.ld + ((size_t)b * D + s) * (size_t)V * es;
        const Stats t = row_stats_global(trow, V, P.bf16, lane);
        Stats d;
        const int slot = k - i0;
        if (slot < kDraftCache && s_dstate[slot] != 0) {
          d.c = s_dc[slot];
          d.S = s_dS[slot];
          d.bad = s_dstate[slot] == 2;
        } else {
          d = row_stats_global(drow, V, P.bf16, lane);
          if (slot < kDraftCache && lane == 0) {
            s_dc[slot] = d.c;
            s_dS[slot] = d.S;
            s_dstate[slot] = d.bad ? 2 : 1;
          }
        }
        int res = 2;
        if (!t.bad && !d.bad && x >= 0 && x < V) {
          const float a = accept_prob(logit_at(trow, x, P.bf16), logit_at(drow, x, P.bf16), t, d);
          res = (P.u_acc[rr + k] < a) ? 0 : 1;
        }
        if (lane == 0) {
          s_res[warp] = res;
          s_st[warp][0] = t.c;
          s_st[warp][1] = t.S;
          s_st[warp][2] = d.c;
          s_st[warp][3] = d.S;
        }
      } else if (lane == 0) {
        s_res[warp] = 3;
      }
      __syncthreads();
      int first = -1, kind = 0;
      for (int w2 = 0; w2 < kRWarps; ++w2) {
        const int v = s_res[w2];
        if (v == 3) break;
        if (v != 0) {
          first = w2;
          kind = v;
          break;
        }
      }
      if (first >= 0) {  // uniform: every thread read the same flags
        stop = kb + first;
        stop_w = first;
        err = (kind == 2);
        break;
      }
      __syncthreads();  // the flags are rewritten by the next group
    }
    if (err) {
      bad = 1;
      break;
    }
    for (int k = i + tid; k < stop; k += kRThreads) out[sig[k]] = P.x[rr + sig[k]];
    if (tid == 0) racc[r] = stop - i;
    if (stop < e) {
      if (warp == 0) {
        const int s = sig[stop];
        const unsigned char* trow = P.lt + (rr + s) * (size_t)V * es;
        const unsigned char* drow = P.ld + ((size_t)b * D + s) * (size_t)V * es;
        const int y = warp_draw(trow, drow, V, P.bf16, s_st[stop_w][0], s_st[stop_w][1],
                                s_st[stop_w][2], s_st[stop_w][3], P.u_s[(size_t)b * R + r], lane);
        if (lane == 0) out[s] = y;
      }
      i = stop + 1;
    } else {
      i = e;
    }
    __syncthreads();  // s_st and s_res are reused by the next round
  }

  if (bad) {
    for (int k = (i0 > 0 ? i0 : 0) + tid; k < e; k += kRThreads) {
      const int s = sig[k];
      if (s >= 0 && s < D) out[s] = -1;
    }
    for (int r = tid; r < R; r += kRThreads) racc[r] = -1;
    if (tid == 0) {
      P.n_out[b] = -1;
      atomicOr(P.status, kStatusInputErr);
    }
    return;
  }
  if (tid == 0) P.n_out[b] = i;
}

// softmax statistics of one logit row, one lane alone (small vocabularies):
// the same quantities as row_stats_global, float-float sum
__device__ __forceinline__ Stats row_stats_lane(const unsigned char* row, int V, int bf16) {
  float m = -INFINITY;
  int odd = 0;
  for (int y = 0; y < V; ++y) {
    const float v = logit_at(row, y, bf16);
    odd |= (v != v) || (v == INFINITY);
    m = fmaxf(m, v);
  }
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  ff a0{0.f, 0.f}, a1{0.f, 0.f};
  int y = 0;
  for (; y + 1 < V; y += 2) {
    a0 = ff_add_f(a0, ex2(fmaf(logit_at(row, y, bf16), kLog2e, -c)));
    a1 = ff_add_f(a1, ex2(fmaf(logit_at(row, y + 1, bf16), kLog2e, -c)));
  }
  if (y < V) a0 = ff_add_f(a0, ex2(fmaf(logit_at(row, y, bf16), kLog2e, -c)));
  Stats s;
  s.S = ff_to_f(ff_add(a0, a1));
  s.c = (m == -INFINITY) ? -INFINITY : c;
  s.bad = odd || !(m > -INFINITY) || !(s.S > 0.f) || !(s.S < INFINITY);
  return s;
}

// The same statistics for an fp32 row of at most 32 logits: the lane copies
// its row into its own shared-memory slot with independent 4-byte cp.async
// copies (one round trip instead of a chain of loads), then reduces it there;
// a slot stride of 33 floats keeps the lanes of a warp in distinct banks.
__device__ __forceinline__ Stats row_stats_lane_staged(const unsigned char* row, int V, float* slot) {
  const float* g = reinterpret_cast<const float*>(row);
  for (int y = 0; y < V; ++y)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(slot + y)), "l"(g + y)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  float m = -INFINITY;
  int odd = 0;
  for (int y = 0; y < V; ++y) {
    const float v = slot[y];
    odd |= (v != v) || (v == INFINITY);
    m = fmaxf(m, v);
  }
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  ff a0{0.f, 0.f}, a1{0.f, 0.f};
  int y = 0;
  for (; y + 1 < V; y += 2) {
    a0 = ff_add_f(a0, ex2(fmaf(slot[y], kLog2e, -c)));
    a1 = ff_add_f(a1, ex2(fmaf(slot[y + 1], kLog2e, -c)));
  }
  if (y < V) a0 = ff_add_f(a0, ex2(fmaf(slot[y], kLog2e, -c)));
  Stats s;
  s.S = ff_to_f(ff_add(a0, a1));
  s.c = (m == -INFINITY) ? -INFINITY : c;
  s.bad = odd || !(m > -INFINITY) || !(s.S > 0.f) || !(s.S < INFINITY);
  return s;
}

// Small vocabularies: one warp per sequence, lane j on window slot j of the
// current group of 32 (sigma index i0 + 32 g + j).  Each active lane forms its
// rows' statistics alone (the draft row's once, kept in registers for the
// first group); a ballot gives the first position that is not accepted, so a
// round needs no block barrier; the whole warp then draws.
__global__ void __launch_bounds__(kLThreads) rounds_lane_kernel(const __grid_constant__ RoundsParams P) {
  __shared__ float s_rowbuf[kLWarps * 32 * 33];
  // one-group fast path: per lane, every round's draft token, accept uniform
  // and the draft logit at that token
  __shared__ int s_xr[kLWarps][kXC][32];
  __shared__ float s_ua[kLWarps][kXC][32];
  __shared__ float s_dx[kLWarps][kXC][32];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  float* const rslot = s_rowbuf + (threadIdx.x >> 5) * 32 * 33 + lane * 33;
  const bool staged = !P.bf16 && P.V <= 32;  // fp32 rows short enough to stage
  const int b = blockIdx.x * kLWarps + (threadIdx.x >> 5);
  if (b >= P.B) return;  // whole warps only: nothing below synchronises the block
  const int R = P.R, D = P.D, V = P.V;
  const size_t es = P.bf16 ? 2 : 4;
  const int32_t* sig = P.order + (size_t)b * D;
  int32_t* out = P.tok_out + (size_t)b * D;
  int32_t* racc = P.racc_out + (size_t)b * R;
  const int i0 = P.i0[b], W = P.win[b];
  int bad = (i0 < 0 || i0 > D || W < 1);
  const int e = bad ? 0 : ((W > D - i0) ? D : i0 + W);
  int odd = 0;
  int s0 = 0;  // sigma of this lane's slot in group 0 (sigma index i0 + lane)
  for (int k = i0 + lane; k < e; k += 32) {
    const int s = sig[k];
    if (k == i0 + lane) s0 = s;
    odd |= (s < 0 || s >= D);
    for (int k2 = i0; k2 < k && !odd; ++k2) odd |= (sig[k2] == s);
  }
  for (int r = lane; r < R; r += 32) racc[r] = -1;
  bad |= __any_sync(0xffffffffu, odd);
  __syncwarp();

  Stats dcache;  // the draft statistics of this lane's slot in group 0
  int have = 0;
  int i = i0;
  // The fast path (fp32 rows of at most 32 logits, a window of at most 32
  // positions, at most kXC rounds): the lane loads every round's draft token
  // and uniform for its slot at once, stages its draft row first and reads
  // the draft logits at those tokens from it; a round is then one staging of
  // its target rows (the target logit at the token read from the stage), the
  // ballot and the draw, and the accepted prefix is written from registers.
  const bool fast = staged && !bad && R <= kXC && e - i0 <= 32;  // warp-uniform
  if (fast && i0 + lane < e) {
    int xv[kXC];
    float uv[kXC];
#pragma unroll
    for (int r = 0; r < kXC; ++r) {
      if (r < R) {
        const size_t rr = ((size_t)b * R + r) * (size_t)D;
        xv[r] = P.x[rr + s0];
        uv[r] = P.u_acc[rr + i0 + lane];
      }
    }
    dcache = row_stats_lane_staged(P.ld + ((size_t)b * D + s0) * (size_t)V * es, V, rslot);
    have = 1;
#pragma unroll
    for (int r = 0; r < kXC; ++r) {
      if (r < R) {
        s_xr[wi][r][lane] = xv[r];
        s_ua[wi][r][lane] = uv[r];
        s_dx[wi][r][lane] = (xv[r] >= 0 && xv[r] < V) ? rslot[xv[r]] : 0.f;
      }
    }
  }
  __syncwarp();
  for (int r = 0; fast && r < R; ++r) {
    if (bad || i >= e) break;  // warp-uniform
    const size_t rr = ((size_t)b * R + r) * (size_t)D;
    const int k = i0 + lane;
    const bool active = (k >= i) && (k < e);
    int res = 0;
    Stats t{0.f, 1.f, 0};
    const Stats d = dcache;
    if (active) {
      t = row_stats_lane_staged(P.lt + (rr + s0) * (size_t)V * es, V, rslot);
      const int x = s_xr[wi][r][lane];
      res = 2;
      if (!t.bad && !d.bad && x >= 0 && x < V) {
        const float a = accept_prob(rslot[x], s_dx[wi][r][lane], t, d);
        res = (s_ua[wi][r][lane] < a) ? 0 : 1;
      }
    }
    const unsigned nacc = __ballot_sync(0xffffffffu, active && res != 0);
    int stop = e;
    if (nacc) {
      const int j = __ffs(nacc) - 1;
      stop = i0 + j;
      if (__shfl_sync(0xffffffffu, res, j) == 2) {
        bad = 1;
        break;
      }
      const float tc = __shfl_sync(0xffffffffu, t.c, j), tS = __shfl_sync(0xffffffffu, t.S, j);
      const float dc = __shfl_sync(0xffffffffu, d.c, j), dS = __shfl_sync(0xffffffffu, d.S, j);
      const int s = __shfl_sync(0xffffffffu, s0, j);
      if (active && k < stop) out[s0] = s_xr[wi][r][lane];
      if (lane == 0) racc[r] = stop - i;
      const int y = warp_draw(P.lt + (rr + s) * (size_t)V * es, P.ld + ((size_t)b * D + s) * (size_t)V * es,
                              V, P.bf16, tc, tS, dc, dS, P.u_s[(size_t)b * R + r], lane);
      if (lane == 0) out[s] = y;
      i = stop + 1;
    } else {
      if (active) out[s0] = s_xr[wi][r][lane];
      if (lane == 0) racc[r] = stop - i;
      i = e;
    }
    __syncwarp();
  }
  for (int r = 0; !fast && r < R; ++r) {
    if (bad || i >= e) break;  // warp-uniform
    const size_t rr = ((size_t)b * R + r) * (size_t)D;
    int stop = e, err = 0;
    Stats st{0.f, 1.f, 0}, sd{0.f, 1.f, 0};  // the stop position's statistics
    for (int g = (i - i0) >> 5; i0 + 32 * g < e; ++g) {
      const int k = i0 + 32 * g + lane;
      const bool active = (k >= i) && (k < e);
      int res = 0;
      Stats t{0.f, 1.f, 0}, d{0.f, 1.f, 0};
      if (active) {
        const int s = sig[k];
        const int x = P.x[rr + s];
        const unsigned char* trow = P.lt + (rr + s) * (size_t)V * es;
        const unsigned char* drow = P.ld + ((size_t)b * D + s) * (size_t)V * es;
        t = staged ? row_stats_lane_staged(trow, V, rslot) : row_stats_lane(trow, V, P.bf16);
        if (g == 0 && have) {
          d = dcache;
        } else {
          d = staged ? row_stats_lane_staged(drow, V, rslot) : row_stats_lane(drow, V, P.bf16);
          if (g == 0) {
            dcache = d;
            have = 1;
          }
        }
        res = 2;
        if (!t.bad && !d.bad && x >= 0 && x < V) {
          const float a = accept_prob(logit_at(trow, x, P.bf16), logit_at(drow, x, P.bf16), t, d);
          res = (P.u_acc[rr + k] < a) ? 0 : 1;
        }
      }
      const unsigned nacc = __ballot_sync(0xffffffffu, active && res != 0);
      if (nacc) {
        const int j = __ffs(nacc) - 1;
        stop = i0 + 32 * g + j;
        err = __shfl_sync(0xffffffffu, res, j) == 2;
        st.c = __shfl_sync(0xffffffffu, t.c, j);
        st.S = __shfl_sync(0xffffffffu, t.S, j);
        sd.c = __shfl_sync(0xffffffffu, d.c, j);
        sd.S = __shfl_sync(0xffffffffu, d.S, j);
        break;
      }
    }
    if (err) {
      bad = 1;
      break;
    }
    for (int k = i + lane; k < stop; k += 32) out[sig[k]] = P.x[rr + sig[k]];
    if (lane == 0) racc[r] = stop - i;
    if (stop < e) {
      const int s = sig[stop];
      const unsigned char* trow = P.lt + (rr + s) * (size_t)V * es;
      const unsigned char* drow = P.ld + ((size_t)b * D + s) * (size_t)V * es;
      const int y = warp_draw(trow, drow, V, P.bf16, st.c, st.S, sd.c, sd.S, P.u_s[(size_t)b * R + r], lane);
      if (lane == 0) out[s] = y;
      i = stop + 1;
    } else {
      i = e;
    }
    __syncwarp();
  }

  if (bad) {
    __syncwarp();
    for (int k = (i0 > 0 ? i0 : 0) + lane; k < e; k += 32) {
      const int s = sig[k];
      if (s >= 0 && s < D) out[s] = -1;
    }
    for (int r = lane; r < R; r += 32) racc[r] = -1;
    if (lane == 0) {
      P.n_out[b] = -1;
      atomicOr(P.status, kStatusInputErr);
    }
    return;
  }
  if (lane == 0) P.n_out[b] = i;
}

}  // namespace

cudaError_t launch_rounds(const RoundsParams& p, cudaStream_t s) {
  if (p.V <= kLaneMaxV) {  // a lane per window position, a warp per sequence
    rounds_lane_kernel<<<(p.B + kLWarps - 1) / kLWarps, kLThreads, 0, s>>>(p);
  } else {  // a warp per window position, a CTA per sequence
    rounds_kernel<<<p.B, kRThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace sv
