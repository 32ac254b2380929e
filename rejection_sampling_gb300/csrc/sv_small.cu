// sv_small.cu -- warp-per-row verification for small vocabularies.
//
// One warp verifies one row (dense) or one sequence window (any-order).  The
// row block is staged in shared memory with an odd row stride, so lane i can
// read position i's row with no bank conflicts; lane i owns position i:
// softmax statistics of its target and draft rows (for a few long rows the
// warp computes them together, one row at a time), the gather at its draft
// token and its accept test.  A ballot gives the first rejection; the whole
// warp then draws the replacement (or the bonus token) by a float-float prefix over
// the fp32 residual values in ascending id order.
//
//  dense     : positions 0..gamma; target rows 0..gamma, draft rows 0..gamma-1;
//              bonus from p_gamma when every draft is accepted (DFlash/DFlash2
//              guide, section 2).
//  any-order : window index i verifies sequence position sigma_i; the round
//              ends at the first rejection, whose position is resampled from
//              max(0, target - draft); no bonus (Self-Speculative Masked
//              Diffusions, key design 2).
#include "sv_common.cuh"

namespace sv {
namespace {

__device__ __forceinline__ float ld_logit(const unsigned char* base, size_t idx, int bf16) {
  if (bf16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ float resid_val(float t, float d, float ct, float cd, float invSt,
                                           float invSd, int mode) {
  const float p = __fmul_rn(ex2(__fmaf_rn(t, kLog2e, -ct)), invSt);
  if (mode != 0) return p;
  const float q = __fmul_rn(ex2(__fmaf_rn(d, kLog2e, -cd)), invSd);
  const float r = __fsub_rn(p, q);
  return r > 0.f ? r : 0.f;
}

// softmax statistics of one shared-memory row, one lane alone:
// c = log2e * max, S = sum 2^(v log2e - c).  Up to 256 terms the sum runs in
// four fp32 partial sums (at most 64 terms each, so its relative error stays
// below 64 units in the last place); longer rows are summed in float-float.
__device__ __forceinline__ void row_stats(const float* row, int V, float& c_out, float& s_out) {
  float m = -INFINITY;
  for (int y = 0; y < V; ++y) m = fmaxf(m, row[y]);
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  int y = 0;
  if (V <= 256) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (; y + 3 < V; y += 4) {
      a0 += ex2(fmaf(row[y], kLog2e, -c));
      a1 += ex2(fmaf(row[y + 1], kLog2e, -c));
      a2 += ex2(fmaf(row[y + 2], kLog2e, -c));
      a3 += ex2(fmaf(row[y + 3], kLog2e, -c));
    }
    for (; y < V; ++y) a0 += ex2(fmaf(row[y], kLog2e, -c));
    s_out = (a0 + a1) + (a2 + a3);
  } else {
    ff a0{0.f, 0.f}, a1{0.f, 0.f};
    for (; y + 1 < V; y += 2) {
      a0 = ff_add_f(a0, ex2(fmaf(row[y], kLog2e, -c)));
      a1 = ff_add_f(a1, ex2(fmaf(row[y + 1], kLog2e, -c)));
    }
    if (y < V) a0 = ff_add_f(a0, ex2(fmaf(row[y], kLog2e, -c)));
    s_out = ff_to_f(ff_add(a0, a1));
  }
  c_out = (m == -INFINITY) ? -INFINITY : c;
}

// the same statistics, the whole warp on one row (lane-strided, then reduced);
// every lane returns them
__device__ __forceinline__ void row_stats_warp(const float* row, int V, int lane, float& c_out,
                                               float& s_out) {
  float m = -INFINITY;
  for (int y = lane; y < V; y += 32) m = fmaxf(m, row[y]);
  m = warp_max(m);
  const float c = (m == -INFINITY) ? 0.f : m * kLog2e;
  ff a{0.f, 0.f};
  for (int y = lane; y < V; y += 32) a = ff_add_f(a, ex2(fmaf(row[y], kLog2e, -c)));
  s_out = ff_to_f(warp_sum_ff(a));
  c_out = (m == -INFINITY) ? -INFINITY : c;
}

__device__ __forceinline__ bool stats_ok(float c, float s) {
  return c > -INFINITY && c < INFINITY && s > 0.f && s < INFINITY;
}

__global__ void small_verify_kernel(const __grid_constant__ SmallParams P) {
  extern __shared__ float smem[];
  pdl_wait_then_release();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= P.B) return;  // whole warp leaves; no block-wide barrier below
  const int R = P.R, VS = P.vstride, V = P.V, NT = P.G;  // NT accept tests
  float* st = smem + (size_t)warp * 2 * R * VS;
  float* sd = st + (size_t)R * VS;

  // ---- rows and validation of the window ----
  int sig = lane, bad = 0;
  if (P.anyorder) {
    if (lane < R) {
      sig = P.order[(size_t)b * R + lane];
      if (sig < 0 || sig >= P.D) bad = 1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, lane < R ? sig : -1 - lane);
    if (lane < R && __popc(same) > 1) bad = 1;
  }
  bad = __any_sync(0xffffffffu, bad);
  // the row's small inputs, issued now so their latency hides behind the
  // staging: lane i's accept uniform and draft token (any-order: the token at
  // sigma_i; when the whole sequence is the window it is read in position
  // order and moved to lane i by a shuffle), and the sample uniform
  const bool xin = P.anyorder && P.D <= 32;
  int xsrc = 0;
  float uacc = 1.f;
  if (lane < NT) uacc = P.u_acc[(size_t)b * NT + lane];
  if (P.anyorder) {
    if (xin) {
      if (lane < P.D) xsrc = P.x[(size_t)b * P.D + lane];
    } else if (lane < R && !bad) {
      xsrc = P.x[(size_t)b * P.D + sig];
    }
  } else if (lane < NT) {
    xsrc = P.x[(size_t)b * NT + lane];
  }
  const float usamp = P.u_s[b];

  // ---- stage the rows in shared memory (row r of the warp = position r) ----
  // The R x V block is walked flat, 32 consecutive elements per step, so every
  // lane works in every step and each row is read contiguously.  fp32 rows
  // move with 4-byte cp.async (all steps in flight at once); bf16 rows are
  // widened in registers, kBatch steps of loads in flight before their stores.
  if (P.flat) {
    // fp32 blocks whose size and start are 16-byte multiples: copied whole, in
    // source order (any-order: sequence positions, read through sigma below)
    const int nt = (P.anyorder ? P.D : NT + 1) * V / 4, nd = (P.anyorder ? P.D : NT) * V / 4;
    const float4* ts = reinterpret_cast<const float4*>(P.lt) + (size_t)b * nt;
    const float4* ds = reinterpret_cast<const float4*>(P.ld) + (size_t)b * nd;
    // two copy groups: the target block, then the draft block -- the target
    // statistics run while the draft block is still arriving
    for (int i = lane; i < nt; i += 32)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(st + 4 * i)), "l"(ts + i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = lane; i < nd; i += 32)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sd + 4 * i)), "l"(ds + i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  } else {
    const int total = R * V;
    int r = lane / V, y = lane - (lane / V) * V;  // (row, column) of element `lane`
    auto rows_of = [&](int rr, size_t& trow, size_t& drow, bool& hasd) {
      if (P.anyorder) {
        int sg = __shfl_sync(0xffffffffu, sig, rr);
        if (bad) sg = 0;
        trow = drow = (size_t)b * P.D + sg;
        hasd = true;
      } else {
        trow = (size_t)b * (NT + 1) + rr;
        drow = (size_t)b * NT + rr;
        hasd = rr < NT;
      }
    };
    auto advance = [&]() {  // the next element of this lane, 32 further on
      y += 32;
      while (y >= V) {
        y -= V;
        ++r;
      }
    };
    if (!P.bf16) {
      const float* lt = reinterpret_cast<const float*>(P.lt);
      const float* ld = reinterpret_cast<const float*>(P.ld);
      for (int base = 0; base < total; base += 32) {
        const bool on = base + lane < total;
        const int rr = on ? r : 0;
        size_t trow, drow;
        bool hasd;
        rows_of(rr, trow, drow, hasd);
        if (on) {
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(st + rr * VS + y)),
                       "l"(lt + trow * V + y)
                       : "memory");
          if (hasd)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sd + rr * VS + y)),
                         "l"(ld + drow * V + y)
                         : "memory");
        }
        advance();
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
      constexpr int kBatch = 8;
      for (int base = 0; base < total; base += 32 * kBatch) {
        float tv[kBatch], dv[kBatch];
        int ri[kBatch], yi[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const bool on = base + 32 * q + lane < total;
          const int rr = on ? r : 0;
          size_t trow, drow;
          bool hasd;
          rows_of(rr, trow, drow, hasd);
          ri[q] = on ? rr : -1;
          yi[q] = y;
          tv[q] = on ? ld_logit(P.lt, trow * V + y, 1) : 0.f;
          dv[q] = (on && hasd) ? ld_logit(P.ld, drow * V + y, 1) : 0.f;
          advance();
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (ri[q] >= 0) {
            st[ri[q] * VS + yi[q]] = tv[q];
            if (P.anyorder || ri[q] < NT) sd[ri[q] * VS + yi[q]] = dv[q];
          }
        }
      }
    }
  }
  __syncwarp();

  // ---- per-position statistics and accept test (lane = position) ----
  // shared-memory row of this lane's position (valid when !bad)
  const int prow = (P.flat && P.anyorder) ? sig : lane;
  float ct = 0.f, St = 1.f, cd = 0.f, Sd = 1.f, a = 0.f;
  int err = bad, acc = 1, x = 0;
  // Lane r computes row r's statistics alone while rows are short next to
  // their count; for few long rows the whole warp takes one row at a time
  // (about R * (V / 32 + 20) steps instead of V).
  const bool by_warp = R * (V + 640) < 32 * V;
  if (P.flat && by_warp) {  // the warp-wide statistics read both blocks at once
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  if (!bad && by_warp) {
    for (int r = 0; r < R; ++r) {
      const int rr = (P.flat && P.anyorder) ? __shfl_sync(0xffffffffu, sig, r) : r;
      float c1, s1;
      row_stats_warp(st + rr * VS, V, lane, c1, s1);
      if (lane == r) ct = c1, St = s1;
      if (r < NT) {
        row_stats_warp(sd + rr * VS, V, lane, c1, s1);
        if (lane == r) cd = c1, Sd = s1;
      }
    }
  }
  if (xin) x = __shfl_sync(0xffffffffu, xsrc, (sig >= 0 && sig < 32) ? sig : 0);
  else x = xsrc;
  if (!bad && lane < R && !by_warp) row_stats(st + prow * VS, V, ct, St);
  if (P.flat && !by_warp) {  // the draft block's copy group
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  if (!bad && lane < R) {
    err |= !stats_ok(ct, St);
    if (lane < NT) {
      if (!by_warp) row_stats(sd + prow * VS, V, cd, Sd);
      err |= !stats_ok(cd, Sd);
      if (x < 0 || x >= V) err = 1;
      if (!err) {
        const float tx = st[prow * VS + x], dx = sd[prow * VS + x];
        float ratio = 0.f;
        if (tx > -INFINITY && dx > -INFINITY) {
          // log2 p(x) - log2 q(x) formed exactly (two-product), rounded once
          const ff ea = ff_add_f(two_prod(tx, kLog2e), -ct);
          const ff ed = ff_add_f(two_prod(dx, kLog2e), -cd);
          ratio = exp2f(ff_to_f(ff_sub(ea, ed))) * __fdiv_rn(Sd, St);
        }
        a = fminf(ratio, 1.f);
        acc = uacc < a;
      }
    }
  }
  err = __any_sync(0xffffffffu, err);
  if (P.acc_out && lane < NT) P.acc_out[(size_t)b * NT + lane] = err ? __int_as_float(0x7fc00000) : a;
  const unsigned rej = __ballot_sync(0xffffffffu, lane < NT && !acc);
  const int n = err ? -1 : (rej ? __ffs(rej) - 1 : NT);

  // ---- draw at the stop position ----
  int y = -1;
  int mode = 2;  // 0 residual, 1 p only, 2 none
  ff T{0.f, 0.f};
  float sct = 0.f, scd = 0.f, sist = 0.f, sisd = 0.f;
  int srow = 0;
  if (n >= 0 && (n < NT || !P.anyorder)) {
    mode = (n < NT) ? 0 : 1;
    srow = (P.flat && P.anyorder) ? __shfl_sync(0xffffffffu, sig, n) : n;  // its shared-memory row
    sct = __shfl_sync(0xffffffffu, ct, n);
    scd = __shfl_sync(0xffffffffu, cd, n);
    sist = 1.f / __shfl_sync(0xffffffffu, St, n);
    sisd = 1.f / __shfl_sync(0xffffffffu, Sd, n);
    const int q = (V + 31) / 32;
    const int e0 = min(V, lane * q), e1 = min(V, e0 + q);
    const float* tr = st + srow * VS;
    const float* dr = sd + srow * VS;
    for (int attempt = 0; attempt < 2; ++attempt) {
      ff ls{0.f, 0.f};
      for (int e = e0; e < e1; ++e) ls = ff_add_f(ls, resid_val(tr[e], dr[e], sct, scd, sist, sisd, mode));
      const ff ex = warp_exclusive_scan_ff(ls, lane);
      T = ff_shfl(ff_add(ex, ls), 31);
      if (!(T.hi > 0.f) && mode == 0) {  // zero residual through rounding: draw from p_n
        mode = 1;
        continue;
      }
      const ff target = ff_mul_f(T, usamp);
      const unsigned hit = __ballot_sync(0xffffffffu, (e1 > e0) && ff_gt(ff_add(ex, ls), target));
      if (hit) {
        const int fl = __ffs(hit) - 1;
        if (lane == fl) {
          ff accm = ex;
          int lastpos = -1;
          for (int e = e0; e < e1; ++e) {
            const float r = resid_val(tr[e], dr[e], sct, scd, sist, sisd, mode);
            if (r > 0.f) lastpos = e;
            accm = ff_add_f(accm, r);
            if (ff_gt(accm, target)) {
              y = e;
              break;
            }
          }
          if (y < 0) y = lastpos >= 0 ? lastpos : e1 - 1;
        }
        y = __shfl_sync(0xffffffffu, y, fl);
      } else {  // u*T at or past the total through rounding: last id with mass
        int lp = -1;
        for (int e = e0; e < e1; ++e)
          if (resid_val(tr[e], dr[e], sct, scd, sist, sisd, mode) > 0.f) lp = e;
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        y = lp < 0 ? 0 : lp;
      }
      break;
    }
  }

  // ---- outputs ----
  if (lane == 0) {
    P.n_out[b] = n;
    if (err) atomicOr(P.status, kStatusInputErr);
  }
  if (P.anyorder) {
    if (lane < R && sig >= 0 && sig < P.D) {
      int v = -1;
      if (n >= 0) v = (lane < n) ? x : (lane == n ? y : -1);
      P.tok_out[(size_t)b * P.D + sig] = v;
    }
  } else {
    for (int j = lane; j <= NT; j += 32) {
      int v = -1;
      if (n >= 0) v = (j < n) ? P.x[(size_t)b * NT + j] : (j == n ? y : -1);
      P.tok_out[(size_t)b * (NT + 1) + j] = v;
    }
  }
  if (P.resid_out) {
    float* o = P.resid_out + (size_t)b * V;
    const bool have = (mode != 2) && (T.hi > 0.f);
    const float invT = have ? __fdiv_rn(1.f, ff_to_f(T)) : 0.f;
    const float* tr = st + srow * VS;
    const float* dr = sd + srow * VS;
    for (int e = lane; e < V; e += 32)
      o[e] = have ? resid_val(tr[e], dr[e], sct, scd, sist, sisd, mode) * invT : 0.f;
  }
}

}  // namespace

size_t small_smem_per_warp(int R, int vstride) { return (size_t)2 * R * vstride * sizeof(float); }

// Warps per CTA for a per-warp shared-memory need: the count (at most 12)
// that keeps the most warps resident per SM, given the SM's shared memory,
// the per-block reservation and the register file (e.g. 9 warps of 8.25 KB:
// 3 CTAs, 27 warps per SM, so 4096 sequences take one wave on 152 SMs).
int small_warps_per_cta(size_t per) {
  static int cap = 0, resv = 0, maxblk = 0;
  if (cap == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&cap, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&maxblk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cap = 0;
      return 8;
    }
  }
  static int regs = 0;  // the kernel's registers per thread, asked once
  if (regs == 0) {
    cudaFuncAttributes fa;
    regs = (cudaFuncGetAttributes(&fa, small_verify_kernel) == cudaSuccess && fa.numRegs > 0) ? fa.numRegs
                                                                                              : 64;
  }
  const int reg_warps = 65536 / (regs * 32);
  int best = 1, best_res = 0;
  for (int w = 1; w <= 12; ++w) {
    const size_t blk = per * w;
    if (blk > (size_t)maxblk) break;
    int ctas = (int)(cap / (blk + resv));
    ctas = min(ctas, reg_warps / w);
    if (ctas * w > best_res) {
      best_res = ctas * w;
      best = w;
    }
  }
  return best;
}

cudaError_t launch_small(const SmallParams& p, cudaStream_t s) {
  const size_t per = small_smem_per_warp(p.R, p.vstride);
  const int warps = small_warps_per_cta(per);
  const size_t smem = per * warps;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(small_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const long long blocks = ((long long)p.B + warps - 1) / warps;
  cudaLaunchAttribute a[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)blocks), dim3(warps * 32), smem, s, a);
  return cudaLaunchKernelEx(&cfg, small_verify_kernel, p);
}

}  // namespace sv
