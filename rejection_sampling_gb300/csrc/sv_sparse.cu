// sv_sparse.cu -- verification on sorted top-k (id, prob) support lists.
//
// The rule as Uno's sampler states it (Uno article, "What 'lossless'
// actually has to mean", _sparse_verify_tensors): p_spec and q_spec are the
// listed probabilities at the draft token (0 where the id is absent), ratio =
// p_spec / q_spec where q_spec > 0 else 0, accept iff u < min(1, ratio); the
// correction after a rejection is clamp(p - q_on_clean, 0) on the target
// ("clean") support, renormalised, q_on_clean being the draft probability of
// the same id.  The block is truncated at the first rejection (DFlash/DFlash2
// guide, 4.4) and an all-accept block draws the bonus from the target list of
// position gamma (same guide, section 2).
//
// One CTA per row, one warp per position (gamma + 1 <= 32 warps).  Warp j
// issues its small loads first, validates its lists (copying a draft list of
// up to kStageK entries into shared memory as it goes) and runs its accept
// test; a shared-memory scan finds the first rejection n; warp n then finds
// each target id's draft probability by binary search in the staged draft
// list (in global memory for longer lists), scans the residual in
// float-float in list order and draws the token.
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kStageK = 128;  // draft lists up to this length are staged in shared memory

// A list is valid if its ids are in [0, V) and strictly ascending and its
// probabilities finite and >= 0; with `sid` / `sp` it is also copied there.
__device__ __forceinline__ bool list_ok(const int32_t* ids, const float* pr, int k, int V,
                                        int lane, int32_t* sid = nullptr, float* sp = nullptr) {
  bool ok = true;
  for (int i = lane; i < k; i += 32) {
    const int id = ids[i];
    const int nx = (i + 1 < k) ? ids[i + 1] : 0x7fffffff;
    const float p = pr[i];
    if (id < 0 || id >= V) ok = false;
    if (nx <= id) ok = false;
    if (!(p >= 0.f) || p == INFINITY) ok = false;
    if (sid) {
      sid[i] = id;
      sp[i] = p;
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// probability of `id` in a sorted list (0 if absent), in shared or global memory
__device__ __forceinline__ float list_lookup(const int32_t* ids, const float* pr, int k, int id) {
  int lo = 0, hi = k;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = ids[mid];
    if (v < id)
      lo = mid + 1;
    else
      hi = mid;
  }
  return (lo < k && ids[lo] == id) ? pr[lo] : 0.f;
}

__global__ void sparse_verify_kernel(const __grid_constant__ SparseParams P) {
  __shared__ int s_acc[32];
  __shared__ int s_err[32];
  __shared__ int s_n;
  extern __shared__ __align__(16) unsigned char s_lists[];  // G x kStageK (id, prob) when staged
  pdl_wait_then_release();
  const int b = blockIdx.x, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = P.G, kt = P.kt, kd = P.kd, V = P.V;
  const int32_t* tid = P.tid + ((size_t)b * (G + 1) + j) * kt;
  const float* tp = P.tp + ((size_t)b * (G + 1) + j) * kt;
  const bool staged = kd <= kStageK;
  int32_t* sid = reinterpret_cast<int32_t*>(s_lists) + (size_t)j * kStageK;
  float* sdp = reinterpret_cast<float*>(s_lists + (size_t)G * kStageK * sizeof(int32_t)) + (size_t)j * kStageK;
  // small inputs first: their latency hides behind the list loads
  const int x = (j < G) ? P.x[(size_t)b * G + j] : 0;
  const float uj = (j < G) ? P.u_acc[(size_t)b * G + j] : 0.f;
  const float us = P.u_s[b];

  bool err = !list_ok(tid, tp, kt, V, lane);
  int acc = 1;
  float a = 0.f;
  if (j < G) {
    const int32_t* did = P.did + ((size_t)b * G + j) * kd;
    const float* dp = P.dp + ((size_t)b * G + j) * kd;
    err |= staged ? !list_ok(did, dp, kd, V, lane, sid, sdp) : !list_ok(did, dp, kd, V, lane);
    if (x < 0 || x >= V) err = true;
    float ps = 0.f, qs = 0.f;
    for (int i = lane; i < kt; i += 32)
      if (tid[i] == x) ps += tp[i];
    for (int i = lane; i < kd; i += 32)
      if (did[i] == x) qs += dp[i];
    ps = warp_sum(ps);
    qs = warp_sum(qs);
    const float ratio = (qs > 0.f) ? __fdiv_rn(ps, qs) : 0.f;
    a = fminf(ratio, 1.f);
    acc = uj < a;
  }
  if (lane == 0) {
    s_acc[j] = acc;
    s_err[j] = err ? 1 : 0;
    if (P.acc_out && j < G) P.acc_out[(size_t)b * G + j] = err ? __int_as_float(0x7fc00000) : a;
  }
  __syncthreads();
  if (j == 0) {
    const int e = (lane <= G) ? s_err[lane] : 0;
    const int r = (lane < G) ? !s_acc[lane] : 0;
    const bool any_err = __any_sync(0xffffffffu, e);
    const unsigned rej = __ballot_sync(0xffffffffu, r);
    if (lane == 0) s_n = any_err ? -1 : (rej ? __ffs(rej) - 1 : G);
  }
  __syncthreads();
  const int n = s_n;
  int32_t* tok = P.tok_out + (size_t)b * (G + 1);
  if (n < 0) {
    if (j == 0) {
      for (int i = lane; i <= G; i += 32) tok[i] = -1;
      if (lane == 0) {
        P.n_out[b] = -1;
        atomicOr(P.status, kStatusInputErr);
      }
      if (P.resid_out)
        for (int i = lane; i < kt; i += 32) P.resid_out[(size_t)b * kt + i] = 0.f;
    }
    return;
  }
  if (j != n) return;

  // ---- warp n: residual on the target support (or the bonus list) ----
  // the draft list of position n: as staged by this warp (shared memory) or in
  // global memory
  __syncwarp();
  const int32_t* did = (n < G) ? (staged ? sid : P.did + ((size_t)b * G + n) * kd) : nullptr;
  const float* dp = (n < G) ? (staged ? sdp : P.dp + ((size_t)b * G + n) * kd) : nullptr;
  const int q = (kt + 31) / 32;
  const int e0 = min(kt, lane * q), e1 = min(kt, e0 + q);
  int mode = (n < G) ? 0 : 1;
  auto weight = [&](int i) -> float {
    const float p = tp[i];
    if (mode != 0) return p;
    const float r = __fsub_rn(p, list_lookup(did, dp, kd, tid[i]));
    return r > 0.f ? r : 0.f;
  };
  ff T{0.f, 0.f}, ls{0.f, 0.f}, ex{0.f, 0.f};
  for (int attempt = 0; attempt < 2; ++attempt) {
    ls = ff{0.f, 0.f};
    for (int i = e0; i < e1; ++i) ls = ff_add_f(ls, weight(i));
    ex = warp_exclusive_scan_ff(ls, lane);
    T = ff_shfl(ff_add(ex, ls), 31);
    if (!(T.hi > 0.f) && mode == 0) {
      mode = 1;  // zero residual through rounding: draw from the target list
      continue;
    }
    break;
  }
  int yi = -1;
  if (T.hi > 0.f) {
    const ff target = ff_mul_f(T, us);
    const unsigned hit = __ballot_sync(0xffffffffu, (e1 > e0) && ff_gt(ff_add(ex, ls), target));
    if (hit) {
      const int fl = __ffs(hit) - 1;
      if (lane == fl) {
        ff accm = ex;
        int lastpos = -1;
        for (int i = e0; i < e1; ++i) {
          const float w = weight(i);
          if (w > 0.f) lastpos = i;
          accm = ff_add_f(accm, w);
          if (ff_gt(accm, target)) {
            yi = i;
            break;
          }
        }
        if (yi < 0) yi = lastpos >= 0 ? lastpos : e1 - 1;
      }
      yi = __shfl_sync(0xffffffffu, yi, fl);
    } else {
      int lp = -1;
      for (int i = e0; i < e1; ++i)
        if (weight(i) > 0.f) lp = i;
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      yi = lp;
    }
  }
  const int y = (yi >= 0) ? tid[yi] : -1;
  for (int i = lane; i <= G; i += 32) tok[i] = (i < n) ? P.x[(size_t)b * G + i] : (i == n ? y : -1);
  if (lane == 0) P.n_out[b] = n;
  if (P.resid_out) {
    const float invT = (T.hi > 0.f) ? __fdiv_rn(1.f, ff_to_f(T)) : 0.f;
    for (int i = lane; i < kt; i += 32) P.resid_out[(size_t)b * kt + i] = weight(i) * invT;
  }
}

}  // namespace

cudaError_t launch_sparse(const SparseParams& p, cudaStream_t s) {
  // G x kStageK x 8 bytes <= 31 KB: within the default dynamic shared memory
  const size_t smem = (p.kd <= kStageK) ? (size_t)p.G * kStageK * (sizeof(int32_t) + sizeof(float)) : 0;
  cudaLaunchAttribute a[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(p.B), dim3(32 * (p.G + 1)), smem, s, a);
  return cudaLaunchKernelEx(&cfg, sparse_verify_kernel, p);
}

}  // namespace sv
