// Expert selection from fp32 router logits, and the balance statistic.
//
// Selection ("Hands-on build guide", step 2; "Implementing Mixed Expert
// (MoE) layers", top-k and routing probabilities; "DeepSeek 5.7", s.2):
// experts are ranked by a key -- the raw logit in the two softmax modes,
// sigmoid(logit) + selection bias in the sigmoid mode -- in descending
// order, ties to the lower expert index, and the first k are taken.
//
// One warp handles one token: lane l holds experts l, l+32, ... (EPL per
// lane).  Each of the k rounds takes every lane's best remaining candidate
// and reduces them across the warp with the total order (key desc, index
// asc); lane 0's winner is authoritative.  Probabilities for the balance
// statistic are accumulated per warp in registers and reduced across warps
// in a fixed order, so the per-partial sums are deterministic.
#include <climits>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRouteWarps = 8;

__device__ __forceinline__ float warp_sum_bcast(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return __shfl_sync(kFull, v, 0);
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

// sigmoid evaluated in double, rounded once to fp32
__device__ __forceinline__ float sigmoid_f32_via_f64(float l) {
  return (float)(1.0 / (1.0 + exp(-(double)l)));
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float* __restrict__ logits, int64_t n_tokens, int n_experts,
             int top_k, int mode, const float* __restrict__ sel_bias,
             int32_t* __restrict__ idx, float* __restrict__ w,
             float* __restrict__ psum_part, int32_t* __restrict__ cnt_part) {
  __shared__ float s_ps[kRouteWarps][EPL * 32];
  __shared__ int s_cnt[EPL * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = n_experts;
  for (int e = threadIdx.x; e < EPL * 32; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();

  float ps[EPL], bias[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    ps[i] = 0.f;
    bias[i] = (mode == 2 && e < E) ? sel_bias[e] : 0.f;
  }

  const int64_t t0 = (int64_t)blockIdx.x * kRouteTokensPerPartial;
  const int64_t t1 = min(n_tokens, t0 + kRouteTokensPerPartial);
  for (int64_t t = t0 + warp; t < t1; t += kRouteWarps) {
    float l[EPL], key[EPL], num[EPL], p[EPL];
    int slot[EPL];
    const float* row = logits + t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = e < E ? row[e] : -INFINITY;
      slot[i] = -1;
    }
    if (mode == 2) {
      float s[EPL];
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const bool v = lane + 32 * i < E;
        s[i] = v ? sigmoid_f32_via_f64(l[i]) : 0.f;
        key[i] = __fadd_rn(s[i], bias[i]);
        num[i] = s[i];
        part += s[i];
      }
      const float ssum = warp_sum_bcast(part);
#pragma unroll
      for (int i = 0; i < EPL; ++i) p[i] = s[i] / ssum;
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i) m = fmaxf(m, l[i]);
      m = warp_max(m);
      float ex[EPL], part = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const bool v = lane + 32 * i < E;
        ex[i] = v ? expf(l[i] - m) : 0.f;
        part += ex[i];
      }
      const float z = warp_sum_bcast(part);
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        p[i] = ex[i] / z;
        key[i] = l[i];
        num[i] = mode == 0 ? p[i] : ex[i];
      }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) ps[i] += (lane + 32 * i < E) ? p[i] : 0.f;

    for (int j = 0; j < top_k; ++j) {
      float bk = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && slot[i] < 0 && (bi == INT_MAX || key[i] > bk)) {
          bk = key[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(kFull, bk, off);
        const int oi = __shfl_xor_sync(kFull, bi, off);
        if (oi != INT_MAX &&
            (bi == INT_MAX || ok > bk || (ok == bk && oi < bi))) {
          bk = ok;
          bi = oi;
        }
      }
      bi = __shfl_sync(kFull, bi, 0);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == bi) slot[i] = j;
    }

    float part = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) part += slot[i] >= 0 ? num[i] : 0.f;
    const float zsel = warp_sum_bcast(part);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (slot[i] >= 0) {
        const int e = lane + 32 * i;
        idx[t * top_k + slot[i]] = e;
        w[t * top_k + slot[i]] = num[i] / zsel;
        atomicAdd(&s_cnt[e], 1);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < EPL; ++i) s_ps[warp][lane + 32 * i] = ps[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kRouteWarps; ++q) acc += s_ps[q][e];
    psum_part[(int64_t)blockIdx.x * E + e] = acc;
    cnt_part[(int64_t)blockIdx.x * E + e] = s_cnt[e];
  }
}

__global__ void balance_finalize_kernel(const float* __restrict__ psum_part,
                                        const int32_t* __restrict__ cnt_part,
                                        int n_parts, int n_experts,
                                        int64_t n_tokens, float coef,
                                        int32_t* __restrict__ counts,
                                        float* __restrict__ balance) {
  __shared__ double s_term[kMaxExperts];
  const int e = threadIdx.x;
  if (e < n_experts) {
    double ps = 0.0;
    long long cnt = 0;
    for (int q = 0; q < n_parts; ++q) {
      ps += (double)psum_part[(int64_t)q * n_experts + e];
      cnt += cnt_part[(int64_t)q * n_experts + e];
    }
    if (counts) counts[e] = (int32_t)cnt;
    const double n = n_tokens > 0 ? (double)n_tokens : 1.0;
    s_term[e] = ((double)cnt / n) * (ps / n);
  }
  __syncthreads();
  if (e == 0 && balance) {
    double acc = 0.0;
    for (int q = 0; q < n_experts; ++q) acc += s_term[q];
    balance[0] = n_tokens > 0 ? (float)((double)coef * acc) : 0.f;
  }
}

}  // namespace

void launch_route_from_logits(const float* logits, int64_t n_tokens, int n_experts,
                              int top_k, int mode, const float* sel_bias,
                              int32_t* idx, float* w, float* psum_part,
                              int32_t* cnt_part, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int parts = (int)ceil_div64(n_tokens, kRouteTokensPerPartial);
  const dim3 grid(parts), block(kRouteWarps * 32);
  if (n_experts <= 32)
    route_kernel<1><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, psum_part, cnt_part);
  else if (n_experts <= 64)
    route_kernel<2><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, psum_part, cnt_part);
  else if (n_experts <= 128)
    route_kernel<4><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, psum_part, cnt_part);
  else
    route_kernel<8><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, psum_part, cnt_part);
}

void launch_balance_finalize(const float* psum_part, const int32_t* cnt_part,
                             int n_parts, int n_experts, int64_t n_tokens,
                             float coef, int32_t* counts, float* balance,
                             cudaStream_t st) {
  if (!counts && !balance) return;
  balance_finalize_kernel<<<1, kMaxExperts, 0, st>>>(
      psum_part, cnt_part, n_parts, n_experts, n_tokens, coef, counts, balance);
}

}  // namespace moe
