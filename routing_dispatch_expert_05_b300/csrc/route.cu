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
// and reduces them across the warp in the total order (key desc, index asc)
// with two warp reductions (redux.sync): the largest key, then the lowest
// index holding it.
//
// The balance statistic ("Tutorial -- MoE SER Expert Routing", section 4):
// per-expert probability sums are accumulated per warp
// in registers, reduced across the CTA's warps in a fixed order, and added
// to running totals in the workspace as integers (fixed point), so the
// totals are the same whatever order the CTAs finish in.  The last CTA of
// the forward turns them into the selection counts and the statistic.
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

// sigmoid evaluated in double, rounded once to fp32 (the selection key's
// definition)
__device__ __forceinline__ float sigmoid_f32_via_f64(float l) {
  return (float)(1.0 / (1.0 + exp(-(double)l)));
}
// fp32 sigmoid: expf (<= 2 ulp), an add and a correctly rounded divide; its
// distance to sigmoid_f32_via_f64 is far below kSlack
__device__ __forceinline__ float sigmoid_fast(float l) { return 1.0f / (1.0f + expf(-l)); }
constexpr float kSlack = 1.0f / 65536.0f;

// Keys as unsigned integers in the same order (x < y  <=>  u(x) < u(y) for
// non-NaN floats); -0 is folded onto +0 first, so the two tie as floats do.
__device__ __forceinline__ uint32_t ordered(float k) {
  const uint32_t b = __float_as_uint(k + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// One selection round: the best remaining candidate of the warp in the total
// order (key desc, index asc) -- a warp max of the keys, then a warp min of
// the indices of the lanes holding that key (two redux.sync).  Returns the
// expert index (INT_MAX if none is left) and its key.
template <int EPL>
__device__ __forceinline__ int warp_best(const uint32_t (&ok)[EPL], const int (&slot)[EPL],
                                         int lane, int E, float* best_key) {
  uint32_t bk = 0u;
  int bi = INT_MAX;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && slot[i] < 0 && (bi == INT_MAX || ok[i] > bk)) {
      bk = ok[i];
      bi = e;
    }
  }
  const uint32_t kmax = __reduce_max_sync(kFull, bi == INT_MAX ? 0u : bk);
  const uint32_t mine = (bi != INT_MAX && bk == kmax) ? (uint32_t)bi : 0xFFFFFFFFu;
  const uint32_t emin = __reduce_min_sync(kFull, mine);
  *best_key = unordered(kmax);
  return emin == 0xFFFFFFFFu ? INT_MAX : (int)emin;
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32, EPL <= 4 ? 4 : 2)
route_kernel(const float* __restrict__ logits, int64_t n_tokens, int n_experts,
             int top_k, int mode, const float* __restrict__ sel_bias,
             int32_t* __restrict__ idx, float* __restrict__ w, int tokens_per_cta,
             const RouteTotals tot, const RouteFinal fin) {
  __shared__ float s_ps[kRouteWarps][EPL * 32];
  __shared__ int s_cnt[EPL * 32];
  __shared__ bool s_last;
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

  const int64_t t0 = (int64_t)blockIdx.x * tokens_per_cta;
  const int64_t t1 = min(n_tokens, t0 + tokens_per_cta);
  // the next token's logits are loaded while this one is ranked
  float l_next[EPL];
  auto load_row = [&](int64_t t) {
    const float* row = logits + t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      l_next[i] = (t < t1 && e < E) ? __ldcs(row + e) : -INFINITY;
    }
  };
  load_row(t0 + warp);
  for (int64_t t = t0 + warp; t < t1; t += kRouteWarps) {
    float l[EPL], key[EPL], num[EPL], p[EPL];
    int slot[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      l[i] = l_next[i];
      slot[i] = -1;
    }
    load_row(t + kRouteWarps);
    if (mode == 2) {
      // Rank fp32 keys first (within kSlack of the exact ones); the exact top
      // k lies among the experts whose fp32 key is within 2 kSlack of the
      // k-th fp32 key, so only those get the double-precision sigmoid.
      float sa[EPL];
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const bool v = lane + 32 * i < E;
        sa[i] = v ? sigmoid_fast(l[i]) : 0.f;
        key[i] = __fadd_rn(sa[i], bias[i]);
        part += sa[i];
      }
      const float ssum = warp_sum_bcast(part);
      uint32_t ok[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) ok[i] = ordered(key[i]);
      float kth = -INFINITY;
      for (int j = 0; j < top_k; ++j) {
        const int bi = warp_best<EPL>(ok, slot, lane, E, &kth);
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (lane + 32 * i == bi) slot[i] = j;
      }
      const float thr = kth - 4.f * kSlack;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const bool cand = lane + 32 * i < E && key[i] >= thr;
        const float s = cand ? sigmoid_f32_via_f64(l[i]) : 0.f;
        num[i] = s;
        key[i] = cand ? __fadd_rn(s, bias[i]) : -INFINITY;
        slot[i] = cand ? -1 : 0x7fff;      // non-candidates never selected
        p[i] = sa[i] / ssum;
      }
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

    uint32_t ok[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) ok[i] = ordered(key[i]);
    for (int j = 0; j < top_k; ++j) {
      float bk;
      const int bi = warp_best<EPL>(ok, slot, lane, E, &bk);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == bi) slot[i] = j;
    }

    float part = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) part += (slot[i] >= 0 && slot[i] < top_k) ? num[i] : 0.f;
    const float zsel = warp_sum_bcast(part);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (slot[i] >= 0 && slot[i] < top_k) {
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
  // this CTA's sums join the running totals: the probability sum (at most
  // 32) in fixed point, 2^-32 units (N * 2^32 stays below 2^63)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kRouteWarps; ++q) acc += s_ps[q][e];
    const unsigned long long fx = __float2ull_rn(acc * 4294967296.0f);
    if (fx != 0ull) atomicAdd(tot.psum_fx + e, fx);
    if (s_cnt[e] != 0) atomicAdd(tot.cnt + e, (unsigned)s_cnt[e]);
  }
  if (!fin.finalize) return;
  // the last CTA to finish (ticket) reads and clears the totals
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(tot.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* s_term = &s_ps[0][0];                  // kRouteWarps * EPL * 32 >= E
  const float n = (float)fin.n_total;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const unsigned long long fx = atomicExch(tot.psum_fx + e, 0ull);
    const unsigned c = atomicExch(tot.cnt + e, 0u);
    if (fin.counts != nullptr) fin.counts[e] = (int32_t)c;
    // frac_e * mean p_e = (count_e / N) * (sum_t p / N)
    s_term[e] = ((float)c / n) * ((float)fx * 2.3283064365386963e-10f / n);
  }
  __syncthreads();
  if (warp == 0) {
    float acc = 0.f;
    for (int e = lane; e < E; e += 32) acc += s_term[e];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) {
      if (fin.balance != nullptr) fin.balance[0] = fin.coef * acc;
      *tot.ticket = 0u;
    }
  }
}

// Between steps: b_e <- b_e + gamma * sign(mean load - load_e) (one fp32
// add; the sign compares E * load_e with the total on integers) and the
// load's coefficient of variation (population std / mean, 0 if nothing was
// routed).  One block, thread e = expert e; the sums run in a fixed order.
__global__ void __launch_bounds__(kMaxExperts)
bias_update_kernel(const int32_t* __restrict__ counts, int n_experts, float gamma,
                   float* __restrict__ sel_bias, float* __restrict__ load_cv) {
  __shared__ long long s_total;
  __shared__ double s_dev[kMaxExperts];
  const int e = threadIdx.x;
  if (e == 0) {
    long long t = 0;
    for (int q = 0; q < n_experts; ++q) t += counts[q];
    s_total = t;
  }
  __syncthreads();
  const long long total = s_total;
  const double mean = (double)total / n_experts;
  if (e < n_experts) {
    const long long c = counts[e];
    const long long diff = total - (long long)n_experts * c;
    const float sgn = diff > 0 ? 1.f : (diff < 0 ? -1.f : 0.f);
    if (sel_bias != nullptr) sel_bias[e] = __fadd_rn(sel_bias[e], gamma * sgn);
    const double dv = (double)c - mean;
    s_dev[e] = dv * dv;
  }
  __syncthreads();
  if (e == 0 && load_cv != nullptr) {
    double acc = 0.0;
    for (int q = 0; q < n_experts; ++q) acc += s_dev[q];
    load_cv[0] = total > 0 ? (float)(sqrt(acc / n_experts) / mean) : 0.f;
  }
}

}  // namespace

void launch_bias_update(const int32_t* counts, int n_experts, float gamma, float* sel_bias,
                        float* load_cv, cudaStream_t st) {
  bias_update_kernel<<<1, kMaxExperts, 0, st>>>(counts, n_experts, gamma, sel_bias, load_cv);
}

void launch_route_from_logits(const float* logits, int64_t n_tokens, int n_experts,
                              int top_k, int mode, const float* sel_bias,
                              int32_t* idx, float* w, const RouteTotals& tot,
                              const RouteFinal& fin, cudaStream_t st) {
  if (n_tokens <= 0) return;
  // a token per warp for small layers (more CTAs); otherwise four per warp,
  // kRouteTokensPerCta per CTA.  Chosen by the whole forward's token count,
  // so the chunks of the host pipeline split tokens into CTAs as one launch
  // over all of them would.
  const int tpc = fin.n_total < 4096 ? kRouteWarps : kRouteTokensPerCta;
  const dim3 grid((unsigned)ceil_div64(n_tokens, tpc)), block(kRouteWarps * 32);
  if (n_experts <= 32)
    route_kernel<1><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, tpc, tot, fin);
  else if (n_experts <= 64)
    route_kernel<2><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, tpc, tot, fin);
  else if (n_experts <= 128)
    route_kernel<4><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, tpc, tot, fin);
  else
    route_kernel<8><<<grid, block, 0, st>>>(logits, n_tokens, n_experts, top_k, mode,
                                            sel_bias, idx, w, tpc, tot, fin);
}

}  // namespace moe
