// Expert selection from fp32 router logits, and the balance statistic.
//
// Selection ("Hands-on build guide", step 2; "Implementing Mixed Expert
// (MoE) layers", top-k and routing probabilities; "DeepSeek 5.7", s.2):
// experts are ranked by a key -- the raw logit in the two softmax modes,
// sigmoid(logit) + selection bias in the sigmoid mode -- in descending
// order, ties to the lower expert index, and the first k are taken.
//
// One warp handles one token: lane l holds experts l, l+32, ... (EPL per
// lane), sorted best first.  Each of the k rounds reduces the lanes' heads
// across the warp in the total order (key desc, index asc) with two warp
// reductions (redux.sync): the largest key, then the lowest index holding
// it; the winning lane drops its head.  The weights divide each chosen
// numerator by their sum taken in slot order.
//
// The balance statistic ("Tutorial -- MoE SER Expert Routing", section 4):
// per-expert probability sums are accumulated per warp
// in registers, reduced across the CTA's warps in a fixed order, and added
// to running totals in the workspace as integers (fixed point), so the
// totals are the same whatever order the CTAs finish in.  The last CTA of
// the forward turns them into the selection counts and the statistic.
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

// sigmoid evaluated in double, rounded once to fp32 (the selection key's
// definition)
__device__ __forceinline__ float sigmoid_f32_via_f64(float l) {
  return (float)(1.0 / (1.0 + exp(-(double)l)));
}
// fp32 sigmoid: expf (<= 2 ulp), an add and a correctly rounded divide; its
// distance to sigmoid_f32_via_f64 is below 2^-22
__device__ __forceinline__ float sigmoid_fast(float l) { return 1.0f / (1.0f + expf(-l)); }
// Bound on |fl(sigmoid_fast(l) + b) - fl(sigmoid_f32_via_f64(l) + b)| for keys
// of magnitude near |key|: the two sigmoids differ by < 2^-22, and the two
// fp32 adds round at most one ulp of the key apart (one ulp <= |key| 2^-23).
// The absolute floor covers keys near zero; the relative part covers large
// selection biases, where one ulp of the key outgrows any absolute slack
// (|key| ~ 10^3 has ulps of 2^-14..2^-13).  Both parts carry a factor of two
// or more of margin.
constexpr float kSlack = 1.0f / 65536.0f;
__device__ __forceinline__ float key_slack(float key) {
  return kSlack + fabsf(key) * (1.0f / 4194304.0f);   // 2^-16 + |key| 2^-22
}

// Keys as unsigned integers in the same order (x < y  <=>  u(x) < u(y) for
// non-NaN floats); -0 is folded onto +0 first, so the two tie as floats do.
__device__ __forceinline__ uint32_t ordered(float k) {
  const uint32_t b = __float_as_uint(k + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Selection keeps, per lane, its candidates sorted best first as 64-bit
// words (ordered key << 32 | ~expert): a larger word is a larger key, or the
// same key and a lower expert index -- the total order of the selection.
// Word 0 marks "none" (every finite key orders above 0).
__device__ __forceinline__ uint64_t cand_word(uint32_t okey, int e) {
  return ((uint64_t)okey << 32) | (uint32_t)~(uint32_t)e;
}
template <int EPL>
__device__ __forceinline__ void sort_desc(uint64_t (&c)[EPL]) {
  // odd-even transposition: EPL rounds of compare-exchange
#pragma unroll
  for (int r = 0; r < EPL; ++r)
#pragma unroll
    for (int i = r & 1; i + 1 < EPL; i += 2) {
      const uint64_t hi = c[i] > c[i + 1] ? c[i] : c[i + 1];
      const uint64_t lo = c[i] > c[i + 1] ? c[i + 1] : c[i];
      c[i] = hi;
      c[i + 1] = lo;
    }
}
// One round: the warp's best remaining candidate -- the largest head key
// (redux.sync max), then the lowest expert index among the heads holding it
// (redux.sync min) -- which its lane then drops from its queue.  Returns the
// expert; *okey_out is its ordered key.
template <int EPL>
__device__ __forceinline__ uint32_t take_best(uint64_t (&c)[EPL], int lane, uint32_t* okey_out) {
  const uint32_t hk = (uint32_t)(c[0] >> 32);
  const uint32_t kmax = __reduce_max_sync(kFull, hk);
  const uint32_t mine = hk == kmax ? ~(uint32_t)c[0] : 0xFFFFFFFFu;
  const uint32_t emin = __reduce_min_sync(kFull, mine);
  if (lane == (int)(emin & 31u)) {
#pragma unroll
    for (int i = 0; i + 1 < EPL; ++i) c[i] = c[i + 1];
    c[EPL - 1] = 0ull;
  }
  *okey_out = kmax;
  return emin;
}

// SIG: the sigmoid mode (its candidate packing keeps the most arrays live),
// compiled apart from the two softmax modes so that each gets its own
// register allocation under the launch bound.
template <int EPL, bool SIG>
__global__ void __launch_bounds__(kRouteWarps * 32, EPL <= 4 ? 4 : 2)
route_kernel(const float* __restrict__ logits, int64_t n_tokens, int n_experts,
             int top_k, int mode, const float* __restrict__ sel_bias,
             int32_t* __restrict__ idx, float* __restrict__ w, int tokens_per_cta,
             const RouteTotals tot, const RouteFinal fin) {
  __shared__ float s_ps[kRouteWarps][EPL * 32];
  __shared__ float s_num[kRouteWarps][EPL * 32];   // this token's numerators, by expert
  __shared__ int s_sel[kRouteWarps][EPL * 32];     // its selected experts, by slot
  __shared__ int s_cnt[EPL * 32];
  __shared__ bool s_last;
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = n_experts;
  for (int e = threadIdx.x; e < EPL * 32; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();

  float ps[EPL], bias[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    ps[i] = 0.f;
    bias[i] = (SIG && e < E) ? sel_bias[e] : 0.f;
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
    float l[EPL], num[EPL], p[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) l[i] = l_next[i];
    load_row(t + kRouteWarps);
    uint64_t c[EPL];
    if constexpr (SIG) {
      // Rank fp32 keys first (within key_slack of the exact ones); the exact
      // top k lies among the experts whose fp32 key is within 2 key_slack of
      // the k-th fp32 key, so only those get the double-precision sigmoid.
      float sa[EPL], ka[EPL];
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        sa[i] = e < E ? sigmoid_fast(l[i]) : 0.f;
        ka[i] = __fadd_rn(sa[i], bias[i]);
        part += sa[i];
        c[i] = e < E ? cand_word(ordered(ka[i]), e) : 0ull;
      }
      const float rs = 1.f / warp_sum_bcast(part);
      sort_desc<EPL>(c);
      uint32_t kth = 0u;
      for (int j = 0; j < top_k; ++j) take_best<EPL>(c, lane, &kth);
      const float kth_key = unordered(kth);
      const float thr = kth_key - 4.f * key_slack(kth_key);
      // The candidates (usually about k of them, spread over the lanes'
      // EPL slots) are packed into consecutive lanes, so that one warp-wide
      // double-precision evaluation serves up to 32 of them, and the results
      // are shuffled back.
      const unsigned lt_mask = (1u << lane) - 1u;
      unsigned cm[EPL];
      int cbase[EPL];
      int nc = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        cm[i] = __ballot_sync(kFull, lane + 32 * i < E && ka[i] >= thr);
        cbase[i] = nc;
        nc += __popc(cm[i]);
      }
      float sx[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) sx[i] = 0.f;
      for (int b0 = 0; b0 < nc; b0 += 32) {
        const int o = b0 + lane;                      // the candidate this lane evaluates
        float lo = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int n = o - cbase[i];
          const bool here = n >= 0 && n < __popc(cm[i]);
          const int src = here ? (int)__fns(cm[i], 0, n + 1) : 0;
          const float v = __shfl_sync(kFull, l[i], src);
          if (here) lo = v;
        }
        const float so = o < nc ? sigmoid_f32_via_f64(lo) : 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int myo = cbase[i] + __popc(cm[i] & lt_mask);
          const float v = __shfl_sync(kFull, so, (myo - b0) & 31);
          if (((cm[i] >> lane) & 1u) && myo >= b0 && myo < b0 + 32) sx[i] = v;
        }
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        const bool cand = (cm[i] >> lane) & 1u;
        num[i] = sx[i];
        c[i] = cand ? cand_word(ordered(__fadd_rn(sx[i], bias[i])), e) : 0ull;
        p[i] = sa[i] * rs;
      }
    } else {
      // key = logit; the numerators are exp(l - max) in both modes: the
      // renormalised top-k of the softmax and the softmax of the top k are
      // the same weights
      uint32_t lmax = 0u;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        const uint32_t ok = ordered(l[i]);
        c[i] = e < E ? cand_word(ok, e) : 0ull;
        lmax = (e < E && ok > lmax) ? ok : lmax;
      }
      const float m = unordered(__reduce_max_sync(kFull, lmax));
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        num[i] = lane + 32 * i < E ? expf(l[i] - m) : 0.f;
        part += num[i];
      }
      const float rz = 1.f / warp_sum_bcast(part);
#pragma unroll
      for (int i = 0; i < EPL; ++i) p[i] = num[i] * rz;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      ps[i] += p[i];
      s_num[warp][lane + 32 * i] = num[i];
    }
    sort_desc<EPL>(c);
    // k rounds; every lane sums the chosen numerators in slot order
    float zsel = 0.f;
    __syncwarp();
    for (int j = 0; j < top_k; ++j) {
      uint32_t kj;
      const uint32_t e = take_best<EPL>(c, lane, &kj);
      zsel += s_num[warp][e];
      if (lane == 0) s_sel[warp][j] = (int)e;
    }
    __syncwarp();
    for (int j = lane; j < top_k; j += 32) {
      const int e = s_sel[warp][j];
      idx[t * top_k + j] = e;
      w[t * top_k + j] = s_num[warp][e] / zsel;
      atomicAdd(&s_cnt[e], 1);
    }
    __syncwarp();
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

template <bool SIG>
void launch_route_epl(dim3 grid, dim3 block, cudaStream_t st, const float* logits,
                      int64_t n_tokens, int n_experts, int top_k, int mode,
                      const float* sel_bias, int32_t* idx, float* w, int tpc,
                      const RouteTotals& tot, const RouteFinal& fin) {
  if (n_experts <= 32)
    launch_pdl(route_kernel<1, SIG>, grid, block, 0, st, logits, n_tokens, n_experts, top_k,
               mode, sel_bias, idx, w, tpc, tot, fin);
  else if (n_experts <= 64)
    launch_pdl(route_kernel<2, SIG>, grid, block, 0, st, logits, n_tokens, n_experts, top_k,
               mode, sel_bias, idx, w, tpc, tot, fin);
  else if (n_experts <= 128)
    launch_pdl(route_kernel<4, SIG>, grid, block, 0, st, logits, n_tokens, n_experts, top_k,
               mode, sel_bias, idx, w, tpc, tot, fin);
  else
    launch_pdl(route_kernel<8, SIG>, grid, block, 0, st, logits, n_tokens, n_experts, top_k,
               mode, sel_bias, idx, w, tpc, tot, fin);
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
  if (mode == 2)
    launch_route_epl<true>(grid, block, st, logits, n_tokens, n_experts, top_k, mode, sel_bias,
                           idx, w, tpc, tot, fin);
  else
    launch_route_epl<false>(grid, block, st, logits, n_tokens, n_experts, top_k, mode, sel_bias,
                            idx, w, tpc, tot, fin);
}

}  // namespace moe
