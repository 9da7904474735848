// The layer's backward pass outside the GEMMs: the weighted combine's and the
// router's gradients, the SwiGLU derivative, the reduction of the expert rows
// back to tokens, and the layout changes the gradient GEMMs need.
//
// The gradient is that of <dout, out> + d_balance * B with the routing held
// fixed ("DeepSeek 5.7: MoE from scratch", Worked example and study lab: the
// router receives gradients through the contribution weights, the top-k
// choice itself is not differentiable, an expert no token chose gets none):
//   dw[t,j] = <dout[t], y[t,j]>,      dy[t,j] = w[t,j] dout[t]
//   softmax modes: dlogit = w * (dw - <w, dw>) on the selected experts
//   sigmoid mode:  dlogit = s (1 - s) (dw - <w, dw>) / sum_sel s
//   balance term:  p (g - <p, g>) (softmax), or through s / sum s (sigmoid),
//                  g_e = d_balance * coef * count_e / N^2
//   SwiGLU:        dg = dh u silu'(g), du = dh silu(g)
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float sigmoid_fast(float z) { return 1.f / (1.f + __expf(-z)); }

// ---------------------------------------------------------------- layouts
// koff[g+1] = koff[g] + max(64, 64 * ceil(m_g / 64)): every group's span of
// the transposed activations is a non-zero number of whole k-blocks.
__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int64_t rows, int G,
                                   int32_t* __restrict__ koff) {
  if (threadIdx.x != 0) return;
  int acc = 0;
  koff[0] = 0;
  for (int g = 0; g < G; ++g) {
    const int m = offsets ? offsets[g + 1] - offsets[g] : (int)rows;
    acc += max(64, (m + 63) / 64 * 64);
    koff[g + 1] = acc;
  }
}

// out[c, koff[g] + l] = in[off[g] + l, c] for l < m_g, 0 on the padding;
// 64 x 64 tiles through shared memory.  TIn is bf16 or float (then
// rounded to bf16).
template <typename TIn>
__global__ void __launch_bounds__(256)
transpose_grouped_kernel(const TIn* __restrict__ in, int C, const int32_t* __restrict__ offsets,
                         int64_t rows, int G, const int32_t* __restrict__ koff,
                         int64_t k_total, bf16* __restrict__ out) {
  __shared__ bf16 tile[64][72];
  __shared__ int64_t s_src[64];
  const int64_t pc0 = (int64_t)blockIdx.x * 64;
  const int c0 = blockIdx.y * 64;
  if (pc0 >= koff[G]) return;
  if (threadIdx.x < 64) {
    const int64_t pc = pc0 + threadIdx.x;
    int lo = 0, hi = G - 1;                        // largest g with koff[g] <= pc
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (koff[mid] <= pc) lo = mid; else hi = mid - 1;
    }
    const int64_t o0 = offsets ? offsets[lo] : 0;
    const int64_t m = offsets ? offsets[lo + 1] - o0 : rows;
    const int64_t l = pc - koff[lo];
    s_src[threadIdx.x] = (pc < koff[G] && l < m) ? o0 + l : -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int r = i >> 6, c = i & 63;
    const int64_t src = s_src[r];
    float v = 0.f;
    if (src >= 0 && c0 + c < C) v = to_f32(in[src * C + c0 + c]);
    tile[r][c] = __float2bfloat16_rn(v);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int c = i >> 6, r = i & 63;
    if (c0 + c < C && pc0 + r < k_total) out[(int64_t)(c0 + c) * k_total + pc0 + r] = tile[r][c];
  }
}

// out[b][c][r] = in[b][r][c]: batched [rows, cols] -> [cols, rows], output
// batch b at out + b * out_stride
__global__ void __launch_bounds__(256)
transpose_batched_kernel(const bf16* __restrict__ in, int rows, int cols,
                         bf16* __restrict__ out, int64_t out_stride) {
  __shared__ bf16 tile[64][72];
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const bf16* src = in + (int64_t)b * rows * cols;
  bf16* dst = out + (int64_t)b * out_stride;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int r = i >> 6, c = i & 63;
    tile[r][c] = (r0 + r < rows && c0 + c < cols) ? src[(int64_t)(r0 + r) * cols + c0 + c]
                                                  : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int c = i >> 6, r = i & 63;
    if (r0 + r < rows && c0 + c < cols) dst[(int64_t)(c0 + c) * rows + r0 + r] = tile[r][c];
  }
}

// ---------------------------------------------------------------- SwiGLU
// h = silu(g) * u for the kept rows (n_rows = offsets[E] rows of F)
__global__ void silu_mul_kernel(const bf16* __restrict__ g, const bf16* __restrict__ u,
                                bf16* __restrict__ h, const int32_t* __restrict__ offsets,
                                int n_experts, int F) {
  const int64_t n = (int64_t)offsets[n_experts] * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float gv = __bfloat162float(g[i]), uv = __bfloat162float(u[i]);
    h[i] = __float2bfloat16_rn(gv * sigmoid_fast(gv) * uv);
  }
}

// dgu[r] = [dg | du]: dg = dh u silu'(g), du = dh silu(g)
__global__ void swiglu_backward_kernel(const bf16* __restrict__ dh, const bf16* __restrict__ g,
                                       const bf16* __restrict__ u, bf16* __restrict__ dgu,
                                       const int32_t* __restrict__ offsets, int n_experts,
                                       int F) {
  const int64_t n = (int64_t)offsets[n_experts] * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / F;
    const int f = (int)(i - r * F);
    const float gv = __bfloat162float(g[i]), uv = __bfloat162float(u[i]);
    const float dv = __bfloat162float(dh[i]);
    const float sg = sigmoid_fast(gv);
    const float silu = gv * sg;
    const float dsilu = sg * (1.f + gv * (1.f - sg));
    dgu[r * 2 * F + f] = __float2bfloat16_rn(dv * uv * dsilu);
    dgu[r * 2 * F + F + f] = __float2bfloat16_rn(dv * silu);
  }
}

// ---------------------------------------------------------------- combine
// Per token (one CTA): dw[t,j] = <dout[t], y[row]> with y compact (fp16 and
// an exponent per 32 columns, row order), dy[row] = w[t,j] dout[t] (bf16).
constexpr int kCbThreads = 256;
__global__ void __launch_bounds__(kCbThreads)
combine_backward_kernel(const __half* __restrict__ y, const uint8_t* __restrict__ y_e8,
                        const int32_t* __restrict__ row_of_slot, const float* __restrict__ w,
                        const bf16* __restrict__ dout, int64_t n_tokens, int top_k, int d,
                        float* __restrict__ dw, bf16* __restrict__ dy) {
  __shared__ float s_red[kCbThreads / 32];
  const int e8_cols = (d + kYScaleBlock - 1) / kYScaleBlock;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    for (int j = 0; j < top_k; ++j) {
      const int r = row_of_slot[t * top_k + j];
      const float wj = w[t * top_k + j];
      float part = 0.f;
      if (r >= 0) {
        for (int c = threadIdx.x; c < d; c += blockDim.x) {
          const float dv = __bfloat162float(dout[t * d + c]);
          const float sc = __uint_as_float((uint32_t)y_e8[(int64_t)r * e8_cols + c / kYScaleBlock] << 23);
          part = fmaf(dv, __half2float(y[(int64_t)r * d + c]) * sc, part);
          dy[(int64_t)r * d + c] = __float2bfloat16_rn(wj * dv);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
      if (lane == 0) s_red[warp] = part;
      __syncthreads();
      if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int q = 0; q < kCbThreads / 32; ++q) acc += s_red[q];
        dw[t * top_k + j] = r >= 0 ? acc : 0.f;
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------- router
// One warp per token: dz[t, :] from dw through the contribution weights and,
// with d_balance, the balance statistic.  p and s are recomputed from the
// fp32 logits.
template <int EPL>
__global__ void __launch_bounds__(256)
router_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                       const float* __restrict__ w, const float* __restrict__ dw,
                       const int32_t* __restrict__ counts, int64_t n_tokens, int E, int k,
                       int mode, float gscale, float* __restrict__ dz,
                       bf16* __restrict__ dz16) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tokens) return;
  const float* lt = logits + t * E;
  float l[EPL], g[EPL], out[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? lt[e] : -INFINITY;
    g[i] = e < E ? gscale * (float)counts[e] : 0.f;       // dB/dp, d_balance folded in
    out[i] = 0.f;
  }
  // selected part: c = <w, dw> over the token's slots
  float wdw = 0.f, ssel = 0.f;
  for (int j = 0; j < k; ++j) {
    wdw += w[t * k + j] * dw[t * k + j];
    if (mode == 2) ssel += sigmoid_fast(lt[idx[t * k + j]]);
  }
  // balance part: p and <p, g>
  float p[EPL], s[EPL], part = 0.f, pz = 0.f;
  if (mode == 2) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      s[i] = lane + 32 * i < E ? sigmoid_fast(l[i]) : 0.f;
      part += s[i];
    }
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, l[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      s[i] = lane + 32 * i < E ? __expf(l[i] - m) : 0.f;
      part += s[i];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    p[i] = s[i] / part;
    pz += p[i] * g[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pz += __shfl_xor_sync(kFull, pz, o);
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if (mode == 2) out[i] = (g[i] - pz) / part * s[i] * (1.f - s[i]);
    else out[i] = p[i] * (g[i] - pz);
  }
  // selected experts
  for (int j = 0; j < k; ++j) {
    const int e = idx[t * k + j];
    if ((e & 31) != lane) continue;
    const float wj = w[t * k + j], dj = dw[t * k + j];
    float add;
    if (mode == 2) {
      const float se = sigmoid_fast(lt[e]);
      add = (dj - wdw) / ssel * se * (1.f - se);
    } else {
      add = wj * (dj - wdw);
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i == (e >> 5)) out[i] += add;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      dz[t * E + e] = out[i];
      if (dz16 != nullptr) dz16[t * E + e] = __float2bfloat16_rn(out[i]);
    }
  }
}

// ---------------------------------------------------------------- dx
// dx[t] = dxr[t] + sum over kept slots of dxp[row] (fp32 out)
__global__ void __launch_bounds__(256)
dx_reduce_kernel(const bf16* __restrict__ dxp, const int32_t* __restrict__ row_of_slot,
                 const float* __restrict__ dxr, int64_t n_tokens, int top_k, int d,
                 float* __restrict__ dx) {
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      float acc = dxr ? dxr[t * d + c] : 0.f;
      for (int j = 0; j < top_k; ++j) {
        const int r = row_of_slot[t * top_k + j];
        if (r >= 0) acc += __bfloat162float(dxp[(int64_t)r * d + c]);
      }
      dx[t * d + c] = acc;
    }
  }
}

__global__ void __launch_bounds__(256)
column_sums_kernel(const float* __restrict__ dz, int64_t n_tokens, int E, float* __restrict__ out) {
  __shared__ float s_red[256];
  const int e = blockIdx.x;
  float acc = 0.f;
  for (int64_t t = threadIdx.x; t < n_tokens; t += blockDim.x) acc += dz[t * E + e];
  s_red[threadIdx.x] = acc;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if (threadIdx.x < h) s_red[threadIdx.x] += s_red[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[e] = s_red[0];
}

}  // namespace

void launch_column_sums(const float* dz, int64_t n_tokens, int E, float* out, cudaStream_t st) {
  column_sums_kernel<<<E, 256, 0, st>>>(dz, n_tokens, E, out);
}

void launch_pad_offsets(const int32_t* offsets, int64_t rows, int G, int32_t* koff,
                        cudaStream_t st) {
  pad_offsets_kernel<<<1, 32, 0, st>>>(offsets, rows, G, koff);
}

void launch_transpose_grouped(const void* in, bool in_f32, int C, const int32_t* offsets,
                              int64_t rows, int G, const int32_t* koff, int64_t k_total,
                              void* out, cudaStream_t st) {
  if (k_total <= 0 || C <= 0) return;
  const dim3 grid((unsigned)(k_total / 64), (unsigned)((C + 63) / 64));
  if (in_f32)
    transpose_grouped_kernel<float><<<grid, 256, 0, st>>>(
        static_cast<const float*>(in), C, offsets, rows, G, koff, k_total, static_cast<bf16*>(out));
  else
    transpose_grouped_kernel<bf16><<<grid, 256, 0, st>>>(
        static_cast<const bf16*>(in), C, offsets, rows, G, koff, k_total, static_cast<bf16*>(out));
}

void launch_transpose_batched(const void* in, int batch, int rows, int cols, void* out,
                              int64_t out_stride, cudaStream_t st) {
  if (batch <= 0 || rows <= 0 || cols <= 0) return;
  const dim3 grid((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64), (unsigned)batch);
  transpose_batched_kernel<<<grid, 256, 0, st>>>(static_cast<const bf16*>(in), rows, cols,
                                                 static_cast<bf16*>(out), out_stride);
}

void launch_silu_mul(const void* g, const void* u, void* h, const int32_t* offsets,
                     int n_experts, int F, int num_sms, cudaStream_t st) {
  silu_mul_kernel<<<num_sms * 8, 256, 0, st>>>(static_cast<const bf16*>(g),
                                               static_cast<const bf16*>(u),
                                               static_cast<bf16*>(h), offsets, n_experts, F);
}

void launch_swiglu_backward(const void* dh, const void* g, const void* u, void* dgu,
                            const int32_t* offsets, int n_experts, int F, int num_sms,
                            cudaStream_t st) {
  swiglu_backward_kernel<<<num_sms * 8, 256, 0, st>>>(
      static_cast<const bf16*>(dh), static_cast<const bf16*>(g), static_cast<const bf16*>(u),
      static_cast<bf16*>(dgu), offsets, n_experts, F);
}

void launch_combine_backward(const void* y16, const uint8_t* y_e8, const int32_t* row_of_slot,
                             const float* w, const void* dout, int64_t n_tokens, int top_k,
                             int d, float* dw, void* dy, int num_sms, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 8);
  combine_backward_kernel<<<blocks, kCbThreads, 0, st>>>(
      static_cast<const __half*>(y16), y_e8, row_of_slot, w, static_cast<const bf16*>(dout),
      n_tokens, top_k, d, dw, static_cast<bf16*>(dy));
}

void launch_router_backward(const float* logits, const int32_t* idx, const float* w,
                            const float* dw, const int32_t* counts, int64_t n_tokens, int E,
                            int k, int mode, float coef, float d_balance, float* dz,
                            void* dz16, cudaStream_t st) {
  bf16* z16 = static_cast<bf16*>(dz16);
  if (n_tokens <= 0) return;
  const double nn = (double)n_tokens;
  const float gscale = (float)((double)d_balance * coef / (nn * nn));
  const dim3 grid((unsigned)ceil_div64(n_tokens, 8)), block(256);
  if (E <= 32)
    router_backward_kernel<1><<<grid, block, 0, st>>>(logits, idx, w, dw, counts, n_tokens, E,
                                                      k, mode, gscale, dz, z16);
  else if (E <= 64)
    router_backward_kernel<2><<<grid, block, 0, st>>>(logits, idx, w, dw, counts, n_tokens, E,
                                                      k, mode, gscale, dz, z16);
  else if (E <= 128)
    router_backward_kernel<4><<<grid, block, 0, st>>>(logits, idx, w, dw, counts, n_tokens, E,
                                                      k, mode, gscale, dz, z16);
  else
    router_backward_kernel<8><<<grid, block, 0, st>>>(logits, idx, w, dw, counts, n_tokens, E,
                                                      k, mode, gscale, dz, z16);
}

void launch_dx_reduce(const void* dxp, const int32_t* row_of_slot, const float* dxr,
                      int64_t n_tokens, int top_k, int d, float* dx, int num_sms,
                      cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 8);
  dx_reduce_kernel<<<blocks, 256, 0, st>>>(static_cast<const bf16*>(dxp), row_of_slot, dxr,
                                           n_tokens, top_k, d, dx);
}

}  // namespace moe
