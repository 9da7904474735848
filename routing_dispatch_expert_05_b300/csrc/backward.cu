// The layer's backward pass outside the GEMMs: the weighted combine's and the
// router's gradients, the SwiGLU derivative, the reduction of the expert rows
// back to tokens, and the small layout changes the gradient GEMMs need.
//
// The gradient is that of <dout, out> + d_balance * B with the routing held
// fixed ("DeepSeek 5.7: MoE from scratch", Worked example and study lab: the
// router receives gradients through the contribution weights, the top-k
// choice itself is not differentiable, an expert no token chose gets none):
//   dw[t,j] = <dout[t], y[t,j]>,      dy[t,j] = w[t,j] dout[t]
//   with y = h W2^T + b2 the first is <dout[t] W2, h> + <dout[t], b2>: the
//   data-gradient GEMM's dh_u = dout W2 (unweighted) gives it as a row dot
//   with h, so y is never recomputed; dh = w dh_u
//   softmax modes: dlogit = w * (dw - <w, dw>) on the selected experts
//   sigmoid mode:  dlogit = s (1 - s) (dw - <w, dw>) / sum_sel s
//   balance term:  p (g - <p, g>) (softmax), or through s / sum s (sigmoid),
//                  g_e = d_balance * coef * count_e / N^2
//   SwiGLU:        dg = dh u silu'(g), du = dh silu(g)
//   SiLU-MLP:      da = dh silu'(a), a = W1 x + b1; db1 = sum of da, db2 = sum
//                  of dy over each expert's rows
//   shared experts (weight 1): the SwiGLU terms with dy = dout, one group of
//                  all tokens
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float sigmoid_fast(float z) { return 1.f / (1.f + __expf(-z)); }

// ---------------------------------------------------------------- layouts
// Rows [offsets[e] + kept[e], offsets[e+1]) of buf0 / buf1 set to zero: the
// rows that round each expert's group up to whole 16-row slices of the
// weight-gradient MMAs.  One block per expert; at most pad - 1 rows each.
__global__ void __launch_bounds__(256)
zero_pad_rows_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ kept,
                     int64_t row_bytes, uint8_t* __restrict__ buf0, uint8_t* __restrict__ buf1) {
  const int e = blockIdx.x;
  const int64_t r0 = (int64_t)offsets[e] + kept[e], r1 = offsets[e + 1];
  const int64_t n16 = row_bytes / 16;
  const int64_t total = r1 > r0 ? (r1 - r0) * n16 : 0;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = threadIdx.x; i < total; i += blockDim.x) {
    const int64_t off = (r0 + i / n16) * row_bytes + (i % n16) * 16;
    *reinterpret_cast<uint4*>(buf0 + off) = z;
    if (buf1 != nullptr) *reinterpret_cast<uint4*>(buf1 + off) = z;
  }
}

// 64 x 64 bf16 tiles through shared memory, 16-byte accesses on both sides:
// a thread loads 8 consecutive elements of a source row and, after the
// barrier, gathers 8 of a column into one 16-byte store; 8 threads cover one
// 128-byte row segment either way.  Rows and columns are multiples of 8.
constexpr int kTp = 64 + 8;                        // padded tile row (elements)

__device__ __forceinline__ void tile_store_t(const bf16 (*tile)[kTp], int i, bf16* dst_row0,
                                             int64_t ld, bool ok) {
  const int c = i >> 3, r8 = (i & 7) * 8;          // output row c, source rows r8..r8+7
  if (!ok) return;
  uint4 v;
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bf16 lo = tile[r8 + 2 * j][c], hi = tile[r8 + 2 * j + 1][c];
    w[j] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
  }
  st_vec16(dst_row0 + (int64_t)c * ld + r8, v);
}

// out[b][c][r] = in[b][r][c]: batched [rows, cols] -> [cols, rows], output
// batch b at out + b * out_stride.  A block owns 64 source rows and walks
// every 64-column tile with the next tile's loads in flight (two shared
// buffers, one barrier per tile).
__global__ void __launch_bounds__(256)
transpose_batched_kernel(const bf16* __restrict__ in, int rows, int cols,
                         bf16* __restrict__ out, int64_t out_stride) {
  __shared__ __align__(16) bf16 tile[2][64][kTp];
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 64;
  const bf16* src = in + (int64_t)b * rows * cols;
  bf16* dst = out + (int64_t)b * out_stride;
  const int r = threadIdx.x >> 3, c8 = (threadIdx.x & 7) * 8;
  const bool ok0 = r0 + r < rows, ok1 = r0 + r + 32 < rows;
  const int n_ct = (cols + 63) / 64;
  uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
  auto load = [&](int ct) {
    const int c = ct * 64 + c8;
    v0 = (ok0 && c < cols) ? ld_vec16_nc(src + (int64_t)(r0 + r) * cols + c)
                           : make_uint4(0u, 0u, 0u, 0u);
    v1 = (ok1 && c < cols) ? ld_vec16_nc(src + (int64_t)(r0 + r + 32) * cols + c)
                           : make_uint4(0u, 0u, 0u, 0u);
  };
  load(0);
  for (int ct = 0; ct < n_ct; ++ct) {
    bf16 (*t)[kTp] = tile[ct & 1];
    *reinterpret_cast<uint4*>(&t[r][c8]) = v0;
    *reinterpret_cast<uint4*>(&t[r + 32][c8]) = v1;
    if (ct + 1 < n_ct) load(ct + 1);
    __syncthreads();
    const int c0 = ct * 64;
    for (int i = threadIdx.x; i < 64 * 8; i += 256) {
      const int c = i >> 3, rr8 = (i & 7) * 8;
      tile_store_t(t, i, dst + (int64_t)c0 * rows + r0, rows, c0 + c < cols && r0 + rr8 < rows);
    }
  }
}

// ---------------------------------------------------------------- SwiGLU
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(p[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Per grouped row r (offsets[E] rows, or `rows` when offsets is null; one
// warp each), from dh_u = dout W2 (unweighted), g, u and the row's routing
// weight w_r (1 when w_row is null: the shared experts):
//   h = silu(g) u (SwiGLU) or silu(g) (u null: SiLU-MLP, g = a = W1 x + b1)
//   dw_row[r] = <dh_u, h>              (the weight's gradient, less <dout, b2>)
//   dh = w_r dh_u;  SwiGLU: dgu[r] = [dg | du] (row stride 2F), dg = dh u
//   silu'(g), du = dh silu(g);  SiLU-MLP: dgu[r] = da = dh silu'(a) (stride F)
//   hw[r] = w_r h                      (dW2 = dout_rows^T hw)
// hw and dw_row are nullable.  Lanes take 8 features at a time (16-byte
// loads and stores).
__global__ void __launch_bounds__(256)
expert_rows_backward_kernel(const bf16* __restrict__ dh_u, const bf16* __restrict__ g,
                            const bf16* __restrict__ u, const float* __restrict__ w_row,
                            const int32_t* __restrict__ offsets, int n_experts, int64_t n_rows,
                            int F, bf16* __restrict__ dgu, bf16* __restrict__ hw,
                            float* __restrict__ dw_row) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = offsets != nullptr ? (int64_t)offsets[n_experts] : n_rows;
  const int ld = u != nullptr ? 2 * F : F;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const float wr = w_row != nullptr ? w_row[r] : 1.f;
    float part = 0.f;
    for (int c = lane * 8; c < F; c += 256) {
      float gv[8], uv[8], dv[8], dg[8], du[8], hv[8];
      unpack8(ld_vec16_nc(g + r * F + c), gv);
      if (u != nullptr) unpack8(ld_vec16_nc(u + r * F + c), uv);
      unpack8(ld_vec16_nc(dh_u + r * F + c), dv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float sg = sigmoid_fast(gv[j]);
        const float sl = gv[j] * sg;                 // silu(g)
        const float uj = u != nullptr ? uv[j] : 1.f;
        const float h = sl * uj;
        part = fmaf(dv[j], h, part);
        const float dh = wr * dv[j];
        dg[j] = dh * uj * sg * (1.f + gv[j] * (1.f - sg));
        du[j] = dh * sl;
        hv[j] = wr * h;
      }
      st_vec16(dgu + r * ld + c, pack8(dg));
      if (u != nullptr) st_vec16(dgu + r * ld + F + c, pack8(du));
      if (hw != nullptr) st_vec16(hw + r * F + c, pack8(hv));
    }
    if (dw_row != nullptr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
      if (lane == 0) dw_row[r] = part;
    }
  }
}

// out[g, c] = sum over rows offsets[g] .. offsets[g+1] of in[row, c] (times
// row_w[row] when row_w is non-null; bf16 in, fp32 out): the bias gradients.
// One thread per column, the rows of a group in order, so the sums are the
// same run to run.
__global__ void __launch_bounds__(256)
group_sums_kernel(const bf16* __restrict__ in, int64_t ld, const int32_t* __restrict__ offsets,
                  const float* __restrict__ row_w, int C, float* __restrict__ out) {
  const int g = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  const int64_t r0 = offsets[g], r1 = offsets[g + 1];
  float acc = 0.f;
  for (int64_t r = r0; r < r1; ++r) {
    const float v = __bfloat162float(in[r * ld + c]);
    acc = row_w != nullptr ? fmaf(row_w[r], v, acc) : acc + v;
  }
  out[(int64_t)g * C + c] = acc;
}

// ---------------------------------------------------------------- combine
// One warp per token t: for each kept slot s = (t, j) with row r,
// dy_u[r] = dout[t] (bf16 rows, unweighted) and w_row[r] = w[s]; dw[s] =
// <dout[t], b2[idx[s]]> (0 without expert biases, and for a dropped slot,
// which has no output).  dout is read once per token (16-byte pieces).
__global__ void __launch_bounds__(256)
scatter_dout_kernel(const bf16* __restrict__ dout, const int32_t* __restrict__ row_of_slot,
                    const float* __restrict__ w, const int32_t* __restrict__ idx,
                    const bf16* __restrict__ b2, int64_t n_tokens, int top_k, int d,
                    bf16* __restrict__ dy_u, float* __restrict__ w_row, float* __restrict__ dw) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tokens;
       t += warps) {
    const int64_t s0 = t * top_k;
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 v = ld_vec16_nc(dout + t * d + c);
      for (int j = 0; j < top_k; ++j) {
        const int r = __ldg(row_of_slot + s0 + j);
        if (r >= 0) st_vec16(dy_u + (int64_t)r * d + c, v);
      }
    }
    for (int j = lane; j < top_k; j += 32) {
      const int r = row_of_slot[s0 + j];
      if (r >= 0) w_row[r] = w[s0 + j];
      if (b2 == nullptr || r < 0) dw[s0 + j] = 0.f;
    }
    if (b2 != nullptr) {
      for (int j = 0; j < top_k; ++j) {
        const int r = __ldg(row_of_slot + s0 + j);
        if (r < 0) continue;
        const bf16* bp = b2 + (int64_t)idx[s0 + j] * d;
        float part = 0.f;
        for (int c = lane * 8; c < d; c += 256) {
          float dv[8], bv[8];
          unpack8(ld_vec16_nc(dout + t * d + c), dv);
          unpack8(ld_vec16_nc(bp + c), bv);
#pragma unroll
          for (int q = 0; q < 8; ++q) part = fmaf(dv[q], bv[q], part);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
        if (lane == 0) dw[s0 + j] = part;
      }
    }
  }
}

// dw[s] += dw_row[row_of_slot[s]] for the kept slots
__global__ void __launch_bounds__(256)
slot_dw_kernel(const float* __restrict__ dw_row, const int32_t* __restrict__ row_of_slot,
               int64_t n_slots, float* __restrict__ dw) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n_slots;
       s += (int64_t)gridDim.x * blockDim.x) {
    const int r = row_of_slot[s];
    if (r >= 0) dw[s] += dw_row[r];
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
// dx[t] = dxr[t] + sum over kept slots of dxp[row] (fp32 out), 8 columns per
// thread
__global__ void __launch_bounds__(256)
dx_reduce_kernel(const bf16* __restrict__ dxp, const int32_t* __restrict__ row_of_slot,
                 const float* __restrict__ dxr, const float* __restrict__ dxs,
                 int64_t n_tokens, int top_k, int d, float* __restrict__ dx) {
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float acc[8];
      const float4* xr = reinterpret_cast<const float4*>(dxr + t * d + c);
      const float4 a0 = xr[0], a1 = xr[1];
      acc[0] = a0.x; acc[1] = a0.y; acc[2] = a0.z; acc[3] = a0.w;
      acc[4] = a1.x; acc[5] = a1.y; acc[6] = a1.z; acc[7] = a1.w;
      if (dxs != nullptr) {                          // the shared experts' part
        const float4* xs = reinterpret_cast<const float4*>(dxs + t * d + c);
        const float4 s0 = xs[0], s1 = xs[1];
        acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
        acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
      }
      for (int j = 0; j < top_k; ++j) {
        const int r = row_of_slot[t * top_k + j];
        if (r < 0) continue;
        float v[8];
        unpack8(ld_vec16_nc(dxp + (int64_t)r * d + c), v);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += v[q];
      }
      float4* o = reinterpret_cast<float4*>(dx + t * d + c);
      o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
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

void launch_zero_pad_rows(const int32_t* offsets, const int32_t* kept, int n_experts,
                          int64_t row_bytes, void* buf0, void* buf1, cudaStream_t st) {
  if (n_experts < 1) return;
  zero_pad_rows_kernel<<<n_experts, 256, 0, st>>>(offsets, kept, row_bytes,
                                                  static_cast<uint8_t*>(buf0),
                                                  static_cast<uint8_t*>(buf1));
}

void launch_transpose_batched(const void* in, int batch, int rows, int cols, void* out,
                              int64_t out_stride, cudaStream_t st) {
  if (batch <= 0 || rows <= 0 || cols <= 0) return;
  const dim3 grid(1u, (unsigned)((rows + 63) / 64), (unsigned)batch);
  transpose_batched_kernel<<<grid, 256, 0, st>>>(static_cast<const bf16*>(in), rows, cols,
                                                 static_cast<bf16*>(out), out_stride);
}

void launch_expert_rows_backward(const void* dh_u, const void* g, const void* u,
                                 const float* w_row, const int32_t* offsets, int n_experts,
                                 int64_t rows, int F, void* dgu, void* hw, float* dw_row,
                                 int num_sms, cudaStream_t st) {
  expert_rows_backward_kernel<<<num_sms * 8, 256, 0, st>>>(
      static_cast<const bf16*>(dh_u), static_cast<const bf16*>(g), static_cast<const bf16*>(u),
      w_row, offsets, n_experts, rows, F, static_cast<bf16*>(dgu), static_cast<bf16*>(hw),
      dw_row);
}

void launch_group_sums(const void* in, int64_t ld, const int32_t* offsets, int G, int C,
                       float* out, cudaStream_t st, const float* row_w) {
  if (G <= 0 || C <= 0) return;
  const dim3 grid((unsigned)((C + 255) / 256), (unsigned)G);
  group_sums_kernel<<<grid, 256, 0, st>>>(static_cast<const bf16*>(in), ld, offsets, row_w, C,
                                          out);
}

void launch_scatter_dout(const void* dout, const int32_t* row_of_slot, const float* w,
                         const int32_t* idx, const void* b2, int64_t n_tokens, int top_k, int d,
                         void* dy_u, float* w_row, float* dw, int num_sms, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)std::min<int64_t>(ceil_div64(n_tokens, 8), (int64_t)num_sms * 8);
  scatter_dout_kernel<<<blocks, 256, 0, st>>>(
      static_cast<const bf16*>(dout), row_of_slot, w, idx, static_cast<const bf16*>(b2),
      n_tokens, top_k, d, static_cast<bf16*>(dy_u), w_row, dw);
}

void launch_slot_dw(const float* dw_row, const int32_t* row_of_slot, int64_t n_slots, float* dw,
                    int num_sms, cudaStream_t st) {
  if (n_slots <= 0) return;
  const int blocks = (int)std::min<int64_t>(ceil_div64(n_slots, 256), (int64_t)num_sms * 4);
  slot_dw_kernel<<<blocks, 256, 0, st>>>(dw_row, row_of_slot, n_slots, dw);
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
                      const float* dxs, int64_t n_tokens, int top_k, int d, float* dx,
                      int num_sms, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 8);
  dx_reduce_kernel<<<blocks, 256, 0, st>>>(static_cast<const bf16*>(dxp), row_of_slot, dxr,
                                           dxs, n_tokens, top_k, d, dx);
}

}  // namespace moe
