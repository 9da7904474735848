// Weighted combine back to token order.
//
// out[t] = sum_{j : row_of_slot[t*k+j] >= 0} w[t,j] * y[row_of_slot[t*k+j]] + S[t]
// ("Implementing Mixed Expert (MoE) layers", weighted aggregation with
// index_add_; "Hands-on build guide", step 5; "DeepSeek 5.7", s.3-4).
//
// Written as a gather-reduce rather than a scatter-add: each token reads its
// own k expert rows, so there are no atomics, the fp32 sum runs in slot order
// j = 0..k-1 and the result is rounded and written once.  The expert outputs
// y are fp32 (the combine continues their fp32 accumulation).  A CTA owns a
// run of whole tokens; a thread owns C consecutive columns (8 for a bf16
// output, 4 for fp32), and the loads of four slots are issued before their
// multiply-adds so they are in flight together.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <int NV>
__device__ __forceinline__ void load_cols(const float* p, float4 (&v)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = __ldcs(reinterpret_cast<const float4*>(p) + i);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ row_of_slot,
               const float* __restrict__ w, const float* __restrict__ shared,
               T* __restrict__ out, int64_t n_tokens, int top_k, int d_model) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int C = sizeof(T) == 2 ? 8 : 4;  // columns per thread step
  constexpr int NV = C / 4;                  // float4 per row segment
  const int nvec = d_model / C;
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    const int32_t* rows = row_of_slot + t * top_k;
    const float* wt = w + t * top_k;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int64_t col = (int64_t)v * C;
      float acc[C];
#pragma unroll
      for (int i = 0; i < C; ++i) acc[i] = 0.f;
      int j = 0;
      for (; j + 4 <= top_k; j += 4) {
        float4 val[4][NV];
        int r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          r[q] = rows[j + q];
          if (r[q] >= 0) load_cols<NV>(y + (int64_t)r[q] * d_model + col, val[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (r[q] < 0) continue;
          const float wj = wt[j + q];
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            acc[4 * i + 0] = fmaf(wj, val[q][i].x, acc[4 * i + 0]);
            acc[4 * i + 1] = fmaf(wj, val[q][i].y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(wj, val[q][i].z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(wj, val[q][i].w, acc[4 * i + 3]);
          }
        }
      }
      for (; j < top_k; ++j) {
        const int r = rows[j];
        if (r < 0) continue;
        float4 val[NV];
        load_cols<NV>(y + (int64_t)r * d_model + col, val);
        const float wj = wt[j];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          acc[4 * i + 0] = fmaf(wj, val[i].x, acc[4 * i + 0]);
          acc[4 * i + 1] = fmaf(wj, val[i].y, acc[4 * i + 1]);
          acc[4 * i + 2] = fmaf(wj, val[i].z, acc[4 * i + 2]);
          acc[4 * i + 3] = fmaf(wj, val[i].w, acc[4 * i + 3]);
        }
      }
      if (shared != nullptr) {
        float4 s[NV];
        load_cols<NV>(shared + t * d_model + col, s);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          acc[4 * i + 0] += s[i].x;
          acc[4 * i + 1] += s[i].y;
          acc[4 * i + 2] += s[i].z;
          acc[4 * i + 3] += s[i].w;
        }
      }
      T* op = out + t * d_model + col;
      if constexpr (C == 4) {
        *reinterpret_cast<float4*>(op) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      } else {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        st_vec16(op, o);
      }
    }
  }
}

// The combine when the down projection has already weighted and placed the
// expert outputs (compact) in slot order: row t*k + j holds w[t,j] * y of
// slot j, so of the weighted sum ("DeepSeek 5.7", s.3) only the sum is left
// here.  out[t] = sum over kept slots j of those rows, in slot order, + S[t].  A token's k rows are contiguous, so the kernel streams
// them; their addresses need no index load.
// row_of_slot == null: the layer has no capacity, every slot is kept (its
// rows are then read without waiting for an index load).
template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
combine_slots_kernel(const __half* __restrict__ y, const uint8_t* __restrict__ y_e8,
                     const int32_t* __restrict__ row_of_slot,
                     const float* __restrict__ shared, T* __restrict__ out,
                     int64_t n_tokens, int top_k, int d_model) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int C = 8;                       // columns per thread step (16 B of fp16)
  constexpr int KB = 8;                      // slots in flight
  const int nvec = d_model / C;
  const int e8_cols = (d_model + kYScaleBlock - 1) / kYScaleBlock;
  for (int64_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int64_t col = (int64_t)v * C;
      const int blk = (int)(col / kYScaleBlock);
      float acc[C];
#pragma unroll
      for (int i = 0; i < C; ++i) acc[i] = 0.f;
      for (int j0 = 0; j0 < top_k; j0 += KB) {
        uint4 val[KB];
        float sc[KB];
        bool keep[KB];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          const int j = j0 + q;
          const int64_t slot = t * top_k + j;
          keep[q] = false;
          sc[q] = 0.f;
          val[q] = make_uint4(0u, 0u, 0u, 0u);
          // dropped slots hold no row: nothing of theirs is read
          if (j < top_k && (row_of_slot == nullptr || row_of_slot[slot] >= 0)) {
            keep[q] = true;
            val[q] = __ldcs(reinterpret_cast<const uint4*>(y + slot * d_model + col));
            sc[q] = __uint_as_float((uint32_t)y_e8[slot * e8_cols + blk] << 23);
          }
        }
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          if (!keep[q]) continue;
          const __half2* h2 = reinterpret_cast<const __half2*>(&val[q]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h2[i]);
            acc[2 * i] = fmaf(sc[q], f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(sc[q], f.y, acc[2 * i + 1]);
          }
        }
      }
      if (shared != nullptr) {
        const float4* sp = reinterpret_cast<const float4*>(shared + t * d_model + col);
        const float4 s0 = __ldcs(sp), s1 = __ldcs(sp + 1);
        acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
        acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
      }
      T* op = out + t * d_model + col;
      if constexpr (sizeof(T) == 4) {
        reinterpret_cast<float4*>(op)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(op)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        st_vec16(op, o);
      }
    }
  }
}

// The same combine with each token's slot rows streamed into shared memory
// by bulk copies: in slot order the k rows of token t are one contiguous
// block of k * d fp16 (and k * d/32 exponent bytes), so one elected thread
// copies a whole token per stage (cp.async.bulk, completing on an mbarrier)
// into a three-stage ring, and the block's threads sum the rows from shared
// memory.  Two blocks per SM keep ~200 KB of y in flight with a handful of
// instructions, where the register-fed kernel holds 128 KB (eight 16-byte
// loads per thread).  Waits are bounded: on expiry the block records
// kDevTimeout and leaves.
constexpr int kBulkStages = 3;
constexpr int kBulkStageMax = 36 * 1024;           // y rows + exponents of one token

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(tc::smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(tc::smem_u32(bar))
      : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
combine_bulk_kernel(const __half* __restrict__ y, const uint8_t* __restrict__ y_e8,
                    const int32_t* __restrict__ row_of_slot,
                    const float* __restrict__ shared, T* __restrict__ out, int64_t n_tokens,
                    int top_k, int d_model, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kBulkStages];
  constexpr int C = 8;
  const int nvec = d_model / C;
  const int e8_cols = d_model / kYScaleBlock;
  const uint32_t y_bytes = (uint32_t)top_k * d_model * 2;
  const uint32_t e_bytes = (uint32_t)top_k * e8_cols;
  const uint32_t s_bytes = shared != nullptr ? (uint32_t)d_model * 4 : 0u;  // the shared row
  const uint32_t stage_bytes = (y_bytes + e_bytes + s_bytes + 127) / 128 * 128;
  if (threadIdx.x == 0) {
    for (int q = 0; q < kBulkStages; ++q) tc::mbar_init(&full[q], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n_mine =
      n_tokens > blockIdx.x ? (n_tokens - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  auto issue = [&](int64_t i) {
    const int64_t t = blockIdx.x + i * gridDim.x;
    const int q = (int)(i % kBulkStages);
    uint8_t* st_y = smem + q * stage_bytes;
    tc::mbar_expect_tx(&full[q], y_bytes + e_bytes + s_bytes);
    bulk_load(st_y, y + t * top_k * d_model, y_bytes, &full[q]);
    bulk_load(st_y + y_bytes, y_e8 + t * top_k * e8_cols, e_bytes, &full[q]);
    if (s_bytes != 0u)
      bulk_load(st_y + y_bytes + e_bytes, shared + t * d_model, s_bytes, &full[q]);
  };
  int64_t issued = 0;                              // (thread 0) tokens whose copies went out
  if (threadIdx.x == 0)
    for (; issued < n_mine && issued < kBulkStages; ++issued) issue(issued);
  int64_t i = 0;
  for (; i < n_mine; ++i) {
    const int q = (int)(i % kBulkStages);
    const uint32_t parity = (uint32_t)((i / kBulkStages) & 1);
    // every thread waits on the stage (bounded); the block leaves together
    // if any of its threads gave up
    const uint64_t t0 = tc::globaltimer();
    bool ok = true;
    while (!tc::mbar_try_wait(&full[q], parity)) {
      if (tc::globaltimer() - t0 > tc::kTimeoutNs) {
        ok = false;
        break;
      }
    }
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) set_device_error(err, kDevTimeout);
      break;
    }
    const int64_t t = blockIdx.x + i * gridDim.x;
    const uint8_t* st_y = smem + q * stage_bytes;
    const uint8_t* st_e = st_y + y_bytes;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int col = v * C;
      const int blk = col / kYScaleBlock;
      float acc[C];
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = 0.f;
      for (int j = 0; j < top_k; ++j) {
        // a dropped slot's row was copied but holds nothing of its own
        if (row_of_slot != nullptr && row_of_slot[t * top_k + j] < 0) continue;
        const uint4 val = *reinterpret_cast<const uint4*>(st_y + ((size_t)j * d_model + col) * 2);
        const float sc = __uint_as_float((uint32_t)st_e[j * e8_cols + blk] << 23);
        const __half2* h2 = reinterpret_cast<const __half2*>(&val);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = __half22float2(h2[c]);
          acc[2 * c] = fmaf(sc, f.x, acc[2 * c]);
          acc[2 * c + 1] = fmaf(sc, f.y, acc[2 * c + 1]);
        }
      }
      if (s_bytes != 0u) {
        const float4* sp = reinterpret_cast<const float4*>(st_e + e_bytes) + col / 4;
        const float4 s0 = sp[0], s1 = sp[1];
        acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
        acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
      }
      T* op = out + t * d_model + col;
      if constexpr (sizeof(T) == 4) {
        reinterpret_cast<float4*>(op)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(op)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        st_vec16(op, o);
      }
    }
    // the stage is read by every thread before it is refilled
    __syncthreads();
    if (threadIdx.x == 0 && issued < n_mine) issue(issued++);
  }
  // after a timeout, the copies already issued land before the block leaves
  // (each waited for once more, bounded)
  if (threadIdx.x == 0) {
    for (int64_t j = i; j < issued; ++j) {
      const uint64_t t0 = tc::globaltimer();
      while (!tc::mbar_try_wait(&full[j % kBulkStages], (uint32_t)((j / kBulkStages) & 1)) &&
             tc::globaltimer() - t0 < tc::kTimeoutNs) {
      }
    }
  }
}

}  // namespace

void launch_combine_slots(const void* y16, const uint8_t* y_e8, const int32_t* row_of_slot,
                          const float* shared, void* out, int64_t n_tokens, int top_k,
                          int d_model, int is_bf16, int num_sms, cudaStream_t st,
                          int32_t* err) {
  if (n_tokens <= 0) return;
  const __half* y = static_cast<const __half*>(y16);
  // whole tokens by bulk copies where a token's rows and exponents fit a
  // stage and the copies keep 16-byte granularity
  const int e8_cols = d_model / kYScaleBlock;
  const int64_t y_bytes = (int64_t)top_k * d_model * 2;
  const int64_t e_bytes = (int64_t)top_k * e8_cols;
  const int64_t s_bytes = shared != nullptr ? (int64_t)d_model * 4 : 0;
  const int64_t stage = (y_bytes + e_bytes + s_bytes + 127) / 128 * 128;
  const bool bulk = err != nullptr && d_model % kYScaleBlock == 0 && e_bytes % 16 == 0 &&
                    stage <= kBulkStageMax &&
                    (reinterpret_cast<uintptr_t>(y16) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(y_e8) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(shared) & 15u) == 0;
  if (bulk) {
    const int smem = (int)(kBulkStages * stage);
    const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 2);
    auto kern = is_bf16 ? reinterpret_cast<const void*>(combine_bulk_kernel<bf16>)
                        : reinterpret_cast<const void*>(combine_bulk_kernel<float>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
        cudaSuccess) {
      const cudaError_t e =
          is_bf16 ? launch_pdl(combine_bulk_kernel<bf16>, dim3(blocks), dim3(kThreads),
                               (size_t)smem, st, y, y_e8, row_of_slot, shared,
                               static_cast<bf16*>(out), n_tokens, top_k, d_model, err)
                  : launch_pdl(combine_bulk_kernel<float>, dim3(blocks), dim3(kThreads),
                               (size_t)smem, st, y, y_e8, row_of_slot, shared,
                               static_cast<float*>(out), n_tokens, top_k, d_model, err);
      if (e == cudaSuccess) return;
    }
    cudaGetLastError();                              // clear, then the register-fed kernel
  }
  const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 4);
  if (is_bf16)
    launch_pdl(combine_slots_kernel<bf16>, dim3(blocks), dim3(kThreads), 0, st, y, y_e8,
               row_of_slot, shared, static_cast<bf16*>(out), n_tokens, top_k, d_model);
  else
    launch_pdl(combine_slots_kernel<float>, dim3(blocks), dim3(kThreads), 0, st, y, y_e8,
               row_of_slot, shared, static_cast<float*>(out), n_tokens, top_k, d_model);
}

void launch_combine(const float* y, const int32_t* row_of_slot, const float* w,
                    const float* shared, void* out, int64_t n_tokens, int top_k,
                    int d_model, int is_bf16, int num_sms, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)std::min<int64_t>(n_tokens, (int64_t)num_sms * 16);
  if (is_bf16)
    combine_kernel<bf16><<<blocks, kThreads, 0, st>>>(
        y, row_of_slot, w, shared, static_cast<bf16*>(out), n_tokens, top_k, d_model);
  else
    combine_kernel<float><<<blocks, kThreads, 0, st>>>(
        y, row_of_slot, w, shared, static_cast<float*>(out), n_tokens, top_k, d_model);
}

}  // namespace moe
