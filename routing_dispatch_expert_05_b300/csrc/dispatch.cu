// Grouping assignments by expert with a capacity limit.
//
// "Expert Networks > Code Implementation", In[10]: assignments are visited in
// token order; expert e processes an assignment while it has processed fewer
// than `capacity`, otherwise the assignment is dropped and counted.  So the
// assignment of token t to expert e is kept iff its rank r -- the number of
// earlier assignments to e -- is below the capacity, and kept assignments
// of e fill rows offsets[e] + r in arrival order ("DeepSeek 5.7", s.3;
// "Implementing Mixed Expert (MoE) layers", grouping by expert).
//
// Three passes over idx (flattened slot order s = t*k + j; an expert occurs
// at most once per token, so slot order within a token does not change any
// rank):
//   1. count:  per chunk of tokens, assignments per expert (smem atomics);
//   2. scan:   per expert, chunk bases (exclusive scan over chunks), totals,
//              kept = min(total, capacity), dropped, offsets = exclusive
//              scan of kept -- one CTA, fixed order;
//   3. rank:   per chunk, each warp owns a contiguous run of slots; ranks
//              inside a 32-slot step come from __match_any_sync (lanes with
//              the same expert) and a running per-(warp, expert) counter;
//              warp bases are an exclusive scan over the chunk's warps.
// A fourth kernel copies x rows into x_perm (32- or 16-byte vectors), either
// row by row of x_perm (gather) or token by token of x (scatter).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(256)
dispatch_count_kernel(const int32_t* __restrict__ idx, int64_t n_tokens, int top_k,
                      int n_experts, int32_t* __restrict__ chunk_cnt,
                      int32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_cnt[kMaxExperts];
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kDispatchTokensPerChunk;
  const int64_t t1 = min(n_tokens, t0 + kDispatchTokensPerChunk);
  for (int64_t s = t0 * top_k + threadIdx.x; s < t1 * top_k; s += blockDim.x) {
    const int e = idx[s];
    if (e < 0 || e >= n_experts) {
      set_device_error(err, kDevBadExpert);
      continue;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x)
    chunk_cnt[(int64_t)blockIdx.x * n_experts + e] = s_cnt[e];
}

__global__ void __launch_bounds__(kMaxExperts)
dispatch_scan_kernel(const int32_t* __restrict__ chunk_cnt, int n_chunks,
                     int n_experts, int64_t capacity,
                     int32_t* __restrict__ chunk_base, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                     int32_t* __restrict__ dropped) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_kept[kMaxExperts];
  const int e = threadIdx.x;
  if (e < n_experts) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int64_t o = (int64_t)c * n_experts + e;
      const int v = chunk_cnt[o];
      chunk_base[o] = run;
      run += v;
    }
    const int kp = capacity < 0 ? run : (int)min((int64_t)run, capacity);
    s_kept[e] = kp;
    if (counts) counts[e] = run;
    if (kept) kept[e] = kp;
    if (dropped) dropped[e] = run - kp;
  }
  __syncthreads();
  if (e == 0) {
    int acc = 0;
    for (int q = 0; q < n_experts; ++q) {
      offsets[q] = acc;
      acc += s_kept[q];
    }
    offsets[n_experts] = acc;
  }
}

__global__ void __launch_bounds__(kRankWarps * 32)
dispatch_rank_kernel(const int32_t* __restrict__ idx, int64_t n_tokens, int top_k,
                     int n_experts, int64_t capacity,
                     const int32_t* __restrict__ chunk_base,
                     const int32_t* __restrict__ offsets,
                     int32_t* __restrict__ row_of_slot,
                     int32_t* __restrict__ token_of_row,
                     int32_t* __restrict__ slot_of_row) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_w[kRankWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kRankWarps * kMaxExperts; i += blockDim.x)
    (&s_w[0][0])[i] = 0;
  __syncthreads();

  const int64_t t0 = (int64_t)blockIdx.x * kDispatchTokensPerChunk;
  const int64_t t1 = min(n_tokens, t0 + kDispatchTokensPerChunk);
  const int64_t s0 = t0 * top_k, s1 = t1 * top_k;
  const int64_t per_warp = ceil_div64(s1 - s0, kRankWarps);
  const int64_t ws0 = s0 + warp * per_warp;
  const int64_t ws1 = min(s1, ws0 + per_warp);
  const unsigned lt_mask = (1u << lane) - 1u;

  // pass 1: assignments per (warp, expert)
  for (int64_t base = ws0; base < ws1; base += 32) {
    const int64_t s = base + lane;
    int e = s < ws1 ? idx[s] : -1;
    if (e >= n_experts) e = -1;
    const unsigned m = __match_any_sync(kFull, e);
    if (e >= 0 && (m & lt_mask) == 0) s_w[warp][e] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  // warp bases: chunk base + exclusive scan over the chunk's warps
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
    int run = chunk_base[(int64_t)blockIdx.x * n_experts + e];
#pragma unroll
    for (int q = 0; q < kRankWarps; ++q) {
      const int v = s_w[q][e];
      s_w[q][e] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 2: ranks, keep/drop, rows
  for (int64_t base = ws0; base < ws1; base += 32) {
    const int64_t s = base + lane;
    int e = s < ws1 ? idx[s] : -1;
    if (e >= n_experts) e = -1;
    const unsigned m = __match_any_sync(kFull, e);
    int rank = 0;
    if (e >= 0) rank = s_w[warp][e] + __popc(m & lt_mask);
    __syncwarp();
    if (e >= 0 && (m & lt_mask) == 0) s_w[warp][e] += __popc(m);
    __syncwarp();
    if (s < ws1) {
      int32_t row = -1;
      if (e >= 0 && (capacity < 0 || rank < capacity)) {
        row = offsets[e] + rank;
        token_of_row[row] = (int32_t)(s / top_k);
        if (slot_of_row != nullptr) slot_of_row[row] = (int32_t)s;
      }
      row_of_slot[s] = row;
    }
  }
}

// x_perm[r] = x[token_of_row[r]] for r < offsets[E]; one warp per row,
// 32-byte (or 16-byte) vectors, up to 4 in flight per lane.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint8_t* __restrict__ x, int64_t row_bytes,
                   const int32_t* __restrict__ token_of_row,
                   const int32_t* __restrict__ offsets, int n_experts,
                   uint8_t* __restrict__ x_perm, bool wide) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t rows = offsets[n_experts];
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nvec = row_bytes >> 4;
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps_total) {
    const int64_t t = token_of_row[r];
    const uint8_t* src = x + t * row_bytes;
    uint8_t* dst = x_perm + r * row_bytes;
    int64_t v = lane;
    if (wide) {
      // 32-byte pieces (256-bit loads and stores), four in flight per lane
      const int64_t n32 = row_bytes >> 5;
      int64_t u = lane;
      for (; u + 96 < n32; u += 128) {
        Vec32 a, b, c, d;
        ld_vec32_nc(src + (u << 5), a);
        ld_vec32_nc(src + ((u + 32) << 5), b);
        ld_vec32_nc(src + ((u + 64) << 5), c);
        ld_vec32_nc(src + ((u + 96) << 5), d);
        st_vec32(dst + (u << 5), a);
        st_vec32(dst + ((u + 32) << 5), b);
        st_vec32(dst + ((u + 64) << 5), c);
        st_vec32(dst + ((u + 96) << 5), d);
      }
      for (; u < n32; u += 32) {
        Vec32 a;
        ld_vec32_nc(src + (u << 5), a);
        st_vec32(dst + (u << 5), a);
      }
      continue;
    }
    for (; v + 96 < nvec; v += 128) {
      const uint4 a = ld_vec16_nc(src + (v << 4));
      const uint4 b = ld_vec16_nc(src + ((v + 32) << 4));
      const uint4 c = ld_vec16_nc(src + ((v + 64) << 4));
      const uint4 d = ld_vec16_nc(src + ((v + 96) << 4));
      st_vec16(dst + (v << 4), a);
      st_vec16(dst + ((v + 32) << 4), b);
      st_vec16(dst + ((v + 64) << 4), c);
      st_vec16(dst + ((v + 96) << 4), d);
    }
    for (; v < nvec; v += 32) st_vec16(dst + (v << 4), ld_vec16_nc(src + (v << 4)));
  }
}

// The same copy driven from the token side: x_perm[row_of_slot[t*k + j]] =
// x[t] for every kept slot.  One warp per token reads its row once (1 KB or
// 4 KB per pass, 32-byte or 16-byte vectors) and writes it to each of its
// rows, so x is read from memory once instead of once per assignment.
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint8_t* __restrict__ x, int64_t row_bytes,
                    const int32_t* __restrict__ row_of_slot, int64_t n_tokens, int top_k,
                    uint8_t* __restrict__ x_perm, bool wide) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int shift = wide ? 5 : 4;
  const int64_t nvec = row_bytes >> shift;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < n_tokens; t += warps_total) {
    const uint8_t* src = x + t * row_bytes;
    for (int64_t u0 = 0; u0 < nvec; u0 += 128) {
      Vec32 a[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t u = u0 + lane + 32 * q;
        if (u < nvec) {
          if (wide) {
            ld_vec32_nc(src + (u << 5), a[q]);
          } else {
            const uint4 v = ld_vec16_nc(src + (u << 4));
            a[q].v[0] = v.x; a[q].v[1] = v.y; a[q].v[2] = v.z; a[q].v[3] = v.w;
          }
        }
      }
      for (int j0 = 0; j0 < top_k; j0 += 32) {
        const int32_t mine = j0 + lane < top_k ? row_of_slot[t * top_k + j0 + lane] : -1;
        const int nj = min(32, top_k - j0);
        for (int j = 0; j < nj; ++j) {
          const int32_t r = __shfl_sync(kFull, mine, j);
          if (r < 0) continue;                       // dropped
          uint8_t* dst = x_perm + (int64_t)r * row_bytes;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t u = u0 + lane + 32 * q;
            if (u >= nvec) continue;
            if (wide) {
              st_vec32(dst + (u << 5), a[q]);
            } else {
              st_vec16(dst + (u << 4), make_uint4(a[q].v[0], a[q].v[1], a[q].v[2], a[q].v[3]));
            }
          }
        }
      }
    }
  }
}

}  // namespace

void launch_scatter_rows(const void* x, int64_t row_bytes, const int32_t* row_of_slot,
                         int64_t n_tokens, int top_k, void* x_perm, int num_sms,
                         cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int64_t blocks_needed = ceil_div64(n_tokens, 8);
  const int blocks = (int)std::min<int64_t>(blocks_needed, (int64_t)num_sms * 8);
  const bool wide = row_bytes % 32 == 0 && (reinterpret_cast<uintptr_t>(x) & 31u) == 0 &&
                    (reinterpret_cast<uintptr_t>(x_perm) & 31u) == 0;
  launch_pdl(scatter_rows_kernel, dim3(blocks), dim3(256), 0, st, static_cast<const uint8_t*>(x), row_bytes,
                                              row_of_slot, n_tokens, top_k,
                                              static_cast<uint8_t*>(x_perm), wide);
}

void launch_dispatch(const int32_t* idx, int64_t n_tokens, int top_k,
                     int n_experts, int64_t capacity, int32_t* chunk_cnt,
                     int32_t* chunk_base, int32_t* offsets, int32_t* row_of_slot,
                     int32_t* token_of_row, int32_t* counts, int32_t* kept,
                     int32_t* dropped, int32_t* err, cudaStream_t st,
                     int32_t* slot_of_row) {
  const int chunks = (int)ceil_div64(n_tokens, kDispatchTokensPerChunk);
  if (chunks > 0)
    launch_pdl(dispatch_count_kernel, dim3(chunks), dim3(256), 0, st, idx, n_tokens, top_k,
               n_experts, chunk_cnt, err);
  launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kMaxExperts), 0, st, chunk_cnt, chunks, n_experts,
                                                  capacity, chunk_base, offsets,
                                                  counts, kept, dropped);
  if (chunks > 0)
    launch_pdl(dispatch_rank_kernel, dim3(chunks), dim3(kRankWarps * 32), 0, st, 
        idx, n_tokens, top_k, n_experts, capacity, chunk_base, offsets,
        row_of_slot, token_of_row, slot_of_row);
}

void launch_gather_rows(const void* x, int64_t row_bytes, const int32_t* token_of_row,
                        const int32_t* offsets, int n_experts, int64_t max_rows,
                        void* x_perm, int num_sms, cudaStream_t st) {
  if (max_rows <= 0) return;
  const int64_t blocks_needed = ceil_div64(max_rows, 8);
  const int blocks = (int)std::min<int64_t>(blocks_needed, (int64_t)num_sms * 8);
  // rows of whole 32-byte pieces at 32-byte aligned bases move as 256-bit
  // accesses (measured ~9% faster than 16-byte ones on 4 KB rows)
  const bool wide = row_bytes % 32 == 0 && (reinterpret_cast<uintptr_t>(x) & 31u) == 0 &&
                    (reinterpret_cast<uintptr_t>(x_perm) & 31u) == 0;
  gather_rows_kernel<<<blocks, 256, 0, st>>>(
      static_cast<const uint8_t*>(x), row_bytes, token_of_row, offsets, n_experts,
      static_cast<uint8_t*>(x_perm), wide);
}

}  // namespace moe
