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
// A fourth kernel copies x rows into x_perm (32- or 16-byte vectors), token
// by token of x: each token row is read once and written to its k rows (a
// copy row by row of x_perm read each token row k times and was slower).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(256)
dispatch_count_kernel(const int32_t* __restrict__ idx, int64_t n_tokens, int top_k,
                      int n_experts, int tpc, int32_t* __restrict__ chunk_cnt,
                      int32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_cnt[kMaxExperts];
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int64_t t1 = min(n_tokens, t0 + tpc);
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

// The capacity of expert e is `capacity` (< 0: none), or room[e] when a
// per-expert room is given (what a shard of a larger batch may still keep).
// One CTA.  The chunks are split into `slices` runs per expert (thread
// (slice, e), experts warp-contiguous so the loads coalesce); each thread
// sums its run, the runs' sums are scanned in slice order, and each thread
// then writes its run's chunk bases.  The group starts are a two-level
// shuffle scan over the experts.  All integer: the order of the additions
// does not change any result.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(const int32_t* __restrict__ chunk_cnt, int n_chunks,
                     int n_experts, int64_t capacity, const int32_t* __restrict__ room,
                     int pad, int32_t* __restrict__ chunk_base, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                     int32_t* __restrict__ dropped) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_part[kScanThreads];             // run sums, [slice][e_span]
  __shared__ int s_kept[kMaxExperts];
  __shared__ int s_wsum[kMaxExperts / 32];
  const int e_span = (n_experts + 31) / 32 * 32;   // <= kMaxExperts
  const int slices = kScanThreads / e_span;        // >= 4
  const int e = threadIdx.x % e_span, sl = threadIdx.x / e_span;
  const bool mine = sl < slices && e < n_experts;
  const int per = (n_chunks + slices - 1) / slices;
  const int c0 = min(n_chunks, sl * per), c1 = min(n_chunks, c0 + per);
  int sum = 0;
  if (mine)
    for (int c = c0; c < c1; ++c) sum += chunk_cnt[(int64_t)c * n_experts + e];
  if (sl < slices) s_part[sl * e_span + e] = sum;
  __syncthreads();
  if (mine) {
    int run = 0;
    for (int q = 0; q < sl; ++q) run += s_part[q * e_span + e];
    for (int c = c0; c < c1; ++c) {
      const int64_t o = (int64_t)c * n_experts + e;
      const int v = chunk_cnt[o];
      chunk_base[o] = run;
      run += v;
    }
  }
  if (sl == 0 && e < n_experts) {
    int total = 0;
    for (int q = 0; q < slices; ++q) total += s_part[q * e_span + e];
    const int64_t cap = room != nullptr ? (int64_t)max(room[e], 0) : capacity;
    const int kp = cap < 0 ? total : (int)min((int64_t)total, cap);
    s_kept[e] = kp;
    if (counts) counts[e] = total;
    if (kept) kept[e] = kp;
    if (dropped) dropped[e] = total - kp;
  }
  __syncthreads();
  // offsets = exclusive scan of the kept rows (pad > 1: rounded up to
  // multiples of pad, zero rows after the kept)
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int v = 0, incl = 0;
  if (threadIdx.x < kMaxExperts) {
    v = threadIdx.x < n_experts ? (s_kept[threadIdx.x] + pad - 1) / pad * pad : 0;
    incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[w] = incl;
  }
  __syncthreads();
  if (threadIdx.x < n_experts) {
    int base = 0;
    for (int q = 0; q < w; ++q) base += s_wsum[q];
    offsets[threadIdx.x] = base + incl - v;
    if (threadIdx.x == n_experts - 1) offsets[n_experts] = base + incl;
  }
}

// An assignment of rank r (arrival index among expert e's) is kept iff
// r < kept_e = offsets[e+1] - offsets[e]: kept_e = min(total_e, capacity_e)
// and r < total_e, so this is r < capacity_e, whichever capacity applied.
// With padded groups kept_e comes from kept_rows instead.
__global__ void __launch_bounds__(kRankWarps * 32)
dispatch_rank_kernel(const int32_t* __restrict__ idx, int64_t n_tokens, int top_k,
                     int n_experts, int tpc,
                     const int32_t* __restrict__ chunk_base,
                     const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ kept_rows,
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

  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int64_t t1 = min(n_tokens, t0 + tpc);
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
      if (e >= 0 && (kept_rows != nullptr ? rank < kept_rows[e]
                                          : offsets[e] + rank < offsets[e + 1])) {
        row = offsets[e] + rank;
        token_of_row[row] = (int32_t)(s / top_k);
        if (slot_of_row != nullptr) slot_of_row[row] = (int32_t)s;
      }
      row_of_slot[s] = row;
    }
  }
}

// The row copy, driven from the token side: x_perm[row_of_slot[t*k + j]] =
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

// Consistency of a grouping ("DeepSeek 5.7", s.3 and Failure modes: most
// implementation bugs are indexing bugs).  One thread per slot s = t*k + j,
// with e = idx[s] and r = row_of_slot[s]:
//   * e in [0, E), and e differs from the token's earlier slots;
//   * r == -1 (dropped), or offsets[e] <= r < offsets[e+1] with
//     token_of_row[r] == t;
// one thread per row r < M = offsets[E]: token_of_row ascending within each
// group (arrival order); block 0 checks offsets (start 0, never decreasing,
// M <= N*k, no group above the capacity).  The kept slots are counted; the
// last CTA (ticket) checks that they number M.  Kept slots map injectively
// (two slots on one row would share both token and expert, which the
// distinct-experts check excludes), so with M of them row_of_slot is a
// bijection of the kept slots onto [0, M).  Any failure sets kDevBadRow.
__global__ void __launch_bounds__(256)
check_grouping_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
                      const int32_t* __restrict__ row_of_slot,
                      const int32_t* __restrict__ token_of_row, int64_t n_tokens, int top_k,
                      int n_experts, int64_t capacity, unsigned* __restrict__ kept_count,
                      unsigned* __restrict__ ticket, int32_t* __restrict__ err) {
  const int64_t n_slots = n_tokens * top_k;
  const int64_t m = offsets[n_experts];
  bool bad = false;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bad |= offsets[0] != 0 || m > n_slots;
    for (int e = 0; e < n_experts; ++e) {
      const int g = offsets[e + 1] - offsets[e];
      bad |= g < 0 || (capacity >= 0 && g > capacity);
    }
  }
  const bool m_ok = m >= 0 && m <= n_slots;
  unsigned kept = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n_slots; s += stride) {
    const int64_t t = s / top_k;
    const int e = idx[s];
    if (e < 0 || e >= n_experts) { bad = true; continue; }
    for (int64_t q = t * top_k; q < s; ++q) bad |= idx[q] == e;
    const int r = row_of_slot[s];
    if (r == -1) continue;
    // (the row is compared with M first: token_of_row is read only inside it)
    if (!m_ok || r < 0 || r >= m || r < offsets[e] || r >= offsets[e + 1] ||
        token_of_row[r] != (int32_t)t) {
      bad = true;
      continue;
    }
    ++kept;
  }
  if (m_ok) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r + 1 < m; r += stride) {
      // rows r and r+1 of one group hold strictly ascending tokens
      const int32_t a = token_of_row[r], b = token_of_row[r + 1];
      bad |= a < 0 || a >= n_tokens;
      int lo = 0, hi = n_experts - 1;              // the group of row r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
      }
      if (r + 1 < offsets[lo + 1]) bad |= b <= a;
    }
  }
  if (bad) set_device_error(err, kDevBadRow);
  // kept slots: a warp sum, one atomic per warp
  for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(kFull, kept, o);
  if ((threadIdx.x & 31) == 0 && kept != 0) atomicAdd(kept_count, kept);
  __threadfence();
  __syncthreads();
  __shared__ bool s_last;
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  const unsigned total = atomicExch(kept_count, 0u);
  if (!m_ok || total != (unsigned)m) set_device_error(err, kDevBadRow);
  *ticket = 0u;
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
                     int32_t* slot_of_row, const int32_t* room, int pad, int tpc) {
  const int chunks = (int)ceil_div64(n_tokens, tpc);
  if (chunks > 0)
    launch_pdl(dispatch_count_kernel, dim3(chunks), dim3(256), 0, st, idx, n_tokens, top_k,
               n_experts, tpc, chunk_cnt, err);
  pad = pad > 1 && kept != nullptr ? pad : 1;      // padding needs the kept counts
  launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, chunk_cnt, chunks,
             n_experts, capacity, room, pad, chunk_base, offsets, counts, kept, dropped);
  if (chunks > 0)
    launch_pdl(dispatch_rank_kernel, dim3(chunks), dim3(kRankWarps * 32), 0, st, idx, n_tokens,
               top_k, n_experts, tpc, chunk_base, offsets,
               pad > 1 ? static_cast<const int32_t*>(kept) : nullptr, row_of_slot,
               token_of_row, slot_of_row);
}

void launch_check_grouping(const int32_t* idx, const int32_t* offsets,
                           const int32_t* row_of_slot, const int32_t* token_of_row,
                           int64_t n_tokens, int top_k, int n_experts, int64_t capacity,
                           unsigned* kept_count, unsigned* ticket, int32_t* err, int num_sms,
                           cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int64_t blocks_needed = ceil_div64(n_tokens * top_k, 256);
  const int blocks = (int)std::min<int64_t>(blocks_needed, (int64_t)num_sms * 8);
  check_grouping_kernel<<<blocks, 256, 0, st>>>(idx, offsets, row_of_slot, token_of_row,
                                                n_tokens, top_k, n_experts, capacity,
                                                kept_count, ticket, err);
}

}  // namespace moe
