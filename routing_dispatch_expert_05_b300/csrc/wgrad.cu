// Weight gradients of the expert (and router / shared) projections on pairs
// of SMs: per group g of token rows [o_g, o_{g+1}),
//
//     C_g[i, j] = sum over rows r of the group of P[r, i] * Q[r, j],
//
// i.e. dW = P_g^T Q_g with P, Q the row-major activations of the forward
// and backward passes ("DeepSeek 5.7: MoE from scratch", Backward pass: each
// expert's weight gradient is accumulated over the tokens routed to it).
//
// Both operands are read in place as MN-major tcgen05 operands: a k-block is
// 64 token rows, and the pair's 256 x 256 tile takes, per CTA, 128 columns
// of P (two TMA boxes of 64 columns x 64 rows, 128-byte swizzle) and 128
// columns of Q the same way, so no transposed copy of any activation is
// made.  Groups are contiguous row ranges of any start; a group whose row
// count is not a multiple of 64 has a last k-block of which only the first
// ceil(rem / 16) slices of 16 rows are multiplied.  The rows after a group
// inside such a slice must be zero: the grouped buffers of the backward pass
// pad every group to a multiple of 16 rows with zero rows, and a group that
// ends at the end of the buffer reads the TMA's zero fill.  A grouping that
// breaks this (or whose offsets are not monotone inside the buffer) sets
// kDevBadRow and its tiles are written as zeros.
//
// The pipeline is the pair kernel's of the grouped GEMM: warp 0 of each CTA
// loads its halves into a 6-stage ring (completing on the leader's full
// barrier), the leader's warp 1 issues tcgen05.mma.cta_group::2 and commits
// to both CTAs' barriers, and eight epilogue warps per CTA read the fp32
// accumulator (two of them in TMEM, 512 columns) and store it; every wait
// is bounded.  With one group, K may be split into chunks whose partial
// sums go to a scratch buffer and are added afterwards (the router's
// gradient: E x d outputs over all N tokens would otherwise be 8 tiles).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace tc {
namespace {

constexpr int kWgTile = 256;                        // output tile (M and N)
constexpr int kWgStages = 6;
constexpr uint32_t kWgHalf = 128 * BK * 2;          // one operand half per CTA: 16 KB
constexpr uint32_t kWgStageBytes = 2 * kWgHalf;     // P half + Q half
constexpr int kWgEpiWarps = 8;
constexpr int kWgThreads = (2 + kWgEpiWarps) * 32;
constexpr uint32_t kWgTmemCols = 2 * kWgTile;       // two accumulators
constexpr int kWgBarBytes = 1024;
constexpr int kWgStgStride = 20;                    // words per staged row (16 fp32 + pad)
constexpr int kWgStgWarpBytes = 32 * kWgStgStride * 4;
constexpr int kWgSmem =
    kWgStages * kWgStageBytes + kWgBarBytes + kWgEpiWarps * kWgStgWarpBytes + 1024;
static_assert(kWgSmem <= 227 * 1024, "shared memory per CTA");

struct WgParams {
  int64_t rows;               // rows of P and Q
  const int32_t* offsets;     // [G+1] or null (one group: all rows)
  int G;
  int m_dim, n_dim;           // output columns of P / Q used
  int mt, nt;                 // 256-wide tiles over m_dim / n_dim
  int splits;                 // chunks of kc rows per group (one group only)
  int64_t kc;
  float* C0;                  // rows i < m_split of each group
  float* C1;                  // rows i >= m_split (null: m_split == m_dim)
  int m_split;
  int32_t* err;
};

struct WgItem {
  int g, s, m, n;
  int64_t k0;
  int cnt;                    // rows to reduce (0: the tile is written as zeros)
  bool bad;
};

__device__ __forceinline__ WgItem wg_item(const WgParams& p, int t) {
  WgItem it;
  const int per_s = p.mt * p.nt;
  const int per_g = p.splits * per_s;
  it.g = t / per_g;
  int l = t - it.g * per_g;
  it.s = l / per_s;
  l -= it.s * per_s;
  it.m = l / p.nt;
  it.n = l - it.m * p.nt;
  int64_t a = 0, b = p.rows;
  if (p.offsets != nullptr) {
    a = __ldg(p.offsets + it.g);
    b = __ldg(p.offsets + it.g + 1);
  }
  it.bad = a < 0 || b < a || b > p.rows;
  if (p.splits > 1) {
    a += (int64_t)it.s * p.kc;
    b = min(b, a + p.kc);
  }
  const int64_t cnt = b > a ? b - a : 0;
  // a partial 16-row slice is only exact where the TMA fills it with zeros
  if (cnt % 16 != 0 && b != p.rows) it.bad = true;
  it.k0 = a;
  it.cnt = it.bad ? 0 : (int)cnt;
  return it;
}

// output row pointer of accumulator row i (i < m_dim) of item `it`
__device__ __forceinline__ float* wg_row(const WgParams& p, const WgItem& it, int i) {
  if (p.splits > 1) return p.C0 + ((int64_t)it.s * p.m_dim + i) * p.n_dim;
  if (p.C1 != nullptr && i >= p.m_split)
    return p.C1 + ((int64_t)it.g * (p.m_dim - p.m_split) + (i - p.m_split)) * p.n_dim;
  const int rows_c0 = p.C1 != nullptr ? p.m_split : p.m_dim;
  return p.C0 + ((int64_t)it.g * rows_c0 + i) * p.n_dim;
}

__global__ void __launch_bounds__(kWgThreads, 1)
tc2_wgrad_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ WgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sP = smem;
  uint8_t* sQ = smem + kWgStages * kWgHalf;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWgStages * kWgStageBytes);
  uint64_t* empty = full + kWgStages;
  uint64_t* tfull = empty + kWgStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  float* s_stage = reinterpret_cast<float*>(smem + kWgStages * kWgStageBytes + kWgBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int total = p.G * p.splits * p.mt * p.nt;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kWgStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 2 * kWgEpiWarps);      // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmP);
    prefetch_map(&tmQ);
  }
  if (warp == 1) tmem_alloc_pair(s_tmem, kWgTmemCols);
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                  // both CTAs' barriers exist
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_phases = 0;
      for (int t = pair; t < total; t += n_pairs) {
        const WgItem it = wg_item(p, t);
        if (it.bad && leader) set_device_error(p.err, kDevBadRow);
        const int nkb = (it.cnt + BK - 1) / BK;
        const int colP = it.m * kWgTile + (int)rank * 128;
        const int colQ = it.n * kWgTile + (int)rank * 128;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1, s_abort, p.err)) { ok = false; break; }
          const uint32_t bar = map_to_rank(&full[stage], 0);
          if (leader) mbar_expect_tx(&full[stage], 2 * kWgStageBytes);
          const int krow = (int)(it.k0 + (int64_t)kb * BK);
          uint8_t* a = sP + stage * kWgHalf;
          uint8_t* b = sQ + stage * kWgHalf;
          tma_load_2d_pair(a, &tmP, bar, colP, krow);
          tma_load_2d_pair(a + 8192, &tmP, bar, colP + 64, krow);
          tma_load_2d_pair(b, &tmQ, bar, colQ, krow);
          tma_load_2d_pair(b + 8192, &tmQ, bar, colQ + 64, krow);
          used |= 1u << stage;
          last_phases = (last_phases & ~(1u << stage)) | (phase << stage);
          if (++stage == kWgStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // the leader's full barriers count both CTAs' copies
      if (leader) {
        for (int s = 0; s < kWgStages; ++s) {
          if (!(used >> s & 1u)) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(&full[s], last_phases >> s & 1u)) {
            if (globaltimer() - t0 > kTimeoutNs) {
              set_device_error(p.err, kDevTimeout);
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
      const uint32_t idesc = idesc_bf16(kWgTile, kWgTile) | kIdescAMnMajor | kIdescBMnMajor;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = pair; t < total; t += n_pairs) {
        const WgItem it = wg_item(p, t);
        const int nkb = (it.cnt + BK - 1) / BK;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kWgTile);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, s_abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sP + stage * kWgHalf);
          const uint32_t b0 = smem_u32(sQ + stage * kWgHalf);
          // slices of 16 rows that hold rows of this group
          const int n16 = kb + 1 < nkb ? BK / 16 : (it.cnt - kb * BK + 15) / 16;
          for (int kk = 0; kk < n16; ++kk)
            umma_pair(d, sdesc_sw128_mn(a0 + kk * 2048), sdesc_sw128_mn(b0 + kk * 2048), idesc,
                      (kb | kk) != 0);
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == kWgStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      umma_commit_pair(drain, 0x1);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(drain, 0)) {
        if (globaltimer() - t0 > kTimeoutNs) {
          set_device_error(p.err, kDevTimeout);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    // warp w reads TMEM lanes 32*(w%4).. (its rows), half (w-2)/4 of the columns
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    float* stg = s_stage + (warp - 2) * (kWgStgWarpBytes / 4);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      const WgItem it = wg_item(p, t);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const int i_base = it.m * kWgTile + (int)rank * 128 + q * 32;  // rows of this warp
      const uint32_t tb = tmem_base + (uint32_t)(acc * kWgTile) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int ci = 0; ci < 4; ++ci) {
        const int c_acc = half * 128 + ci * 32;    // accumulator column
        const int col0 = it.n * kWgTile + c_acc;   // output column
        uint32_t r[32];
        if (it.cnt > 0) {
          MOE_TMEM_LD32(tb + (uint32_t)c_acc, r);
          MOE_TMEM_WAIT32(r);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (col0 >= p.n_dim) continue;
        // two halves of 16 columns through the staging rows: lane = row
        // when staging, then (row of an 8-row group, 16-byte piece) when
        // storing, so each row's 64 bytes go out as one segment
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float4* dst = reinterpret_cast<float4*>(stg + lane * kWgStgStride);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(__uint_as_float(r[16 * hh + 4 * j]),
                                 __uint_as_float(r[16 * hh + 4 * j + 1]),
                                 __uint_as_float(r[16 * hh + 4 * j + 2]),
                                 __uint_as_float(r[16 * hh + 4 * j + 3]));
          __syncwarp();
          const int c4 = lane & 3;
          const int col = col0 + 16 * hh + c4 * 4;
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8) {
            const int rr = k8 * 8 + (lane >> 2);
            const int i = i_base + rr;
            if (i < p.m_dim && col < p.n_dim) {
              const float4 v = *reinterpret_cast<const float4*>(stg + rr * kWgStgStride + c4 * 4);
              *reinterpret_cast<float4*>(wg_row(p, it, i) + col) = v;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cluster(map_to_rank(&tempty[acc], 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();                                  // no CTA leaves while its peer works
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kWgTmemCols);
  }
}

// out[i] = sum over s of part[s * n + i] (the split-K partial sums), float4
__global__ void __launch_bounds__(256)
sum_partials_kernel(const float* __restrict__ part, int splits, int64_t n,
                    float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n4 = n / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = reinterpret_cast<const float4*>(part + (int64_t)s * n)[i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    reinterpret_cast<float4*>(out)[i] = a;
  }
}

int wg_pairs(int num_sms) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(kWgThreads);
  cfg.dynamicSmemBytes = kWgSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void*>(tc2_wgrad_kernel),
                                     &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return std::min(clusters, num_sms / 2);
}

}  // namespace
}  // namespace tc

int wgrad_splits(const WgradProblem& q, int num_sms) {
  if (q.offsets != nullptr || q.n_groups != 1) return 1;
  const int64_t tiles = (int64_t)((q.m_dim + 255) / 256) * ((q.n_dim + 255) / 256);
  const int64_t want = std::max<int64_t>(1, (num_sms / 2) / std::max<int64_t>(tiles, 1));
  // at least 8 k-blocks per chunk
  const int64_t most = std::max<int64_t>(1, q.rows / (8 * tc::BK));
  return (int)std::min<int64_t>({want, most, 64});
}

size_t wgrad_partial_floats(const WgradProblem& q, int num_sms) {
  const int s = wgrad_splits(q, num_sms);
  return s > 1 ? (size_t)s * q.m_dim * q.n_dim : 0;
}

bool launch_wgrad(const WgradProblem& q, int num_sms, cudaStream_t st) {
  using namespace tc;
  // TMA: 16-byte aligned bases and row pitches, column counts in 16-byte units
  auto aligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (q.rows < 1 || q.m_dim < 8 || q.n_dim < 8 || q.m_dim % 8 != 0 || q.n_dim % 8 != 0 ||
      q.p_ld < q.m_dim || q.q_ld < q.n_dim || q.p_ld % 8 != 0 || q.q_ld % 8 != 0 ||
      !aligned(q.P) || !aligned(q.Q) || !aligned(q.C0) || q.n_groups < 1 ||
      q.rows > (int64_t)INT32_MAX - 2 * BK || encode_fn() == nullptr)
    return false;
  if (q.C1 != nullptr && (q.m_split <= 0 || q.m_split >= q.m_dim || !aligned(q.C1)))
    return false;
  WgParams p{};
  p.rows = q.rows;
  p.offsets = q.offsets;
  p.G = q.offsets != nullptr ? q.n_groups : 1;
  p.m_dim = q.m_dim;
  p.n_dim = q.n_dim;
  p.mt = (q.m_dim + kWgTile - 1) / kWgTile;
  p.nt = (q.n_dim + kWgTile - 1) / kWgTile;
  p.splits = wgrad_splits(q, num_sms);
  if (p.splits > 1 && (size_t)p.splits * q.m_dim * q.n_dim > q.partial_floats)
    p.splits = (int)std::min<size_t>((size_t)p.splits, q.partial_floats /
                                                           ((size_t)q.m_dim * q.n_dim));
  if (p.splits < 2) p.splits = 1;
  p.kc = p.splits > 1 ? ((q.rows + p.splits - 1) / p.splits + BK - 1) / BK * BK : q.rows;
  if (p.splits > 1) {
    if (q.partial == nullptr || q.C1 != nullptr || !aligned(q.partial)) return false;
    p.splits = (int)((q.rows + p.kc - 1) / p.kc);  // chunks that hold rows
    p.C0 = q.partial;
  } else {
    p.C0 = q.C0;
  }
  p.C1 = q.C1;
  p.m_split = q.C1 != nullptr ? q.m_split : q.m_dim;
  p.err = q.err;
  CUtensorMap mp, mq;
  if (!make_map(&mp, q.P, (uint64_t)q.m_dim, (uint64_t)q.rows, (uint64_t)q.p_ld * 2, 64u) ||
      !make_map(&mq, q.Q, (uint64_t)q.n_dim, (uint64_t)q.rows, (uint64_t)q.q_ld * 2, 64u))
    return false;
  if (cudaFuncSetAttribute(tc2_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kWgSmem) != cudaSuccess)
    return false;
  const int n_pairs = wg_pairs(num_sms);
  if (n_pairs < 1) return false;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kWgThreads);
  cfg.dynamicSmemBytes = kWgSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, tc2_wgrad_kernel, mp, mq, p) != cudaSuccess) return false;
  if (p.splits > 1) {
    const int64_t n = (int64_t)q.m_dim * q.n_dim;
    const int blocks = (int)std::min<int64_t>((n / 4 + 255) / 256, (int64_t)num_sms * 4);
    if (launch_pdl(tc::sum_partials_kernel, dim3(blocks), dim3(256), 0, st, q.partial,
                   p.splits, n, q.C0) != cudaSuccess)
      return false;
  }
  return true;
}

}  // namespace moe
