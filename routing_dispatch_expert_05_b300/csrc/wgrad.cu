// Weight gradients of the expert (and router / shared) projections on pairs
// of SMs: per group g of token rows [o_g, o_{g+1}),
//
//     C_g[i, j] = sum over rows r of the group of P[r, i] * Q[r, j],
//
// i.e. dW = P_g^T Q_g with P, Q the row-major activations of the forward
// and backward passes ("DeepSeek 5.7: MoE from scratch", Backward pass: each
// expert's weight gradient is accumulated over the tokens routed to it).
//
// Both operands are read in place as MN-major tcgen05 operands: a stage is
// 128 token rows, and the pair's 256 x 256 tile takes, per CTA, 128 columns
// of P (two TMA boxes of 64 columns x 128 rows, 128-byte swizzle) and 128
// columns of Q the same way, so no transposed copy of any activation is
// made.  Groups are contiguous row ranges of any start; a group whose row
// count is not a multiple of 128 has a last stage of which only the first
// ceil(rem / 16) slices of 16 rows are multiplied.  The rows after a group
// inside such a slice must be zero: the grouped buffers of the backward pass
// pad every group to a multiple of 16 rows with zero rows, and a group that
// ends at the end of the buffer reads the TMA's zero fill.  A grouping that
// breaks this (or whose offsets are not monotone inside the buffer) sets
// kDevBadRow and its tiles are written as zeros.
//
// The pipeline is the pair kernel's of the grouped GEMM: warp 0 of each CTA
// loads its halves into a 3-stage ring (completing on the leader's full
// barrier), the leader's warp 1 issues tcgen05.mma.cta_group::2 and commits
// to both CTAs' barriers, and eight epilogue warps per CTA read the fp32
// accumulator (two of them in TMEM, 512 columns); every wait is bounded.
// An epilogue warp loads its 32 rows x 128 columns into registers and hands
// the accumulator back at once (the MMA never waits for stores), then writes
// each 32 x 32 chunk with a TMA tensor store from a 128-byte-swizzled
// staging buffer.  The output maps are 3-D (group, row, column), so a chunk
// is clipped at its group's last row and column; the weight gradients are
// written once, in fp32, without a pass through the load/store unit.
// With one group, K may be split into chunks whose partial sums go to a
// scratch buffer and are added afterwards (the router's gradient: E x d
// outputs over all N tokens would otherwise be 8 tiles).
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
// A stage holds 128 token rows: per CTA and operand two TMA boxes of 64
// columns x 128 rows (16 KB each).  (With 64-row k-blocks, four 8 KB boxes
// per CTA and k-block, issuing the copies took nearly as long as the MMAs.)
constexpr int kWgK = 128;                            // token rows per stage
constexpr int kWgStages = 3;
constexpr uint32_t kWgBox = 64 * kWgK * 2;           // one 64-column box: 16 KB
constexpr uint32_t kWgHalf = 2 * kWgBox;             // one operand half per CTA: 32 KB
constexpr uint32_t kWgStageBytes = 2 * kWgHalf;     // P half + Q half
constexpr int kWgEpiWarps = 8;
constexpr int kWgThreads = (2 + kWgEpiWarps) * 32;
constexpr uint32_t kWgTmemCols = 2 * kWgTile;       // two accumulators
constexpr int kWgBarBytes = 1024;                   // barriers; group order at +512
constexpr int kWgStgWarpBytes = 32 * 32 * 4;        // one 32 x 32 fp32 chunk, swizzled
constexpr int kWgSmem =
    kWgStages * kWgStageBytes + kWgBarBytes + kWgEpiWarps * kWgStgWarpBytes + 1024;
static_assert(kWgSmem <= 227 * 1024, "shared memory per CTA");
static_assert((kWgStages * kWgStageBytes + kWgBarBytes) % 1024 == 0,
              "swizzled staging must start on a 1024-byte boundary");

struct WgParams {
  int64_t rows;               // rows of P and Q
  const int32_t* offsets;     // [G+1] or null (one group: all rows)
  int G;
  int m_dim, n_dim;           // output columns of P / Q used
  int mt, nt;                 // 256-wide tiles over m_dim / n_dim
  int splits;                 // chunks of kc rows per group (one group only)
  int64_t kc;
  int has_c1;                 // rows i >= m_split go to the second output
  int m_split;                // (m_dim without it); a multiple of 32
  int32_t* err;
};

struct WgItem {
  int g, s, m, n;
  int64_t k0;
  int cnt;                    // rows to reduce (0: the tile is written as zeros)
  bool bad;
};

// Tile t belongs to the group of rank t / per_g in order of decreasing row
// count (s_order; equal counts by index): a tile's cost is its group's rows,
// and with the heaviest groups' tiles dealt out first the pairs' loads even
// out (the routing of a real layer is far from uniform).
__device__ __forceinline__ WgItem wg_item(const WgParams& p, const uint8_t* s_order, int t) {
  WgItem it;
  const int per_s = p.mt * p.nt;
  const int per_g = p.splits * per_s;
  const int gi = t / per_g;
  it.g = p.G > 1 ? (int)s_order[gi] : gi;
  int l = t - gi * per_g;
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

__global__ void __launch_bounds__(kWgThreads, 1)
tc2_wgrad_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmC0,
                 const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ WgParams p) {
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
  uint8_t* s_order = reinterpret_cast<uint8_t*>(smem + kWgStages * kWgStageBytes + 512);
  uint8_t* s_stage = smem + kWgStages * kWgStageBytes + kWgBarBytes;

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
    prefetch_map(&tmC0);
    if (p.has_c1) prefetch_map(&tmC1);
  }
  if (warp == 1) tmem_alloc_pair(s_tmem, kWgTmemCols);
  pdl_wait();
  pdl_launch_dependents();
  if (p.G > 1) {
    // group ranks by decreasing rows (the staging area is free until the
    // epilogue starts); every CTA computes the same order
    int* s_rows = reinterpret_cast<int*>(s_stage);
    for (int g = threadIdx.x; g < p.G; g += blockDim.x)
      s_rows[g] = __ldg(p.offsets + g + 1) - __ldg(p.offsets + g);
    __syncthreads();
    for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
      const int rg = s_rows[g];
      int rank = 0;
      for (int h = 0; h < p.G; ++h) {
        const int rh = s_rows[h];
        rank += (rh > rg) | ((rh == rg) & (h < g));
      }
      s_order[rank] = (uint8_t)g;
    }
  }
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
        const WgItem it = wg_item(p, s_order, t);
        if (it.bad && leader) set_device_error(p.err, kDevBadRow);
        const int nkb = (it.cnt + kWgK - 1) / kWgK;
        const int colP = it.m * kWgTile + (int)rank * 128;
        const int colQ = it.n * kWgTile + (int)rank * 128;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1, s_abort, p.err)) { ok = false; break; }
          const uint32_t bar = map_to_rank(&full[stage], 0);
          if (leader) mbar_expect_tx(&full[stage], 2 * kWgStageBytes);
          const int krow = (int)(it.k0 + (int64_t)kb * kWgK);
          uint8_t* a = sP + stage * kWgHalf;
          uint8_t* b = sQ + stage * kWgHalf;
          tma_load_2d_pair(a, &tmP, bar, colP, krow);
          tma_load_2d_pair(a + kWgBox, &tmP, bar, colP + 64, krow);
          tma_load_2d_pair(b, &tmQ, bar, colQ, krow);
          tma_load_2d_pair(b + kWgBox, &tmQ, bar, colQ + 64, krow);
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
        const WgItem it = wg_item(p, s_order, t);
        const int nkb = (it.cnt + kWgK - 1) / kWgK;
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
          const int n16 = kb + 1 < nkb ? kWgK / 16 : (it.cnt - kb * kWgK + 15) / 16;
          for (int kk = 0; kk < n16; ++kk)
            umma_pair(d, sdesc_sw128_mn(a0 + kk * 2048, kWgBox),
                      sdesc_sw128_mn(b0 + kk * 2048, kWgBox), idesc, (kb | kk) != 0);
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
    uint8_t* stg = s_stage + (warp - 2) * kWgStgWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      const WgItem it = wg_item(p, s_order, t);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * kWgTile) + ((uint32_t)(q * 32) << 16);
      uint32_t r[4][32];
      if (it.cnt > 0) {
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) MOE_TMEM_LD32(tb + (uint32_t)(half * 128 + ci * 32), r[ci]);
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) MOE_TMEM_WAIT32(r[ci]);
      } else {
#pragma unroll
        for (int ci = 0; ci < 4; ++ci)
#pragma unroll
          for (int j = 0; j < 32; ++j) r[ci][j] = 0u;
      }
      // the accumulator is in registers: hand it back before any store
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive_relaxed(&tempty[acc]);
        else mbar_arrive_relaxed_cluster(map_to_rank(&tempty[acc], 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      // rows i0 .. i0+31 of the group's output, in the first or second map
      const int i0 = it.m * kWgTile + (int)rank * 128 + q * 32;
      if (i0 >= p.m_dim) continue;
      const bool second = p.has_c1 && i0 >= p.m_split;
      const CUtensorMap* map = second ? &tmC1 : &tmC0;
      const int y = second ? i0 - p.m_split : i0;
      const int z = p.splits > 1 ? it.s : it.g;
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int col0 = it.n * kWgTile + half * 128 + ci * 32;
        if (col0 >= p.n_dim) continue;
        if (lane == 0) bulk_wait_read();           // the previous chunk has left
        __syncwarp();
        // row `lane` = 128 bytes; its 16-byte piece j sits at j ^ (lane % 8)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_uint4(r[ci][4 * j], r[ci][4 * j + 1], r[ci][4 * j + 2], r[ci][4 * j + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(map, stg, col0, y, z);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();                // every store of this warp is done
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

// 3-D fp32 map [z][rows][cols] with 32 x 32 boxes in the 128-byte swizzle
bool make_out_map(CUtensorMap* m, const float* base, uint64_t cols, uint64_t rows, uint64_t z) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, rows, z};
  const cuuint64_t strides[2] = {cols * 4, cols * rows * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
      q.rows > (int64_t)INT32_MAX - 2 * kWgK || q.n_groups > 256 || encode_fn() == nullptr)
    return false;
  if (q.C1 != nullptr && (q.m_split <= 0 || q.m_split >= q.m_dim || q.m_split % 32 != 0 ||
                         !aligned(q.C1)))
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
  }
  float* c0 = p.splits > 1 ? q.partial : q.C0;
  p.has_c1 = q.C1 != nullptr;
  p.m_split = q.C1 != nullptr ? q.m_split : q.m_dim;
  p.err = q.err;
  CUtensorMap mp, mq, mc0, mc1;
  if (!make_map(&mp, q.P, (uint64_t)q.m_dim, (uint64_t)q.rows, (uint64_t)q.p_ld * 2,
                (uint32_t)kWgK) ||
      !make_map(&mq, q.Q, (uint64_t)q.n_dim, (uint64_t)q.rows, (uint64_t)q.q_ld * 2,
                (uint32_t)kWgK))
    return false;
  // outputs: [z][rows][n_dim] fp32, z = group (or split), boxes 32 x 32
  const uint64_t zc = p.splits > 1 ? (uint64_t)p.splits : (uint64_t)p.G;
  if (!make_out_map(&mc0, c0, (uint64_t)q.n_dim, (uint64_t)p.m_split, zc)) return false;
  if (p.has_c1) {
    if (!make_out_map(&mc1, q.C1, (uint64_t)q.n_dim, (uint64_t)(q.m_dim - q.m_split), zc))
      return false;
  } else {
    mc1 = mc0;
  }
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
  if (cudaLaunchKernelEx(&cfg, tc2_wgrad_kernel, mp, mq, mc0, mc1, p) != cudaSuccess)
    return false;
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
