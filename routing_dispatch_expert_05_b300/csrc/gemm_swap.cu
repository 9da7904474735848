// Grouped expert GEMMs for layers whose experts hold few rows each (the
// decode-shaped layer: 64 tokens, top-8 of 128 experts, about four rows per
// expert), on the 5th-generation tensor cores with the operands swapped.
//
// The layer is the same as in gemm_tc.cu ("Implementing Mixed Expert (MoE)
// layers", expert forward pass: silu(fc1 x) * fc2 x, then fc3; "Expert
// Networks", In[7]: the SiLU-MLP with biases): per expert e, out rows
// [offsets[e], offsets[e+1]) of C = epilogue(X W^T).  With a handful of
// rows per expert, a tile of 128 token rows would be almost all padding.
// Here the MMA's M side holds 128 weight rows (output features) and its N
// side the expert's token rows, rounded up to 16: D^T = W X^T, so the
// padding is at most 15 token columns and the work is the streaming of the
// expert weights, each read once.
//
// Structure (one persistent CTA per SM, 10 warps, the pipeline of the
// single-CTA kernel): warp 0 loads, per k-block of 64, the weight tile (128 x
// 64 bf16; for SwiGLU the gate and the up tile of the same 128 features) and
// the token tile (16-row boxes, up to 64 rows) into a ring of stages; one
// lane of warp 1 issues tcgen05.mma (M = 128, N = tokens, K = 16) into one
// of two TMEM accumulators (SwiGLU: a gate and an up accumulator side by
// side); warps 2-9 read them back (TMEM lane = output feature, column =
// token row).  Few, large copies per stage: the copy engine's cost per
// instruction, not per byte, limits 16-row boxes.
//
// Tiles are (expert, block of 64 token rows, block of output features); the
// feature block is fastest, so CTAs working at the same time share the
// token rows and stream disjoint weight rows.
//
// Epilogues:
//   * SwiGLU: the same TMEM lane of the gate and the up accumulator holds
//     one feature, h = silu(gate) * up (128 features per tile);
//   * SiLU + bias: h = silu(v + b1), 128 features per tile;
//   * compact (down projection): each warp's 32 lanes are one 32-column block
//     of an output row, scaled by the row's routing weight; the block's
//     largest magnitude (a warp max) picks the power of two that brings it
//     into [2^14, 2^15), the values are rounded once to fp16 and written to
//     the row's slot, with the exponent byte beside them -- the format of
//     the single-CTA kernel's compact epilogue.
//
// Waits are bounded in time as in gemm_tc.cu.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace sw {

using namespace tc;

constexpr int kWRows = 128;                         // MMA M: weight rows per tile
constexpr int kTokRows = 64;                        // token rows per tile (MMA N <= 64)
constexpr uint32_t kTileW1 = kWRows * BK * 2;       // one weight tile: 16 KB
constexpr uint32_t kTileX = kTokRows * BK * 2;      // 8 KB
constexpr uint32_t kBox = 16 * BK * 2;              // one 16-row token box: 2 KB
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kBarBytes = 1024;
constexpr int kTableBytes = (2 * (kMaxExperts + 1) * 4 + 127) / 128 * 128;
// Ring geometry: SwiGLU stages hold a gate and an up weight tile (5 stages
// of 40 KB), the others one weight tile (8 stages of 24 KB).  TMEM: two
// accumulators of 64 columns (SwiGLU: gate at +0, up at +64 of each).
template <bool SWIGLU> struct Geo {
  static constexpr int kStages = SWIGLU ? 5 : 8;
  static constexpr uint32_t kTileW = (SWIGLU ? 2 : 1) * kTileW1;
  static constexpr uint32_t kStageBytes = kTileW + kTileX;
  static constexpr uint32_t kAccCols = (SWIGLU ? 2 : 1) * kTokRows;
  static constexpr uint32_t kTmemCols = SWIGLU ? 256 : 128;
  static constexpr int kSmem = kStages * kStageBytes + kBarBytes + kTableBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static_assert((kStages * kTileW) % 1024 == 0 && kTileX % 1024 == 0, "swizzle atoms");
};

struct Params {
  const int32_t* offsets;     // [G+1] device
  int n_groups;
  int rows;                   // rows of the grouped buffers (offsets[G] <= rows)
  int K;
  int n_out;                  // output features per group
  int swiglu;                 // 1: W0 gate, W1 up, h = silu(gate) * up
  int epilogue;               // kEpiSwiglu / kEpiSiluBias / kEpiNone (compact)
  const bf16* bias;           // [G][n_out] or null
  int64_t bias_stride;
  void* C;                    // h [rows, n_out] bf16, or compact y16 [*, n_out] fp16
  uint8_t* c_e8;              // compact: exponent bytes [*, e8_cols]
  int e8_cols;
  const int32_t* c_row_map;   // compact: output row of grouped row r (null: r)
  const float* c_row_scale;   // compact: scale of output row o (null: 1)
  int32_t* err;
};

struct Tile {
  int g, row0, row_end, fb;
};

__device__ __forceinline__ Tile tile_of(int t, const int* tile_start, const int* off, int G,
                                        int nfb) {
  int lo = 0, hi = G - 1;  // largest g with tile_start[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  Tile r;
  r.g = lo;
  r.row0 = off[lo] + (local / nfb) * kTokRows;
  r.row_end = min(off[lo + 1], r.row0 + kTokRows);
  r.fb = local % nfb;
  return r;
}

// token columns of a tile's MMA: its rows rounded up to 16
__device__ __forceinline__ int tile_n(const Tile& tl) {
  return (tl.row_end - tl.row0 + 15) & ~15;
}

// ---------------------------------------------------------------- epilogues
// SwiGLU, one 16-column chunk: lane j holds gate (g) and up (u) of feature
// f0 + 32 q + j for token columns c0 .. c0 + 15.
__device__ __forceinline__ void swiglu_chunk(const Params& p, const Tile& tl, int lane, int q,
                                             int c0, const uint32_t (&g)[16],
                                             const uint32_t (&u)[16]) {
  const int f = tl.fb * kWRows + q * 32 + lane;
  if (f >= p.n_out) return;
  bf16* C = static_cast<bf16*>(p.C);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int row = tl.row0 + c0 + i;
    if (row < tl.row_end)
      C[(int64_t)row * p.n_out + f] =
          __float2bfloat16_rn(silu_fast(__uint_as_float(g[i])) * __uint_as_float(u[i]));
  }
}

// SiLU + bias, one 16-column chunk: lane j holds feature f0 + 32 q + j.
__device__ __forceinline__ void silu_bias_chunk(const Params& p, const Tile& tl, int lane, int q,
                                                int c0, const uint32_t (&r)[16]) {
  const int f = tl.fb * kWRows + q * 32 + lane;
  if (f >= p.n_out) return;
  const float b = p.bias ? __bfloat162float(p.bias[(int64_t)tl.g * p.bias_stride + f]) : 0.f;
  bf16* C = static_cast<bf16*>(p.C);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int row = tl.row0 + c0 + i;
    if (row < tl.row_end)
      C[(int64_t)row * p.n_out + f] = __float2bfloat16_rn(silu_fast(__uint_as_float(r[i]) + b));
  }
}

// Compact output, one 16-column chunk: lane j holds feature f0 + 32 q + j of
// token columns c0 .. c0 + 15; the warp's 32 lanes are one exponent block.
__device__ __forceinline__ void compact_chunk(const Params& p, const Tile& tl, int lane, int q,
                                              int c0, const uint32_t (&r)[16]) {
  // n_out is a multiple of 32, so a warp's block of features lies wholly
  // inside or wholly past it; past it there is nothing to write (not even
  // the exponent byte, which would land on the next row's)
  if (tl.fb * kWRows + q * 32 >= p.n_out) return;
  const int f = tl.fb * kWRows + q * 32 + lane;
  const bool f_ok = f < p.n_out;
  const float b = (p.bias && f_ok)
                      ? __bfloat162float(p.bias[(int64_t)tl.g * p.bias_stride + f]) : 0.f;
  // lane i < 16 fetches column i's output row and scale
  int my_orow = -1;
  float my_scale = 1.f;
  {
    const int row = tl.row0 + c0 + lane;
    if (lane < 16 && row < tl.row_end) {
      my_orow = p.c_row_map ? __ldg(p.c_row_map + row) : row;
      if (p.c_row_scale) my_scale = __ldg(p.c_row_scale + my_orow);
    }
  }
  __half* Y = static_cast<__half*>(p.C);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int orow = __shfl_sync(0xffffffffu, my_orow, i);
    const float rscale = __shfl_sync(0xffffffffu, my_scale, i);
    if (orow < 0) continue;                       // warp-uniform
    const float v = f_ok ? __uint_as_float(r[i]) + b : 0.f;
    // the block's largest |v * rscale| is |rscale| * max |v|; non-negative
    // floats order as their bit patterns
    const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
    const float mx = __uint_as_float(mb) * fabsf(rscale);
    int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
    e = min(max(e, -100), 127);
    const float scale = rscale * __uint_as_float((uint32_t)(127 + 14 - e) << 23);
    if (f_ok) Y[(int64_t)orow * p.n_out + f] = __float2half_rn(v * scale);
    if (lane == 0) p.c_e8[(int64_t)orow * p.e8_cols + (f >> 5)] = (uint8_t)(e + 113);
  }
}

// ---------------------------------------------------------------- kernel
template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
swap_gemm_kernel(const __grid_constant__ CUtensorMap tmW0,
                 const __grid_constant__ CUtensorMap tmW1,
                 const __grid_constant__ CUtensorMap tmX, const __grid_constant__ Params p) {
  using Gm = Geo<SWIGLU>;
  constexpr int kStages = Gm::kStages;
  constexpr uint32_t kTileW = Gm::kTileW;
  constexpr uint32_t kStageBytes = Gm::kStageBytes;
  constexpr uint32_t kAccCols = Gm::kAccCols;
  constexpr uint32_t kTmemCols = Gm::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sX = smem + kStages * kTileW;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_tile_start = reinterpret_cast<int*>(smem + kStages * kStageBytes + kBarBytes);
  int* s_off = s_tile_start + kMaxExperts + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.n_groups;
  const int nfb = (p.n_out + kWRows - 1) / kWRows;   // 128 output features per tile
  const int nkb = (p.K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], kEpiWarps);
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmW0);
    if (SWIGLU) prefetch_map(&tmW1);
    prefetch_map(&tmX);
  }
  if (warp == 1) tmem_alloc(s_tmem, kTmemCols);
  pdl_wait();                 // the grouping (offsets) and X come from predecessors
  pdl_launch_dependents();
  if (warp == 2) {
    // tile table: per group, token blocks x feature blocks; the grouping is
    // checked as in the single-CTA kernel (start 0, never decreasing, within
    // the buffer), a bad one runs no tile
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < G; base += 32) {
      const int gg = base + lane;
      int m = 0;
      if (gg < G) {
        const int o0 = p.offsets[gg], o1 = p.offsets[gg + 1];
        s_off[gg] = o0;
        m = o1 - o0;
        bad |= m < 0 || (gg == 0 && o0 != 0);
      }
      const int tiles = m > 0 ? (m + kTokRows - 1) / kTokRows * nfb : 0;
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (gg < G) s_tile_start[gg] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    const int m_total = p.offsets[G];
    bad = __any_sync(0xffffffffu, bad) || m_total > p.rows;
    if (lane == 0) {
      s_tile_start[G] = bad ? 0 : carry;
      s_off[G] = m_total;
      if (bad) set_device_error(p.err, kDevBadRow);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = s_tile_start[G];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_phases = 0;             // per-stage bits
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile tl = tile_of(t, s_tile_start, s_off, G, nfb);
        const int nb = tile_n(tl) >> 4;               // 16-row token boxes
        const int wrow = tl.g * p.n_out + tl.fb * kWRows;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1, s_abort, p.err)) { ok = false; break; }
          mbar_expect_tx(&full[stage], kTileW + (uint32_t)nb * kBox);
          uint8_t* w = sW + stage * kTileW;
          tma_load_2d(w, &tmW0, &full[stage], kb * BK, wrow);
          if (SWIGLU) tma_load_2d(w + kTileW1, &tmW1, &full[stage], kb * BK, wrow);
          uint8_t* x = sX + stage * kTileX;
          for (int i = 0; i < nb; ++i)
            tma_load_2d(x + i * kBox, &tmX, &full[stage], kb * BK, tl.row0 + 16 * i);
          used |= 1u << stage;
          last_phases = (last_phases & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // every issued copy has landed before the CTA can exit
      for (int s = 0; s < kStages; ++s) {
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
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile tl = tile_of(t, s_tile_start, s_off, G, nfb);
        const uint32_t idesc = idesc_bf16(kWRows, tile_n(tl));
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, s_abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sW + stage * kTileW);
          const uint32_t b0 = smem_u32(sX + stage * kTileX);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc,
                 (kb | kk) != 0);
            if (SWIGLU)         // the up accumulator, 64 columns on
              umma(d + kTokRows, sdesc_sw128(a0 + kTileW1 + kk * 32), sdesc_sw128(b0 + kk * 32),
                   idesc, (kb | kk) != 0);
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // all MMAs issued by this thread are complete before TMEM is freed
      umma_commit(drain);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(drain, 0)) {
        if (globaltimer() - t0 > kTimeoutNs) {
          set_device_error(p.err, kDevTimeout);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int q = warp & 3;                          // TMEM lane quadrant
    const int half = (warp - 2) >> 2;                // which 16-column chunks
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = tile_of(t, s_tile_start, s_off, G, nfb);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * kAccCols) + ((uint32_t)(q * 32) << 16);
      const int nch = tile_n(tl) >> 4;
      for (int ch = half; ch < nch; ch += 2) {
        uint32_t r[16];
        MOE_TMEM_LD16(tb + ch * 16, r);
        if constexpr (SWIGLU) {
          uint32_t u[16];
          MOE_TMEM_LD16(tb + kTokRows + ch * 16, u);
          MOE_TMEM_WAIT16(r);
          MOE_TMEM_WAIT16(u);
          swiglu_chunk(p, tl, lane, q, ch * 16, r, u);
        } else {
          MOE_TMEM_WAIT16(r);
          if (p.c_e8 != nullptr) compact_chunk(p, tl, lane, q, ch * 16, r);
          else silu_bias_chunk(p, tl, lane, q, ch * 16, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace sw

bool swap_gemm_supported(const TcProblem& q) {
  if (q.K < 1 || q.n_out < 16 || q.n_out % 16 != 0 || q.n_groups < 1 ||
      q.n_groups > kMaxExperts)
    return false;
  if (q.swiglu && (q.B1 == nullptr || q.c_e8 != nullptr)) return false;
  if (!q.swiglu && q.c_e8 == nullptr && q.epilogue != kEpiSiluBias) return false;
  if (q.c_e8 != nullptr && (q.e8_cols != (q.n_out + 31) / 32 || q.n_out % 32 != 0)) return false;
  return tc::encode_fn() != nullptr;
}

bool launch_swap_gemm(const TcProblem& q, int num_sms, cudaStream_t st) {
  using namespace sw;
  if (!swap_gemm_supported(q)) return false;
  Params p{};
  p.offsets = q.offsets;
  p.n_groups = q.n_groups;
  p.rows = (int)q.rows;
  p.K = q.K;
  p.n_out = q.n_out;
  p.swiglu = q.swiglu;
  p.epilogue = q.swiglu ? kEpiSwiglu : q.epilogue;
  p.bias = static_cast<const bf16*>(q.bias);
  p.bias_stride = q.bias_stride;
  p.C = q.C;
  p.c_e8 = q.c_e8;
  p.e8_cols = q.e8_cols;
  p.c_row_map = q.c_row_map;
  p.c_row_scale = q.c_row_scale;
  p.err = q.err;
  // weights [G * n_out, K] in 128-row boxes; token rows [rows, K] in 16-row
  // boxes
  const uint64_t wrows = (uint64_t)q.n_groups * q.n_out;
  CUtensorMap mw0, mw1, mx;
  if (!make_map(&mw0, q.B0, (uint64_t)q.K, wrows, (uint64_t)q.K * 2, (uint32_t)kWRows))
    return false;
  if (q.swiglu) {
    if (!make_map(&mw1, q.B1, (uint64_t)q.K, wrows, (uint64_t)q.K * 2, (uint32_t)kWRows))
      return false;
  } else {
    mw1 = mw0;
  }
  if (!make_map(&mx, q.A, (uint64_t)q.K, (uint64_t)q.a_rows, (uint64_t)q.K * 2, 16u))
    return false;
  auto kern = q.swiglu ? swap_gemm_kernel<true> : swap_gemm_kernel<false>;
  const int smem = q.swiglu ? Geo<true>::kSmem : Geo<false>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return false;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, st, mw0, mw1, mx, p) ==
         cudaSuccess;
}

}  // namespace moe
