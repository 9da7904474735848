// Grouped bf16 GEMM on the 5th-generation tensor cores (sm_103a):
//   C = epilogue(A B^T), A rows grouped by expert, fp32 accumulation in TMEM.
//
// This is the expert FFN of the layer ("Implementing Mixed Expert (MoE)
// layers", expert forward pass: silu(fc1 x) * fc2 x, then fc3; "DeepSeek
// 5.7", s.1 and s.5: grouped GEMMs over expert-sorted token buffers;
// "Expert Networks", In[7]: the SiLU-MLP with biases).
//
// Structure (one persistent CTA per SM, 6 warps):
//   warp 0     TMA producer: A tile 128 x 64 and B tile 256 x 64 (bf16,
//              128-byte swizzle) per k-block into a 4-stage smem ring;
//   warp 1     owns 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//              one lane issues tcgen05.mma (M=128, N=256, K=16, kind::f16);
//   warps 2-5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31 = tile rows), apply the activation, store bf16.
// The accumulator is double-buffered, so the epilogue of one tile overlaps
// the main loop of the next.
//
// SwiGLU: the B tile holds 128 rows of W1 (gate) and the same 128 rows of
// W3 (up); accumulator columns 0..127 are gate, 128..255 up, and the
// epilogue writes h = silu(gate) * up -- 128 output columns per tile.
//
// Groups: expert e owns rows offsets[e] .. offsets[e+1]-1 (read on the
// device).  Tile t is mapped to (expert, m-tile, n-tile) through a prefix of
// per-expert tile counts; rows of a tile past the expert's end are computed
// (they read the next expert's rows, or zeros past the buffer) but never
// stored.  Empty experts own no tile.
//
// Every wait on an mbarrier is bounded in time: on expiry the CTA records
// kDevTimeout in the error word, the other roles leave their loops, in-flight
// copies and MMAs are waited for (again bounded) and TMEM is freed.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, kStages = 4;
// warp 0 TMA producer, warp 1 MMA issuer, warps 2.. epilogue: two epilogue
// warps per TMEM lane quadrant (warp w may read lanes 32*(w%4)..), each
// taking half of the tile's output columns
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTileA = BM * BK * 2;            // 16 KB
constexpr uint32_t kTileB = BN * BK * 2;            // 32 KB
constexpr uint32_t kStageBytes = kTileA + kTileB;   // 48 KB
constexpr uint32_t kTmemCols = 2 * BN;              // two accumulators
constexpr int kBarBytes = 1024;
// per-group tile starts and row offsets, padded so what follows stays
// 128-byte aligned
constexpr int kTableBytes = (2 * (kMaxExperts + 1) * 4 + 127) / 128 * 128;
// Epilogue staging: each epilogue warp turns its 32 rows x 32 columns chunk
// (one row per lane after tcgen05.ld) into row-contiguous global stores.
// Rows are padded (fp32: 36 words, bf16: 20 words) so that both the
// row-per-lane writes and the column-per-lane reads are free of bank
// conflicts (up to a 2-way conflict on a quarter of the bf16 reads).
constexpr int kStgF32Stride = 20;                  // words per staged row (16 fp32)
constexpr int kStgB16Stride = 20;                  // words per staged row (32 x 16-bit)
constexpr int kStgWarpBytes = 32 * kStgB16Stride * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes + kTableBytes +
                           kEpiWarps * kStgWarpBytes + 1024 /* alignment */;
static_assert((kStages * kStageBytes + kBarBytes + kTableBytes) % 16 == 0,
              "epilogue staging must be 16-byte aligned (vector stores)");
static_assert(kStgWarpBytes % 16 == 0 && (kStgF32Stride * 4) % 16 == 0 &&
                  (kStgB16Stride * 4) % 16 == 0 && kStgF32Stride >= 16 && kStgB16Stride >= 16,
              "staged rows must keep 16-byte alignment and hold 64 bytes");
static_assert(kEpiWarps == 8, "two epilogue warps per TMEM lane quadrant");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// Ring geometry of the single-CTA kernel.  The wide form holds a 256-row B
// tile per stage (4 stages of 48 KB); the narrow form, for one n-tile of at
// most 128 columns without SwiGLU (the router GEMM: N = E), holds a 128-row
// B tile (6 stages of 32 KB): 50% more bytes of A in flight for a GEMM whose
// time is the streaming of A from memory.
template <bool NARROW> struct Ring {
  static constexpr int kStages = NARROW ? 6 : 4;
  static constexpr uint32_t kTileB = NARROW ? 128 * BK * 2 : BN * BK * 2;
  static constexpr uint32_t kStageBytes = kTileA + kTileB;
  static constexpr int kSmem = kStages * kStageBytes + kBarBytes + kTableBytes +
                               kEpiWarps * kStgWarpBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static_assert((kStages * kStageBytes + kBarBytes + kTableBytes) % 16 == 0, "staging alignment");
};

struct Params {
  const int32_t* offsets;     // [G+1] device or null (one group of `rows`)
  int n_groups;
  int rows;
  int a_rows;                 // rows of the A tensor map (a row past them reads zeros)
  int K;                      // reduction length (multiple of 64 per sub-block)
  int n_out;                  // output columns
  int swiglu;                 // 1: B = (W1 rows, W3 rows), epilogue silu(g)*u
  int epilogue;               // kEpiNone / kEpiSiluBias / kEpiSwiglu
  int b_rows;                 // rows of B per group (and per sub-block)
  int k_sub;                  // K-split width (K itself unless split)
  int n_sub;                  // K / k_sub
  const bf16* bias;           // [G][n_out] or null
  int64_t bias_stride;
  void* C;                    // [rows, n_out]
  int c_is_f32;
  uint8_t* c_e8;              // compact fp16 output: per (row, 32 columns) exponent
  int e8_cols;                // ceil(n_out / 32)
  int b_mn;                   // B MN-major (TMA boxes of 64 columns x 64 K-rows)
  int mma_n;                  // MMA N / B rows per tile (single CTA, no SwiGLU):
                              // 256, or n_out rounded up to 16 when a single n-tile
                              // is narrower (the router: N = E)
  int32_t* err;
  const int32_t* a_row_map;   // null: A rows are the tile rows; else A row r
                              // is row a_row_map[r] of the A tensor
  const int32_t* c_row_map;   // compact output only: row r goes to output row
                              // c_row_map[r] (null: row r)
  const float* c_row_scale;   // compact output only: output row o is scaled by
                              // c_row_scale[o] before compacting (null: 1)
};

// ---------------------------------------------------------------- tiles
struct Tile {
  int g, row0, row_end, n;
};

__device__ __forceinline__ Tile tile_of(int t, const int* tile_start, const int* off,
                                        int G, int nt, int bm = BM) {
  int lo = 0, hi = G - 1;  // largest g with tile_start[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  Tile r;
  r.g = lo;
  r.row0 = off[lo] + (local / nt) * bm;
  r.row_end = off[lo + 1];
  r.n = local % nt;
  return r;
}

// ------------------------------------------------------- epilogue helpers
// Writes the warp's staged 32 rows x 16 fp32 columns (row r at
// stg + r * kStgF32Stride) as whole 64-byte row segments: lane = (row of an
// 8-row group, 16-byte piece).
__device__ __forceinline__ void store_staged_f32(const float* stg, int lane, int row_base,
                                                 int row_end, int col0, int n_out, float* C) {
  const int c4 = lane & 3;
  const bool col_ok = col0 + c4 * 4 < n_out;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2);
    const int row = row_base + r;
    if (col_ok && row < row_end) {
      const float4 val = *reinterpret_cast<const float4*>(stg + r * kStgF32Stride + c4 * 4);
      *reinterpret_cast<float4*>(C + (int64_t)row * n_out + col0 + c4 * 4) = val;
    }
  }
}

// Writes the warp's staged 32 rows x 32 16-bit columns (row r at
// stg + r * kStgB16Stride words) as whole 64-byte row segments.
__device__ __forceinline__ void store_staged_b16(const uint32_t* stg, int lane, int row_base,
                                                 int row_end, int col0, int n_out, void* C) {
  const int c8 = lane & 3;
  const bool col_ok = col0 + c8 * 8 < n_out;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2);
    const int row = row_base + r;
    if (col_ok && row < row_end) {
      const uint4 val = *reinterpret_cast<const uint4*>(stg + r * kStgB16Stride + c8 * 4);
      st_vec16(static_cast<uint16_t*>(C) + (int64_t)row * n_out + col0 + c8 * 8, val);
    }
  }
}

// The same 64-byte row segments to output rows given per lane: lane r holds
// the output row of staged row r (negative: not stored).
__device__ __forceinline__ void store_staged_b16_rows(const uint32_t* stg, int lane, int orow,
                                                      int col0, int n_out, void* C) {
  const int c8 = lane & 3;
  const bool col_ok = col0 + c8 * 8 < n_out;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2);
    const int o = __shfl_sync(0xffffffffu, orow, r);
    if (col_ok && o >= 0) {
      const uint4 val = *reinterpret_cast<const uint4*>(stg + r * kStgB16Stride + c8 * 4);
      st_vec16(static_cast<uint16_t*>(C) + (int64_t)o * n_out + col0 + c8 * 8, val);
    }
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The epilogues below read the accumulator in 32-column chunks; the load of
// chunk c+1 is issued before chunk c is converted and stored, so its TMEM
// latency overlaps that work (tcgen05.wait::ld then finds it complete).

// Compact output of one tile, one pass over the accumulator: for each 32
// columns of a row, the largest |v| picks a power of two 2^s that brings it
// into [2^14, 2^15); v * 2^s (exact) is rounded once to fp16, and the biased
// exponent of 2^-s (one byte, an E8 shared exponent) is stored beside it.
// The warp takes half `half` of the tile's 256 columns (4 exponents).
__device__ __forceinline__ void compact_chunk(const Params& p, int lane, int orow, float rscale,
                                              const bf16* bp, int ci, int c0,
                                              const uint32_t (&r)[32], uint32_t* stg,
                                              uint32_t& e8w) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  // the bias test sits outside the per-value loop (tested per value it cost
  // the down projection 4% on a layer without biases); a whole block's 32
  // biases come in four 16-byte loads where they are 16-byte aligned
  if (bp != nullptr) {
    if (c0 + 32 <= p.n_out && (reinterpret_cast<uintptr_t>(bp + c0) & 15u) == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bp + c0) + q);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(b2[i]);
          v[8 * q + 2 * i] += f.x;
          v[8 * q + 2 * i + 1] += f.y;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < p.n_out) v[j] += __bfloat162float(bp[c0 + j]);
    }
  }
  float mx0 = 0.f, mx1 = 0.f, mx2 = 0.f, mx3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    // four independent max chains (columns past n_out hold 0)
    mx0 = fmaxf(mx0, fabsf(v[j]));
    mx1 = fmaxf(mx1, fabsf(v[j + 1]));
    mx2 = fmaxf(mx2, fabsf(v[j + 2]));
    mx3 = fmaxf(mx3, fabsf(v[j + 3]));
  }
  // the block's largest |v * rscale| is |rscale| * max |v| (rounding is
  // monotone); rscale * 2^(14-e) is exact, so v * it rounds as (v * rscale) * 2^(14-e)
  const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * fabsf(rscale);
  int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
  e = min(max(e, -100), 127);                      // zero / tiny blocks: bounded scale
  const float scale = rscale * __uint_as_float((uint32_t)(127 + 14 - e) << 23);
  e8w |= (uint32_t)(e + 113) << (8 * ci);                                // 2^(e-14)
  uint4* dst = reinterpret_cast<uint4*>(stg + lane * kStgB16Stride);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    dst[j] = make_uint4(pack_half2(v[8 * j] * scale, v[8 * j + 1] * scale),
                        pack_half2(v[8 * j + 2] * scale, v[8 * j + 3] * scale),
                        pack_half2(v[8 * j + 4] * scale, v[8 * j + 5] * scale),
                        pack_half2(v[8 * j + 6] * scale, v[8 * j + 7] * scale));
  __syncwarp();
  store_staged_b16_rows(stg, lane, orow, c0, p.n_out, p.C);
  __syncwarp();
}

__device__ __forceinline__ void compact_tile(const Params& p, const Tile& tl, int lane, int half,
                                             int row_base, uint32_t tb, uint32_t* stg) {
  constexpr int kCh = BN / 32 / 2;                 // chunks per half
  const int row = row_base + lane;
  // this lane's output row (rows past the group are not stored) and scale
  int orow = -1;
  float rscale = 1.f;
  if (row < tl.row_end) {
    orow = p.c_row_map != nullptr ? __ldg(p.c_row_map + row) : row;
    if (p.c_row_scale != nullptr) rscale = __ldg(p.c_row_scale + orow);
  }
  const bf16* bp = p.bias ? p.bias + (int64_t)tl.g * p.bias_stride : nullptr;
  const int ch0 = half * kCh;
  uint32_t e8w = 0u;                               // this row's 4 exponents
  uint32_t ra[32], rb[32];
  MOE_TMEM_LD32(tb + ch0 * 32, ra);
  MOE_TMEM_WAIT32(ra);
#pragma unroll
  for (int ci = 0; ci < kCh; ++ci) {
    const int c0 = tl.n * BN + (ch0 + ci) * 32;
    // chunk ci is in ra (even ci) or rb (odd ci); load the next one first
    if (ci % 2 == 0) {
      if (ci + 1 < kCh) MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, rb);
      if (c0 < p.n_out) compact_chunk(p, lane, orow, rscale, bp, ci, c0, ra, stg, e8w);
      if (ci + 1 < kCh) MOE_TMEM_WAIT32(rb);
    } else {
      if (ci + 1 < kCh) MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, ra);
      if (c0 < p.n_out) compact_chunk(p, lane, orow, rscale, bp, ci, c0, rb, stg, e8w);
      if (ci + 1 < kCh) MOE_TMEM_WAIT32(ra);
    }
  }
  if (orow >= 0) {
    const int b0 = tl.n * (BN / 32) + half * kCh;  // first exponent index
    const int n4 = min(kCh, p.e8_cols - b0);
    uint8_t* ep = p.c_e8 + (int64_t)orow * p.e8_cols + b0;
    if (n4 == 4 && (reinterpret_cast<uintptr_t>(ep) & 3u) == 0) {
      *reinterpret_cast<uint32_t*>(ep) = e8w;
    } else {
      for (int i = 0; i < n4; ++i) ep[i] = (uint8_t)(e8w >> (8 * i));
    }
  }
}

// One 32-column chunk of the plain output: v holds the values (activation
// applied); stage them and write whole row segments.
__device__ __forceinline__ void store_chunk(const Params& p, const Tile& tl, int lane,
                                            int row_base, int col0, const float (&v)[32],
                                            float* stg_f, uint32_t* stg_w) {
  if (p.c_is_f32) {
    // two 16-column halves through the staging rows
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float4* dst = reinterpret_cast<float4*>(stg_f + lane * kStgF32Stride);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(v[16 * hh + 4 * j], v[16 * hh + 4 * j + 1],
                             v[16 * hh + 4 * j + 2], v[16 * hh + 4 * j + 3]);
      __syncwarp();
      store_staged_f32(stg_f, lane, row_base, tl.row_end, col0 + 16 * hh, p.n_out,
                       static_cast<float*>(p.C));
      __syncwarp();
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(stg_w + lane * kStgB16Stride);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                          pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                          pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                          pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    __syncwarp();
    store_staged_b16(stg_w, lane, row_base, tl.row_end, col0, p.n_out, p.C);
    __syncwarp();
  }
}

// Plain output of one tile (bf16, or fp32 if c_is_f32): SwiGLU / SiLU+bias /
// identity epilogue.  The warp takes half `half` of the tile's output columns.
template <bool WITH_SWIGLU = true>
__device__ __forceinline__ void store_tile(const Params& p, const Tile& tl, int lane, int half,
                                           int row_base, uint32_t tb, float* stg_f,
                                           uint32_t* stg_w) {
  if (WITH_SWIGLU && p.swiglu) {
    // 128 output columns per tile: gate in accumulator columns 0..127, up in
    // 128..255; two chunks per half
    constexpr int kCh = BN / 2 / 32 / 2;
    const int ch0 = half * kCh;
    uint32_t ga[32], ua[32], gb[32], ub[32];
    MOE_TMEM_LD32(tb + ch0 * 32, ga);
    MOE_TMEM_LD32(tb + BN / 2 + ch0 * 32, ua);
    MOE_TMEM_WAIT32(ga);
    MOE_TMEM_WAIT32(ua);
#pragma unroll
    for (int ci = 0; ci < kCh; ++ci) {
      const int col0 = tl.n * (BN / 2) + (ch0 + ci) * 32;
      const uint32_t(&g)[32] = ci % 2 == 0 ? ga : gb;
      const uint32_t(&u)[32] = ci % 2 == 0 ? ua : ub;
      if (ci + 1 < kCh) {
        if (ci % 2 == 0) {
          MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, gb);
          MOE_TMEM_LD32(tb + BN / 2 + (ch0 + ci + 1) * 32, ub);
        } else {
          MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, ga);
          MOE_TMEM_LD32(tb + BN / 2 + (ch0 + ci + 1) * 32, ua);
        }
      }
      if (col0 < p.n_out) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          v[j] = silu_fast(__uint_as_float(g[j])) * __uint_as_float(u[j]);
        store_chunk(p, tl, lane, row_base, col0, v, stg_f, stg_w);
      }
      if (ci + 1 < kCh) {
        if (ci % 2 == 0) {
          MOE_TMEM_WAIT32(gb);
          MOE_TMEM_WAIT32(ub);
        } else {
          MOE_TMEM_WAIT32(ga);
          MOE_TMEM_WAIT32(ua);
        }
      }
    }
    return;
  }
  constexpr int kCh = BN / 32 / 2;
  const int ch0 = half * kCh;
  uint32_t ra[32], rb[32];
  MOE_TMEM_LD32(tb + ch0 * 32, ra);
  MOE_TMEM_WAIT32(ra);
#pragma unroll
  for (int ci = 0; ci < kCh; ++ci) {
    const int col0 = tl.n * BN + (ch0 + ci) * 32;
    const uint32_t(&r)[32] = ci % 2 == 0 ? ra : rb;
    if (ci + 1 < kCh) {
      if (ci % 2 == 0) MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, rb);
      else MOE_TMEM_LD32(tb + (ch0 + ci + 1) * 32, ra);
    }
    if (col0 < p.n_out) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      if (p.bias) {
        const bf16* bp = p.bias + (int64_t)tl.g * p.bias_stride + col0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < p.n_out) v[j] += __bfloat162float(bp[j]);
      }
      if (p.epilogue == kEpiSiluBias) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = silu_fast(v[j]);
      }
      store_chunk(p, tl, lane, row_base, col0, v, stg_f, stg_w);
    }
    if (ci + 1 < kCh) {
      if (ci % 2 == 0) MOE_TMEM_WAIT32(rb);
      else MOE_TMEM_WAIT32(ra);
    }
  }
}

// The tile table of a grouped problem, built by one warp: s_off[g] = first
// row of group g (s_off[G] = rows in all), s_tile_start[g] = first tile of
// group g (s_tile_start[G] = tiles in all), nt n-tiles per bm-row m-tile.
// The grouping is checked on the way ("DeepSeek 5.7", Failure modes: most
// bugs are indexing bugs): offsets must start at 0, never decrease and end
// within the rows the buffers hold (p.rows).  A grouping that breaks this
// sets kDevBadRow in the error word and gets no tiles, so nothing is read or
// written through it.
__device__ __forceinline__ void build_tile_table(const Params& p, int G, int nt, int bm, int lane,
                                                 int* s_tile_start, int* s_off) {
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < G; base += 32) {
    const int gg = base + lane;
    int m = 0;
    if (gg < G) {
      const int o0 = p.offsets ? p.offsets[gg] : 0;
      const int o1 = p.offsets ? p.offsets[gg + 1] : p.rows;
      s_off[gg] = o0;
      m = o1 - o0;
      bad |= m < 0 || (gg == 0 && o0 != 0);
    }
    const int tiles = m > 0 ? (m + bm - 1) / bm * nt : 0;
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (gg < G) s_tile_start[gg] = carry + incl - tiles;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int m_total = p.offsets ? p.offsets[G] : p.rows;
  bad = __any_sync(0xffffffffu, bad) || m_total > p.rows;
  if (lane == 0) {
    s_tile_start[G] = bad ? 0 : carry;
    s_off[G] = m_total;
    if (bad) set_device_error(p.err, kDevBadRow);
  }
}

// ---------------------------------------------------------------- kernel
// Epilogue kinds, one kernel instantiation each.
enum : int { kEkStore = 0, kEkCompact = 1 };

template <int EK, bool NARROW>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ Params p) {
  using R = Ring<NARROW>;
  constexpr int kStages = R::kStages;
  constexpr uint32_t kTileB = R::kTileB;
  constexpr uint32_t kStageBytes = R::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kTileA;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_tile_start = reinterpret_cast<int*>(smem + kStages * kStageBytes + kBarBytes);
  int* s_off = s_tile_start + kMaxExperts + 1;
  uint8_t* s_stage = smem + kStages * kStageBytes + kBarBytes + kTableBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.offsets ? p.n_groups : 1;
  const int nt_cols = p.swiglu ? BN / 2 : BN;       // output columns per tile
  const int nt = (p.n_out + nt_cols - 1) / nt_cols;  // n-tiles per group
  const int nkb = (p.K + BK - 1) / BK;
  const int kb_per_sub = p.k_sub / BK;

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
    prefetch_map(&tmA);
    prefetch_map(&tmB0);
    if (p.swiglu) prefetch_map(&tmB1);
  }
  if (warp == 1) tmem_alloc(s_tmem, kTmemCols);
  pdl_wait();                 // the grouping (offsets) and A come from predecessors
  pdl_launch_dependents();
  if (warp == 2) build_tile_table(p, G, nt, BM, lane, s_tile_start, s_off);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = s_tile_start[G];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // Lane 0 waits for free stages and loads B (and a plain A tile).  With a
    // row map, the A tile is gathered: lane l loads rows 4l..4l+3 of the
    // tile (tokens row_map[row]) with one gather4 per k-block.
    const bool gather = p.a_row_map != nullptr;
    const int m_total = s_off[G];
    int stage = 0;
    uint32_t phase = 0;
    uint32_t used = 0, last_phases = 0;             // per-stage bits
    if (gather || lane == 0) {
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile tl = tile_of(t, s_tile_start, s_off, G, nt);
        int src[4] = {0, 0, 0, 0};
        if (gather) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // rows past the last kept row read token 0; they are never stored
            const int row = tl.row0 + lane * 4 + i;
            src[i] = row < m_total ? __ldg(p.a_row_map + row) : 0;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          int good = 1;
          if (lane == 0) good = wait_bounded(&empty[stage], phase ^ 1, s_abort, p.err);
          if (gather) good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) { ok = false; break; }
          uint8_t* a = sA + stage * kTileA;
          if (lane == 0) {
            // an MN-major B arrives as 64-column boxes of 8 KB
            const uint32_t b_bytes = p.b_mn ? (uint32_t)((p.mma_n + 63) / 64) * 8192u
                                            : (uint32_t)p.mma_n * BK * 2;
            mbar_expect_tx(&full[stage], kTileA + b_bytes);
            uint8_t* b = sB + stage * kTileB;
            if (!gather) tma_load_2d(a, &tmA, &full[stage], kb * BK, tl.row0);
            if (p.b_mn) {
              // group g, sub-block s: K-rows g*k_sub + kk of B0 / B1
              const int sub = p.n_sub > 1 ? kb / kb_per_sub : 0;
              const int kk = (kb - sub * kb_per_sub) * BK;
              const int krow = tl.g * p.k_sub + kk;
              for (int pc = 0; pc * 64 < p.mma_n; ++pc)
                tma_load_2d(b + pc * 8192, sub ? &tmB1 : &tmB0, &full[stage],
                            tl.n * BN + pc * 64, krow);
            } else if (!NARROW && p.swiglu) {
              const int brow = tl.g * p.b_rows + tl.n * (BN / 2);
              tma_load_2d(b, &tmB0, &full[stage], kb * BK, brow);
              tma_load_2d(b + kTileB / 2, &tmB1, &full[stage], kb * BK, brow);
            } else {
              // K split into n_sub blocks of B (whole k-blocks each); with
              // one block, K itself (of any length)
              const int sub = p.n_sub > 1 ? kb / kb_per_sub : 0;
              const int kk = (kb - sub * kb_per_sub) * BK;
              const int brow = (tl.g * p.n_sub + sub) * p.b_rows + tl.n * BN;
              tma_load_2d(b, &tmB0, &full[stage], kk, brow);
            }
            used |= 1u << stage;
            last_phases = (last_phases & ~(1u << stage)) | (phase << stage);
          }
          if (gather) {
            __syncwarp();
            tma_gather4(a + lane * 4 * (BK * 2), &tmA, &full[stage], kb * BK, src[0], src[1],
                        src[2], src[3]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
    // every issued copy has landed before the CTA can exit
    if (lane == 0) {
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
      const uint32_t idesc = idesc_bf16(BM, p.mma_n) | (p.b_mn ? kIdescBMnMajor : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, s_abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kTileA);
          const uint32_t b0 = smem_u32(sB + stage * kTileB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma(d, sdesc_sw128(a0 + kk * 32),
                 p.b_mn ? sdesc_sw128_mn(b0 + kk * 2048) : sdesc_sw128(b0 + kk * 32), idesc,
                 (kb | kk) != 0);
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
    const int half = (warp - 2) >> 2;                // which half of the columns
    float* stg_f = reinterpret_cast<float*>(s_stage + (warp - 2) * kStgWarpBytes);
    uint32_t* stg_w = reinterpret_cast<uint32_t*>(stg_f);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = tile_of(t, s_tile_start, s_off, G, nt);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const int row_base = tl.row0 + q * 32;         // this warp's 32 rows
      const uint32_t tb = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if constexpr (EK == kEkCompact) {
        compact_tile(p, tl, lane, half, row_base, tb, stg_w);
      } else {
        store_tile<!NARROW>(p, tl, lane, half, row_base, tb, stg_f, stg_w);
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

// The same grouped GEMM on pairs of SMs (a cluster of two CTAs) with
// tcgen05.mma.cta_group::2: a pair computes a 256-row x 256-column tile.
// CTA r of the pair loads rows 128r..128r+127 of A and half of the B tile
// (SwiGLU: r = 0 the gate rows, r = 1 the up rows; otherwise columns
// 128r..128r+127), each 128 x 64 per k-block into a 6-stage ring, and holds
// rows 128r.. of the accumulator in its own TMEM.  Per SM, a k-block moves 32
// KB through shared memory instead of 48 KB for the same tensor work, which
// is what bounds the single-CTA kernel.
//   * both CTAs' copies complete on the leader's (rank 0) full barrier, which
//     expects the bytes of both; the leader's MMA thread issues the MMAs and
//     commits to the empty / accumulator-full barriers of both CTAs at once;
//   * each CTA's epilogue warps read their own TMEM rows and release the
//     accumulator on the leader's barrier (remote arrive from rank 1);
//   * TMEM is allocated and freed by one warp in each CTA, collectively.
// Waits are bounded exactly as in the single-CTA kernel.
constexpr int BM2 = 256;
constexpr int kStages2 = 6;
constexpr uint32_t kTileA2 = 128 * BK * 2;         // this CTA's 128 rows of A
constexpr uint32_t kTileB2 = 128 * BK * 2;         // this CTA's half of B
constexpr uint32_t kStageBytes2 = kTileA2 + kTileB2;
constexpr int kSmemBytes2 =
    kStages2 * kStageBytes2 + kBarBytes + kTableBytes + kEpiWarps * kStgWarpBytes + 1024;
static_assert(kSmemBytes2 <= 227 * 1024, "shared memory per CTA (pairs)");
static_assert((kStages2 * kStageBytes2 + kBarBytes + kTableBytes) % 16 == 0, "staging alignment");

template <int EK>
__global__ void __launch_bounds__(kThreads, 1)
tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages2 * kTileA2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages2 * kStageBytes2);
  uint64_t* empty = full + kStages2;
  uint64_t* tfull = empty + kStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_tile_start = reinterpret_cast<int*>(smem + kStages2 * kStageBytes2 + kBarBytes);
  int* s_off = s_tile_start + kMaxExperts + 1;
  uint8_t* s_stage = smem + kStages2 * kStageBytes2 + kBarBytes + kTableBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int G = p.offsets ? p.n_groups : 1;
  const int nt_cols = p.swiglu ? BN / 2 : BN;       // output columns per tile
  const int nt = (p.n_out + nt_cols - 1) / nt_cols;  // n-tiles per group
  const int nkb = (p.K + BK - 1) / BK;
  const int kb_per_sub = p.k_sub / BK;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 2 * kEpiWarps);        // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmA);
    prefetch_map(&tmB0);
    if (p.swiglu) prefetch_map(&tmB1);
  }
  if (warp == 1) tmem_alloc_pair(s_tmem, kTmemCols);
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 2) build_tile_table(p, G, nt, BM2, lane, s_tile_start, s_off);
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                  // both CTAs' barriers exist
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total = s_tile_start[G];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // Lane 0 waits for free stages and loads B (and a plain A tile).  With a
    // row map, this CTA's 128 A rows are gathered: lane l loads rows
    // 4l..4l+3 of them (tokens row_map[row]) with one gather4 per k-block.
    const bool gather = p.a_row_map != nullptr;
    const int m_total = s_off[G];
    if (gather || lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_phases = 0;
      for (int t = pair; t < total; t += n_pairs) {
        const Tile tl = tile_of(t, s_tile_start, s_off, G, nt, BM2);
        int src[4] = {0, 0, 0, 0};
        if (gather) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // rows past the last kept row read token 0; they are never stored
            const int row = tl.row0 + (int)rank * 128 + lane * 4 + i;
            src[i] = row < m_total ? __ldg(p.a_row_map + row) : 0;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          int good = 1;
          if (lane == 0) good = wait_bounded(&empty[stage], phase ^ 1, s_abort, p.err);
          if (gather) good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) { ok = false; break; }
          const uint32_t bar = map_to_rank(&full[stage], 0);
          uint8_t* a = sA + stage * kTileA2;
          if (lane == 0) {
            if (leader) mbar_expect_tx(&full[stage], 2 * kStageBytes2);
            uint8_t* b = sB + stage * kTileB2;
            if (!gather) {
              // a CTA whose 128 rows all lie past the group's end multiplies
              // padding: it loads from past the end of A, which TMA fills
              // with zeros without reading memory (no traffic, and zero
              // operands cost the tensor cores less power)
              const int arow = tl.row0 + (int)rank * 128;
              tma_load_2d_pair(a, &tmA, bar, kb * BK, arow < tl.row_end ? arow : p.a_rows);
            }
            if (p.b_mn) {
              // this CTA's 128 columns as two 64-column boxes, K-rows
              // g*k_sub + kk of B0 / B1
              const int sub = p.n_sub > 1 ? kb / kb_per_sub : 0;
              const int kk = (kb - sub * kb_per_sub) * BK;
              const int krow = tl.g * p.k_sub + kk;
              const int col = tl.n * BN + (int)rank * 128;
              tma_load_2d_pair(b, sub ? &tmB1 : &tmB0, bar, col, krow);
              tma_load_2d_pair(b + 8192, sub ? &tmB1 : &tmB0, bar, col + 64, krow);
            } else if (p.swiglu) {
              const int brow = tl.g * p.b_rows + tl.n * (BN / 2);
              tma_load_2d_pair(b, rank ? &tmB1 : &tmB0, bar, kb * BK, brow);
            } else {
              // K split into n_sub blocks of B (whole k-blocks each); with
              // one block, K itself (of any length)
              const int sub = p.n_sub > 1 ? kb / kb_per_sub : 0;
              const int kk = (kb - sub * kb_per_sub) * BK;
              const int brow = (tl.g * p.n_sub + sub) * p.b_rows + tl.n * BN + (int)rank * 128;
              tma_load_2d_pair(b, &tmB0, bar, kk, brow);
            }
            used |= 1u << stage;
            last_phases = (last_phases & ~(1u << stage)) | (phase << stage);
          }
          if (gather) {
            __syncwarp();
            tma_gather4_pair(a + lane * 4 * (BK * 2), &tmA, bar, kb * BK, src[0], src[1],
                             src[2], src[3]);
          }
          if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // the leader's full barriers count both CTAs' copies: every issued
      // copy of the pair has landed once they complete
      if (leader && lane == 0) {
        for (int s = 0; s < kStages2; ++s) {
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
      const uint32_t idesc = idesc_bf16(BM2, BN) | (p.b_mn ? kIdescBMnMajor : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = pair; t < total; t += n_pairs) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1, s_abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, s_abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kTileA2);
          const uint32_t b0 = smem_u32(sB + stage * kTileB2);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_pair(d, sdesc_sw128(a0 + kk * 32),
                      p.b_mn ? sdesc_sw128_mn(b0 + kk * 2048) : sdesc_sw128(b0 + kk * 32),
                      idesc, (kb | kk) != 0);
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == kStages2) { stage = 0; phase ^= 1; }
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
    const int q = warp & 3;                          // TMEM lane quadrant
    const int half = (warp - 2) >> 2;                // which half of the columns
    float* stg_f = reinterpret_cast<float*>(s_stage + (warp - 2) * kStgWarpBytes);
    uint32_t* stg_w = reinterpret_cast<uint32_t*>(stg_f);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      const Tile tl = tile_of(t, s_tile_start, s_off, G, nt, BM2);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const int row_base = tl.row0 + (int)rank * 128 + q * 32;
      const uint32_t tb = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if constexpr (EK == kEkCompact) {
        compact_tile(p, tl, lane, half, row_base, tb, stg_w);
      } else {
        store_tile(p, tl, lane, half, row_base, tb, stg_f, stg_w);
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
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------- wait self-check
// The bounded-wait path of the GEMM kernels, made to run out on purpose: two
// roles wait on mbarriers nothing will ever complete; the first gives up
// after limit_ns, records kDevTimeout and raises the CTA's abort flag; the
// second (with a 4x longer limit of its own) leaves on that flag.  flags[r]
// = 1 if role r's wait succeeded (it never should).  No trap, no endless
// loop: the kernel returns and the context stays usable.
__global__ void __launch_bounds__(64)
wait_check_kernel(int32_t* err, uint64_t limit_ns, int32_t* flags) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* ab = &s_abort;
  if (lane == 0 && warp < 2) {
    const bool ok = wait_bounded(&bar[warp], 0, ab, err, warp == 0 ? limit_ns : 4 * limit_ns);
    flags[warp] = ok ? 1 : 0;
  }
}

}  // namespace tc

bool launch_wait_check(int32_t* err, uint64_t limit_ns, int32_t* flags, cudaStream_t st) {
  tc::wait_check_kernel<<<1, 64, 0, st>>>(err, limit_ns, flags);
  return cudaGetLastError() == cudaSuccess;
}

bool tc_gemm_supported(const TcProblem& q) {
  if (q.K < 1 || q.n_out < 8 || q.n_out % 8 != 0) return false;
  if (q.k_sub % tc::BK != 0 && q.n_sub > 1) return false;
  if (q.n_groups > kMaxExperts) return false;
  // compact output: one exponent per 32 columns, no SwiGLU pairing
  if (q.c_e8 != nullptr && (q.swiglu || q.e8_cols != (q.n_out + 31) / 32)) return false;
  if (q.c_e8 == nullptr && (q.c_row_map != nullptr || q.c_row_scale != nullptr)) return false;
  // MN-major B: whole k-blocks per sub-block, not with SwiGLU or a gathered A
  if (q.b_mn_major && (q.swiglu || q.a_row_map != nullptr || q.k_sub % tc::BK != 0 ||
                       (q.n_sub > 1 && q.B1 == nullptr)))
    return false;
  return tc::encode_fn() != nullptr;
}

namespace {
// CTA pairs that can be resident at once for the pair kernel (0: none)
int pair_grid(const void* kern, int num_sms) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = tc::kSmemBytes2;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return std::min(clusters, num_sms / 2);
}
}  // namespace

bool launch_tc_gemm(const TcProblem& q, int num_sms, cudaStream_t st) {
  using namespace tc;
  Params p{};
  p.offsets = q.offsets;
  p.n_groups = q.n_groups;
  p.rows = (int)q.rows;
  p.a_rows = (int)q.a_rows;
  p.K = q.K;
  p.n_out = q.n_out;
  p.swiglu = q.swiglu;
  p.epilogue = q.epilogue;
  p.b_rows = q.b_rows;
  p.k_sub = q.n_sub > 1 ? q.k_sub : q.K;
  p.n_sub = q.n_sub;
  p.bias = static_cast<const bf16*>(q.bias);
  p.bias_stride = q.bias_stride;
  p.C = q.C;
  p.c_is_f32 = q.c_is_f32;
  p.c_e8 = q.c_e8;
  p.e8_cols = q.e8_cols;
  // a single n-tile narrower than 256 columns multiplies only its own width
  p.mma_n = (!q.swiglu && q.n_out < BN) ? (q.n_out + 15) / 16 * 16 : BN;
  p.b_mn = q.b_mn_major;
  p.err = q.err;
  p.a_row_map = q.a_row_map;
  p.c_row_map = q.c_row_map;
  p.c_row_scale = q.c_row_scale;
  const int ksub = p.k_sub;
  const uint64_t brows_total = (uint64_t)q.b_groups * q.n_sub * q.b_rows;
  // A [a_rows, K] (a gathered A is read one row per box, four per gather4);
  // B: SwiGLU halves of 128 rows, otherwise 256 rows (128 per CTA of a pair)
  auto maps = [&](bool pair_tiles, CUtensorMap* ma, CUtensorMap* mb0, CUtensorMap* mb1) {
    if (!make_map(ma, q.A, (uint64_t)q.K, (uint64_t)q.a_rows, (uint64_t)q.K * 2,
                  q.a_row_map ? 1u : (uint32_t)BM))
      return false;
    if (q.b_mn_major) {
      // [b_groups * k_sub K-rows, n_out columns], boxes of 64 columns x 64 rows
      const uint64_t krows = (uint64_t)q.b_groups * q.k_sub;
      if (!make_map(mb0, q.B0, (uint64_t)q.n_out, krows, (uint64_t)q.n_out * 2, 64u))
        return false;
      if (q.n_sub > 1)
        return make_map(mb1, q.B1, (uint64_t)q.n_out, krows, (uint64_t)q.n_out * 2, 64u);
      *mb1 = *mb0;
      return true;
    }
    if (q.swiglu)
      return make_map(mb0, q.B0, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2, BN / 2) &&
             make_map(mb1, q.B1, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2, BN / 2);
    if (!make_map(mb0, q.B0, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2,
                  pair_tiles ? BN / 2 : (uint32_t)p.mma_n))
      return false;
    *mb1 = *mb0;
    return true;
  };
  CUtensorMap ma, mb0, mb1;
  // CTA pairs; the single-CTA kernel runs if pairs cannot be launched here
  if (q.use_pairs) {
    auto kern2 = q.c_e8 != nullptr ? tc2_gemm_kernel<kEkCompact> : tc2_gemm_kernel<kEkStore>;
    int n_pairs = 0;
    if (cudaFuncSetAttribute(kern2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes2) == cudaSuccess)
      n_pairs = pair_grid(reinterpret_cast<const void*>(kern2), num_sms);
    if (n_pairs >= 1 && maps(true, &ma, &mb0, &mb1)) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(2 * n_pairs);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemBytes2;
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
      if (cudaLaunchKernelEx(&cfg, kern2, ma, mb0, mb1, p) == cudaSuccess) return true;
    }
    cudaGetLastError();   // clear, then run on single CTAs
  }
  if (!maps(false, &ma, &mb0, &mb1)) return false;
  // one n-tile of at most 128 columns (the router GEMM): the narrow ring
  const bool narrow = !q.swiglu && p.mma_n <= 128;
  auto kern = q.c_e8 != nullptr
                  ? (narrow ? tc_gemm_kernel<kEkCompact, true> : tc_gemm_kernel<kEkCompact, false>)
                  : (narrow ? tc_gemm_kernel<kEkStore, true> : tc_gemm_kernel<kEkStore, false>);
  const int smem = narrow ? Ring<true>::kSmem : Ring<false>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return false;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, st, ma, mb0, mb1, p) ==
         cudaSuccess;
}

}  // namespace moe
