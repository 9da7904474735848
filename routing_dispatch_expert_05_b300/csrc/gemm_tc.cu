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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kTileA = BM * BK * 2;            // 16 KB
constexpr uint32_t kTileB = BN * BK * 2;            // 32 KB
constexpr uint32_t kStageBytes = kTileA + kTileB;   // 48 KB
constexpr uint32_t kTmemCols = 2 * BN;              // two accumulators
constexpr uint64_t kTimeoutNs = 2000000000ull;      // 2 s
constexpr int kBarBytes = 1024;
// per-group tile starts and row offsets, padded so what follows stays
// 128-byte aligned
constexpr int kTableBytes = (2 * (kMaxExperts + 1) * 4 + 127) / 128 * 128;
// Epilogue staging: each epilogue warp turns its 32 rows x 32 columns chunk
// (one row per lane after tcgen05.ld) into row-contiguous global stores.
// Rows are padded (fp32: 36 words, bf16: 20 words) so that both the
// row-per-lane writes and the column-per-lane reads are free of bank
// conflicts (up to a 2-way conflict on a quarter of the bf16 reads).
constexpr int kStgF32Stride = 36;                  // floats per staged row
constexpr int kStgB16Stride = 20;                  // 32-bit words per staged row
constexpr int kStgWarpBytes = 32 * kStgF32Stride * 4;
// Routing epilogue: per-warp selection counters (each epilogue warp owns the
// statistics partial of its 32 tokens, so the warps never wait on each other)
// and the router / selection biases as fp32.
constexpr int kRouteSmemBytes = 4 * kMaxExperts * 4 + 2 * kMaxExperts * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes + kTableBytes +
                           4 * kStgWarpBytes + kRouteSmemBytes + 1024 /* alignment */;
static_assert((kStages * kStageBytes + kBarBytes + kTableBytes) % 16 == 0,
              "epilogue staging must be 16-byte aligned (vector stores)");
static_assert(kStgWarpBytes % 16 == 0 && (kStgF32Stride * 4) % 16 == 0 &&
                  (kStgB16Stride * 4) % 16 == 0,
              "staged rows must keep 16-byte alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

struct Params {
  const int32_t* offsets;     // [G+1] device or null (one group of `rows`)
  int n_groups;
  int rows;
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
  int32_t* err;
  const int32_t* a_row_map;   // null: A rows are the tile rows; else A row r
                              // is row a_row_map[r] of the A tensor
  RouteEpilogue route;        // route.idx != null: the routing epilogue
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `bar` with parity `parity` to complete, giving up
// when another role aborted or after kTimeoutNs (then abort everyone).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        set_device_error(err, kDevTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
        "r"(c0), "r"(c1)
      : "memory");
}
// Four rows r0..r3 (each one box of BK columns starting at column c0) into
// consecutive 128-byte rows of shared memory; the map's box is one row high.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int r0, int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
        "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               ::"r"(taddr), "r"(ncols) : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core-matrix groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                             // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;                   // stride byte offset
  d |= (uint64_t)1 << 46;                             // descriptor version
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b,
                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      ::"r"(smem_u32(bar)) : "memory");
}
#define MOE_TMEM_LD32(taddr, r)                                                     \
  asm volatile(                                                                     \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                     \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"                     \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"    \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),     \
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),   \
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),            \
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),            \
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),            \
        "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
      : "r"(taddr))
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- tiles
struct Tile {
  int g, row0, row_end, n;
};

__device__ __forceinline__ Tile tile_of(int t, const int* tile_start, const int* off,
                                        int G, int nt) {
  int lo = 0, hi = G - 1;  // largest g with tile_start[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  Tile r;
  r.g = lo;
  r.row0 = off[lo] + (local / nt) * BM;
  r.row_end = off[lo + 1];
  r.n = local % nt;
  return r;
}

// ------------------------------------------------------- epilogue helpers
// Writes the warp's staged 32 rows x 32 fp32 columns (row r at
// stg + r * kStgF32Stride) as whole 128-byte row segments: lane = (row
// quarter, 16-byte piece).
__device__ __forceinline__ void store_staged_f32(const float* stg, int lane, int row_base,
                                                 int row_end, int col0, int n_out, float* C) {
  const int c4 = lane & 7;
  const bool col_ok = col0 + c4 * 4 < n_out;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + (lane >> 3);
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

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Compact output of one tile, one pass over the accumulator: for each 32
// columns of a row, the largest |v| picks a power of two 2^s that brings it
// into [2^14, 2^15); v * 2^s (exact) is rounded once to fp16, and the biased
// exponent of 2^-s (one byte, an E8 shared exponent) is stored beside it.
__device__ __forceinline__ void compact_tile(const Params& p, const Tile& tl, int lane,
                                             int row_base, uint32_t tb, uint32_t* stg) {
  const int row = row_base + lane;
  const bf16* bp = p.bias ? p.bias + (int64_t)tl.g * p.bias_stride : nullptr;
  uint32_t e8lo = 0u, e8hi = 0u;                   // this row's 8 exponents of the tile
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    const int c0 = tl.n * BN + ch * 32;
    if (c0 >= p.n_out) break;                      // warp-uniform
    uint32_t r[32];
    MOE_TMEM_LD32(tb + ch * 32, r);
    tmem_ld_wait();
    float v[32];
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = __uint_as_float(r[j]);
      if (bp != nullptr && c0 + j < p.n_out) v[j] += __bfloat162float(bp[c0 + j]);
      mx = fmaxf(mx, fabsf(v[j]));                 // columns past n_out hold 0
    }
    int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
    e = min(max(e, -100), 127);                    // zero / tiny blocks: bounded scale
    const float scale = __uint_as_float((uint32_t)(127 + 14 - e) << 23);   // 2^(14-e)
    const uint32_t e8 = (uint32_t)(e + 113) << (8 * (ch & 3));             // 2^(e-14)
    if (ch < 4) e8lo |= e8; else e8hi |= e8;
    uint4* dst = reinterpret_cast<uint4*>(stg + lane * kStgB16Stride);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[j] = make_uint4(pack_half2(v[8 * j] * scale, v[8 * j + 1] * scale),
                          pack_half2(v[8 * j + 2] * scale, v[8 * j + 3] * scale),
                          pack_half2(v[8 * j + 4] * scale, v[8 * j + 5] * scale),
                          pack_half2(v[8 * j + 6] * scale, v[8 * j + 7] * scale));
    __syncwarp();
    store_staged_b16(stg, lane, row_base, tl.row_end, c0, p.n_out, p.C);
    __syncwarp();
  }
  if (row < tl.row_end) {
    uint8_t* ep = p.c_e8 + (int64_t)row * p.e8_cols + tl.n * (BN / 32);
    const int n8 = min(BN / 32, p.e8_cols - tl.n * (BN / 32));
    if (n8 == 8 && (reinterpret_cast<uintptr_t>(ep) & 7u) == 0) {
      *reinterpret_cast<uint2*>(ep) = make_uint2(e8lo, e8hi);
    } else {
      for (int i = 0; i < n8; ++i) ep[i] = (uint8_t)((i < 4 ? e8lo : e8hi) >> (8 * (i & 3)));
    }
  }
}

// Sum of 32 per-lane vectors, transposed: on return v[0] of lane l is the
// sum over the 32 lanes of their v[l].  A fixed butterfly (31 shuffles), so
// the summation order -- and the result -- is the same on every run.
__device__ __forceinline__ void warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
}

// Insert (key, e, aux) into a list sorted by key descending in which equal
// keys keep arrival order.  Experts arrive in ascending index order, so ties
// go to the lower expert index.  Slots >= k are never filled (idx -1 = empty).
template <int KM>
__device__ __forceinline__ void topk_insert(float (&tk)[KM], int (&ti)[KM], float (&ta)[KM],
                                            int k, float key, int e, float aux) {
  bool shifting = false;   // once placed, every later entry moves down one slot
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    if (i < k && (shifting || ti[i] < 0 || key > tk[i])) {
      const float kk = tk[i], aa = ta[i];
      const int ii = ti[i];
      tk[i] = key; ti[i] = e; ta[i] = aux;
      key = kk; e = ii; aux = aa;
      shifting = true;
      if (e < 0) break;    // filled an empty slot: nothing left to move
    }
  }
}

// sigmoid in double, rounded once to fp32: the selection key's definition
__device__ __forceinline__ float sigmoid_exact(float l) {
  return (float)(1.0 / (1.0 + exp(-(double)l)));
}
// fp32 sigmoid: expf (<= 2 ulp), one add and a correctly rounded divide; its
// distance to sigmoid_exact stays far below kSigmoidSlack
__device__ __forceinline__ float sigmoid_fast(float l) {
  return 1.0f / (1.0f + expf(-l));
}
constexpr float kSigmoidSlack = 1.0f / 65536.0f;   // bound used for candidates

// The routing epilogue of the router GEMM: the accumulator holds the fp32
// logits of 128 tokens x E experts (E <= 256, one n-tile).  Lane = token.
//   pass 1: logits (+ router bias), optional logits store, selection keys,
//           running top-k, softmax max / normaliser (online) or sum of s;
//   pass 2 (sigmoid mode): exact keys for the candidates (see below);
//   pass 3: routing probabilities p[t, e] -> per-expert sums over the
//           warp's 32 tokens (one statistics partial per warp).
// The sigmoid key is sigmoid(l) + b with sigmoid evaluated in double and
// rounded to fp32.  Double is slow here, so pass 1 ranks fp32 keys ka whose
// distance to the exact keys is below delta = kSigmoidSlack; every expert of
// the exact top k then has ka >= (k-th largest ka) - 2 delta, and only those
// candidates get exact keys -- the selection equals the all-double one.
__device__ __forceinline__ void route_tile(const Params& p, const Tile& tl, int q, int lane,
                                           uint32_t tb, float* stg, int* cnt,
                                           const float* s_rb, const float* s_sb) {
  constexpr int KM = kRouteMaxK;
  const RouteEpilogue& R = p.route;
  const int E = p.n_out, k = R.top_k, mode = R.mode;
  const int nch = (E + 31) / 32;
  const int row_base = tl.row0 + q * 32;
  const int row = row_base + lane;
  const bool valid = row < tl.row_end;
  const bool warp_has_rows = row_base < tl.row_end;
  const int part = row_base / kRouteTokensPerPartial;   // this warp's statistics partial

  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();

  float tk[KM], ta[KM];
  int ti[KM];
#pragma unroll
  for (int i = 0; i < KM; ++i) tk[i] = -INFINITY, ta[i] = 0.f, ti[i] = -1;
  float m = -INFINITY, z = 0.f;                     // softmax max and sum exp(l - m)
  float ssum = 0.f;                                 // sigmoid: sum of s (fp32 s)

  // ---- pass 1
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const int col0 = ch * 32;
    uint32_t r[32];
    MOE_TMEM_LD32(tb + col0, r);
    tmem_ld_wait();
    float l[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = col0 + j;
      l[j] = __uint_as_float(r[j]) + s_rb[e];
    }
    if (p.C != nullptr) {
      float4* dst = reinterpret_cast<float4*>(stg + lane * kStgF32Stride);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(l[4 * j], l[4 * j + 1], l[4 * j + 2], l[4 * j + 3]);
      __syncwarp();
      store_staged_f32(stg, lane, row_base, tl.row_end, col0, E, static_cast<float*>(p.C));
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = col0 + j;
      if (e >= E) break;
      if (mode == 2) {
        const float sa = sigmoid_fast(l[j]);
        ssum += sa;
        topk_insert<KM>(tk, ti, ta, k, __fadd_rn(sa, s_sb[e]), e, 0.f);
      } else {
        if (l[j] > m) {
          z = z * expf(m - l[j]) + 1.f;
          m = l[j];
        } else {
          z += expf(l[j] - m);
        }
        topk_insert<KM>(tk, ti, ta, k, l[j], e, 0.f);
      }
    }
  }

  // ---- pass 2 (sigmoid): exact keys of the candidates
  if (mode == 2) {
    float kth = tk[0];                              // the k-th fp32 key (unrolled pick)
#pragma unroll
    for (int i = 1; i < KM; ++i)
      if (i == k - 1) kth = tk[i];
    const float thr = kth - 4.f * kSigmoidSlack;
#pragma unroll
    for (int i = 0; i < KM; ++i) tk[i] = -INFINITY, ta[i] = 0.f, ti[i] = -1;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      const int col0 = ch * 32;
      uint32_t r[32];
      MOE_TMEM_LD32(tb + col0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = col0 + j;
        if (e >= E) break;
        const float l = __uint_as_float(r[j]) + s_rb[e];
        const float b = s_sb[e];
        if (__fadd_rn(sigmoid_fast(l), b) >= thr) {
          const float s = sigmoid_exact(l);
          topk_insert<KM>(tk, ti, ta, k, __fadd_rn(s, b), e, s);
        }
      }
    }
  }

  // ---- selection outputs: idx, weights, counts
  if (valid) {
    float wsum = 0.f, wv[KM];
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      wv[i] = 0.f;
      if (i < k) {
        wv[i] = mode == 2 ? ta[i] : expf(tk[i] - tk[0]);
        wsum += wv[i];
      }
    }
    const int64_t o = (int64_t)row * k;
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      if (i < k) {
        R.idx[o + i] = ti[i];
        R.w[o + i] = wv[i] / wsum;
        atomicAdd(&cnt[ti[i]], 1);
      }
    }
  }

  // ---- pass 3: probabilities, summed per expert over this warp's tokens
  const float inv = mode == 2 ? 1.f / ssum : 1.f / z;
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const int col0 = ch * 32;
    uint32_t r[32];
    MOE_TMEM_LD32(tb + col0, r);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = col0 + j;
      float pv = 0.f;
      if (valid && e < E) {
        const float l = __uint_as_float(r[j]) + s_rb[e];
        pv = (mode == 2 ? sigmoid_fast(l) : expf(l - m)) * inv;
      }
      v[j] = pv;
    }
    warp_transpose_sum32(v, lane);
    if (warp_has_rows && col0 + lane < E)
      R.psum_part[(int64_t)part * E + col0 + lane] = v[0];
  }
  __syncwarp();
  if (warp_has_rows)
    for (int e = lane; e < E; e += 32) R.cnt_part[(int64_t)part * E + e] = cnt[e];
  __syncwarp();
}

// ---------------------------------------------------------------- kernel
// Epilogue kinds, one kernel instantiation each.
enum : int { kEkStore = 0, kEkCompact = 1, kEkRoute = 2 };

template <int EK>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ Params p) {
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
  int* s_rcnt = reinterpret_cast<int*>(s_stage + 4 * kStgWarpBytes);  // [4][kMaxExperts]
  float* s_rb = reinterpret_cast<float*>(s_rcnt + 4 * kMaxExperts);   // router bias [256]
  float* s_sb = s_rb + kMaxExperts;                                    // selection bias

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
      mbar_init(&tempty[s], 4);
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&tmA);
    prefetch_map(&tmB0);
    if (p.swiglu) prefetch_map(&tmB1);
  }
  if (warp == 1) tmem_alloc(s_tmem, kTmemCols);
  if (EK == kEkRoute && warp == 3) {
    for (int e = lane; e < kMaxExperts; e += 32) {
      const bool in = e < p.n_out;
      s_rb[e] = in && p.bias != nullptr ? __bfloat162float(p.bias[e]) : 0.f;
      s_sb[e] = in && p.route.mode == 2 ? p.route.sel_bias[e] : 0.f;
    }
  }
  if (warp == 2) {
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int gg = base + lane;
      int m = 0;
      if (gg < G) {
        const int o0 = p.offsets ? p.offsets[gg] : 0;
        const int o1 = p.offsets ? p.offsets[gg + 1] : p.rows;
        s_off[gg] = o0;
        m = o1 - o0;
      }
      const int tiles = (m + BM - 1) / BM * nt;
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (gg < G) s_tile_start[gg] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_tile_start[G] = carry;
      s_off[G] = p.offsets ? p.offsets[G] : p.rows;
    }
  }
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
            mbar_expect_tx(&full[stage], kStageBytes);
            uint8_t* b = sB + stage * kTileB;
            if (!gather) tma_load_2d(a, &tmA, &full[stage], kb * BK, tl.row0);
            if (p.swiglu) {
              const int brow = tl.g * p.b_rows + tl.n * (BN / 2);
              tma_load_2d(b, &tmB0, &full[stage], kb * BK, brow);
              tma_load_2d(b + kTileB / 2, &tmB1, &full[stage], kb * BK, brow);
            } else {
              const int sub = kb / kb_per_sub;
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
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
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
            umma(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc,
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
    const int q = warp & 3;
    float* stg_f = reinterpret_cast<float*>(s_stage + (warp - 2) * kStgWarpBytes);
    uint32_t* stg_w = reinterpret_cast<uint32_t*>(stg_f);
    const int cols_tile = p.swiglu ? BN / 2 : BN;   // output columns per tile
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = tile_of(t, s_tile_start, s_off, G, nt);
      if (!wait_bounded(&tfull[acc], acc_phase, s_abort, p.err)) break;
      tc_fence_after();
      const int row_base = tl.row0 + q * 32;         // this warp's 32 rows
      const uint32_t tb = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if constexpr (EK == kEkRoute) {
        route_tile(p, tl, q, lane, tb, stg_f, s_rcnt + (warp - 2) * kMaxExperts, s_rb, s_sb);
      } else if constexpr (EK == kEkCompact) {
        compact_tile(p, tl, lane, row_base, tb, stg_w);
      } else {
#pragma unroll 1
      for (int ch = 0; ch < cols_tile / 32; ++ch) {
        const int col0 = tl.n * cols_tile + ch * 32;
        if (col0 >= p.n_out) break;                  // warp-uniform
        float v[32];
        if (p.swiglu) {
          uint32_t g[32], u[32];
          MOE_TMEM_LD32(tb + ch * 32, g);
          MOE_TMEM_LD32(tb + BN / 2 + ch * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = silu_f32(__uint_as_float(g[j])) * __uint_as_float(u[j]);
        } else {
          uint32_t r[32];
          MOE_TMEM_LD32(tb + ch * 32, r);
          tmem_ld_wait();
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
            for (int j = 0; j < 32; ++j) v[j] = silu_f32(v[j]);
          }
        }
        // lane = row: stage the row's 32 values
        if (p.c_is_f32) {
          float4* dst = reinterpret_cast<float4*>(stg_f + lane * kStgF32Stride);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(stg_w + lane * kStgB16Stride);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        }
        __syncwarp();
        // lane = 16-byte column piece: whole row segments per store
        if (p.c_is_f32) {
          store_staged_f32(stg_f, lane, row_base, tl.row_end, col0, p.n_out,
                           static_cast<float*>(p.C));
        } else {
          const int c8 = lane & 3;
          const bool col_ok = col0 + c8 * 8 < p.n_out;
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int r = it * 8 + (lane >> 2);
            const int row = row_base + r;
            if (col_ok && row < tl.row_end) {
              const uint4 val =
                  *reinterpret_cast<const uint4*>(stg_w + r * kStgB16Stride + c8 * 4);
              st_vec16(static_cast<bf16*>(p.C) + (int64_t)row * p.n_out + col0 + c8 * 8,
                       val);
            }
          }
        }
        __syncwarp();
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

// ---------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 2-D bf16 map: `inner` contiguous elements per row, `outer` rows
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_gemm_supported(const TcProblem& q) {
  if (q.K < 1 || q.n_out < 8 || q.n_out % 8 != 0) return false;
  if (q.k_sub % tc::BK != 0 && q.n_sub > 1) return false;
  if (q.n_groups > kMaxExperts) return false;
  // the routing epilogue: one group, all E columns in one accumulator tile
  // compact output: one exponent per 32 columns, no SwiGLU pairing
  if (q.c_e8 != nullptr && (q.swiglu || q.e8_cols != (q.n_out + 31) / 32)) return false;
  if (q.route.idx != nullptr &&
      (q.n_out > tc::BN || q.offsets != nullptr || q.swiglu || q.n_sub != 1 ||
       q.route.top_k < 1 || q.route.top_k > kRouteMaxK || q.route.top_k > q.n_out))
    return false;
  return tc::encode_fn() != nullptr;
}

bool launch_tc_gemm(const TcProblem& q, int num_sms, cudaStream_t st) {
  using namespace tc;
  CUtensorMap ma, mb0, mb1;
  // A [a_rows, K]
  // a gathered A is read one row per box (four boxes per gather4)
  if (!make_map(&ma, q.A, (uint64_t)q.K, (uint64_t)q.a_rows, (uint64_t)q.K * 2,
                q.a_row_map ? 1u : (uint32_t)BM))
    return false;
  const int ksub = q.n_sub > 1 ? q.k_sub : q.K;
  const uint64_t brows_total = (uint64_t)q.b_groups * q.n_sub * q.b_rows;
  if (q.swiglu) {
    if (!make_map(&mb0, q.B0, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2, BN / 2) ||
        !make_map(&mb1, q.B1, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2, BN / 2))
      return false;
  } else {
    if (!make_map(&mb0, q.B0, (uint64_t)ksub, brows_total, (uint64_t)ksub * 2, BN))
      return false;
    mb1 = mb0;
  }
  Params p{};
  p.offsets = q.offsets;
  p.n_groups = q.n_groups;
  p.rows = (int)q.rows;
  p.K = q.K;
  p.n_out = q.n_out;
  p.swiglu = q.swiglu;
  p.epilogue = q.epilogue;
  p.b_rows = q.b_rows;
  p.k_sub = ksub;
  p.n_sub = q.n_sub;
  p.bias = static_cast<const bf16*>(q.bias);
  p.bias_stride = q.bias_stride;
  p.C = q.C;
  p.c_is_f32 = q.c_is_f32;
  p.c_e8 = q.c_e8;
  p.e8_cols = q.e8_cols;
  p.err = q.err;
  p.a_row_map = q.a_row_map;
  p.route = q.route;
  auto kern = q.route.idx != nullptr ? tc_gemm_kernel<kEkRoute>
             : q.c_e8 != nullptr       ? tc_gemm_kernel<kEkCompact>
                                       : tc_gemm_kernel<kEkStore>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return false;
  kern<<<num_sms, kThreads, kSmemBytes, st>>>(ma, mb0, mb1, p);
  return cudaGetLastError() == cudaSuccess;
}

}  // namespace moe
