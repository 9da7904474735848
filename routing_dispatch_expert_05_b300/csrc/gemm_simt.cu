// CUDA-core grouped GEMM with fp32 accumulation: C = epilogue(A B^T).
//
// Used for the fp32 layers (tensor-core TF32 would not meet a 1e-4 relative
// error bound) and for small or unaligned shapes.  Groups are row ranges of A
// given by device offsets (expert e owns rows offsets[e] .. offsets[e+1]-1);
// the grid's x extent is an upper bound on the m-tiles over all groups and
// each CTA maps its tile index to (group, m-tile) from a prefix over the
// groups' tile counts, so no host synchronisation is needed to size it.
// Empty groups own no tile.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;
constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

template <typename T>
__device__ __forceinline__ float ld_elem(const void* base, int64_t i) {
  return to_f32(static_cast<const T*>(base)[i]);
}

template <typename T, int EPI>
__global__ void __launch_bounds__(kThreads) simt_gemm_kernel(GemmProblem p) {
  constexpr int NB = EPI == kEpiSwiglu ? 2 : 1;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[NB][BK][BN + 4];
  __shared__ int s_tile_start[kMaxExperts + 1];

  const int tid = threadIdx.x;
  int g = 0;
  int64_t row0, row_end;
  if (p.offsets == nullptr) {
    row0 = (int64_t)blockIdx.x * BM;
    row_end = p.rows;
    if (row0 >= row_end) return;
  } else {
    const int G = p.n_groups;
    if (tid < 32) {
      int carry = 0;
      for (int base = 0; base < G; base += 32) {
        const int gg = base + tid;
        int tiles = 0;
        if (gg < G) tiles = (p.offsets[gg + 1] - p.offsets[gg] + BM - 1) / BM;
        int incl = tiles;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(kFull, incl, off);
          if (tid >= off) incl += v;
        }
        if (gg < G) s_tile_start[gg] = carry + incl - tiles;
        carry += __shfl_sync(kFull, incl, 31);
      }
      if (tid == 0) s_tile_start[G] = carry;
    }
    __syncthreads();
    const int vt = blockIdx.x;
    if (vt >= s_tile_start[G]) return;
    int lo = 0, hi = G - 1;  // largest g with s_tile_start[g] <= vt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile_start[mid] <= vt) lo = mid; else hi = mid - 1;
    }
    g = lo;
    row0 = p.offsets[g] + (int64_t)(vt - s_tile_start[g]) * BM;
    row_end = p.offsets[g + 1];
  }
  const int col0 = blockIdx.y * BN;
  const int K = p.K, N = p.N;
  const int ksub = p.k_sub;
  const int64_t bgo = (int64_t)g * p.b_group_stride;

  const int tx = tid & 15, ty = tid >> 4;
  float acc[NB][4][4];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[b][i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    // A tile: 64 x 16, thread loads 4 (k fastest)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int li = tid + q * kThreads;
      const int r = li >> 4, kk = li & 15;
      const int64_t gr = row0 + r;
      const int gk = k0 + kk;
      float v = 0.f;
      if (gr < row_end && gk < K) {
        const int64_t src = p.a_row_map ? (int64_t)p.a_row_map[gr] : gr;
        v = ld_elem<T>(p.A, src * K + gk);
      }
      As[kk][r] = v;
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const void* B = b == 0 ? p.B0 : p.B1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int li = tid + q * kThreads;
        const int n = li >> 4, kk = li & 15;
        const int gn = col0 + n, gk = k0 + kk;
        float v = 0.f;
        if (gn < N && gk < K) {
          const int sub = gk / ksub, kin = gk - sub * ksub;
          v = ld_elem<T>(B, bgo + (int64_t)sub * p.sub_stride + (int64_t)gn * ksub + kin);
        }
        Bs[b][kk][n] = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[b][kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[b][i][j] = fmaf(a[i], bv[j], acc[b][i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = col0 + tx * 4 + j;
      if (c >= N) continue;
      float v;
      if (EPI == kEpiSwiglu) {
        v = silu_f32(acc[0][i][j]) * acc[NB - 1][i][j];
      } else {
        v = acc[0][i][j];
        if (p.bias) v += ld_elem<T>(p.bias, (int64_t)g * p.bias_group_stride + c);
        if (EPI == kEpiSiluBias) v = silu_f32(v);
      }
      if (p.c_is_f32)
        static_cast<float*>(p.C)[r * N + c] = v;
      else
        static_cast<T*>(p.C)[r * N + c] = from_f32<T>(v);
    }
  }
}

template <typename T>
void launch_typed(const GemmProblem& p, cudaStream_t st) {
  const int64_t mtiles = p.offsets == nullptr
                             ? ceil_div64(p.rows, BM)
                             : ceil_div64(p.rows, BM) + p.n_groups;
  if (mtiles <= 0 || p.N <= 0) return;
  const dim3 grid((unsigned)mtiles, (unsigned)ceil_div64(p.N, BN));
  switch (p.epilogue) {
    case kEpiNone: simt_gemm_kernel<T, kEpiNone><<<grid, kThreads, 0, st>>>(p); break;
    case kEpiSiluBias: simt_gemm_kernel<T, kEpiSiluBias><<<grid, kThreads, 0, st>>>(p); break;
    default: simt_gemm_kernel<T, kEpiSwiglu><<<grid, kThreads, 0, st>>>(p); break;
  }
}

// Router logits for a few tokens: logits[t, e] = sum_i x[t, i] W[e, i] (+ b[e]),
// fp32 accumulation.  A CTA takes kSmallTok tokens (staged in shared memory);
// its warps walk the experts, lanes splitting d so that each router row is
// read as whole 512-byte warp loads, and a warp reduction finishes each
// (token, expert) sum.  With few tokens the tensor-core router is one tile
// whose k-loop is a serial chain; here all experts proceed at once.
constexpr int kSmallTok = 4;
constexpr int kSmallWarps = 8;
template <typename T>
__global__ void __launch_bounds__(kSmallWarps * 32)
router_small_kernel(const T* __restrict__ x, const T* __restrict__ W, const T* __restrict__ b,
                    float* __restrict__ logits, int64_t n_tokens, int n_experts, int d) {
  extern __shared__ __align__(16) uint8_t sx_raw[];
  T* sx = reinterpret_cast<T*>(sx_raw);              // [kSmallTok][d]
  const int64_t t0 = (int64_t)blockIdx.x * kSmallTok;
  const int nt = (int)min((int64_t)kSmallTok, n_tokens - t0);
  constexpr int V = 16 / sizeof(T);                  // elements per 16 bytes
  const int nv = d / V;
  for (int i = threadIdx.x; i < kSmallTok * nv; i += blockDim.x) {
    const int tt = i / nv, v = i - tt * nv;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (tt < nt) val = reinterpret_cast<const uint4*>(x + (t0 + tt) * d)[v];
    reinterpret_cast<uint4*>(sx + (int64_t)tt * d)[v] = val;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = warp; e < n_experts; e += kSmallWarps) {
    const uint4* wr = reinterpret_cast<const uint4*>(W + (int64_t)e * d);
    float acc[kSmallTok];
#pragma unroll
    for (int tt = 0; tt < kSmallTok; ++tt) acc[tt] = 0.f;
    for (int v = lane; v < nv; v += 32) {
      const uint4 wv = __ldg(wr + v);
      const T* wp = reinterpret_cast<const T*>(&wv);
#pragma unroll
      for (int tt = 0; tt < kSmallTok; ++tt) {
        const uint4 xv = reinterpret_cast<const uint4*>(sx + (int64_t)tt * d)[v];
        const T* xp = reinterpret_cast<const T*>(&xv);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[tt] = fmaf(to_f32(xp[j]), to_f32(wp[j]), acc[tt]);
      }
    }
#pragma unroll
    for (int tt = 0; tt < kSmallTok; ++tt)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc[tt] += __shfl_xor_sync(kFull, acc[tt], off);
    if (lane == 0) {
      const float bias = b ? to_f32(b[e]) : 0.f;
      for (int tt = 0; tt < nt; ++tt) logits[(t0 + tt) * n_experts + e] = acc[tt] + bias;
    }
  }
}

}  // namespace

void launch_router_small(const void* x, const void* w, const void* b, float* logits,
                         int64_t n_tokens, int n_experts, int d, int is_bf16, cudaStream_t st) {
  if (n_tokens <= 0) return;
  const int blocks = (int)ceil_div64(n_tokens, kSmallTok);
  const int threads = kSmallWarps * 32;
  const size_t smem = (size_t)kSmallTok * d * (is_bf16 ? 2 : 4);
  if (is_bf16)
    router_small_kernel<bf16><<<blocks, threads, smem, st>>>(
        static_cast<const bf16*>(x), static_cast<const bf16*>(w), static_cast<const bf16*>(b),
        logits, n_tokens, n_experts, d);
  else
    router_small_kernel<float><<<blocks, threads, smem, st>>>(
        static_cast<const float*>(x), static_cast<const float*>(w),
        static_cast<const float*>(b), logits, n_tokens, n_experts, d);
}

void launch_simt_gemm(const GemmProblem& p, cudaStream_t st) {
  if (p.is_bf16) launch_typed<bf16>(p, st);
  else launch_typed<float>(p, st);
}

}  // namespace moe
