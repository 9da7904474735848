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
  pdl_wait();
  pdl_launch_dependents();
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
      // the grouping must start at 0, never decrease and end within the
      // buffer's rows; otherwise flag it and run no tile
      int carry = 0;
      bool bad = false;
      for (int base = 0; base < G; base += 32) {
        const int gg = base + tid;
        int tiles = 0;
        if (gg < G) {
          const int m = p.offsets[gg + 1] - p.offsets[gg];
          bad |= m < 0 || (gg == 0 && p.offsets[0] != 0);
          tiles = m > 0 ? (m + BM - 1) / BM : 0;
        }
        int incl = tiles;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(kFull, incl, off);
          if (tid >= off) incl += v;
        }
        if (gg < G) s_tile_start[gg] = carry + incl - tiles;
        carry += __shfl_sync(kFull, incl, 31);
      }
      bad = __any_sync(kFull, bad) || p.offsets[G] > p.rows;
      if (tid == 0) {
        s_tile_start[G] = bad ? 0 : carry;
        if (bad && blockIdx.x == 0 && blockIdx.y == 0) set_device_error(p.err, kDevBadRow);
      }
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
// fp32 accumulation.  A CTA takes EB experts and 8 * TPW tokens; each lane
// holds its slice of the EB router rows in registers (16-byte pieces
// lane, lane + 32, ...; MAXV of them per pass over d), each warp walks TPW
// tokens reading their x rows from L2, and a warp reduction finishes each
// (token, expert) sum.  With few tokens the weights are read once per CTA
// column and the work spreads over E / EB x N / (8 TPW) CTAs.
template <typename T, int EB, int TPW, int MAXV>
__global__ void __launch_bounds__(256)
router_small_kernel(const T* __restrict__ x, const T* __restrict__ W, const T* __restrict__ b,
                    float* __restrict__ logits, int64_t n_tokens, int n_experts, int d) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int V = 16 / sizeof(T);                  // elements per 16 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * EB;
  const int64_t tw = ((int64_t)blockIdx.y * 8 + warp) * TPW;   // this warp's first token
  const int nv = d / V;
  float acc[EB][TPW];
#pragma unroll
  for (int eb = 0; eb < EB; ++eb)
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) acc[eb][tt] = 0.f;
  for (int c0 = 0; c0 < nv; c0 += 32 * MAXV) {
    uint4 wv[EB][MAXV];
#pragma unroll
    for (int eb = 0; eb < EB; ++eb)
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        const int v = c0 + lane + 32 * i;
        wv[eb][i] = (v < nv && e0 + eb < n_experts)
                        ? __ldg(reinterpret_cast<const uint4*>(W + (int64_t)(e0 + eb) * d) + v)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
      const int64_t t = tw + tt;
      if (t >= n_tokens) break;
      const uint4* xr = reinterpret_cast<const uint4*>(x + t * d);
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        const int v = c0 + lane + 32 * i;
        if (v >= nv) break;
        const uint4 xv = __ldg(xr + v);
        const T* xp = reinterpret_cast<const T*>(&xv);
#pragma unroll
        for (int eb = 0; eb < EB; ++eb) {
          const T* wp = reinterpret_cast<const T*>(&wv[eb][i]);
#pragma unroll
          for (int j = 0; j < V; ++j) acc[eb][tt] = fmaf(to_f32(xp[j]), to_f32(wp[j]), acc[eb][tt]);
        }
      }
    }
  }
#pragma unroll
  for (int eb = 0; eb < EB; ++eb)
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc[eb][tt] += __shfl_xor_sync(kFull, acc[eb][tt], off);
  if (lane == 0) {
#pragma unroll
    for (int eb = 0; eb < EB; ++eb) {
      const int e = e0 + eb;
      if (e >= n_experts) break;
      const float bias = b ? to_f32(b[e]) : 0.f;
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
        if (tw + tt < n_tokens) logits[(tw + tt) * n_experts + e] = acc[eb][tt] + bias;
    }
  }
}

template <typename T, int EB, int TPW, int MAXV>
void launch_router_small_t(const void* x, const void* w, const void* b, float* logits,
                           int64_t n_tokens, int n_experts, int d, cudaStream_t st) {
  const dim3 grid((unsigned)ceil_div64(n_experts, EB), (unsigned)ceil_div64(n_tokens, 8 * TPW));
  launch_pdl(router_small_kernel<T, EB, TPW, MAXV>, grid, dim3(256), 0, st,
             static_cast<const T*>(x), static_cast<const T*>(w), static_cast<const T*>(b), logits,
             n_tokens, n_experts, d);
}

}  // namespace

void launch_router_small(const void* x, const void* w, const void* b, float* logits,
                         int64_t n_tokens, int n_experts, int d, int is_bf16, cudaStream_t st) {
  if (n_tokens <= 0) return;
  // up to 128 tokens: 2 experts x 8 tokens per CTA (more CTAs); beyond, 4 x
  // 64 (fewer re-reads of x)
  const bool few = n_tokens <= 128;
  if (is_bf16) {
    if (few) launch_router_small_t<bf16, 2, 1, 8>(x, w, b, logits, n_tokens, n_experts, d, st);
    else launch_router_small_t<bf16, 4, 8, 4>(x, w, b, logits, n_tokens, n_experts, d, st);
  } else {
    if (few) launch_router_small_t<float, 2, 1, 8>(x, w, b, logits, n_tokens, n_experts, d, st);
    else launch_router_small_t<float, 4, 8, 4>(x, w, b, logits, n_tokens, n_experts, d, st);
  }
}

void launch_simt_gemm(const GemmProblem& p, cudaStream_t st) {
  if (p.is_bf16) launch_typed<bf16>(p, st);
  else launch_typed<float>(p, st);
}

}  // namespace moe
