// Shared device helpers of the MoE library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Device error word codes (the first int32 of the workspace).  The host maps
// them to MOE_ERR_DEVICE_CHECK / MOE_ERR_TIMEOUT.
enum : int32_t {
  kDevOk = 0,
  kDevBadExpert = 1,   // an expert index outside [0, E)
  kDevTimeout = 2,     // a bounded wait ran out
  kDevBadRow = 3,      // a row index outside the grouped buffer
};

__device__ __forceinline__ void set_device_error(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) {
  return __float2bfloat16_rn(v);
}

// silu(z) = z / (1 + exp(-z)); for z -> -inf, exp overflows to +inf and the
// quotient is -0, the correct limit.
__device__ __forceinline__ float silu_f32(float z) {
  return z / (1.0f + expf(-z));
}
// silu for the tensor-core epilogues, whose results are rounded to bf16: the
// fast exponential and divide intrinsics are a few fp32 ulps off, far below
// that rounding, and take the SwiGLU epilogue off the up projection's
// critical path (0.641 -> 0.610 ms on the Qwen3-style layer).  For z below
// about -88 the divisor overflows to infinity and the result is -0.
__device__ __forceinline__ float silu_fast(float z) {
  return __fdividef(z, 1.0f + __expf(-z));
}

// 16-byte vector of the element type: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  float4 v;
  __device__ __forceinline__ float get(int i) const {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
  }
};
template <> struct Vec16<bf16> {
  static constexpr int N = 8;
  uint4 v;
  __device__ __forceinline__ float get(int i) const {
    uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
    uint32_t bits = (i & 1) ? (w & 0xFFFF0000u) : (w << 16);
    return __uint_as_float(bits);
  }
};

__device__ __forceinline__ uint4 ld_vec16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint4 ld_vec16_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
// 32-byte vectors (256-bit global loads / stores)
struct Vec32 {
  uint32_t v[8];
};
__device__ __forceinline__ void ld_vec32_nc(const void* p, Vec32& r) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]),
                 "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
               : "l"(p));
}
__device__ __forceinline__ void st_vec32(void* p, const Vec32& r) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r.v[0]),
               "r"(r.v[1]), "r"(r.v[2]), "r"(r.v[3]), "r"(r.v[4]), "r"(r.v[5]), "r"(r.v[6]),
               "r"(r.v[7])
               : "memory");
}
__device__ __forceinline__ void st_vec16(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}
// streaming store (evict-first): written once, read by a later kernel
__device__ __forceinline__ void st_vec16_cs(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

// Programmatic dependent launch.  The layer's kernels are launched with
// programmatic stream serialization, so a kernel's CTAs may start while its
// predecessor's last CTAs still run; pdl_wait() (griddepcontrol.wait) blocks
// until the predecessor grid has completed and its memory is visible, and
// every such kernel calls it before reading anything a predecessor wrote.
// pdl_launch_dependents() lets the next kernel's CTAs be scheduled as soon
// as resources free up (their own pdl_wait keeps them correct).  Launched
// without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifndef __CUDACC_RTC__
// kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization (the kernel must call pdl_wait before reading its inputs)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
#endif

}  // namespace moe
