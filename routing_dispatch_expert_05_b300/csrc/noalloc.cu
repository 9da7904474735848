// moe_dispatch_permute_noalloc: the grouping stage for callers that cannot
// hand the library any scratch memory.
//
// Some callers of this library cannot allocate device memory when they call
// it: a serving engine that reserves all of the GPU's memory up front for its
// own pool, or a latency-critical loop that must not call cudaMalloc (which
// can synchronise the whole device).  The usual moe_dispatch_permute needs a
// workspace for its per-chunk histogram; this variant keeps that histogram in
// a fixed array compiled into the library instead, so the caller supplies
// only the inputs and outputs.
//
// The array (kNoAllocBytes, 512 KB) lives in every GPU that loads the library
// until the process exits, and it bounds the layer size: n_tokens <=
// kNoAllocMaxTokens.  All calls share it, so calls whose GPU work overlaps
// (two streams, or two host threads) race on it and must be ordered.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int64_t kNoAllocMaxTokens = 65536;
// tokens per histogram chunk here: wider than moe_dispatch_permute's, so the
// fixed array stays at 512 KB
constexpr int kNoAllocTokensPerChunk = 256;
constexpr int64_t kNoAllocMaxChunks = kNoAllocMaxTokens / kNoAllocTokensPerChunk;  // 256
// per-chunk counts and per-chunk bases, [chunks][E] int32 each
constexpr size_t kNoAllocBytes = 2 * (size_t)kNoAllocMaxChunks * kMaxExperts * 4;
static_assert(kNoAllocMaxTokens % kNoAllocTokensPerChunk == 0, "whole chunks");

// The scratch.  In host code this name is only a stand-in for the device
// array: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_dispatch_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per
// device, on that device's first call).
moe_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool ok16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok16_or_null(const void* p) { return p == nullptr || ok16(p); }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_permute_noalloc(const moe_config_t* cfg,
                                                     const int32_t* idx, const void* x,
                                                     int32_t* offsets, int32_t* row_of_slot,
                                                     int32_t* token_of_row, void* x_perm,
                                                     moe_stats_t* stats, void* stream) {
  size_t unused = 0;
  const moe_status_t valid = moe_scratch_size(cfg, &unused);   // validates cfg
  if (valid != MOE_OK) return valid;
  const moe_config_t& c = *cfg;
  if (c.n_tokens > kNoAllocMaxTokens) return MOE_ERR_UNSUPPORTED;
  if (!ok16(offsets)) return MOE_ERR_INVALID_ARG;
  if (stats != nullptr && !(ok16_or_null(stats->counts) && ok16_or_null(stats->kept) &&
                            ok16_or_null(stats->dropped) && ok16_or_null(stats->balance)))
    return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) {
    const size_t eb = (size_t)c.n_experts * 4;
    cudaMemsetAsync(offsets, 0, eb + 4, st);
    if (stats != nullptr) {
      if (stats->counts) cudaMemsetAsync(stats->counts, 0, eb, st);
      if (stats->kept) cudaMemsetAsync(stats->kept, 0, eb, st);
      if (stats->dropped) cudaMemsetAsync(stats->dropped, 0, eb, st);
      if (stats->balance) cudaMemsetAsync(stats->balance, 0, 4, st);
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (!ok16(idx) || !ok16(row_of_slot) || !ok16(token_of_row)) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr) || !ok16_or_null(x) || !ok16_or_null(x_perm))
    return MOE_ERR_INVALID_ARG;

  void* scratch = nullptr;
  const moe_status_t s = scratch_address(&scratch);
  if (s != MOE_OK) return s;
  const int chunks = (int)ceil_div64(c.n_tokens, kNoAllocTokensPerChunk);
  int32_t* chunk_cnt = static_cast<int32_t*>(scratch);
  int32_t* chunk_base = chunk_cnt + (size_t)chunks * c.n_experts;
  int64_t capacity = -1;
  if (c.capacity_factor > 0.f)
    capacity = (int64_t)((double)c.capacity_factor * (double)(c.n_tokens / c.n_experts));
  // every scratch entry the kernels read is written earlier in the same call
  // (counts by the histogram, bases by the scan): nothing needs clearing.  An
  // expert index outside [0, E) is dropped; with no workspace there is no
  // device error word to flag it.
  launch_dispatch(idx, c.n_tokens, c.top_k, c.n_experts, capacity, chunk_cnt, chunk_base,
                  offsets, row_of_slot, token_of_row, stats ? stats->counts : nullptr,
                  stats ? stats->kept : nullptr, stats ? stats->dropped : nullptr,
                  /*err=*/nullptr, st, /*slot_of_row=*/nullptr, /*room=*/nullptr, /*pad=*/1,
                  kNoAllocTokensPerChunk);
  if (x_perm != nullptr) {
    // the row copy from the token side, as moe_dispatch_permute makes it:
    // each token row is read once and written to each of its kept rows
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    launch_scatter_rows(x, (int64_t)c.d_model * (c.dtype == MOE_BF16 ? 2 : 4), row_of_slot,
                        c.n_tokens, c.top_k, x_perm, sms, st);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
