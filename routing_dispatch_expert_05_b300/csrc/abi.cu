// The exported C ABI (include/moe.h): argument checks, workspace layout and
// the order of launches.  No entry point allocates, frees or waits (except
// moe_read_device_error, which waits to read one word back).
#include <cmath>
#include <cstring>
#include <mutex>
#include <algorithm>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

size_t elem_size(const moe_config_t& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  // scratch (shared by all stage calls)
  size_t err, fin_ticket, route_psum, route_cnt, chunk_cnt, chunk_base, logits,
      scratch_end;
  // intermediates of moe_forward
  size_t idx, w, offsets, row_of_slot, token_of_row, slot_of_row, x_perm, h, y, y_e8,
      h_shared,
      shared_out, x_stage, out_stage, total;
  int chunks;
};

// extra_rows: room for groups padded past N*k rows (the backward's grouping);
// backward: without the forward's expert outputs and staging buffers
Layout layout_of(const moe_config_t& c, int64_t extra_rows = 0, bool backward = false) {
  Layout L{};
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const int64_t N = c.n_tokens, E = c.n_experts, k = c.top_k, d = c.d_model,
                F = c.d_ff;
  const size_t es = elem_size(c);
  L.chunks = (int)ceil_div64(N, kDispatchTokensPerChunk);
  L.err = take(kAlign);
  L.fin_ticket = L.err + 64;   // inside the first (zero-filled) block
  // running selection totals (zero between forwards, like the ticket)
  L.route_psum = take((size_t)E * 8);
  L.route_cnt = take((size_t)E * 4);
  L.chunk_cnt = take((size_t)L.chunks * E * 4);
  L.chunk_base = take((size_t)L.chunks * E * 4);
  L.logits = take((size_t)N * E * 4);
  L.scratch_end = o;
  L.idx = take((size_t)N * k * 4);
  L.w = take((size_t)N * k * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.row_of_slot = take((size_t)N * k * 4);
  const int64_t R = N * k + extra_rows;            // grouped rows
  L.token_of_row = take((size_t)R * 4);
  L.slot_of_row = take((size_t)R * 4);
  L.x_perm = take((size_t)R * d * es);
  L.h = take((size_t)R * F * es);
  // expert outputs: fp32, or (bf16 layers on the tensor cores) fp16 with an
  // exponent byte per (row, 32-column block) -- either fits here
  if (backward) {
    L.total = o;
    return L;
  }
  L.y = take((size_t)R * d * 4);
  L.y_e8 = take((size_t)R * ceil_div64(d, kYScaleBlock));
  if (c.n_shared > 0) {
    L.h_shared = take((size_t)N * c.n_shared * c.d_ff_shared * es);
    L.shared_out = take((size_t)N * d * 4);
  }
  L.x_stage = take((size_t)N * d * es);
  L.out_stage = take((size_t)N * d * es);
  L.total = o;
  return L;
}

// The scratch areas of a workspace laid out for config `c`.
struct Scratch {
  int32_t* err;
  RouteTotals totals;  // running selection statistics
  int32_t* chunk_cnt;  // dispatch per-chunk histogram and bases
  int32_t* chunk_base;
  float* logits;
};

Scratch scratch_of(const Layout& L, void* ws) {
  char* b = static_cast<char*>(ws);
  Scratch sc;
  sc.err = reinterpret_cast<int32_t*>(b + L.err);
  sc.totals.ticket = reinterpret_cast<unsigned*>(b + L.fin_ticket);
  sc.totals.psum_fx = reinterpret_cast<unsigned long long*>(b + L.route_psum);
  sc.totals.cnt = reinterpret_cast<unsigned*>(b + L.route_cnt);
  sc.chunk_cnt = reinterpret_cast<int32_t*>(b + L.chunk_cnt);
  sc.chunk_base = reinterpret_cast<int32_t*>(b + L.chunk_base);
  sc.logits = reinterpret_cast<float*>(b + L.logits);
  return sc;
}

moe_status_t check_config(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens < 0 || c->d_model < 1 || c->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->n_experts > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->route < MOE_ROUTE_SOFTMAX_TOPK || c->route > MOE_ROUTE_SIGMOID_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (c->expert != MOE_EXPERT_SILU_MLP && c->expert != MOE_EXPERT_SWIGLU)
    return MOE_ERR_INVALID_ARG;
  if (c->has_bias != 0 && c->has_bias != 1) return MOE_ERR_INVALID_ARG;
  if (c->has_bias && c->expert != MOE_EXPERT_SILU_MLP) return MOE_ERR_INVALID_ARG;
  const int vec = c->dtype == MOE_BF16 ? 8 : 4;  // elements per 16 bytes
  if (c->d_model % vec != 0 || c->d_ff % vec != 0) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && (c->d_ff_shared < 1 || c->d_ff_shared % vec != 0))
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->capacity_factor) || !std::isfinite(c->balance_coef))
    return MOE_ERR_INVALID_ARG;
  // row indices are int32: every assignment must fit
  if ((double)c->n_tokens * (double)c->top_k > 2147483647.0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// all listed pointers non-null and 16-byte aligned
moe_status_t need(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
// listed pointers may be null; non-null ones must be aligned
moe_status_t maybe(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

#define MOE_TRY(expr)                        \
  do {                                       \
    const moe_status_t s_ = (expr);          \
    if (s_ != MOE_OK) return s_;             \
  } while (0)

moe_status_t check_router_weights(const moe_config_t& c, const moe_weights_t* w) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need({w->w_router}));
  MOE_TRY(maybe({w->b_router}));
  if (c.route == MOE_ROUTE_SIGMOID_BIAS) MOE_TRY(need({w->sel_bias}));
  return MOE_OK;
}
moe_status_t check_up_weights(const moe_config_t& c, const moe_weights_t* w) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need({w->w1}));
  if (c.expert == MOE_EXPERT_SWIGLU) MOE_TRY(need({w->w3}));
  if (c.has_bias) MOE_TRY(need({w->b1}));
  return MOE_OK;
}
moe_status_t check_down_weights(const moe_config_t& c, const moe_weights_t* w) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need({w->w2}));
  if (c.has_bias) MOE_TRY(need({w->b2}));
  return MOE_OK;
}
moe_status_t check_shared_weights(const moe_config_t& c, const moe_weights_t* w) {
  if (c.n_shared == 0) return MOE_OK;
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  return need({w->ws1, w->ws3, w->ws2});
}
moe_status_t check_stats(const moe_stats_t* s) {
  if (s == nullptr) return MOE_OK;
  return maybe({s->counts, s->kept, s->dropped, s->balance});
}

moe_status_t check_ws(void* ws, size_t ws_bytes, size_t needed) {
  if (ws == nullptr || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < needed) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t last_cuda() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return n > 0 ? n : 148;
}

template <typename T> T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int32_t* err_word(void* ws) { return static_cast<int32_t*>(ws); }

int64_t capacity_of(const moe_config_t& c) {
  if (!(c.capacity_factor > 0.f)) return -1;
  const int64_t base = c.n_tokens / c.n_experts;
  return (int64_t)((double)c.capacity_factor * (double)base);
}

// zero the requested per-expert stats (used when there are no tokens)
moe_status_t zero_stats(const moe_config_t& c, moe_stats_t* s, cudaStream_t st) {
  if (s == nullptr) return MOE_OK;
  const size_t eb = (size_t)c.n_experts * 4;
  if (s->counts) cudaMemsetAsync(s->counts, 0, eb, st);
  if (s->kept) cudaMemsetAsync(s->kept, 0, eb, st);
  if (s->dropped) cudaMemsetAsync(s->dropped, 0, eb, st);
  if (s->balance) cudaMemsetAsync(s->balance, 0, 4, st);
  return last_cuda();
}

// ---- stage bodies (arguments already checked) -----------------------------
// The router and the selection of c.n_tokens tokens.  Their statistics join
// the running totals of the scratch; with `finalize` the totals (over
// n_total tokens, all launches since the last finalize) become the counts
// and the balance statistic in stats, and are cleared.
void router_body(const moe_config_t& c, const void* x, const moe_weights_t& w,
                 float* logits, int32_t* idx, float* wts, moe_stats_t* stats,
                 const Scratch& sc, cudaStream_t st, bool gemm, bool finalize = true,
                 int64_t n_total = -1) {
  float* lg = logits ? logits : sc.logits;
  if (gemm && c.n_tokens < kRouterSmallTokens) {
    // a few tokens: every expert's dot product at once on the CUDA cores
    launch_router_small(x, w.w_router, w.b_router, lg, c.n_tokens, c.n_experts, c.d_model,
                        c.dtype == MOE_BF16, st);
    gemm = false;
  }
  if (gemm && c.dtype == MOE_BF16) {
    // bf16 router: one dense tcgen05 GEMM (N = E columns) writing fp32
    // logits; the selection kernel reads them.  (Selecting inside the GEMM's
    // epilogue, one thread per token, measured 1.8x slower: the serial
    // insertion chains of four warps per SM cannot hide their latency.)
    TcProblem q{};
    q.A = x;
    q.a_rows = c.n_tokens;
    q.K = c.d_model;
    q.B0 = w.w_router;
    q.b_groups = 1;
    q.b_rows = c.n_experts;
    q.k_sub = c.d_model;
    q.n_sub = 1;
    q.n_groups = 1;
    q.rows = c.n_tokens;
    q.n_out = c.n_experts;
    q.epilogue = kEpiNone;
    q.bias = w.b_router;
    q.bias_stride = 0;
    q.C = lg;
    q.c_is_f32 = 1;
    q.err = sc.err;
    if (tc_gemm_supported(q) && launch_tc_gemm(q, num_sms(), st)) gemm = false;
  }
  if (gemm) {
    GemmProblem p{};
    p.A = x;
    p.B0 = w.w_router;
    p.k_sub = c.d_model;
    p.bias = w.b_router;
    p.bias_group_stride = 0;
    p.C = lg;
    p.c_is_f32 = 1;
    p.offsets = nullptr;
    p.n_groups = 1;
    p.rows = c.n_tokens;
    p.N = c.n_experts;
    p.K = c.d_model;
    p.epilogue = kEpiNone;
    p.is_bf16 = c.dtype == MOE_BF16;
    launch_simt_gemm(p, st);
  }
  RouteFinal fin{};
  fin.finalize = finalize;
  fin.n_total = n_total < 0 ? c.n_tokens : n_total;
  fin.coef = c.balance_coef;
  fin.counts = stats ? stats->counts : nullptr;
  fin.balance = stats ? stats->balance : nullptr;
  launch_route_from_logits(lg, c.n_tokens, c.n_experts, c.top_k, c.route, w.sel_bias, idx,
                           wts, sc.totals, fin, st);
}

void dispatch_body(const moe_config_t& c, const int32_t* idx, const void* x,
                   int32_t* offsets, int32_t* ros, int32_t* tor, void* x_perm,
                   moe_stats_t* stats, const Scratch& sc, cudaStream_t st,
                   int32_t* slot_of_row = nullptr, const int32_t* room = nullptr,
                   int pad = 1, int32_t* kept = nullptr) {
  launch_dispatch(idx, c.n_tokens, c.top_k, c.n_experts, capacity_of(c), sc.chunk_cnt,
                  sc.chunk_base, offsets, ros, tor, stats ? stats->counts : nullptr,
                  kept != nullptr ? kept : (stats ? stats->kept : nullptr),
                  stats ? stats->dropped : nullptr, sc.err, st, slot_of_row, room, pad);
  if (x_perm != nullptr)
    launch_scatter_rows(x, (int64_t)c.d_model * elem_size(c), ros, c.n_tokens, c.top_k,
                        x_perm, num_sms(), st);
}

// CTA pairs (256-row tiles) pay off when experts hold enough rows; with a
// few rows per expert most of a 256-row tile would be padding
bool pairs_pay(const moe_config_t& c) {
  return (double)c.n_tokens * c.top_k / c.n_experts >= 128.0;
}

// Experts of a few rows each (a decode-shaped layer): the swapped-operand
// kernel, whose tiles are 128 weight rows by the expert's token rows rounded
// up to 16, instead of 128- or 256-row token tiles that would be almost all
// padding.
bool swap_pays(const moe_config_t& c) {
  return (double)c.n_tokens * c.top_k / c.n_experts <= 16.0;
}

// bf16 expert GEMMs run on the tensor cores; fp32 ones on the CUDA cores
moe_status_t run_gemm(const moe_config_t& c, const TcProblem& tq, const GemmProblem& sq,
                      cudaStream_t st) {
  if (c.dtype == MOE_BF16 && tc_gemm_supported(tq))
    return launch_tc_gemm(tq, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
  GemmProblem p = sq;
  p.err = tq.err;
  launch_simt_gemm(p, st);
  return MOE_OK;
}

// The up projection reads its rows either from the expert-sorted buffer
// (row_map == null, a = x_perm) or straight from the token rows
// (a = x, row r reads token row_map[r]).
moe_status_t up_body(const moe_config_t& c, const void* a, const int32_t* row_map,
                     const int32_t* offsets, const moe_weights_t& w, void* h,
                     int32_t* err, cudaStream_t st) {
  const bool swiglu = c.expert == MOE_EXPERT_SWIGLU;
  const int64_t a_rows = row_map ? c.n_tokens : c.n_tokens * c.top_k;
  GemmProblem p{};
  p.A = a;
  p.a_row_map = row_map;
  p.B0 = w.w1;
  p.B1 = swiglu ? w.w3 : nullptr;
  p.b_group_stride = (int64_t)c.d_ff * c.d_model;
  p.k_sub = c.d_model;
  p.bias = c.has_bias ? w.b1 : nullptr;
  p.bias_group_stride = c.d_ff;
  p.C = h;
  p.offsets = offsets;
  p.n_groups = c.n_experts;
  p.rows = c.n_tokens * c.top_k;
  p.N = c.d_ff;
  p.K = c.d_model;
  p.epilogue = swiglu ? kEpiSwiglu : kEpiSiluBias;
  p.is_bf16 = c.dtype == MOE_BF16;
  TcProblem q{};
  q.A = a;
  q.a_rows = a_rows;
  q.a_row_map = row_map;
  q.K = c.d_model;
  q.B0 = w.w1;
  q.B1 = p.B1;
  q.b_groups = c.n_experts;
  q.b_rows = c.d_ff;
  q.k_sub = c.d_model;
  q.n_sub = 1;
  q.offsets = offsets;
  q.n_groups = c.n_experts;
  q.rows = c.n_tokens * c.top_k;
  q.n_out = c.d_ff;
  q.swiglu = swiglu;
  q.epilogue = p.epilogue;
  q.bias = p.bias;
  q.bias_stride = c.d_ff;
  q.C = h;
  q.err = err;
  q.use_pairs = pairs_pay(c);
  if (c.dtype == MOE_BF16 && row_map == nullptr && swap_pays(c) && swap_gemm_supported(q))
    return launch_swap_gemm(q, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
  return run_gemm(c, q, p, st);
}

// y_e8 != null asks for the compact expert outputs (fp16 + exponents); it
// returns MOE_ERR_UNSUPPORTED (nothing launched) where only fp32 y is made.
// With slot_of_row and wts (compact output only) row r is written, scaled by
// its routing weight, to row slot_of_row[r] = t*k + j: the weighted expert
// outputs in slot order, for launch_combine_slots.
moe_status_t down_body(const moe_config_t& c, const void* h, const int32_t* offsets,
                       const moe_weights_t& w, void* y, uint8_t* y_e8, int32_t* err,
                       cudaStream_t st, const int32_t* slot_of_row = nullptr,
                       const float* wts = nullptr, int64_t rows = -1) {
  if (rows < 0) rows = c.n_tokens * c.top_k;
  GemmProblem p{};
  p.A = h;
  p.B0 = w.w2;
  p.b_group_stride = (int64_t)c.d_model * c.d_ff;
  p.k_sub = c.d_ff;
  p.bias = c.has_bias ? w.b2 : nullptr;
  p.bias_group_stride = c.d_model;
  p.C = y;
  p.c_is_f32 = 1;
  p.offsets = offsets;
  p.n_groups = c.n_experts;
  p.rows = rows;
  p.N = c.d_model;
  p.K = c.d_ff;
  p.epilogue = kEpiNone;
  p.is_bf16 = c.dtype == MOE_BF16;
  TcProblem q{};
  q.A = h;
  q.a_rows = rows;
  q.K = c.d_ff;
  q.B0 = w.w2;
  q.b_groups = c.n_experts;
  q.b_rows = c.d_model;
  q.k_sub = c.d_ff;
  q.n_sub = 1;
  q.offsets = offsets;
  q.n_groups = c.n_experts;
  q.rows = q.a_rows;
  q.n_out = c.d_model;
  q.epilogue = kEpiNone;
  q.bias = p.bias;
  q.bias_stride = c.d_model;
  q.C = y;
  q.c_is_f32 = 1;
  q.err = err;
  q.use_pairs = pairs_pay(c);
  if (y_e8 != nullptr) {
    q.c_is_f32 = 0;
    q.c_e8 = y_e8;
    q.e8_cols = (int)ceil_div64(c.d_model, kYScaleBlock);
    q.c_row_map = slot_of_row;
    q.c_row_scale = wts;
    if (c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (swap_pays(c) && swap_gemm_supported(q))
      return launch_swap_gemm(q, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
    if (!tc_gemm_supported(q)) return MOE_ERR_UNSUPPORTED;
    return launch_tc_gemm(q, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
  }
  return run_gemm(c, q, p, st);
}

moe_status_t shared_body(const moe_config_t& c, const void* x, const moe_weights_t& w,
                         void* h_shared, float* shared_out, int32_t* err,
                         cudaStream_t st) {
  const int fs_total = c.n_shared * c.d_ff_shared;
  GemmProblem up{};
  up.A = x;
  up.B0 = w.ws1;  // [S, Fs, d] read as [S*Fs, d]
  up.B1 = w.ws3;
  up.k_sub = c.d_model;
  up.C = h_shared;
  up.n_groups = 1;
  up.rows = c.n_tokens;
  up.N = fs_total;
  up.K = c.d_model;
  up.epilogue = kEpiSwiglu;
  up.is_bf16 = c.dtype == MOE_BF16;
  TcProblem uq{};
  uq.A = x;
  uq.a_rows = c.n_tokens;
  uq.K = c.d_model;
  uq.B0 = w.ws1;
  uq.B1 = w.ws3;
  uq.b_groups = 1;
  uq.b_rows = fs_total;
  uq.k_sub = c.d_model;
  uq.n_sub = 1;
  uq.n_groups = 1;
  uq.rows = c.n_tokens;
  uq.n_out = fs_total;
  uq.swiglu = 1;
  uq.epilogue = kEpiSwiglu;
  uq.C = h_shared;
  uq.err = err;
  uq.use_pairs = c.n_tokens >= 128;
  MOE_TRY(run_gemm(c, uq, up, st));
  GemmProblem dn{};
  dn.A = h_shared;
  dn.B0 = w.ws2;  // [S, d, Fs]: column block s of the concatenated down
  dn.k_sub = c.d_ff_shared;
  dn.sub_stride = (int64_t)c.d_model * c.d_ff_shared;
  dn.C = shared_out;
  dn.c_is_f32 = 1;
  dn.n_groups = 1;
  dn.rows = c.n_tokens;
  dn.N = c.d_model;
  dn.K = fs_total;
  dn.epilogue = kEpiNone;
  dn.is_bf16 = c.dtype == MOE_BF16;
  TcProblem dq{};
  dq.A = h_shared;
  dq.a_rows = c.n_tokens;
  dq.K = fs_total;
  dq.B0 = w.ws2;  // viewed as [S*d, Fs]
  dq.b_groups = 1;
  dq.b_rows = c.d_model;
  dq.k_sub = c.d_ff_shared;
  dq.n_sub = c.n_shared;
  dq.n_groups = 1;
  dq.rows = c.n_tokens;
  dq.n_out = c.d_model;
  dq.epilogue = kEpiNone;
  dq.C = shared_out;
  dq.c_is_f32 = 1;
  dq.err = err;
  dq.use_pairs = c.n_tokens >= 128;
  return run_gemm(c, dq, dn, st);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_scratch_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(*cfg).scratch_end;
  return MOE_OK;
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x,
                             const moe_weights_t* weights, float* logits,
                             int32_t* idx, float* w, moe_stats_t* stats, void* ws,
                             size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_router_weights(c, weights));
  MOE_TRY(check_stats(stats));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) return zero_stats(c, stats, st);
  MOE_TRY(need({x, idx, w}));
  MOE_TRY(maybe({logits}));
  router_body(c, x, *weights, logits, idx, w, stats, scratch_of(layout_of(c), ws), st, true);
  return last_cuda();
}

moe_status_t moe_route_logits(const moe_config_t* cfg, const float* logits,
                              const float* sel_bias, int32_t* idx, float* w,
                              moe_stats_t* stats, void* ws, size_t ws_bytes,
                              void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (c.route == MOE_ROUTE_SIGMOID_BIAS) MOE_TRY(need({sel_bias}));
  MOE_TRY(check_stats(stats));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) return zero_stats(c, stats, st);
  MOE_TRY(need({logits, idx, w}));
  moe_weights_t wt{};
  wt.sel_bias = sel_bias;
  router_body(c, nullptr, wt, const_cast<float*>(logits), idx, w, stats,
              scratch_of(layout_of(c), ws), st, false);
  return last_cuda();
}

moe_status_t moe_dispatch_permute(const moe_config_t* cfg, const int32_t* idx,
                                  const void* x, int32_t* offsets,
                                  int32_t* row_of_slot, int32_t* token_of_row,
                                  void* x_perm, moe_stats_t* stats, void* ws,
                                  size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_stats(stats));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  MOE_TRY(need({offsets}));
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) {
    cudaMemsetAsync(offsets, 0, (size_t)(c.n_experts + 1) * 4, st);
    MOE_TRY(last_cuda());
    return zero_stats(c, stats, st);
  }
  MOE_TRY(need({idx, row_of_slot, token_of_row}));
  // x and x_perm: both present (rows are gathered) or both NULL (no gather)
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(maybe({x, x_perm}));
  dispatch_body(c, idx, x, offsets, row_of_slot, token_of_row, x_perm, stats,
                scratch_of(layout_of(c), ws), st);
  return last_cuda();
}

moe_status_t moe_dispatch_permute_room(const moe_config_t* cfg, const int32_t* idx,
                                       const void* x, const int32_t* room,
                                       int32_t* offsets, int32_t* row_of_slot,
                                       int32_t* token_of_row, void* x_perm,
                                       moe_stats_t* stats, void* ws, size_t ws_bytes,
                                       void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_stats(stats));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  MOE_TRY(need({offsets, room}));
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) {
    cudaMemsetAsync(offsets, 0, (size_t)(c.n_experts + 1) * 4, st);
    MOE_TRY(last_cuda());
    return zero_stats(c, stats, st);
  }
  MOE_TRY(need({idx, row_of_slot, token_of_row}));
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(maybe({x, x_perm}));
  dispatch_body(c, idx, x, offsets, row_of_slot, token_of_row, x_perm, stats,
                scratch_of(layout_of(c), ws), st, nullptr, room);
  return last_cuda();
}

moe_status_t moe_expert_up(const moe_config_t* cfg, const void* x_perm,
                           const int32_t* offsets, const moe_weights_t* weights,
                           void* h, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_up_weights(c, weights));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({x_perm, offsets, h}));
  MOE_TRY(up_body(c, x_perm, nullptr, offsets, *weights, h, err_word(ws),
                  static_cast<cudaStream_t>(stream)));
  return last_cuda();
}

moe_status_t moe_expert_up_gather(const moe_config_t* cfg, const void* x,
                                  const int32_t* token_of_row, const int32_t* offsets,
                                  const moe_weights_t* weights, void* h, void* ws,
                                  size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_up_weights(c, weights));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({x, token_of_row, offsets, h}));
  MOE_TRY(up_body(c, x, token_of_row, offsets, *weights, h, err_word(ws),
                  static_cast<cudaStream_t>(stream)));
  return last_cuda();
}

moe_status_t moe_expert_down(const moe_config_t* cfg, const void* h,
                             const int32_t* offsets, const moe_weights_t* weights,
                             float* y, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_down_weights(c, weights));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({h, offsets, y}));
  MOE_TRY(down_body(c, h, offsets, *weights, y, nullptr, err_word(ws),
                    static_cast<cudaStream_t>(stream)));
  return last_cuda();
}

moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm,
                             const int32_t* offsets, const moe_weights_t* weights,
                             void* h, float* y, void* ws, size_t ws_bytes,
                             void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_up_weights(c, weights));
  MOE_TRY(check_down_weights(c, weights));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({x_perm, offsets, h, y}));
  auto st = static_cast<cudaStream_t>(stream);
  MOE_TRY(up_body(c, x_perm, nullptr, offsets, *weights, h, err_word(ws), st));
  MOE_TRY(down_body(c, h, offsets, *weights, y, nullptr, err_word(ws), st));
  return last_cuda();
}

moe_status_t moe_shared_ffn(const moe_config_t* cfg, const void* x,
                            const moe_weights_t* weights, void* h_shared,
                            float* shared_out, void* ws, size_t ws_bytes,
                            void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (c.n_shared == 0) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_shared_weights(c, weights));
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({x, h_shared, shared_out}));
  MOE_TRY(shared_body(c, x, *weights, h_shared, shared_out, err_word(ws),
                      static_cast<cudaStream_t>(stream)));
  return last_cuda();
}

moe_status_t moe_combine(const moe_config_t* cfg, const float* y,
                         const int32_t* row_of_slot, const float* w,
                         const float* shared_out, void* out, void* ws,
                         size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({y, row_of_slot, w, out}));
  MOE_TRY(maybe({shared_out}));
  launch_combine(y, row_of_slot, w, shared_out, out, c.n_tokens, c.top_k, c.d_model,
                 c.dtype == MOE_BF16, num_sms(), static_cast<cudaStream_t>(stream));
  return last_cuda();
}

}  // extern "C"

namespace {
// The whole layer; ev (if not null) receives kForwardEvents events: the
// start, then one after each stage (router, dispatch, up, down, shared,
// combine -- "shared" coincides with "down" when there is none).
// The whole layer for the n_tokens of `c`, on stream st, with buffers from
// the workspace layout L (laid out for at least c.n_tokens tokens) and its
// scratch sc.  The selection statistics join the scratch's running totals;
// with `finalize` they become (over n_total tokens) the counts and balance
// statistic in stats (else only kept/dropped are set).
// ev (if not null) receives MOE_FORWARD_EVENTS events around the stages.
moe_status_t forward_core(const moe_config_t& c, const Layout& L, const Scratch& sc,
                          bool finalize, int64_t n_total, const void* x,
                          const moe_weights_t& w, void* out, moe_stats_t* stats, void* ws,
                          cudaStream_t st, cudaEvent_t const* ev) {
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* wts = at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* ros = at<int32_t>(ws, L.row_of_slot);
  int32_t* tor = at<int32_t>(ws, L.token_of_row);
  void* x_perm = at<char>(ws, L.x_perm);
  void* h = at<char>(ws, L.h);
  float* y = at<float>(ws, L.y);
  float* shared_out = c.n_shared > 0 ? at<float>(ws, L.shared_out) : nullptr;
  // the balance statistic and pre-drop counts come from the router, the
  // kept/dropped counts from the dispatch
  moe_stats_t rs{};
  if (stats) {
    rs.counts = stats->counts;
    rs.balance = stats->balance;
  }
  auto mark = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], st);
  };
  mark(0);
  router_body(c, x, w, nullptr, idx, wts, &rs, sc, st, true, finalize, n_total);
  mark(1);
  moe_stats_t ds{};
  if (stats) {
    ds.kept = stats->kept;
    ds.dropped = stats->dropped;
  }
  // the expert-sorted copy of the token rows is written once and read by
  // the up projection as whole 128-row TMA boxes.  Gathering the rows inside
  // the GEMM instead (moe_expert_up_gather: tile::gather4, one 128-byte row
  // piece per row and k-block) saves that memory but measured 3.3x slower
  // on the Qwen3-style layer.
  int32_t* sor = at<int32_t>(ws, L.slot_of_row);
  dispatch_body(c, idx, x, offsets, ros, tor, x_perm, &ds, sc, st, sor);
  mark(2);
  MOE_TRY(up_body(c, x_perm, nullptr, offsets, w, h, sc.err, st));
  mark(3);
  // bf16 layers keep the expert outputs compact (half the bytes of fp32)
  uint8_t* y_e8 = at<uint8_t>(ws, L.y_e8);
  // (weighted and in slot order, so that the combine streams a token's rows)
  moe_status_t ds_ = c.dtype == MOE_BF16
                         ? down_body(c, h, offsets, w, y, y_e8, sc.err, st, sor, wts)
                         : MOE_ERR_UNSUPPORTED;
  const bool compact = ds_ == MOE_OK;
  if (ds_ == MOE_ERR_UNSUPPORTED) ds_ = down_body(c, h, offsets, w, y, nullptr, sc.err, st);
  MOE_TRY(ds_);
  mark(4);
  if (c.n_shared > 0)
    MOE_TRY(shared_body(c, x, w, at<char>(ws, L.h_shared), shared_out, sc.err, st));
  mark(5);
  // without a capacity nothing is dropped: the combine need not read row_of_slot
  if (compact)
    launch_combine_slots(y, y_e8, capacity_of(c) < 0 ? nullptr : ros, shared_out, out,
                         c.n_tokens, c.top_k, c.d_model, c.dtype == MOE_BF16, num_sms(), st,
                         sc.err);
  else
    launch_combine(y, ros, wts, shared_out, out, c.n_tokens, c.top_k, c.d_model,
                   c.dtype == MOE_BF16, num_sms(), st);
  mark(6);
  return last_cuda();
}

moe_status_t check_forward_args(const moe_config_t* cfg, const moe_weights_t* weights,
                                moe_stats_t* stats, void* ws, size_t ws_bytes) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_router_weights(c, weights));
  MOE_TRY(check_up_weights(c, weights));
  MOE_TRY(check_down_weights(c, weights));
  MOE_TRY(check_shared_weights(c, weights));
  MOE_TRY(check_stats(stats));
  return check_ws(ws, ws_bytes, layout_of(c).total);
}

moe_status_t forward_impl(const moe_config_t* cfg, const void* x,
                          const moe_weights_t* weights, void* out, moe_stats_t* stats,
                          void* ws, size_t ws_bytes, void* stream, cudaEvent_t const* ev) {
  MOE_TRY(check_forward_args(cfg, weights, stats, ws, ws_bytes));
  const moe_config_t& c = *cfg;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.n_tokens == 0) return zero_stats(c, stats, st);
  MOE_TRY(need({x, out}));
  const Layout L = layout_of(c);
  return forward_core(c, L, scratch_of(L, ws), true, c.n_tokens, x, *weights, out, stats, ws,
                      st, ev);
}

// ---- the host-buffer forward, pipelined over token chunks ------------------
// Without a capacity limit every token's output depends on that token alone,
// so moe_forward_host can split the tokens into chunks and overlap the copy
// of chunk i+1 to the device and of chunk i-1 back with the compute of chunk
// i.  The copies run on two streams of the library's own (created once per
// device); the compute runs on the caller's stream, in chunk order, and the
// statistics are reduced once over all chunks' partials -- the same results,
// bit for bit, as one moe_forward over all tokens.
constexpr int kHostChunks = 4;
constexpr int64_t kHostChunkMin = 4096;     // smaller chunks re-stream the weights too often
constexpr int kMaxDevices = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in[kHostChunks] = {}, done[kHostChunks] = {}, out_done = nullptr;
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

// the current device's pipeline objects, created on its first use (lock held)
HostPipe* host_pipe() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  HostPipe& hp = g_pipe[dev];
  if (hp.ready) return &hp;
  bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.out_done, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kHostChunks; ++i)
    ok = cudaEventCreateWithFlags(&hp.in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return nullptr;
  }
  hp.ready = true;
  return &hp;
}

moe_status_t forward_host_pipelined(const moe_config_t& c, const char* xh,
                                    const moe_weights_t& w, char* oh, moe_stats_t* stats,
                                    void* ws, cudaStream_t st, HostPipe& hp) {
  const Layout L = layout_of(c);
  const Scratch sc = scratch_of(L, ws);
  const size_t row = (size_t)c.d_model * elem_size(c);
  char* xd = at<char>(ws, L.x_stage);
  char* od = at<char>(ws, L.out_stage);
  const int nch = (int)std::min<int64_t>(kHostChunks, c.n_tokens / kHostChunkMin);
  // Chunk sizes in the proportions kChunkShare[nch]: the first chunk's copy
  // in (the fill) and the last chunk's compute and copy out (the drain)
  // overlap nothing, so with three or four chunks those two are smaller.
  // Chunks start on selection-CTA boundaries (the same per-CTA sums as one
  // launch over all tokens).
  static constexpr int kChunkShare[kHostChunks + 1][kHostChunks] = {
      {0, 0, 0, 0}, {1, 0, 0, 0}, {1, 1, 0, 0}, {3, 5, 3, 0}, {3, 5, 5, 3}};
  int64_t bound[kHostChunks + 1] = {};
  {
    int total = 0, acc = 0;
    for (int i = 0; i < nch; ++i) total += kChunkShare[nch][i];
    for (int i = 1; i < nch; ++i) {
      acc += kChunkShare[nch][i - 1];
      const int64_t b = c.n_tokens * acc / total;
      bound[i] = b / kRouteTokensPerCta * kRouteTokensPerCta;
    }
    bound[nch] = c.n_tokens;
  }
  const int nrun = nch;
  bool ok = cudaEventRecord(hp.start, st) == cudaSuccess &&
            cudaStreamWaitEvent(hp.h2d, hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.d2h, hp.start, 0) == cudaSuccess;
  // the last chunk's selection turns the running totals of all chunks into
  // the counts and the balance statistic; no capacity, so every selection
  // is kept
  moe_stats_t none{}, last{};
  if (stats != nullptr) {
    last.counts = stats->counts ? stats->counts : stats->kept;
    last.balance = stats->balance;
  }
  moe_status_t status = MOE_OK;
  for (int i = 0; ok && status == MOE_OK && i < nrun; ++i) {
    const int64_t s0 = bound[i];
    const int64_t n = bound[i + 1] - s0;
    ok = cudaMemcpyAsync(xd + s0 * row, xh + s0 * row, n * row, cudaMemcpyHostToDevice,
                         hp.h2d) == cudaSuccess &&
         cudaEventRecord(hp.in[i], hp.h2d) == cudaSuccess &&
         cudaStreamWaitEvent(st, hp.in[i], 0) == cudaSuccess;
    if (!ok) break;
    moe_config_t ci = c;
    ci.n_tokens = n;
    const bool fin = i == nrun - 1;
    status = forward_core(ci, L, sc, fin, c.n_tokens, xd + s0 * row, w, od + s0 * row,
                          fin ? &last : &none, ws, st, nullptr);
    if (status != MOE_OK) break;
    ok = cudaEventRecord(hp.done[i], st) == cudaSuccess &&
         cudaStreamWaitEvent(hp.d2h, hp.done[i], 0) == cudaSuccess &&
         cudaMemcpyAsync(oh + s0 * row, od + s0 * row, n * row, cudaMemcpyDeviceToHost,
                         hp.d2h) == cudaSuccess;
  }
  if (ok && status == MOE_OK && stats != nullptr) {
    int32_t* counts = last.counts;
    const size_t eb = (size_t)c.n_experts * 4;
    if (stats->kept && counts != stats->kept)
      ok = cudaMemcpyAsync(stats->kept, counts, eb, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
    if (ok && stats->dropped) ok = cudaMemsetAsync(stats->dropped, 0, eb, st) == cudaSuccess;
  }
  // The caller's stream completes with the last copy back, and with every
  // other copy the call enqueued even when an enqueue above failed, so the
  // caller's buffers outlive the copies whatever the call returns.
  const bool joined = cudaEventRecord(hp.out_done, hp.d2h) == cudaSuccess &&
                      cudaStreamWaitEvent(st, hp.out_done, 0) == cudaSuccess &&
                      cudaEventRecord(hp.start, hp.h2d) == cudaSuccess &&
                      cudaStreamWaitEvent(st, hp.start, 0) == cudaSuccess;
  if (status != MOE_OK) return status;
  return ok && joined ? last_cuda() : MOE_ERR_CUDA;
}

// ---- backward -------------------------------------------------------------
// Buffers of moe_backward after the forward's own layout (which holds the
// recomputed routing, grouping, x_perm, h and compact y).
// The backward's grouping pads every expert's rows to whole 16-row slices
// (zero rows), so the weight-gradient MMAs can stop at a group's end.
constexpr int kBwPad = 16;

// The router's weight-gradient problem: dWr [E, d] = dlogits^T x over all
// tokens, one group, K split over CTA pairs (partials in the workspace).
WgradProblem router_wgrad_problem(const moe_config_t& c, const void* dz16, const void* x,
                                  float* d_wr, float* partial, int32_t* err) {
  WgradProblem q{};
  q.P = dz16;
  q.p_ld = c.n_experts;
  q.m_dim = c.n_experts;
  q.Q = x;
  q.q_ld = c.d_model;
  q.n_dim = c.d_model;
  q.rows = c.n_tokens;
  q.n_groups = 1;
  q.C0 = d_wr;
  q.partial = partial;
  q.err = err;
  return q;
}

struct BwLayout {
  Layout fw;             // grouped buffers with room for the padded rows
  int64_t rows;          // grouped rows: N*k + (kBwPad - 1) * E
  size_t counts, kept, g, u, dy, dh, dgu, dxp, dz, dz16, dxr, dw, w_row, dw_row, wrT, part;
  // shared experts (S * Fs columns, one group of all tokens)
  size_t gs, us, hs, dhs, dgus, dxs, ws2T, total;
};

BwLayout bw_layout_of(const moe_config_t& c) {
  BwLayout B{};
  const int64_t N = c.n_tokens, E = c.n_experts, k = c.top_k, d = c.d_model, F = c.d_ff;
  B.rows = N * k + (kBwPad - 1) * E;
  B.fw = layout_of(c, (kBwPad - 1) * E, true);
  size_t o = B.fw.total;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const int64_t R = B.rows;
  B.counts = take((size_t)E * 4);
  B.kept = take((size_t)E * 4);
  B.g = take((size_t)R * F * 2);
  B.u = take((size_t)R * F * 2);
  B.dy = take((size_t)R * d * 2);
  B.dh = take((size_t)R * F * 2);
  B.dgu = take((size_t)R * 2 * F * 2);
  B.dxp = take((size_t)R * d * 2);
  B.dz = take((size_t)N * E * 4);
  B.dz16 = take((size_t)N * E * 2);
  B.dxr = take((size_t)N * d * 4);
  B.dw = take((size_t)N * k * 4);
  B.w_row = take((size_t)R * 4);
  B.dw_row = take((size_t)R * 4);
  B.wrT = take((size_t)d * E * 2);
  B.part = take(std::max<size_t>(
      4, wgrad_partial_floats(router_wgrad_problem(c, nullptr, nullptr, nullptr, nullptr,
                                                   nullptr),
                              num_sms()) * 4));
  const int64_t SF = (int64_t)c.n_shared * c.d_ff_shared;
  if (SF > 0) {
    B.gs = take((size_t)N * SF * 2);
    B.us = take((size_t)N * SF * 2);
    B.hs = take((size_t)N * SF * 2);
    B.dhs = take((size_t)N * SF * 2);
    B.dgus = take((size_t)N * 2 * SF * 2);
    B.dxs = take((size_t)N * d * 4);
    B.ws2T = take((size_t)SF * d * 2);
  }
  B.total = o;
  return B;
}

moe_status_t check_backward_args(const moe_config_t* cfg, const moe_weights_t* w) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  // the tensor-core path: bf16 layers, feature widths in whole k-blocks, E a
  // multiple of 8 (the router's gradient GEMMs read E-wide rows)
  if (c.dtype != MOE_BF16 || c.d_ff % 64 != 0 || c.d_model % 64 != 0 ||
      c.n_experts % 8 != 0 || (c.n_shared > 0 && c.d_ff_shared % 64 != 0))
    return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_router_weights(c, w));
  MOE_TRY(check_up_weights(c, w));
  MOE_TRY(check_shared_weights(c, w));
  return check_down_weights(c, w);
}

TcProblem plain_problem(const void* A, int64_t a_rows, int K, const void* B0, int b_groups,
                        int b_rows, const int32_t* offsets, int n_groups, int64_t rows,
                        int n_out, void* C, int c_is_f32, int32_t* err) {
  TcProblem q{};
  q.A = A;
  q.a_rows = a_rows;
  q.K = K;
  q.B0 = B0;
  q.b_groups = b_groups;
  q.b_rows = b_rows;
  q.k_sub = K;
  q.n_sub = 1;
  q.offsets = offsets;
  q.n_groups = n_groups;
  q.rows = rows;
  q.n_out = n_out;
  q.epilogue = kEpiNone;
  q.C = C;
  q.c_is_f32 = c_is_f32;
  q.err = err;
  return q;
}

moe_status_t tc_run(const TcProblem& q, cudaStream_t st) {
  if (!tc_gemm_supported(q)) return MOE_ERR_UNSUPPORTED;
  return launch_tc_gemm(q, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t wgrad_run(const WgradProblem& q, cudaStream_t st) {
  return launch_wgrad(q, num_sms(), st) ? MOE_OK : MOE_ERR_CUDA;
}

// The backward pass (routing held fixed): the forward's routing, grouping
// and expert activations are recomputed, then the gradients run back
// through the combine, the experts and the router.
moe_status_t backward_impl(const moe_config_t& c, const void* x, const moe_weights_t& w,
                           const void* dout, float d_balance, moe_grads_t& gr, void* ws,
                           cudaStream_t st) {
  const BwLayout B = bw_layout_of(c);
  const Layout& L = B.fw;
  const Scratch sc = scratch_of(L, ws);
  const int64_t N = c.n_tokens, M = B.rows;        // M: grouped rows (padded)
  const int E = c.n_experts, k = c.top_k, d = c.d_model, F = c.d_ff;
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* wts = at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* ros = at<int32_t>(ws, L.row_of_slot);
  int32_t* tor = at<int32_t>(ws, L.token_of_row);
  void* x_perm = at<char>(ws, L.x_perm);
  void* hw = at<char>(ws, L.h);                     // w h, per grouped row
  int32_t* counts = at<int32_t>(ws, B.counts);
  int32_t* kept = at<int32_t>(ws, B.kept);
  void* g = at<char>(ws, B.g);
  void* u = at<char>(ws, B.u);
  void* dy_u = at<char>(ws, B.dy);                  // dout per grouped row
  float* w_row = at<float>(ws, B.w_row);
  float* dw_row = at<float>(ws, B.dw_row);
  void* dh = at<char>(ws, B.dh);
  void* dgu = at<char>(ws, B.dgu);
  void* dxp = at<char>(ws, B.dxp);
  float* dz = at<float>(ws, B.dz);
  void* dz16 = at<char>(ws, B.dz16);
  float* dxr = at<float>(ws, B.dxr);
  float* dw = at<float>(ws, B.dw);
  char* wrT = at<char>(ws, B.wrT);
  const int ns = num_sms();

  const bool swiglu = c.expert == MOE_EXPERT_SWIGLU;
  const int S = c.n_shared, SF = c.n_shared * c.d_ff_shared;
  float* dxs = SF > 0 ? at<float>(ws, B.dxs) : nullptr;

  // 1. recompute: routing (counts for the balance term), grouping (each
  //    expert's rows padded to whole 16-row slices, the padding zero in
  //    x_perm and dy_u), x_perm, g = x W1^T (+ b1 for the SiLU-MLP: a), and
  //    for SwiGLU u = x W3^T.  Neither h nor y is recomputed: the gradient of
  //    the routing weights is a row dot of dh_u and h, formed from g and u
  //    where they are read anyway.
  moe_stats_t rs{};
  rs.counts = counts;
  router_body(c, x, w, nullptr, idx, wts, &rs, sc, st, true);
  dispatch_body(c, idx, x, offsets, ros, tor, x_perm, nullptr, sc, st, nullptr, nullptr,
                kBwPad, kept);
  launch_zero_pad_rows(offsets, kept, E, (int64_t)d * 2, x_perm, dy_u, st);
  TcProblem q = plain_problem(x_perm, M, d, w.w1, E, F, offsets, E, M, F, g, 0, sc.err);
  q.use_pairs = pairs_pay(c);
  if (!swiglu && c.has_bias) {
    q.bias = w.b1;
    q.bias_stride = F;
  }
  MOE_TRY(tc_run(q, st));
  if (swiglu) {
    q.B0 = w.w3;
    q.C = u;
    MOE_TRY(tc_run(q, st));
  }

  // 2. dout to the expert rows: dy_u[row] = dout[t] (unweighted), w_row[row]
  //    = w[t, j] (0 on the padding), dw = <dout, b2> (biases) or 0
  cudaMemsetAsync(w_row, 0, (size_t)M * 4, st);
  MOE_TRY(last_cuda());
  launch_scatter_dout(dout, ros, wts, idx, c.has_bias ? w.b2 : nullptr, N, k, d, dy_u, w_row,
                      dw, ns, st);

  // 3. data gradients: dh_u = dy_u W2; per row dw += <dh_u, h>, dh = w dh_u,
  //    SwiGLU: [dg | du] = SwiGLU', SiLU-MLP: da = dh silu'(a), and hw = w h
  //    (for dW2); dlogits from dw; dx_perm = dg W1 + du W3 (SiLU-MLP: da W1);
  //    the shared experts' part of dx (below); dx = sum over slots +
  //    dlogits Wr (+ shared).  The expert weights are read in place as
  //    MN-major B operands: W2 [E, d, F] is, per expert, d K-rows of F
  //    output columns; W1 / W3 [E, F, d] are F K-rows of d columns (the two
  //    K sub-blocks of [dg | du]); Wr [E, d] likewise when E fills whole
  //    k-blocks, else it is transposed.
  q = plain_problem(dy_u, M, d, w.w2, E, F, offsets, E, M, F, dh, 0, sc.err);
  q.b_mn_major = 1;
  q.use_pairs = pairs_pay(c);
  MOE_TRY(tc_run(q, st));
  launch_expert_rows_backward(dh, g, swiglu ? u : nullptr, w_row, offsets, E, 0, F, dgu, hw,
                              dw_row, ns, st);
  launch_slot_dw(dw_row, ros, N * k, dw, ns, st);
  launch_router_backward(sc.logits, idx, wts, dw, counts, N, E, k, c.route, c.balance_coef,
                         d_balance, dz, dz16, st);
  q = plain_problem(dgu, M, swiglu ? 2 * F : F, w.w1, E, d, offsets, E, M, d, dxp, 0, sc.err);
  q.b_mn_major = 1;
  q.k_sub = F;
  if (swiglu) {
    q.B1 = w.w3;
    q.n_sub = 2;
  }
  q.use_pairs = pairs_pay(c);
  MOE_TRY(tc_run(q, st));
  if (E % 64 == 0) {                               // whole 64-row k-blocks of Wr
    q = plain_problem(dz16, N, E, w.w_router, 1, d, nullptr, 1, N, d, dxr, 1, sc.err);
    q.b_mn_major = 1;
  } else {
    launch_transpose_batched(w.w_router, 1, E, d, wrT, (int64_t)d * E, st);
    q = plain_problem(dz16, N, E, wrT, 1, d, nullptr, 1, N, d, dxr, 1, sc.err);
  }
  MOE_TRY(tc_run(q, st));
  if (SF > 0) {
    // shared experts: one SwiGLU of width S*Fs over all tokens, weight one,
    // so its output gradient is dout itself.  gs = x Ws1^T, us = x Ws3^T;
    // dhs = dout Ws2 (one shared expert: Ws2 [d, Fs] read MN-major; more:
    // Ws2 [S, d, Fs] transposed to the K-major [S*Fs, d]); [dgs | dus] and
    // hs = silu(gs) us; dxs = dgs Ws1 + dus Ws3
    char* gs = at<char>(ws, B.gs);
    char* us = at<char>(ws, B.us);
    char* hs = at<char>(ws, B.hs);
    char* dhs = at<char>(ws, B.dhs);
    char* dgus = at<char>(ws, B.dgus);
    char* ws2T = at<char>(ws, B.ws2T);
    const int Fs = c.d_ff_shared;
    q = plain_problem(x, N, d, w.ws1, 1, SF, nullptr, 1, N, SF, gs, 0, sc.err);
    q.use_pairs = N >= 128;
    MOE_TRY(tc_run(q, st));
    q.B0 = w.ws3;
    q.C = us;
    MOE_TRY(tc_run(q, st));
    if (S == 1) {
      q = plain_problem(dout, N, d, w.ws2, 1, SF, nullptr, 1, N, SF, dhs, 0, sc.err);
      q.b_mn_major = 1;
    } else {
      launch_transpose_batched(w.ws2, S, d, Fs, ws2T, (int64_t)Fs * d, st);
      q = plain_problem(dout, N, d, ws2T, 1, SF, nullptr, 1, N, SF, dhs, 0, sc.err);
    }
    q.use_pairs = N >= 128;
    MOE_TRY(tc_run(q, st));
    launch_expert_rows_backward(dhs, gs, us, nullptr, nullptr, 0, N, SF, dgus, hs, nullptr, ns,
                                st);
    // Ws1 / Ws3 [S*Fs, d] read in place (MN-major: S*Fs K-rows of d columns)
    q = plain_problem(dgus, N, 2 * SF, w.ws1, 1, d, nullptr, 1, N, d, dxs, 1, sc.err);
    q.b_mn_major = 1;
    q.B1 = w.ws3;
    q.k_sub = SF;
    q.n_sub = 2;
    q.use_pairs = N >= 128;
    MOE_TRY(tc_run(q, st));
  }
  launch_dx_reduce(dxp, ros, dxr, dxs, N, k, d, gr.dx, ns, st);

  // 4. weight gradients, read in place: dW2[e] = dy_u,e^T hw_e (= dy^T h);
  //    [dW1 | dW3][e]
  //    = [dg | du]_e^T x_e (one launch, rows F.. of each group's output to
  //    dW3); the router's dWr = dlogits^T x and the shared experts' over all
  //    tokens as one group
  WgradProblem wq{};
  wq.P = dy_u;
  wq.p_ld = d;
  wq.m_dim = d;
  wq.Q = hw;
  wq.q_ld = F;
  wq.n_dim = F;
  wq.rows = M;
  wq.offsets = offsets;
  wq.n_groups = E;
  wq.C0 = gr.d_w2;
  wq.err = sc.err;
  MOE_TRY(wgrad_run(wq, st));
  wq.P = dgu;
  wq.p_ld = swiglu ? 2 * F : F;
  wq.m_dim = swiglu ? 2 * F : F;
  wq.Q = x_perm;
  wq.q_ld = d;
  wq.n_dim = d;
  wq.C0 = gr.d_w1;
  if (swiglu) {
    wq.C1 = gr.d_w3;
    wq.m_split = F;
  }
  MOE_TRY(wgrad_run(wq, st));
  if (c.has_bias) {
    // db1[e] = sum of da, db2[e] = sum of w dy_u over expert e's rows (the
    // padding rows are zero)
    launch_group_sums(dgu, F, offsets, E, F, gr.d_b1, st);
    launch_group_sums(dy_u, d, offsets, E, d, gr.d_b2, st, w_row);
  }
  WgradProblem rq = router_wgrad_problem(c, dz16, x, gr.d_w_router, at<float>(ws, B.part),
                                         sc.err);
  rq.partial_floats = wgrad_partial_floats(rq, ns);
  MOE_TRY(wgrad_run(rq, st));
  if (gr.d_b_router != nullptr) launch_column_sums(dz, N, E, gr.d_b_router, st);
  if (SF > 0) {
    // shared: dWs2[s] = dout^T hs[:, s], [dWs1 | dWs3] = [dgs | dus]^T x
    const int Fs = c.d_ff_shared;
    WgradProblem sq{};
    sq.rows = N;
    sq.n_groups = 1;
    sq.err = sc.err;
    sq.P = dout;
    sq.p_ld = d;
    sq.m_dim = d;
    sq.q_ld = SF;
    sq.n_dim = Fs;
    for (int sx = 0; sx < S; ++sx) {
      sq.Q = at<char>(ws, B.hs) + (size_t)sx * Fs * 2;
      sq.C0 = gr.d_ws2 + (size_t)sx * d * Fs;
      MOE_TRY(wgrad_run(sq, st));
    }
    sq.P = at<char>(ws, B.dgus);
    sq.p_ld = 2 * SF;
    sq.m_dim = 2 * SF;
    sq.Q = x;
    sq.q_ld = d;
    sq.n_dim = d;
    sq.C0 = gr.d_ws1;
    sq.C1 = gr.d_ws3;
    sq.m_split = SF;
    MOE_TRY(wgrad_run(sq, st));
  }
  return last_cuda();
}

}  // namespace

extern "C" {

moe_status_t moe_forward(const moe_config_t* cfg, const void* x,
                         const moe_weights_t* weights, void* out,
                         moe_stats_t* stats, void* ws, size_t ws_bytes,
                         void* stream) {
  return forward_impl(cfg, x, weights, out, stats, ws, ws_bytes, stream, nullptr);
}

moe_status_t moe_forward_timed(const moe_config_t* cfg, const void* x,
                               const moe_weights_t* weights, void* out,
                               moe_stats_t* stats, void* ws, size_t ws_bytes,
                               void* stream, void* const* events, int32_t n_events) {
  if (events == nullptr || n_events != MOE_FORWARD_EVENTS) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i)
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, x, weights, out, stats, ws, ws_bytes, stream,
                      reinterpret_cast<cudaEvent_t const*>(events));
}


moe_status_t moe_forward_host(const moe_config_t* cfg, const void* x_host,
                              const moe_weights_t* weights, void* out_host,
                              moe_stats_t* stats, void* ws, size_t ws_bytes,
                              void* stream) {
  MOE_TRY(check_forward_args(cfg, weights, stats, ws, ws_bytes));
  const moe_config_t& c = *cfg;
  const Layout L = layout_of(c);
  if (c.n_tokens > 0 && (x_host == nullptr || out_host == nullptr))
    return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (capacity_of(c) < 0 && c.n_tokens >= 2 * kHostChunkMin) {
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* hp = host_pipe();
    if (hp != nullptr)
      return forward_host_pipelined(c, static_cast<const char*>(x_host), *weights,
                                    static_cast<char*>(out_host), stats, ws, st, *hp);
  }
  const size_t bytes = (size_t)c.n_tokens * c.d_model * elem_size(c);
  void* xd = at<char>(ws, L.x_stage);
  void* od = at<char>(ws, L.out_stage);
  if (bytes > 0 && cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  MOE_TRY(moe_forward(cfg, xd, weights, od, stats, ws, ws_bytes, stream));
  if (bytes > 0 && cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_update_selection_bias(const moe_config_t* cfg, const int32_t* counts,
                                       float* sel_bias, float gamma, float* load_cv,
                                       void* stream) {
  MOE_TRY(check_config(cfg));
  if (!std::isfinite(gamma)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need({counts}));
  if (sel_bias == nullptr && load_cv == nullptr) return MOE_ERR_INVALID_ARG;
  if ((sel_bias != nullptr && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) ||
      (load_cv != nullptr && (reinterpret_cast<uintptr_t>(load_cv) & 3u)))
    return MOE_ERR_INVALID_ARG;
  launch_bias_update(counts, cfg->n_experts, gamma, sel_bias, load_cv,
                     static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status_t moe_backward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = bw_layout_of(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t* cfg, const void* x, const moe_weights_t* weights,
                          const void* dout, float d_balance, moe_grads_t* grads, void* ws,
                          size_t ws_bytes, void* stream) {
  MOE_TRY(check_backward_args(cfg, weights));
  const moe_config_t& c = *cfg;
  if (grads == nullptr || !std::isfinite(d_balance)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(ws, ws_bytes, bw_layout_of(c).total));
  if (c.n_tokens == 0) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(need({x, dout, grads->dx, grads->d_w_router, grads->d_w1, grads->d_w2}));
  if (c.expert == MOE_EXPERT_SWIGLU) MOE_TRY(need({grads->d_w3}));
  if (c.has_bias) MOE_TRY(need({grads->d_b1, grads->d_b2}));
  if (c.n_shared > 0) MOE_TRY(need({grads->d_ws1, grads->d_ws3, grads->d_ws2}));
  MOE_TRY(maybe({grads->d_b_router}));
  if (grads->d_b_router != nullptr && weights->b_router == nullptr) return MOE_ERR_INVALID_ARG;
  return backward_impl(c, x, *weights, dout, d_balance, *grads, ws,
                       static_cast<cudaStream_t>(stream));
}

moe_status_t moe_check_grouping(const moe_config_t* cfg, const int32_t* idx,
                               const int32_t* offsets, const int32_t* row_of_slot,
                               const int32_t* token_of_row, void* ws, size_t ws_bytes,
                               void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_ws(ws, ws_bytes, layout_of(c).scratch_end));
  MOE_TRY(need({offsets}));
  if (c.n_tokens == 0) return MOE_OK;
  MOE_TRY(need({idx, row_of_slot, token_of_row}));
  // two words of the workspace's first (zero-filled) block: the kept-slot
  // count and the last-CTA ticket, both left zero
  unsigned* words = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 192);
  launch_check_grouping(idx, offsets, row_of_slot, token_of_row, c.n_tokens, c.top_k,
                        c.n_experts, capacity_of(c), words, words + 1, err_word(ws), num_sms(),
                        static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status_t moe_check_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                    void* stream) {
  if (ws == nullptr || ws_bytes < kAlign || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 1000000000) return MOE_ERR_INVALID_ARG;
  int32_t* err = static_cast<int32_t*>(ws);
  int32_t* flags = err + 32;                       // bytes 128..135 of the first block
  return launch_wait_check(err, (uint64_t)limit_ns, flags, static_cast<cudaStream_t>(stream))
             ? last_cuda()
             : MOE_ERR_CUDA;
}

moe_status_t moe_read_device_error(void* ws, int32_t* code, void* stream) {
  if (ws == nullptr || code == nullptr) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(ws, 0, sizeof(v), st) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v == kDevOk ? MOE_OK : v == kDevTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

int32_t moe_version(void) { return 200; }

}  // extern "C"
