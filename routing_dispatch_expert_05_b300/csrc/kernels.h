// Internal (C++) launch interface between the ABI layer and the kernels.
// Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Tokens per CTA of the selection kernel from 4096 tokens on (8 below).  The
// host pipeline starts its chunks on multiples of it, so every CTA sums the
// same tokens either way.
constexpr int kRouteTokensPerCta = 32;
// Tokens per dispatch chunk (the unit of the per-chunk histogram).
constexpr int kDispatchTokensPerChunk = 128;
constexpr int kMaxExperts = 256;

// ---- router ---------------------------------------------------------------
// Running per-expert totals of one forward's selection statistics, in the
// workspace: probability sums in units of 2^-32 (integers, so the totals do
// not depend on the order in which CTAs add them), selection counts, and a
// ticket.  All three are zero between forwards.
struct RouteTotals {
  unsigned long long* psum_fx;   // [E]
  unsigned* cnt;                 // [E]
  unsigned* ticket;
};
// With `finalize`, the last CTA of the launch turns the totals (of every
// launch since they were last cleared) into counts[E] and the balance
// statistic over n_total tokens (either output nullable) and clears them.
struct RouteFinal {
  bool finalize;
  int64_t n_total;
  float coef;
  int32_t* counts;
  float* balance;
};
// logits[N, E] (fp32) -> idx, w; adds this launch's statistics to `tot`.
void launch_route_from_logits(const float* logits, int64_t n_tokens, int n_experts,
                              int top_k, int mode, const float* sel_bias,
                              int32_t* idx, float* w, const RouteTotals& tot,
                              const RouteFinal& fin, cudaStream_t st);

// between steps: selection-bias update from the per-expert counts and the
// load's coefficient of variation (either output nullable)
void launch_bias_update(const int32_t* counts, int n_experts, float gamma, float* sel_bias,
                        float* load_cv, cudaStream_t st);

// ---- dispatch -------------------------------------------------------------
// capacity: one for every expert (< 0: none); room (device [E], nullable):
// a capacity per expert instead.  pad > 1 (with kept non-null): each
// expert's group of rows is rounded up to a multiple of pad, so
// offsets[e+1] - offsets[e] = pad * ceil(kept[e] / pad); the rows after the
// kept ones are not written (launch_zero_pad_rows clears them)
void launch_dispatch(const int32_t* idx, int64_t n_tokens, int top_k,
                     int n_experts, int64_t capacity /* <0: none */,
                     int32_t* chunk_cnt, int32_t* chunk_base, int32_t* offsets,
                     int32_t* row_of_slot, int32_t* token_of_row,
                     int32_t* counts, int32_t* kept, int32_t* dropped,
                     int32_t* err, cudaStream_t st, int32_t* slot_of_row = nullptr,
                     const int32_t* room = nullptr, int pad = 1,
                     int tokens_per_chunk = kDispatchTokensPerChunk);
// x_perm[row_of_slot[t*k + j]] = x[t] for every kept slot (one warp per token,
// 32- or 16-byte vectors; a TMA bulk-copy version measured slower)
void launch_scatter_rows(const void* x, int64_t row_bytes, const int32_t* row_of_slot,
                         int64_t n_tokens, int top_k, void* x_perm, int num_sms,
                         cudaStream_t st);
// Device-side consistency check of a grouping (offsets monotone and within
// the buffer, row_of_slot a bijection of the kept slots onto [0, M) that
// agrees with idx and token_of_row, groups in arrival order); a failure sets
// kDevBadRow.  kept_count and ticket: two zeroed words, left zero.
void launch_check_grouping(const int32_t* idx, const int32_t* offsets,
                           const int32_t* row_of_slot, const int32_t* token_of_row,
                           int64_t n_tokens, int top_k, int n_experts, int64_t capacity,
                           unsigned* kept_count, unsigned* ticket, int32_t* err, int num_sms,
                           cudaStream_t st);

// ---- SIMT GEMM (fp32 and bf16 storage, fp32 accumulation) ----------------
enum Epilogue : int {
  kEpiNone = 0,      // C = A B^T (+ bias)
  kEpiSiluBias = 1,  // C = silu(A B^T + bias)
  kEpiSwiglu = 2,    // C = silu(A B0^T) * (A B1^T)
};

struct GemmProblem {
  const void* A;             // [rows, K] row-major, lda = K
  const void* B0;            // group g: B0 + g * b_group_stride, [N, ...]
  const void* B1;            // second operand (SwiGLU up), same layout
  int64_t b_group_stride;    // elements between groups
  // element (n, k) of group g's B sits at
  //   B + g*b_group_stride + (k / k_sub) * sub_stride + n * k_sub + (k % k_sub)
  // (k_sub = K for one plain [N, K] matrix; the shared down projection is
  // S column blocks of width k_sub = Fs)
  int k_sub;
  int64_t sub_stride;
  const void* bias;          // [G][N] or null
  int64_t bias_group_stride;
  void* C;                   // [rows, N] row-major
  int c_is_f32;              // 1: C is fp32 regardless of the storage type
  const int32_t* offsets;    // [G+1] device (row ranges) or null: one group
  int n_groups;
  int64_t rows;              // rows when offsets == null, else max rows
  int N, K;
  int epilogue;
  int is_bf16;               // storage type of A, B, bias (and C unless c_is_f32)
  // Optional row map (fused dispatch gather): row r of the grouped problem
  // reads row a_row_map[r] of A.  null: A is in grouped row order.
  const int32_t* a_row_map;
  int32_t* err;              // device error word (nullable): a bad grouping
};
void launch_simt_gemm(const GemmProblem& p, cudaStream_t st);
// router logits [N, E] fp32 for a few tokens (CUDA cores, one thread per
// expert); x [N, d], w [E, d], b [E] or null, in the layer dtype
void launch_router_small(const void* x, const void* w, const void* b, float* logits,
                         int64_t n_tokens, int n_experts, int d, int is_bf16, cudaStream_t st);
// below this many tokens the router GEMM runs on the CUDA cores
constexpr int64_t kRouterSmallTokens = 512;

// ---- tcgen05 grouped GEMM (bf16 storage, fp32 accumulation in TMEM) -------
struct TcProblem {
  const void* A;             // [a_rows, K] bf16 row-major
  int64_t a_rows;
  int K;
  const void* B0;            // [b_groups * n_sub * b_rows, k_sub] bf16
  const void* B1;            // SwiGLU up projection, same layout as B0
  int b_groups;              // groups stacked in B
  int b_rows;                // rows of B per (group, sub-block)
  int k_sub;                 // K-split width (K when n_sub == 1)
  int n_sub;                 // K = n_sub * k_sub; block s of K reads sub-block s
  const int32_t* offsets;    // [n_groups+1] device row ranges, or null
  int n_groups;
  int64_t rows;              // rows when offsets == null
  int n_out;                 // output columns (multiple of 8)
  int swiglu;                // 1: out = silu(A B0^T) * (A B1^T)
  int epilogue;              // Epilogue
  const void* bias;          // [n_groups][n_out] bf16 or null
  int64_t bias_stride;
  void* C;                   // [rows, n_out] bf16 (or fp32 if c_is_f32, fp16 if c_scale)
  int c_is_f32;
  // Compact output (non-SwiGLU only): C holds fp16 values v * 2^s with one
  // power of two per (row, 32-column block), chosen so that the block's
  // largest magnitude lands in [2^14, 2^15); c_e8[row * e8_cols + block] is
  // the biased fp32 exponent of 2^-s (value = fp16 * 2^(c_e8 - 127)).
  uint8_t* c_e8;
  int e8_cols;               // ceil(n_out / 32)
  int32_t* err;              // device error word
  // Optional row map (fused dispatch gather): A row r of the grouped problem
  // is row a_row_map[r] of A ([a_rows, K], e.g. the token rows x), for
  // r < offsets[n_groups].  null: A is already in grouped row order.
  const int32_t* a_row_map;
  // 1: run on CTA pairs (tcgen05 cta_group::2, 256-row tiles) where the
  // problem allows it
  int use_pairs;
  // Compact output only: row r of the grouped problem is written to output
  // row c_row_map[r] (e.g. its assignment slot t*k + j), scaled by
  // c_row_scale[output row] (e.g. the routing weight) before compacting.
  const int32_t* c_row_map;
  const float* c_row_scale;
  // 1: B is MN-major: group g (sub-block s) is rows g*k_sub .. of B0 (s = 0)
  // or B1 (s = 1), each row n_out contiguous elements -- e.g. a weight
  // [E, K, N] used without a transpose.  Not with SwiGLU.
  int b_mn_major;
};
bool tc_gemm_supported(const TcProblem& p);
bool launch_tc_gemm(const TcProblem& p, int num_sms, cudaStream_t st);
// The same grouped problem with the operands swapped (gemm_swap.cu), for
// experts of a few rows each: weight rows on the MMA's M side, each expert's
// token rows (A, up to 64 per tile) on N.  Supports the SwiGLU and SiLU+bias
// up projections (bf16 C) and the compact down projection (c_e8 set, with
// c_row_map / c_row_scale); n_out a multiple of 16 (32 when compact).
bool swap_gemm_supported(const TcProblem& p);
bool launch_swap_gemm(const TcProblem& p, int num_sms, cudaStream_t st);

// Weight gradients on the tensor cores: for each group g,
//   C[g*rows_a + i, j] = sum_{c in [k_offsets[g], k_offsets[g+1])} A[i, c] B[j, c]
// A [rows_a, k_total] and B [rows_b, k_total] bf16 row-major (the grouped
// activations transposed, every group's column span a non-zero multiple of
// 64, zero-padded); C fp32 [n_groups * rows_a, rows_b].
// Weight gradients, per group g of rows [offsets[g], offsets[g+1]) of P and
// Q (null offsets: one group of all rows): C_g = P_g^T Q_g in fp32, from the
// first m_dim columns of P [rows, p_ld] and n_dim of Q [rows, q_ld] (bf16),
// both read in place (MN-major tcgen05 operands, CTA pairs).  Output rows i
// < m_split of group g go to C0[g][i][:], the rest (C1 non-null) to
// C1[g][i - m_split][:]; without C1, C0 is [G][m_dim][n_dim].  Each group's
// row count must be a multiple of 16, or the group must end at `rows`, and
// the rows that pad a group to 16 must be zero.  One group over few tiles is
// split over K into `partial` (wgrad_partial_floats(q) floats) and summed.
struct WgradProblem {
  const void* P;
  int64_t p_ld;
  int m_dim;
  const void* Q;
  int64_t q_ld;
  int n_dim;
  int64_t rows;
  const int32_t* offsets;
  int n_groups;
  float* C0;
  float* C1;
  int m_split;
  float* partial;
  size_t partial_floats;      // room at `partial` (fewer splits if it holds less)
  int32_t* err;
};
int wgrad_splits(const WgradProblem& q, int num_sms);
size_t wgrad_partial_floats(const WgradProblem& q, int num_sms);
bool launch_wgrad(const WgradProblem& q, int num_sms, cudaStream_t st);
// the GEMM kernels' bounded mbarrier wait, run out on purpose (see moe.h)
bool launch_wait_check(int32_t* err, uint64_t limit_ns, int32_t* flags, cudaStream_t st);

// ---- combine ----------------------------------------------------------------
// y: fp32 expert outputs [N*k, d]; out: layer dtype [N, d]
void launch_combine(const float* y, const int32_t* row_of_slot, const float* w,
                    const float* shared, void* out, int64_t n_tokens, int top_k,
                    int d_model, int is_bf16, int num_sms, cudaStream_t st);
// the same with compact expert outputs: y16 [N*k, d] fp16 and
// y_e8 [N*k, ceil(d/32)] (value = y16 * 2^(y_e8 - 127) for its 32 columns)
// compact expert outputs already weighted and in slot order (row t*k + j);
// row_of_slot null: no slot was dropped (a layer without capacity)
// err (nullable): the bulk-copy kernel's timeout word; without it, or where
// a token's rows do not fit a stage, the register-fed kernel runs
void launch_combine_slots(const void* y16, const uint8_t* y_e8, const int32_t* row_of_slot,
                          const float* shared, void* out, int64_t n_tokens, int top_k,
                          int d_model, int is_bf16, int num_sms, cudaStream_t st,
                          int32_t* err = nullptr);
constexpr int kYScaleBlock = 32;    // columns per compact-output exponent

// ---- backward (backward.cu) -----------------------------------------------
// zero rows [offsets[e] + kept[e], offsets[e+1]) of buf0 and buf1 (rows of
// row_bytes, a multiple of 16; buf1 nullable): the padding of a padded grouping
void launch_zero_pad_rows(const int32_t* offsets, const int32_t* kept, int n_experts,
                          int64_t row_bytes, void* buf0, void* buf1, cudaStream_t st);
// out[b][c][r] = in[b][r][c] (bf16), batch b of the output at out + b * out_stride
void launch_transpose_batched(const void* in, int batch, int rows, int cols, void* out,
                              int64_t out_stride, cudaStream_t st);
// Per grouped row (offsets[E] rows, or `rows` with offsets null): from dh_u
// (= dout W2, unweighted), g, u (null: SiLU-MLP) and the row's routing weight
// (w_row null: 1), h = silu(g) u; dw_row = <dh_u, h>; dh = w dh_u; dgu =
// [dh u silu'(g) | dh silu(g)] (SiLU-MLP: dh silu'(g), row stride F); hw = w h.
// hw and dw_row nullable.
void launch_expert_rows_backward(const void* dh_u, const void* g, const void* u,
                                 const float* w_row, const int32_t* offsets, int n_experts,
                                 int64_t rows, int F, void* dgu, void* hw, float* dw_row,
                                 int num_sms, cudaStream_t st);
// out[g] = sum over group g's rows of in[row] (times row_w[row] if non-null)
void launch_group_sums(const void* in, int64_t ld, const int32_t* offsets, int G, int C,
                       float* out, cudaStream_t st, const float* row_w = nullptr);
// dy_u[row] = dout[t] and w_row[row] = w[s] for each kept slot s = (t, j);
// dw[s] = <dout[t], b2[idx[s]]> (b2 non-null) or 0
void launch_scatter_dout(const void* dout, const int32_t* row_of_slot, const float* w,
                         const int32_t* idx, const void* b2, int64_t n_tokens, int top_k, int d,
                         void* dy_u, float* w_row, float* dw, int num_sms, cudaStream_t st);
// dw[s] += dw_row[row_of_slot[s]] for the kept slots
void launch_slot_dw(const float* dw_row, const int32_t* row_of_slot, int64_t n_slots, float* dw,
                    int num_sms, cudaStream_t st);
void launch_router_backward(const float* logits, const int32_t* idx, const float* w,
                            const float* dw, const int32_t* counts, int64_t n_tokens, int E,
                            int k, int mode, float coef, float d_balance, float* dz,
                            void* dz16 /* nullable bf16 copy */, cudaStream_t st);
// dx = dxr (+ dxs, nullable) + the token's kept rows of dxp
void launch_dx_reduce(const void* dxp, const int32_t* row_of_slot, const float* dxr,
                      const float* dxs, int64_t n_tokens, int top_k, int d, float* dx,
                      int num_sms, cudaStream_t st);
// d_b_router[e] = sum_t dz[t, e] (fixed-order tree per expert)
void launch_column_sums(const float* dz, int64_t n_tokens, int E, float* out, cudaStream_t st);

}  // namespace moe
