// Host-side launchers shared between the translation units of libmok.
#pragma once

#include <climits>

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mok.h"

namespace mok {

// Routes per plan chunk (one CTA of the count / place kernels).
constexpr int kPlanChunk = 1024;

int plan_chunks(int64_t R);
size_t plan_scratch_bytes(int64_t R, int E);
size_t plan_ranks_scratch_bytes(int64_t R, int E, int ranks);
// the pull schedule with `ranks` virtual source ranks of T / ranks tokens
mok_status launch_plan_ranks(const int32_t* topk, int64_t T, int K, int E, int ranks, int32_t* counts,
                             int32_t* offsets, int32_t* table, int32_t* route_dst, int* scratch,
                             cudaStream_t st);

mok_status launch_route(const float* s, int T, int E, int K, int32_t* topk, float* g,
                        cudaStream_t st);
mok_status launch_plan(const int32_t* topk, int64_t R, int E, int32_t* counts, int32_t* offsets,
                       int32_t* table, int32_t* route_dst, int* hist, cudaStream_t st);

// xg[route_dst[t K + k]] = x[t] (each token row read once, stored K times;
// K <= 32); when g_route is non-null also g_route[route_dst[r]] = g[r].
mok_status launch_dispatch_bf16(const void* x, const int32_t* route_dst, int T, int K, int D, void* xg,
                                const float* g, float* g_route, cudaStream_t st);
// The same with MXFP8 quantisation: codes [R][D] and grouped scale words
// (expert of position p: table[p].e).
mok_status launch_dispatch_mxfp8(const void* x, const int32_t* route_dst, const int32_t* table,
                                 const int32_t* offsets, int T, int K, int D, int E, void* xg_q, uint8_t* xg_scale,
                                 cudaStream_t st);
mok_status launch_quantize_mxfp8(const void* src, int64_t rows, int64_t cols, void* q,
                                 uint8_t* scale, cudaStream_t st);
// out[t] = bf16(base[t] + sum_k w[t,k] * rows[route_dst[t*K+k]]); base and w
// nullable (0 and 1).
mok_status launch_combine(const void* rows, const void* base, const float* w,
                          const int32_t* route_dst, int T, int K, int D, void* out,
                          cudaStream_t st);

// Kept activations of the forward's routed up/gate (mok_plan_buf::act): h, u
// fp32 [rows][2I] of every group whose rows end at or below `rows`; null /
// 0: none kept.
struct KeptAct {
  float* act = nullptr;
  int64_t rows = 0;
  int32_t limit() const {  // the row limit as the kernels compare it
    return act ? static_cast<int32_t>(rows < INT32_MAX ? rows : INT32_MAX) : 0;
  }
};

// Whether a layer of R routed rows in G groups averages fewer than 512 rows
// per group: its forward GEMMs then take the routed rows as the MMA's N
// dimension (no padding rows, HBM-bound), else run row-major 256-row tiles.
inline bool routed_rows_as_n(int64_t R, int G) { return R < static_cast<int64_t>(512) * G; }

// Forward grouped GEMMs (CTA pairs, gemm_pair.cu).  offsets == nullptr: one
// group of m_total rows.
//  up/gate: a[rows][I] = bf16(SiLU(A W_gate^T) * (A W_up^T)), A [rows][D]
//  down   : y[rows][D] = bf16(a W_down^T)
// max_sms > 0: the grid takes at most that many SMs (the rest stay free for
// kernels of other streams).
mok_status launch_upgate(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                         const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                         cudaStream_t st, int max_sms = 0, KeptAct kept = {});
mok_status launch_down(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets,
                       int G, int64_t m_total, int D, int I, void* y_out, cudaStream_t st, int max_sms = 0);
// The shared expert as an extra group of a routed launch: A [rows][K],
// weights w0 (, w1) with `inner` = I_shared, output [rows][N].
struct SharedOperands {
  const void* A;
  int64_t rows;
  const void* w0;
  const void* w1;
  int inner;
  void* out;
};
// The same two GEMMs with the shared expert's tiles (sh) spread through the
// routed launch (cta_group::2, 256-row tiles).
mok_status launch_upgate_pair(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                              const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                              cudaStream_t st, const SharedOperands* sh = nullptr, KeptAct kept = {},
                              int max_sms = 0);
// Router scores s = softmax(x W_r^T) [T][E] fp32 (E <= 256): x [T][D], W_r
// [E][D] bf16, on CTA pairs with the softmax in the epilogue.
mok_status launch_router_pair(const void* x, int64_t T, const void* w_router, int E, int D, float* s_out,
                              cudaStream_t st);
// Ring dispatch fused into the routed up/gate (BF16): producer warps in the
// same launch gather x rows into `ring` ([ring_rows + 128][D] bf16) in
// chunks of chunk_rows routed rows; counters: 2 * ceil(R / chunk_rows) ints.
mok_status launch_upgate_ring(const void* x, const int32_t* table, int K, const void* w_gate, const void* w_up,
                              const int32_t* offsets, int G, int64_t R, int D, int I, void* a_out, void* ring,
                              int64_t ring_rows, int chunk_rows, int32_t* counters, cudaStream_t st,
                              KeptAct kept = {});
// Ring geometry for R routed rows and chunk b (0: 2048): 4 slots of b rows,
// or fewer when that already holds every row (then no slot is reused).
constexpr int64_t kRingSlots = 4;
inline int64_t ring_chunk(int chunk_rows) { return chunk_rows > 0 ? chunk_rows : 2048; }
inline int64_t ring_rows_for(int64_t R, int64_t b) {
  int64_t all = (R + b - 1) / b;
  if (all < 1) all = 1;
  return (all < kRingSlots ? all : kRingSlots) * b;
}
inline size_t ring_bytes(int64_t R, int64_t D, int64_t b, int elem_bytes = 2) {
  return static_cast<size_t>(ring_rows_for(R, b) + 128) * D * elem_bytes;
}
inline size_t ring_counter_bytes(int64_t R, int64_t b) { return static_cast<size_t>((R + b - 1) / b) * 8; }
mok_status launch_down_pair(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets, int G,
                            int64_t m_total, int D, int I, void* y_out, cudaStream_t st,
                            const SharedOperands* sh = nullptr, int max_sms = 0);

// Backward (max_sms > 0: the persistent grid takes at most that many SMs).
// dgrad+replay: dh, du, ag [rows][I] bf16 and, when dgp is
// non-null, dgp [rows][I/32] partials of <t, a> (32 I columns each);
// g_route null = weight 1.  skip_rows_below > 0: only the groups with a row
// at or above it (the others were kept by the forward).
mok_status launch_bwd_dgrad(const void* xg, const void* dyg, int64_t rows, const void* w_gate,
                            const void* w_up, const void* w_down, const int32_t* offsets, int G,
                            int D, int I, const float* g_route, void* dh, void* du, void* ag,
                            float* dgp, cudaStream_t st, int32_t skip_rows_below = 0, int max_sms = 0);
// The same outputs for the groups whose rows all lie below kept_rows, from
// the forward's kept h, u (act fp32 [rows][2I]) and t = dYg W_down.
mok_status launch_bwd_dgrad_kept(const void* dyg, int64_t rows, const void* w_down, const int32_t* offsets, int G,
                                 int D, int I, const float* g_route, const float* act, int32_t kept_rows, void* dh,
                                 void* du, void* ag, float* dgp, cudaStream_t st, int max_sms = 0);
// dx [rows][D] = bf16(dh W_gate + du W_up)
//  launch_bwd_dx: routed groups averaging under 512 rows, and ungrouped rows
//  (offsets null), run on CTA pairs with the rows as the MMA's N dimension
//  (launch_dx_pair_t, gemm_pair.cu), others on single-CTA 128-row tiles.
mok_status launch_dx_pair_t(const void* dh, const void* du, int64_t rows, const void* w_gate, const void* w_up,
                            const int32_t* offsets, int G, int D, int I, void* dx, cudaStream_t st, int max_sms = 0);
mok_status launch_bwd_dx(const void* dh, const void* du, int64_t rows, const void* w_gate,
                         const void* w_up, const int32_t* offsets, int G, int D, int I, void* dx,
                         cudaStream_t st, int max_sms = 0);
// dw [G][M][N] = bf16(sum over each group's rows of pm[p][m] qn[p][n])
mok_status launch_wgrad(const void* pm, const void* qn, int64_t rows, const int32_t* offsets,
                        int G, int M, int N, void* dw, cudaStream_t st, int max_sms = 0);
// MXFP8 backward.  Replay: h, u fp32 [rows][I] from the up/gate pair GEMM
// (operands as launch_upgate_mx); skip_rows_below > 0: only the groups with
// a row at or above it.  Activation gradient: from fp32 h, u, t [R][I] and
// g_route (null = 1): dh, du, a_g bf16 [R][I], the codes of [dh | du]
// [R][2I] with grouped scale words (ld = mx_scale_ld(R, E)) and dgp [R] =
// <t, a>; the rows of groups that end at or below kept.rows read h, u from
// kept.act ([rows][2I]) instead.
mok_status launch_replay_mx(const void* xq, const void* xsc, int64_t rows, const void* qg, const void* sg,
                            const void* qu, const void* su, const int32_t* offsets, int G, int D, int I, void* h,
                            void* u, cudaStream_t st, int32_t skip_rows_below = 0);
mok_status launch_act_grad_mx(const void* h, const void* u, const void* t, const float* g_route,
                              const int32_t* table, const int32_t* offsets, int64_t R, int I, int E, void* dh,
                              void* du, void* ag, void* dhu_q, uint8_t* dhu_sc, float* dgp, cudaStream_t st,
                              KeptAct kept = {});
// Codes of src^T per matrix: src bf16 [G][M][N]; output row g N + n holds
// src[g][:, n] quantised along M at columns [col0, col0 + M) of out_cols,
// plain scale layout of G*N rows (M, col0, out_cols multiples of 128, N of 64).
mok_status launch_quantize_cols_mxfp8(const void* src, int G, int M, int N, void* q, uint8_t* scale, int out_cols,
                                      int col0, cudaStream_t st);
// ds [T][E], dg [T][K] (nullable) from the partials dgp [R][nI]
mok_status launch_router_grad(const float* dgp, int nI, const int32_t* route_dst,
                              const int32_t* topk, const float* g, const float* s, int T, int E,
                              int K, float* ds, float* dg, cudaStream_t st);

// MXFP8 scale storage of a [rows][K] tensor: int32 words [K/128][ld] with
// ld a multiple of 128; word (g, r) holds the E8M0 scales of row r for K
// columns [128 g, 128 g + 128), byte b = 32-column block b.  Within each
// aligned block of 128 rows, row 32 c + l sits at word 4 l + c: the order in
// which tcgen05.cp (32x128b, warpx4) puts a block where the block-scaled MMA
// reads it (lane 32 q + l, column c).
//  plain   : row r at position r, ld = rows rounded up to 128;
//  grouped : expert-contiguous rows (expert e owns [offsets[e], offsets[e+1]))
//            with each expert starting a new block: row offsets[e] + i at
//            position 128 (offsets[e] / 128 + e) + i, ld = 128 (ceil(rows/128) + E).
__host__ __device__ inline int64_t mx_scale_pos(int64_t r) {
  return (r & ~int64_t(127)) | ((r & 31) << 2) | ((r >> 5) & 3);
}
__host__ __device__ inline int64_t mx_group_row0(int64_t offset, int e) {
  return 128 * (offset / 128 + e);
}
inline int64_t mx_scale_ld(int64_t rows, int groups = 0) {
  return groups > 0 ? 128 * ((rows + 127) / 128 + groups) : (rows + 127) / 128 * 128;
}
inline size_t mx_scale_bytes(int64_t rows, int64_t K, int groups = 0) {
  return static_cast<size_t>(K / 128) * static_cast<size_t>(mx_scale_ld(rows, groups)) * 4;
}
// MXFP8 grouped GEMMs: a codes [rows][I] + scales, y [rows][D] (bf16, or
// fp32 when f32_out: the backward's t)
mok_status launch_upgate_mx(const void* xq, const void* xsc, int64_t rows, const void* qg,
                            const void* sg, const void* qu, const void* su, const int32_t* offsets,
                            int G, int D, int I, void* aq, void* asc, cudaStream_t st, KeptAct kept = {},
                            const void* sp = nullptr);
// The same (row-major tiles) with the quantising dispatch fused in as a ring:
// producer warps quantise routed rows of x (bf16 [T][D], row r from
// x[table[r].src / K]) into `ring` ([ring_rows + 128][D] codes) chunk by
// chunk, and their scale words into xsc (the grouped layout, R rows);
// counters: 2 * ceil(R / chunk_rows) ints.
mok_status launch_upgate_mx_ring(const void* x, const int32_t* table, int K, const void* qg, const void* sg,
                                 const void* qu, const void* su, const int32_t* offsets, int G, int64_t R, int D, int I,
                                 void* aq, void* asc, void* xsc, void* ring, int64_t ring_rows, int chunk_rows,
                                 int32_t* counters, cudaStream_t st, KeptAct kept = {});
// Paired scale blocks of W_up / W_gate (plain-layout scale words sg, su of
// G*I rows, K = D) for the up/gate with the routed rows as N: block
// b = e (I / 64) + s holds the words of W_up rows e I + 64 s .. + 63, then
// of the same W_gate rows; plain layout of 2 G I virtual rows.
mok_status launch_pair_scales(const void* sg, const void* su, int G, int I, int D, void* sp, cudaStream_t st);
mok_status launch_down_mx(const void* aq, const void* asc, int64_t rows, const void* qd,
                          const void* sd, const int32_t* offsets, int G, int D, int I, void* y,
                          cudaStream_t st, bool f32_out = false, int max_sms = 0);

bool shape_ok(const mok_shape* s);
// SMs the shared expert's side-stream launches may take (0: all): every SM
// but shape.producer_sms, which stay free for route, plan and the dispatch.
int shared_expert_sms(const mok_shape& s);
// SMs the shared expert's backward takes on mok_moe_bwd's side stream
// (0: no side stream, it runs after the routed dX on every SM):
// shape.bwd_shared_sms, at most a third of the SMs.
int bwd_shared_split(const mok_shape& s);

// Device address of a __device__ variable (its host-side stand-in `symbol`)
// on the current device.  cudaGetSymbolAddress is called once per device and
// context: the result is cached with the id of the context it was made in
// and looked up again when another context is current (for instance the new
// primary context after cudaDeviceReset, which reloads the module), so a
// stale address is never handed out.  Null on failure.
struct SymbolCache {
  void* addr[64] = {};
  unsigned long long ctx[64] = {};
};
void* symbol_address(const void* symbol, SymbolCache& cache);

}  // namespace mok
