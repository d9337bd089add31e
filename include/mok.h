/*
 * mok.h -- C ABI of the single-GPU MoE layer (GB300, sm_103a).
 *
 * The layer (Mixture-of-Kittens blog, "Overlapping computation and
 * communication in MoE", the MoE(x, s) equation):
 *
 *   MoE(x, s) = E_shared(x) + sum_{i in topk(s)} g_i E_i(x),
 *   E_i(x)    = W_down_i (SiLU(W_gate_i x) * (W_up_i x)),
 *   g_i       = s_i / sum_{j in topk(s)} s_j.
 *
 * Notation: T tokens, D model dim, I expert intermediate dim, E routed
 * experts, K experts per token, I_shared shared-expert intermediate dim,
 * R = T*K routes.  A route is a (token t, slot k) pair, numbered t*K + k.
 *
 * Conventions for every entry point:
 *  - All matrices are row-major and densely packed (leading dim = row width).
 *    bf16 buffers are IEEE bfloat16 bit patterns; fp32 buffers are IEEE
 *    binary32.  Device pointers unless stated otherwise.
 *  - The caller owns every buffer.  The library never allocates device
 *    memory, never frees, and never synchronises the host, except
 *    mok_get_error(), which synchronises the given stream.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued on it in order; results are valid once the
 *    stream reaches that point.
 *  - Argument errors (null pointers, misalignment, unsupported sizes,
 *    workspace too small) are detected on the host and returned at once;
 *    nothing is enqueued then.  Errors the GPU detects (an expert index
 *    outside [0, E), a pipeline wait that timed out) set a device status
 *    word that mok_get_error() reads and clears.  MOK_ERR_CUDA means a launch
 *    or CUDA runtime call failed.
 *  - Results are bitwise deterministic: every reduction runs in a fixed
 *    order and no floating-point atomics are used.
 *  - Pointers must be 16-byte aligned.  Size rules: D % 256 == 0,
 *    I % 128 == 0, I_shared % 128 == 0, 1 <= K <= min(E, 32), E <= 1024,
 *    T*K < 2^31.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = 1,
  MOK_ERR_UNSUPPORTED = 2,
  MOK_ERR_WORKSPACE = 3,
  MOK_ERR_CUDA = 4,
  MOK_ERR_TIMEOUT = 5,
  MOK_ERR_BAD_ROUTE = 6
} mok_status;

typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1 } mok_dtype;

/* Operation codes for mok_workspace_bytes(). */
typedef enum {
  MOK_OP_PLAN = 0,
  MOK_OP_EXPERT_FFN = 1,
  MOK_OP_SHARED_FFN = 2,
  MOK_OP_FWD = 3,
  MOK_OP_BWD = 4,
  MOK_OP_RING = 5
} mok_op;

/* Layer shape.  I_shared = 0 means no shared expert.  dtype selects the
 * arithmetic of the routed experts (the shared expert is always BF16).
 * chunk_rows: routed rows per dispatch chunk b (the overlap granularity of
 * the Mixture-of-Kittens paper note, "Granularity as a tunable"):
 * 512..32768 = the forward gathers through a ring of 4 chunks that producer
 * warps fill while the up/gate GEMM consumes it (mok_expert_upgate_ring;
 * MXFP8: the producers quantise the rows, their scales going to the grouped
 * layout in full); -1 = the dispatch gathers the whole batch before the
 * expert GEMMs; 0 = automatic: for BF16 the whole-batch dispatch when the
 * layer averages fewer than 512 routed rows per expert (the GEMMs then take
 * the routed rows as the MMA's N and stream weights at HBM speed), else the
 * ring with b = 2048 (measured faster there on a GB300); for MXFP8 the
 * whole-batch quantising dispatch.
 * producer_sms: the split of the GPU between the dispatch (producers) and
 * the shared expert in the first dispatch window (paper note, "The
 * production details": the shared expert fills the first dispatch window).
 * mok_moe_fwd runs the shared expert's launches on a side stream next to
 * route, plan and the dispatch; with producer_sms > 0 those launches take
 * every SM but producer_sms (at least 2), which stay free so that the
 * dispatch runs beside them instead of queueing behind; 0 = the shared
 * expert's launches take every SM.  The same holds for mok_shared_ffn and
 * the shared-only call of mok_expert_upgate.  0..4096.
 * bwd_shared_sms: the split of the GPU in mok_moe_bwd.  The shared expert's
 * backward (its dgrad, dX and three weight gradients) needs only x, dY and
 * its own weights; with bwd_shared_sms > 0 it runs on a side stream on that
 * many SMs (at most a third of them) while the routed experts' dgrad and dX
 * run on the others, and the caller's stream waits for it before the
 * reverse combine, the first launch that reads its output.  0 = no side
 * stream: the shared expert's backward runs after the routed dX on every
 * SM, which measured faster on a GB300 at every split (the routed dgrad and
 * dX lose more bandwidth on fewer SMs than the overlap hides).  0..4096;
 * every setting gives the same bits. */
typedef struct {
  int32_t T, D, I, E, K, I_shared;
  int32_t dtype;
  int32_t chunk_rows;
  int32_t producer_sms;
  int32_t bwd_shared_sms;
} mok_shape;

/* MXFP8 tensors (paper note, "The production details").  A [rows][cols]
 * tensor quantised along cols is E4M3 ("fn") codes [rows][cols] plus E8M0
 * scales, one per 32 consecutive elements of a row.  Element value =
 * code * 2^(scale - 127).  cols must be a multiple of 128.  The scales are
 * 32-bit words [cols/128][ld], ld a multiple of 128: the word of row
 * position p for columns [128 g, 128 g + 128) holds, byte b (the least
 * significant first), the scale of columns [128 g + 32 b, 128 g + 32 b + 32),
 * and sits at index g * ld + (p & ~127) + 4 * (p % 32) + (p % 128) / 32
 * (within each block of 128 positions, position 32 c + l at word 4 l + c: the
 * order the tensor cores read scale blocks in).  Row r has position
 *   plain layout   : p = r, ld = rows rounded up to 128
 *                    (mok_quantize_mxfp8, the weights' sc_*);
 *   grouped layout : rows grouped by expert as mok_plan's offsets (expert e
 *                    owns rows [offsets[e], offsets[e+1])), every expert
 *                    starting a new block: p = 128 (offsets[e] / 128 + e) +
 *                    r - offsets[e], ld = 128 (ceil(rows / 128) + E)
 *                    (the routed activations xg_scale, a_scale).
 * Positions that hold no row are never read for a valid output.
 * mok_mxfp8_scale_bytes gives the size of either layout.
 *
 * Weights (device, bf16 unless noted).  Routed: w_gate, w_up [E][I][D];
 * w_down [E][D][I].  MXFP8 copies (used when shape.dtype = MOK_MXFP8, may be
 * NULL otherwise): q_gate, q_up, q_down codes of the same shapes (as
 * [E*I][D], [E*I][D], [E*D][I] tensors quantised along the last dim) and
 * sc_* their scale words (mok_quantize_mxfp8 writes both).  Shared expert,
 * always BF16: ws_gate, ws_up [I_shared][D]; ws_down [D][I_shared] (NULL
 * when I_shared = 0).  MXFP8 backward (mok_moe_bwd with dtype MOK_MXFP8;
 * may be NULL otherwise), written by mok_quantize_mxfp8_bwd_weights:
 * qt_down the codes of W_down^T [E][I][D] (as [E*I][D] quantised along D)
 * and sct_down its scale words (plain layout); qt_gu the codes of
 * [W_gate^T | W_up^T] [E][D][2I] (as [E*D][2I] quantised along 2I) and
 * sct_gu its scale words. */
typedef struct {
  const void *w_gate, *w_up, *w_down;
  const void *q_gate, *q_up, *q_down;
  const uint8_t *sc_gate, *sc_up, *sc_down;
  const void *ws_gate, *ws_up, *ws_down;
  const void *qt_down;
  const uint8_t *sct_down;
  const void *qt_gu;
  const uint8_t *sct_gu;
  const uint8_t *sc_gu_pair;
} mok_weights;

/* State saved by the forward for the backward.
 * topk_idx int32 [T][K]; g fp32 [T][K]; counts int32 [E]; offsets int32
 * [E+1]; table int32 [R][3]; route_dst int32 [R].
 *
 * act, act_rows (optional; paper note, "A ring buffer instead of a host
 * round-trip": the backward replays only the forward activations it no
 * longer has): a caller-owned fp32 store of act_rows rows of 2I floats.
 * The forward writes h = W_gate x (columns [0, I)) and u = W_up x (columns
 * [I, 2I)), unrounded, for the routed rows of every expert whose rows all
 * lie below act_rows in expert order (offsets[e+1] <= act_rows), at row
 * offsets[e] + j.  The backward reads them for those experts and replays
 * h, u (streaming W_gate and W_up again) only for the others.  act = NULL
 * or act_rows = 0 keeps nothing: the backward replays every expert.  With
 * act_rows >= T*K every expert is kept.  act must be 16-byte aligned and
 * stay untouched between the forward and the backward.
 *
 * act_shared (optional): the same for the shared expert, fp32 [T][2 I_shared]
 * (h in columns [0, I_shared), u in [I_shared, 2 I_shared), row = token);
 * with it the backward's shared dgrad reads h, u there instead of
 * recomputing them from x.  NULL: the backward replays them.  16-byte
 * aligned; ignored when I_shared = 0. */
typedef struct {
  int32_t *topk_idx;
  float *g;
  int32_t *counts, *offsets, *table, *route_dst;
  float *act;
  int64_t act_rows;
  float *act_shared;
} mok_plan_buf;

/* Bytes of caller-provided device workspace `op` needs for `shape`
 * (0 for an invalid shape).  The workspace needs 256-byte alignment. */
size_t mok_workspace_bytes(const mok_shape *shape, int op);

/* Intermediates of mok_moe_bwd that stay in its workspace after the call,
 * for inspection (the pages have no counterpart; the parity tests read
 * them): dh, du and a_g = bf16(g a) of the routed experts, each bf16
 * [T*K][I] in expert order (row = mok_plan's dst). */
typedef enum { MOK_WS_BWD_DH = 1, MOK_WS_BWD_DU = 2, MOK_WS_BWD_AG = 3 } mok_ws_region;
/* Byte offset of `region` in the MOK_OP_BWD workspace of `shape`, or
 * (size_t)-1 for an invalid shape or region.  The contents are those of the
 * last mok_moe_bwd that used the workspace, until the next call writes it. */
size_t mok_workspace_offset(const mok_shape *shape, int region);

/* Top-K routing (blog, "Overlapping computation and communication in MoE":
 * the router selects the top-k routed experts and their weights).
 * s: fp32 [T][E] router weights.  Writes topk_idx int32 [T][K] (descending
 * s, lowest expert index first among equal s) and g fp32 [T][K]
 * (g_k = s_k / (((s_0 + s_1) + s_2) + ...), fp32 sum in k order, IEEE
 * division).  Scores must be finite. */
mok_status mok_route(const float *s, int32_t T, int32_t E, int32_t K,
                     int32_t *topk_idx, float *g, void *stream);

/* Router (blog, "Overlapping computation and communication in MoE": the
 * gate is formed from router weights s over the routed experts).  s =
 * softmax(x W_r^T) over the E experts, x bf16 [T][D], w_router bf16 [E][D],
 * logits summed in fp32 on the tensor cores, the softmax (exp(l - max) /
 * sum, fast exponential, one IEEE reciprocal per row) in the same launch;
 * s fp32 [T][E] is written, then mok_route's top-K and g run on it
 * (topk_idx, g as for mok_route).  E <= 256, else MOK_ERR_UNSUPPORTED. */
mok_status mok_router(const mok_shape *shape, const void *x, const void *w_router, float *s,
                      int32_t *topk_idx, float *g, void *stream);

/* Device-side plan (blog, "Scheduling": the pull schedule with one source
 * rank).  From topk_idx int32 [T][K] writes counts int32 [E] (routes per
 * expert), offsets int32 [E+1] (exclusive scan, offsets[E] = R), table
 * int32 [R][3] (row dst = {src_index = t*K + k, expert, dst}; an expert's
 * routes are contiguous and in ascending t*K + k order) and route_dst int32
 * [R] (route_dst[t*K + k] = dst).  ws: mok_workspace_bytes(MOK_OP_PLAN)
 * bytes of scratch.  An index outside [0, E) sets MOK_ERR_BAD_ROUTE in the
 * device status word; the outputs are then unspecified. */
mok_status mok_plan(const int32_t *topk_idx, int32_t T, int32_t E, int32_t K,
                    int32_t *counts, int32_t *offsets, int32_t *table,
                    int32_t *route_dst, void *ws, size_t ws_bytes, void *stream);

/* mok_plan without caller-provided scratch: the same outputs, computed by
 * the same kernels, for callers that cannot hand over device memory as
 * workspace (their device memory belongs to another allocator they may not
 * call from here, or the code path must not allocate).  The pages have no
 * counterpart to this entry point.
 * The scratch is a fixed 1 MiB array inside the library's device image
 * (held on every GPU that loads the library until the process exits); it
 * allows ceil(T*K / 1024) * E <= 262144, else MOK_ERR_WORKSPACE and nothing
 * is enqueued.  Nothing is allocated.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) and caches it with the
 * id of the current context; a call under another context (after
 * cudaDeviceReset the device gets a new one, and the library's module is
 * reloaded) looks it up again.  Make the first call in each context before
 * any stream capture.  All calls share the one array, so
 * calls that overlap on the GPU (different streams, no ordering between
 * them) race and give wrong plans; order them.  Arguments and errors
 * otherwise as mok_plan. */
mok_status mok_plan_static(const int32_t *topk_idx, int32_t T, int32_t E, int32_t K,
                           int32_t *counts, int32_t *offsets, int32_t *table,
                           int32_t *route_dst, void *stream);

/* The pull schedule with several source ranks on one GPU (blog,
 * "Scheduling": a destination's slots for local expert l are ordered by the
 * per-source ordinal o, then the source rank r (paper note, "Pull dispatch,
 * push combine"); the pages' garbled in-rank position read as
 * p = sum_r' min(M[l][r'], o) + |{r' < r : M[l][r'] > o}|).  The T tokens
 * form `ranks` contiguous virtual source ranks of T / ranks tokens (ranks
 * must divide T); with ranks = 1 this is mok_plan.  Outputs as mok_plan;
 * within each expert the rows follow the round-robin order.  ws:
 * mok_plan_ranks_workspace_bytes(T, E, K, ranks) bytes (0 when invalid). */
size_t mok_plan_ranks_workspace_bytes(int32_t T, int32_t E, int32_t K, int32_t ranks);
mok_status mok_plan_ranks(const int32_t *topk_idx, int32_t T, int32_t E, int32_t K, int32_t ranks,
                          int32_t *counts, int32_t *offsets, int32_t *table, int32_t *route_dst,
                          void *ws, size_t ws_bytes, void *stream);

/* Dispatch (blog, "Scheduling": tokens land expert-contiguous, zero local
 * copies).  xg[p] = x[table[p].src_index / K] for p < R, computed token by
 * token: row t of x is read once and stored at its K positions
 * route_dst[t*K + k] (mok_plan's inverse of the table; BF16 by bulk copies
 * through shared memory, a row piece loaded once and stored K times);
 * x bf16 [T][D], xg bf16 [R][D].  route_dst is required.  With dtype MOK_MXFP8 xg receives
 * the E4M3 codes [R][D] of the dispatched rows and xg_scale their scale
 * words in the grouped layout (quantisation fused into the dispatch, once
 * per token), for which table and offsets (mok_plan's) are required; table,
 * xg_scale and offsets are ignored for BF16. */
mok_status mok_dispatch(const mok_shape *shape, const void *x, const int32_t *table,
                        const int32_t *route_dst, const int32_t *offsets, void *xg, uint8_t *xg_scale,
                        void *stream);

/* Grouped expert FFN over expert-contiguous rows: expert e owns rows
 * [offsets[e], offsets[e+1]) of xg.  a = bf16(SiLU(xg W_gate^T) * (xg W_up^T))
 * [R][I] (written to a_out when non-null, else to the workspace), then
 * yg = bf16(a W_down^T) [R][D].  fp32 accumulation on the tensor cores.
 * MOK_MXFP8: xg / xg_scale are MXFP8 (from mok_dispatch), the weights are
 * q_* / sc_*, a is quantised to MXFP8 along I before the down projection
 * and kept in the workspace (a_out must be NULL); yg stays bf16. */
mok_status mok_expert_ffn(const mok_shape *shape, const mok_weights *w, const void *xg,
                          const uint8_t *xg_scale, const int32_t *offsets, void *a_out,
                          void *yg, void *ws, size_t ws_bytes, void *stream);

/* The two halves of mok_expert_ffn, for callers that schedule them apart.
 * mok_expert_upgate: a = bf16(SiLU(xg W_gate^T) * (xg W_up^T)) [R][I].
 * mok_expert_down: yg = bf16(a W_down^T) [R][D].  Same rules as
 * mok_expert_ffn.  For MOK_MXFP8, a is written as codes [R][I] plus scale
 * words a_scale (grouped layout) and read back that way by
 * mok_expert_down; xg_scale / a_scale are ignored for BF16.
 * Shared expert in the same launch (paper note, "The production details":
 * the shared expert fills compute while routed rows stream): when
 * shape.I_shared > 0 and x_shared / a_shared (resp. a_shared / ys) are
 * non-NULL, the shared expert's up/gate (x_shared bf16 [T][D] -> a_shared
 * bf16 [T][I_shared]) or down (a_shared -> ys bf16 [T][D]) tiles are spread
 * through the routed launch (BF16; after the routed launch for MXFP8).
 * mok_expert_upgate with xg, offsets and a all NULL runs the shared
 * expert's up/gate alone (x_shared -> a_shared), e.g. on a second stream
 * while the routing, plan and dispatch run. */
mok_status mok_expert_upgate(const mok_shape *shape, const mok_weights *w, const void *xg,
                             const uint8_t *xg_scale, const int32_t *offsets, void *a,
                             uint8_t *a_scale, const void *x_shared, void *a_shared, void *stream);
/* mok_expert_upgate with the dispatch fused in as a ring (BF16; blog,
 * "Scheduling": rows land expert-contiguous with no second local copy;
 * paper note, "Granularity as a tunable" and "A ring buffer instead of a
 * host round-trip").  Routed row p (expert order) is x[table[p].src_index /
 * K], x bf16 [T][D], table mok_plan's [R][3].  Inside the same launch,
 * warps 2 and 3 of every CTA are producers: chunk by chunk (b =
 * shape.chunk_rows routed rows, 0 or -1 = 2048) they copy their share of the
 * chunk's rows into a ring of 4 chunks in `ws` with coalesced 16-byte vector
 * loads and stores and count themselves in on a per-chunk device counter.
 * Before loading a tile's rows the GEMM's TMA warp waits for their chunks;
 * once a tile's loads have landed its MMA thread counts the rows as read, and
 * a producer refills a slot only after every N tile has read the chunk it
 * holds.  All waits are bounded (MOK_ERR_TIMEOUT on expiry) and the launch
 * is cooperative, so producers and consumers are resident together.
 * a bf16 [R][I], bit-identical to mok_dispatch followed by mok_expert_upgate.
 * ws: mok_workspace_bytes(MOK_OP_RING) bytes (the ring, 4 b + 128 rows of
 * D bf16, and 2 ceil(R / b) counters), 256-byte aligned. */
mok_status mok_expert_upgate_ring(const mok_shape *shape, const mok_weights *w, const void *x,
                                  const int32_t *table, const int32_t *offsets, void *a, void *ws,
                                  size_t ws_bytes, void *stream);
mok_status mok_expert_down(const mok_shape *shape, const mok_weights *w, const void *a,
                           const uint8_t *a_scale, const int32_t *offsets, void *yg,
                           const void *a_shared, void *ys, void *stream);

/* Shared expert (paper note, "The production details": kept in BF16).
 * ys = bf16(W_sd bf16(SiLU(W_sg x) * (W_su x))) [T][D]. */
mok_status mok_shared_ffn(const mok_shape *shape, const mok_weights *w, const void *x,
                          void *ys, void *ws, size_t ws_bytes, void *stream);

/* Combine (blog layer equation; paper note "The production details":
 * fixed-order reduction).  out[t] = bf16(ys[t] + sum_{k=0..K-1}
 * g[t,k] * yg[route_dst[t*K+k]]), fp32 accumulation in that order.  ys may
 * be NULL (no shared expert); g may be NULL (all weights 1). */
mok_status mok_combine(const mok_shape *shape, const void *yg, const void *ys, const float *g,
                       const int32_t *route_dst, void *out, void *stream);

/* Whole forward: route -> plan -> dispatch -> shared FFN -> grouped FFN ->
 * combine.  x bf16 [T][D]; s fp32 [T][E]; out bf16 [T][D].  Ordered on
 * `stream` as one operation: the shared expert's up/gate (and, for MXFP8,
 * its down projection) runs on an internal side stream (one per device and
 * host thread, created on first use), forked from `stream` after the work
 * already queued there, beside route, plan and the dispatch, and joined
 * back before the routed up/gate (BF16 with the whole-batch dispatch) or
 * before its output is read (otherwise).  `saved`
 * (nullable) receives the routing and plan for mok_moe_bwd.  With
 * shape.dtype = MOK_MXFP8 the routed experts run in MXFP8 (dispatch
 * quantises x, the up/gate epilogue quantises a) and the shared expert in
 * BF16.  The forward gathers through a ring instead of a whole-batch
 * dispatch as shape.chunk_rows says. */
mok_status mok_moe_fwd(const mok_shape *shape, const mok_weights *w, const void *x,
                       const float *s, void *out, mok_plan_buf *saved, void *ws,
                       size_t ws_bytes, void *stream);

/* Backward of L = <dy, MoE(x, s)>.  saved: the forward's routing and
 * plan.  dy bf16 [T][D].  Writes dx bf16 [T][D]; dw_gate, dw_up bf16
 * [E][I][D]; dw_down bf16 [E][D][I]; dws_* the shared expert's (ignored
 * when I_shared = 0); ds fp32 [T][E] (zero outside the top-k);
 * dg fp32 [T][K] (nullable) = <t, a> per route with t = W_down^T dy (paper
 * note, "The production details": the router-gradient inner product; the
 * down-projection output is not formed).  h and u are read from saved->act
 * for the experts the forward kept there and recomputed for the rest.  Weight
 * gradients of experts with no routes are written as zeros.
 * With shape.dtype = MOK_MXFP8 the routed experts' replay (h, u), t and dX
 * products run in MXFP8, each operand quantised along that product's
 * reduction dim (x, dY per row along D; w's q_gate, q_up, qt_down; the
 * activation gradient quantises [dh | du] along 2I for qt_gu); h, u and t
 * stay fp32 between the products and the activation gradient.  The
 * weight gradients are BF16 products (of bf16 x, dY, dh, du, g a) and the
 * shared expert is BF16.  MXFP8 needs I % 256 == 0 (the t and dX products
 * run on 256-column tiles; MOK_ERR_UNSUPPORTED otherwise) and w's q_* and
 * qt_* copies (MOK_ERR_INVALID_ARG without them).  With
 * shape.bwd_shared_sms > 0 the shared expert's backward runs on the side
 * stream of mok_moe_fwd, on mok_bwd_shared_sms SMs, while the routed dgrad
 * and dX take the others; the caller's stream waits for it before the
 * reverse combine, so on return all work is queued on `stream` as for a
 * single-stream call. */
mok_status mok_moe_bwd(const mok_shape *shape, const mok_weights *w, const void *x,
                       const float *s, const mok_plan_buf *saved, const void *dy, void *dx,
                       void *dw_gate, void *dw_up, void *dw_down, void *dws_gate,
                       void *dws_up, void *dws_down, float *ds, float *dg, void *ws,
                       size_t ws_bytes, void *stream);

/* SMs that mok_moe_bwd gives the shared expert's backward on its side
 * stream on the current device: shape.bwd_shared_sms, at most a third of the
 * SMs; 0 when the backward runs without a side stream (I_shared = 0, T = 0,
 * or shape.bwd_shared_sms under 2); -1 for an invalid shape.  Host-only. */
int32_t mok_bwd_shared_sms(const mok_shape *shape);

/* Bytes of MXFP8 scale storage for a [rows][cols] tensor: plain layout
 * when groups = 0, grouped layout over `groups` experts otherwise (see the
 * MXFP8 layout above).  0 for invalid sizes (cols not a positive multiple
 * of 128, negative rows or groups).  Host-only. */
size_t mok_mxfp8_scale_bytes(int64_t rows, int64_t cols, int32_t groups);

/* The MXFP8 routed up/gate with the routed rows as the MMA's N dimension
 * (no padding rows in its MMAs; used when w->sc_gu_pair is given and the
 * experts average fewer than 512 routed rows) takes each CTA's A operand as
 * 64 W_up rows followed by the same 64 W_gate rows, whose scales it reads
 * from one 512-byte block of this paired copy: block b of expert e =
 * b / (I/64), s = b % (I/64), holds the scale words of W_up rows 64 s ..
 * 64 s + 63 and then of the same W_gate rows, in the plain layout of 2 E I
 * rows (the block order of the 32x128b copy).  Writes sc_gu_pair
 * (mok_mxfp8_scale_bytes(2*E*I, D, 0) bytes) from w->sc_gate and w->sc_up
 * (mok_quantize_mxfp8's words); a permutation, no arithmetic.  Weights are
 * parameters: call once after quantising them.  The pages have no
 * counterpart; the layout serves the tensor cores' scale placement.  The
 * routed-rows-as-N up/gate gives the row-major one's bytes; on a GB300 it
 * measured slower (DSV3 MXFP8 up/gate 1.89 vs 1.55 ms): its quantising
 * epilogue holds the single accumulator longer than the MMAs it saves. */
mok_status mok_mxfp8_pair_scales(const mok_shape *shape, const mok_weights *w, uint8_t *sc_gu_pair,
                                 void *stream);

/* The MXFP8 weight copies of the backward, from the bf16 w_gate, w_up,
 * w_down of `w`: qt_down = codes of W_down^T [E][I][D] quantised along D
 * (E*I*D bytes) with sct_down (mok_mxfp8_scale_bytes(E*I, D, 0) bytes);
 * qt_gu = codes of [W_gate^T | W_up^T] [E][D][2I] quantised along 2I
 * (E*D*2I bytes) with sct_gu (mok_mxfp8_scale_bytes(E*D, 2I, 0) bytes).
 * Same rounding as mok_quantize_mxfp8.  D and I multiples of 128. */
mok_status mok_quantize_mxfp8_bwd_weights(const mok_shape *shape, const mok_weights *w, void *qt_down,
                                          uint8_t *sct_down, void *qt_gu, uint8_t *sct_gu, void *stream);

/* MXFP8 quantiser: src bf16 [rows][cols] (cols % 128 == 0) -> q E4M3 codes
 * [rows][cols] and scale words in the plain layout (see the MXFP8 layout
 * above; mok_mxfp8_scale_bytes(rows, cols, 0) bytes).  Per 1x32 block the
 * scale is 2^e with e the smallest integer such that amax <= 448 * 2^e
 * (all-zero block: byte 0); codes round to nearest even. */
mok_status mok_quantize_mxfp8(const void *src, int64_t rows, int64_t cols, void *q,
                              uint8_t *scale, void *stream);

/* Failure-detection check (no counterpart on the pages).  Enqueues on
 * `stream` one pipeline wait on an mbarrier that nothing arrives on and one
 * ring-counter wait on a counter that nothing increments: both give up after
 * the 2 s budget of every device wait and record MOK_ERR_TIMEOUT, which the
 * next mok_get_error returns; the GPU context stays usable.  About 4 s of
 * one thread's time; no fault, trap or hang. */
mok_status mok_check_wait_timeout(void *stream);

/* Synchronises `stream`, returns the device status word of the current
 * device (MOK_OK, MOK_ERR_BAD_ROUTE or MOK_ERR_TIMEOUT) and clears it. */
mok_status mok_get_error(void *stream);

/* Static description of a status code. */
const char *mok_status_string(mok_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOK_H */
