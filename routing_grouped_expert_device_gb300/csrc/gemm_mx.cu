// MXFP8 grouped expert GEMMs on CTA pairs (Mixture-of-Kittens paper note,
// "The production details": MXFP8 with quantisation fused into the
// dispatch, the grouped GEMMs and the gated activation).
//
// Operands are E4M3 codes with one E8M0 scale per 1x32 block along K, scale
// words in 128-row blocks (layout in kernels.h): the A operand (routed rows)
// in the grouped layout, in which every expert starts a new block, and the
// weights in the plain layout.
//
// A cluster of two CTAs computes a 256-row x 256-column tile as the BF16
// pair kernel does: CTA rank r loads its 128 rows of A and one half of B
// (up/gate: rank 0 the 128 W_gate rows, rank 1 the 128 W_up rows; down:
// output columns [128 r, 128 r + 128)), and the leader issues
// cta_group::2 block-scaled MMAs (M 256, N 256, K 32, four per 128-column
// stage).  Per stage each CTA also loads three scale blocks of 512 B: its
// own 128 rows of A, and B's two halves (every CTA needs the scales of all
// 256 B rows).  All loads of both CTAs complete on the leader's
// full[stage]; the MMA thread then copies the three blocks into a TMEM ring
// with tcgen05.cp (each CTA from its own shared memory) and issues the four
// MMAs, which read
//   A row m : lane m (own 128 rows), column sfa + m / 32
//   B row n : lane 32 q + n % 32 for every quarter q, column sfb + n / 32
// with the byte of the 32-bit scale word chosen by the MMA's scale id.
// The copy and the MMAs that follow it from the same thread execute in
// order; the ring slot of a stage is refilled only after the MMAs that read
// it have committed (the stage's empty barrier), as for its shared memory.
//
// up/gate : the epilogue forms a = bf16(SiLU(h) u) and quantises it to E4M3
//           per 32 columns (one TMEM load of 32 columns is one block),
//           writing a's scale words in the grouped layout.
// replay  : the up/gate products of the backward, h and u written as fp32.
// down    : y = bf16(acc), or the fp32 accumulator (the backward's t).
#include <cuda_fp8.h>

#include "gemm_core.cuh"
#include "kernels.h"
#include "mx_quant.cuh"
#include "pair.cuh"

namespace mok {
namespace {

constexpr int BKB = 128;  // K columns (bytes) of one K block: one 128-byte swizzled box
// The quantising up/gate keeps three stages of two K blocks (eight MMAs per
// stage: the MMA thread's wait, fences and commit per stage cost about a
// third of one K block's MMA time; six stages of one K block took 1.55 ms
// at DSV3 size against 1.47-1.49 ms), and so do the modes that store their
// output straight from registers: fp32 (t, the replay) and the bf16 down
// and dX with the routed rows as N, each warp store 32 consecutive columns
// of one row.  The row-major bf16 down keeps four stages of one K block and
// uses 64 KB per CTA to drain the accumulator into shared memory, so that
// it is free for the next tile's MMAs while TMA stores write the tile out.
constexpr int kMaxStages = 3;
constexpr int STAGING_BYTES = 4 * 4 * 4096;  // 4 lane quarters x 4 boxes of 32 rows x 64 bf16
// The quantising up/gate with the routed rows as N passes u from the warps
// that drain it to the warps that drain h through shared memory: 32 rows x
// 32 columns of fp32 for each of the 2 x 2 (column half, lane-quarter pair)
// warp pairs.
constexpr int XCH_BYTES = 4 * 32 * 32 * 4;
// `staged`: the modes that drain a bf16 tile through STAGING_BYTES of
// shared memory
__host__ __device__ constexpr int mx_stages(bool staged) { return staged ? 4 : kMaxStages; }
// K blocks (of BKB bytes) per stage
__host__ __device__ constexpr int mx_ksub(bool staged) { return staged ? 1 : 2; }
constexpr int A_BYTES = 128 * BKB;  // this CTA's 128 rows, one K block
constexpr int B_BYTES = 128 * BKB;  // this CTA's half of B, one K block
constexpr int CODE_BYTES = A_BYTES + B_BYTES;
constexpr int SF_BLOCK = 512;           // one 128-row block of scale words
constexpr int SF_BYTES = 3 * SF_BLOCK;  // A's block, B's two halves (one K block)
constexpr uint32_t ACC_COLS = 256;
constexpr uint32_t SF_COLS = 12;  // per K block: A 4, B 8
// Eight epilogue warps: warps 4 + 4h + q drain TMEM lane quarter q (the
// hardware ties a warp to quarter warp % 4), columns of half h of the
// accumulator, so each warp holds the accumulator for half as long.
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 128 + EPI_WARPS * 32;

// Block-scaled instruction descriptor, kind::mxf8f6f4: B scale id (bits
// 4-5), A and B format E4M3 = 0 (7-9, 10-12), both K-major, N >> 3 (17-22),
// scale format UE8M0 (23), M >> 4 (24-28), A scale id (29-30).
__device__ __forceinline__ uint32_t idesc_mx(uint32_t sf_id, uint32_t n = 256) {
  return (sf_id << 4) | ((n >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mx2(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

struct MxParams {
  SchedArgs sched;  // bm = 256
  int* status;
  CUtensorMap tmA;    // codes [rows][K] u8, box 128 x 128
  CUtensorMap tmSA;   // A scale words, grouped layout [K/128][lda], box 128 x 1
  CUtensorMap tmB0;   // codes [G*NB][K], box 128 x 128
  CUtensorMap tmB1;
  CUtensorMap tmSB0;  // scale words of B0, plain layout [K/128][G*NB], box 128 x 1
  CUtensorMap tmSB1;  // scale words of B1
  int32_t b_group_rows, b_tile_rows, b1_off;
  uint8_t* aq;    // up/gate: a codes [rows][I]
  uint32_t* asc;  // up/gate: a scale words, grouped layout [I/128][a_ld]
  int64_t a_ld;
  __nv_bfloat16* y;  // down: y [rows][D]
  __nv_bfloat16* h_out;  // bf16 replay outputs h, u [rows][I] (unused: the replay stores fp32)
  __nv_bfloat16* u_out;
  float* h32;  // kF32: replay h, u [rows][I], or y [rows][D]
  float* u32;
  float* y32;
  float* act;  // up/gate: kept h, u fp32 [rows][2 out_ld] of groups ending at or below act_rows
  int32_t act_rows;
  // up/gate with the routed rows as N: W_up, W_gate codes in 64-row boxes
  // and the paired scale blocks (mok_mxfp8_pair_scales: block b of expert
  // e = b / (I / 64) holds the scale words of W_up rows 64 s .. 64 s + 63
  // and then of the same W_gate rows, s = b % (I / 64))
  CUtensorMap tmU64, tmG64, tmSP;
  int32_t out_ld;
  // bf16 outputs as [rows][out_ld], boxes 32 rows x 64 columns, 128-byte
  // swizzle: y (down), or h and u (replay)
  CUtensorMap tmO0, tmO1;
  // Ring dispatch (kRing, the row-major quantising up/gate): tmA maps the
  // ring of codes, [ring_rows + 128][D]; routed row r sits at ring row
  // r % ring_rows (ring rows 0..127 repeated after the end, so no 128-row
  // box wraps), and its scale words go to the grouped layout that tmSA
  // maps (xsc, ld xs_ld), in full.
  const uint4* x;         // [T][D] bf16, as 16-byte vectors
  const int32_t* table;   // the plan's [R][3]
  int32_t K, D8;          // top-k; D / 8
  uint2* ring;            // codes, 8 per uint2
  uint32_t* xsc;
  int64_t xs_ld, ring_rows;
  int32_t chunk_rows, nchunks, n_tiles;
  int32_t* ready;         // [nchunks]: producer warps done with the chunk
  int32_t* done;          // [nchunks]: (row, N tile) reads of the chunk completed
};

// ---------------------------------------------------------------------------
// Ring dispatch with the quantisation in the producers (Mixture-of-Kittens
// paper note, "The production details": MXFP8 quantisation fused into the
// dispatch; "Granularity as a tunable": chunks of b rows signalled through
// device counters).  Warps 2 and 3 of every CTA take chunk after chunk of b
// routed rows in expert order: producer warp w quantises rows w, w + np, ...
// of the chunk from x[table[r].src / K] (the dispatch's per-row rule) into
// ring row r mod ring_rows and the row's grouped scale position, fences the
// generic-to-async proxy and release-increments ready[c].  Before writing
// chunk c it waits until chunk c - slots (same ring slot) has been read by
// every N tile.  All CTAs are resident (cooperative launch); every wait is
// bounded.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int mx_chunk_rows(const MxParams& P, int c) {
  const int64_t r0 = static_cast<int64_t>(c) * P.chunk_rows;
  const int64_t R = P.sched.m_total;
  return static_cast<int>((r0 + P.chunk_rows < R ? r0 + P.chunk_rows : R) - r0);
}

__device__ void mx_ring_produce(const MxParams& P, int pw, int np, int lane, volatile int* abort) {
  const int64_t slots = P.ring_rows / P.chunk_rows;
  const int D8 = P.D8;
  for (int c = 0; c < P.nchunks; ++c) {
    if (c >= slots) {
      bool ok = true;
      if (lane == 0)
        ok = wait_count(P.done + (c - slots), mx_chunk_rows(P, c - static_cast<int>(slots)) * P.n_tiles, abort,
                        P.status, SITE_RING_SLOT);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    }
    const int64_t r0 = static_cast<int64_t>(c) * P.chunk_rows;
    const int64_t r1 = r0 + mx_chunk_rows(P, c);
    for (int64_t r = r0 + pw; r < r1; r += np) {
      const int src = __ldg(P.table + r * 3) / P.K;
      const int e = __ldg(P.table + r * 3 + 1);
      const int64_t off = __ldg(P.sched.offsets + e);
      const int64_t pos = mx_scale_pos(mx_group_row0(off, e) + (r - off));
      const uint4* in = P.x + static_cast<int64_t>(src) * D8;
      const int64_t q = r % P.ring_rows;
      uint2* out = P.ring + q * D8;
      uint2* mirror = q < 128 ? P.ring + (P.ring_rows + q) * D8 : nullptr;
#pragma unroll 1
      for (int v0 = 0; v0 < D8; v0 += 128) {  // 4 passes of 256 columns in flight
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int vi = v0 + 32 * u + lane;
          v[u] = vi < D8 ? ld_nc_v4(in + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int vi = v0 + 32 * u + lane;
          if (v0 + 32 * u >= D8) break;  // warp-uniform: D is a multiple of 128 (16 vectors)
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          float f[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16lo(w[j]);
            f[2 * j + 1] = bf16hi(w[j]);
          }
          int ex;
          const uint2 codes = mx_codes8(f, ex);
          const uint32_t word = mx_word16(ex, lane);
          out[vi] = codes;
          if (mirror) mirror[vi] = codes;
          if ((lane & 15) == 0) P.xsc[static_cast<int64_t>(vi / 16) * P.xs_ld + pos] = word;
        }
      }
    }
    // the chunk's rows of this warp are written: visible to the consumers'
    // TMA (async proxy) reads, then this warp is counted in
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0) red_release_add(P.ready + c, 1);
  }
}

// Rows [max(r0, g0), min(r0 + 128, g1)) of a 128-row box that lie inside its
// group [g0, g1): their chunks, and per chunk the count of those rows.
template <class F>
__device__ __forceinline__ void mx_box_chunks(const MxParams& P, int64_t r0, int64_t g0, int64_t g1, F f) {
  const int64_t v0 = r0 > g0 ? r0 : g0;
  const int64_t v1 = r0 + 128 < g1 ? r0 + 128 : g1;
  for (int64_t v = v0; v < v1;) {
    const int c = static_cast<int>(v / P.chunk_rows);
    const int64_t e = (static_cast<int64_t>(c) + 1) * P.chunk_rows < v1 ? (static_cast<int64_t>(c) + 1) * P.chunk_rows : v1;
    f(c, static_cast<int>(e - v));
    v = e;
  }
}

// kT with kSwiglu (the quantising up/gate): A is the tile's 64 W_up rows
// (A rows 0-63) and the same 64 W_gate rows (64-127) of this CTA's half of
// the tile's 128 I columns, with their paired scale block; TMEM lane
// quarters 0, 1 then hold u and 2, 3 the matching h, one column per routed
// row.  The u warps pass their chunk to the h warps through shared memory;
// the h warps form a = bf16(SiLU(h) u), find each row's amax over their 32
// columns (one 1x32 block of a) with a transposing butterfly, and write the
// codes (32 bytes of a row per warp) and the scale byte of their block.
//
// kT (the forms with bf16 outputs: down, replay): the routed rows are the
// MMA's N dimension.  A is 128 weight rows per CTA with the scale block of
// those rows (down: rows 128 r .. of the tile's 256 W_down rows; replay:
// the tile's 128 W_gate rows in CTA 0 and the same W_up rows in CTA 1, so
// CTA 0 produces h and CTA 1 u), B is half of the tile's N routed rows per
// CTA, and B's scales are the two grouped 128-row blocks of the tile (every
// CTA copies both); N = the tile's rows rounded up to 16, so the padding
// rows of a group's last tile cost no MMA work.  The epilogue transposes
// each 32-row chunk into two boxes.
//
// kF32 (forms with bf16 outputs): the accumulator is stored unrounded as
// fp32 (h32 / u32 for the replay, y32 for down) straight from registers;
// in the transposed form each warp store writes 32 consecutive columns of
// one row (128 bytes), in the row-major form each thread 128 bytes of its
// row.
//
// kRing (the row-major quantising up/gate): A's codes come from the ring
// that warps 2 and 3 of every CTA fill (mx_ring_produce); the TMA warp waits
// for the chunks a tile's rows lie in, and the MMA thread counts the rows
// as read once the tile's last stage has landed.
template <bool kSwiglu, bool kReplay = false, bool kT = false, bool kF32 = false, bool kRing = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_mx_pair_persistent(const __grid_constant__ MxParams P) {
  static_assert(!kRing || (kSwiglu && !kReplay && !kT && !kF32), "the ring feeds the row-major up/gate");
  constexpr bool kBf16Out = !kSwiglu || kReplay;
  constexpr bool kSwigluT = kT && kSwiglu && !kReplay;
  static_assert(!kF32 || kBf16Out, "fp32 outputs replace the bf16 ones");
  // the bf16 down / dX with the routed rows as N store from registers too
  constexpr bool kDirect16 = kT && kBf16Out && !kF32 && !kReplay;
  constexpr bool kStaged = kBf16Out && !kF32 && !kDirect16;  // bf16 tiles drained through shared memory
  static_assert(!kT || kSwigluT || kDirect16 || kF32, "the transposed down and replay store from registers");
  constexpr int STAGES = mx_stages(kStaged);
  // a stage holds KSUB K blocks: A's KSUB boxes, then B's, then KSUB sets of
  // three scale blocks, copied to KSUB sets of SF_COLS TMEM columns
  constexpr int KSUB = mx_ksub(kStaged);
  constexpr int STAGE_CODE = KSUB * CODE_BYTES;
  constexpr int STAGE_SF = KSUB * SF_BYTES;
  constexpr uint32_t STAGE_TX = 2 * (STAGE_CODE + STAGE_SF);
  constexpr uint32_t STAGE_SF_COLS = KSUB * SF_COLS;
  static_assert(ACC_COLS + STAGES * STAGE_SF_COLS <= 512, "accumulator and scale ring in TMEM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sf_smem = smem + STAGES * STAGE_CODE;
  uint8_t* staging = sf_smem + STAGES * STAGE_SF;  // 1024-byte aligned; STAGING_BYTES when kStaged
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + (kStaged ? STAGING_BYTES : (kSwigluT ? XCH_BYTES : 0)));
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* total_holder = reinterpret_cast<int*>(tmem_holder + 2);
  int* tstart = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * EPI_WARPS * 32);  // both CTAs' epilogue threads
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc2(tmem_holder, 512);
  if (warp == 3) {
    const int total = build_tile_table(P.sched, tstart, lane);
    if (lane == 0) *total_holder = total;
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_parity[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false;
      bool ok = true;
      const CUtensorMap* tmB = rank ? &P.tmB1 : &P.tmB0;
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileCoord c = walk.at(tile);
        const int local0 = c.mt * 256 + static_cast<int>(rank) * 128;  // this CTA's first row in the group
        const int arow = c.row0 + local0;
        const int sfrow = static_cast<int>(mx_group_row0(c.row0, c.g)) + local0;  // a multiple of 128
        const int brow0 = c.g * P.b_group_rows + c.nt * P.b_tile_rows;
        const int brow = brow0 + (rank ? P.b1_off : 0);
        int ay = arow;
        if (kRing) {
          // this CTA's rows of the tile must be in the ring
          mx_box_chunks(P, arow, c.row0, static_cast<int64_t>(c.row0) + c.rows, [&](int ch, int) {
            if (ok) ok = wait_count(P.ready + ch, 2 * static_cast<int>(gridDim.x), abort_flag, P.status, SITE_RING_CHUNK);
          });
          if (!ok) break;
          fence_proxy_async_global();
          ay = static_cast<int>(arow % P.ring_rows);
        }
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], STAGE_TX);
          const uint32_t lbar = map_to_rank(smem_u32(&full[stage]), 0);
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
          const int kk = kb * KSUB + sub;  // the K block
          uint8_t* st = smem + stage * STAGE_CODE + sub * A_BYTES;  // A of K block kk; B at + KSUB A_BYTES
          uint8_t* sf = sf_smem + stage * STAGE_SF + sub * SF_BYTES;
          if (kSwigluT) {
            // A: 64 W_up rows then the same 64 W_gate rows (this CTA's half of
            // the tile's I columns) with their paired scale block; B: half of
            // the tile's routed rows, scales from the tile's two grouped blocks
            const int urow = brow0 + static_cast<int>(rank) * 64;
            const int xrow = c.row0 + c.mt * 256 + static_cast<int>(rank) * (t_ncols(c) / 2);
            const int gb = static_cast<int>(mx_group_row0(c.row0, c.g)) + c.mt * 256;
            const int pblk = (brow0 / 64 + static_cast<int>(rank)) * 128;  // virtual row of the paired block
            tma_load_2d_pair(st, &P.tmU64, kk * BKB, urow, lbar);
            tma_load_2d_pair(st + 64 * BKB, &P.tmG64, kk * BKB, urow, lbar);
            tma_load_2d_pair(st + KSUB * A_BYTES, &P.tmA, kk * BKB, xrow, lbar);
            tma_load_2d_pair(sf, &P.tmSP, pblk, kk, lbar);
            tma_load_2d_pair(sf + SF_BLOCK, &P.tmSA, gb, kk, lbar);
            tma_load_2d_pair(sf + 2 * SF_BLOCK, &P.tmSA, gb + 128, kk, lbar);
          } else if (kT) {
            // this CTA's weight rows (A): down rows 128 r .. of the tile, replay
            // the tile's rows of W_gate (CTA 0) or W_up (CTA 1)
            const int wrow = brow0 + (kReplay ? 0 : static_cast<int>(rank) * 128);
            const int xrow = c.row0 + c.mt * 256 + static_cast<int>(rank) * (t_ncols(c) / 2);
            const int gb = static_cast<int>(mx_group_row0(c.row0, c.g)) + c.mt * 256;  // the tile's scale blocks
            tma_load_2d_pair(st, kReplay ? tmB : &P.tmB0, kk * BKB, wrow, lbar);
            tma_load_2d_pair(st + KSUB * A_BYTES, &P.tmA, kk * BKB, xrow, lbar);
            tma_load_2d_pair(sf, kReplay && rank ? &P.tmSB1 : &P.tmSB0, wrow, kk, lbar);
            tma_load_2d_pair(sf + SF_BLOCK, &P.tmSA, gb, kk, lbar);
            tma_load_2d_pair(sf + 2 * SF_BLOCK, &P.tmSA, gb + 128, kk, lbar);
          } else {
            tma_load_2d_pair(st, &P.tmA, kk * BKB, ay, lbar);
            tma_load_2d_pair(st + KSUB * A_BYTES, tmB, kk * BKB, brow, lbar);
            tma_load_2d_pair(sf, &P.tmSA, sfrow, kk, lbar);
            tma_load_2d_pair(sf + SF_BLOCK, &P.tmSB0, brow0, kk, lbar);
            tma_load_2d_pair(sf + 2 * SF_BLOCK, &P.tmSB1, brow0 + P.b1_off, kk, lbar);
          }
          }
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && leader) {
        for (int i = 0; i < STAGES; ++i) {
          if (!issued[i]) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(&full[i], issued_parity[i]) && globaltimer() - t0 < kWaitBudgetNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- scale copies + MMA issuer (leader only) ----------------
    if (leader) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, any = false;
      int it = 0;
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
        const TileCoord c = walk.at(tile);
        const uint32_t ncols = kT ? static_cast<uint32_t>(t_ncols(c)) : 256u;
        ok = __all_sync(0xffffffffu, mbar_wait(tempty, (it & 1) ^ 1, abort_flag, P.status, SITE_MMA));
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < c.kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA));
          if (!ok) break;
          tc_fence_after();
          if (kRing && kb == c.kblocks - 1 && lane == 0) {
            // every load of this tile (both CTAs) has landed: its ring rows
            // are read for this N tile
            for (int h = 0; h < 2; ++h)
              mx_box_chunks(P, static_cast<int64_t>(c.row0) + c.mt * 256 + h * 128, c.row0,
                            static_cast<int64_t>(c.row0) + c.rows, [&](int ch, int n) { red_release_add(P.done + ch, n); });
          }
          if (lane == 0) {
#pragma unroll
            for (int sub = 0; sub < KSUB; ++sub) {
              const uint32_t sft = tmem_base + ACC_COLS + stage * STAGE_SF_COLS + sub * SF_COLS;
              const uint32_t sfs = smem_u32(sf_smem + stage * STAGE_SF + sub * SF_BYTES);
              tmem_cp_block2(sft, sfs);                     // A: columns sft .. sft + 3
              tmem_cp_block2(sft + 4, sfs + SF_BLOCK);      // B rows 0..127: sft + 4 .. sft + 7
              tmem_cp_block2(sft + 8, sfs + 2 * SF_BLOCK);  // B rows 128..255: sft + 8 .. sft + 11
              const uint32_t a = smem_u32(smem + stage * STAGE_CODE + sub * A_BYTES);
              const uint32_t b = a + KSUB * A_BYTES;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_mx2(tmem_base, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(b + k * 32, 16, 1024),
                        idesc_mx(k, ncols), sft, sft + 4, (kb | sub | k) != 0);
            }
            commit2(&empty[stage], 0x3);
            any = true;
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if (lane == 0) commit2(tfull, 0x3);
        __syncwarp();
      }
      any = __shfl_sync(0xffffffffu, any, 0);
      if (any) {
        if (lane == 0) commit2(drain, 0x1);
        __syncwarp();
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitBudgetNs) {
        }
      }
    }
  } else if (kRing && (warp == 2 || warp == 3)) {
    // ---------------- ring producers (every CTA: warps 2 and 3) ----------------
    mx_ring_produce(P, static_cast<int>(blockIdx.x) * 2 + (warp - 2), 2 * static_cast<int>(gridDim.x), lane,
                    abort_flag);
  } else if (kSwigluT && warp >= 4) {
    // ---------------- epilogue, quantising up/gate with the routed rows as N ----------------
    // Warp 4 + 4 h + q: TMEM lane quarter q, accumulator columns (routed
    // rows) [128 h, 128 h + 128).  Quarters 0, 1 hold u of I columns
    // i0 + 64 r + 32 q + lane, quarters 2, 3 h of the same columns; warp
    // pair (q & 1, half) meets at named barrier 4 + 2 half + (q & 1).
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const bool hwarp = q >= 2;
    const int pair = 2 * half + (q & 1);
    float* xb = reinterpret_cast<float*>(staging) + pair * 1024;  // [32 rows][32 columns]
    const uint32_t pbar = 4 + pair;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      bool ok = __all_sync(0xffffffffu, mbar_wait(tfull, it & 1, abort_flag, P.status, SITE_EPILOGUE));
      ok = named_bar_and(3, 256, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int nrows = min(c.rows - c.mt * 256, 256);
      const int64_t row0 = c.row0 + c.mt * 256;
      const int icol = c.nt * 128 + static_cast<int>(rank) * 64 + 32 * (q & 1) + lane;  // this lane's I column
      const int ch0 = 4 * half;
      const int ch_end = min((t_ncols(c) + 31) / 32, ch0 + 4);
      const bool keep = P.act && c.row0 + c.rows <= P.act_rows;
      float* kept = keep ? P.act + row0 * (2 * P.out_ld) + (hwarp ? 0 : P.out_ld) + icol : nullptr;
      // the scale word of grouped row g, byte of this warp pair's 32-column block
      uint8_t* scb = reinterpret_cast<uint8_t*>(P.asc + static_cast<int64_t>(c.nt) * P.a_ld) +
                     (2 * static_cast<int>(rank) + (q & 1));
      const int64_t grow0 = mx_group_row0(c.row0, c.g) + c.mt * 256;
#pragma unroll 1
      for (int ch = ch0; ch < ch_end; ++ch) {
        const int nv = min(nrows - ch * 32, 32);  // valid rows of the chunk (at least 1)
        uint32_t v[32];
        tmem_ld32(taddr + ch * 32, v);
        tmem_ld_wait();
        if (keep) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) kept[static_cast<int64_t>(ch * 32 + j) * (2 * P.out_ld)] = __uint_as_float(v[j]);
        }
        if (!hwarp) {
#pragma unroll
          for (int j = 0; j < 32; ++j) xb[j * 32 + lane] = __uint_as_float(v[j]);
        }
        named_bar(pbar, 64);  // u of the chunk in shared memory
        if (hwarp) {
          float a[32], m[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            a[j] = __bfloat162float(__float2bfloat16_rn(silu_f(__uint_as_float(v[j])) * xb[j * 32 + lane]));
            m[j] = fabsf(a[j]);
          }
          // m[0] of lane l = amax over the 32 columns of row l
#pragma unroll
          for (int sh = 16; sh >= 1; sh >>= 1) {
            const bool upper = (lane & sh) != 0;
#pragma unroll
            for (int j = 0; j < sh; ++j) {
              const float send = upper ? m[j] : m[j + sh];
              const float keepv = upper ? m[j + sh] : m[j];
              m[j] = fmaxf(keepv, __shfl_xor_sync(0xffffffffu, send, sh));
            }
          }
          const int e = mx_exponent(m[0]);
          uint8_t* arow = P.aq + (row0 + ch * 32) * P.out_ld + icol;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int ej = __shfl_sync(0xffffffffu, e, j);
            const float inv = __uint_as_float(static_cast<uint32_t>(127 - ej) << 23);  // 2^-e
            if (j < nv)
              arow[static_cast<int64_t>(j) * P.out_ld] =
                  static_cast<uint8_t>(__nv_cvt_float_to_fp8(a[j] * inv, __NV_SATFINITE, __NV_E4M3));
          }
          if (lane < nv) scb[4 * mx_scale_pos(grow0 + ch * 32 + lane)] = static_cast<uint8_t>(e + 127);
        }
        named_bar(pbar, 64);  // the chunk's u consumed
      }
      tc_fence_before();
      if (leader) mbar_arrive(tempty);  // the accumulator is free for the next tile
      else remote_arrive(map_to_rank(smem_u32(tempty), 0));
    }
    __syncwarp();
  } else if (kT && warp >= 4) {
    // ---------------- epilogue, transposed form (both CTAs) ----------------
    // Warp 4 + 4 h + q: TMEM lane quarter q (output columns 32 q .. of the
    // CTA's 128), accumulator columns (routed rows) [128 h, 128 h + 128).
    // Each warp stores its chunks straight from registers (lane = column,
    // one row per store: 32 neighbouring columns, bf16 or fp32) and the
    // accumulator is released once every chunk is out; the eight warps
    // first combine their accumulator waits at barrier 3.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      bool ok = __all_sync(0xffffffffu, mbar_wait(tfull, it & 1, abort_flag, P.status, SITE_EPILOGUE));
      ok = named_bar_and(3, 256, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int nrows = min(c.rows - c.mt * 256, 256);
      const int row0 = c.row0 + c.mt * 256;
      // first output column of this CTA; the replay's CTA 1 writes u, CTA 0 h
      const int dcol = c.nt * P.b_tile_rows + (kReplay ? 0 : static_cast<int>(rank) * 128);
      const int ch0 = 4 * half;
      const int ch_end = min((t_ncols(c) + 31) / 32, ch0 + 4);
      if constexpr (kDirect16) {
        // lane = output column 32 q + lane.  The warp's chunks (at most
        // four) are first drained into registers, rounded to bf16 (word j
        // of chunk cc holds rows 2 j, 2 j + 1 of chunk ch0 + cc), and the
        // accumulator is released before any store, so the next tile's MMAs
        // do not wait for the stores; each warp store then writes 32
        // neighbouring bf16 columns of one row.
        uint32_t pk[4][16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (ch0 + cc < ch_end) {
            uint32_t v[32];
            tmem_ld32(taddr + (ch0 + cc) * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[cc][j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          }
        }
        tc_fence_before();
        if (leader) mbar_arrive(tempty);  // the accumulator is free for the next tile
        else remote_arrive(map_to_rank(smem_u32(tempty), 0));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = ch0 + cc;
          if (ch < ch_end) {
            const int nv = min(nrows - ch * 32, 32);  // valid rows of the chunk (at least 1)
            uint16_t* o = reinterpret_cast<uint16_t*>(P.y) + static_cast<int64_t>(row0 + ch * 32) * P.out_ld +
                          dcol + 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv)
                o[static_cast<int64_t>(j) * P.out_ld] =
                    static_cast<uint16_t>((j & 1) ? pk[cc][j >> 1] >> 16 : pk[cc][j >> 1] & 0xFFFFu);
          }
        }
        continue;
      }
      if constexpr (kF32) {
        // lane = output column 32 q + lane; register j = row ch * 32 + j
        float* out32 = kReplay ? (rank ? P.u32 : P.h32) : P.y32;
#pragma unroll 1
        for (int ch = ch0; ch < ch_end; ++ch) {
          const int nv = min(nrows - ch * 32, 32);  // valid rows of the chunk (at least 1)
          uint32_t v[32];
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait();
          float* o = out32 + static_cast<int64_t>(row0 + ch * 32) * P.out_ld + dcol + 32 * q + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) o[static_cast<int64_t>(j) * P.out_ld] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        if (leader) mbar_arrive(tempty);  // the accumulator is free for the next tile
        else remote_arrive(map_to_rank(smem_u32(tempty), 0));
        continue;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, own 128 rows) ----------------
    const int q = warp & 3;             // TMEM lane quarter of this warp
    const int half = (warp - 4) >> 2;  // column half of the accumulator
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      if (!__all_sync(0xffffffffu, mbar_wait(tfull, it & 1, abort_flag, P.status, SITE_EPILOGUE))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int local = c.mt * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;  // row within the group
      const bool valid = local < c.rows;
      const int64_t row = c.row0 + local;
      if (kF32) {
        // 256 fp32 columns per row: y (down), or h then u (replay); this
        // warp drains 128 of them, 32 per TMEM load, each thread storing its
        // row's 128 bytes
#pragma unroll 1
        for (int ch = 4 * half; ch < 4 * half + 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait();
          if (valid) {
            float* dst = kReplay ? (ch < 4 ? P.h32 : P.u32) + row * P.out_ld + c.nt * 128 + (ch & 3) * 32
                                 : P.y32 + row * P.out_ld + c.nt * 256 + ch * 32;
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
              st_global_v4(dst + qq * 4, v[4 * qq], v[4 * qq + 1], v[4 * qq + 2], v[4 * qq + 3]);
          }
        }
        tc_fence_before();
        if (leader) mbar_arrive(tempty);
        else remote_arrive(map_to_rank(smem_u32(tempty), 0));
        continue;
      }
      if (kBf16Out) {
        // 256 bf16 columns per row: y (down), or h then u (replay); this
        // warp drains 128 of them.  A full 32-row slab is drained into the
        // warp's two 4 KB boxes (128-byte swizzle: 16-byte chunk c of row r
        // at chunk c ^ (r % 8)), the accumulator is released, and two TMA
        // stores write the boxes.  A slab that crosses the group's end is
        // written row by row (a TMA store would overwrite the next group's
        // rows).
        const int nvalid = min(max(c.rows - (local - lane), 0), 32);
        uint8_t* boxes = staging + q * (4 * 4096);  // boxes 2 half, 2 half + 1 are this warp's
        if (nvalid == 32) {
          if (lane == 0) bulk_wait_read0();  // the previous tile's stores have read the boxes
          __syncwarp();
        }
#pragma unroll 1
        for (int ch = 4 * half; ch < 4 * half + 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          if (nvalid == 32) {
            uint8_t* rowp = boxes + (ch >> 1) * 4096 + lane * 128;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int chunk = (ch & 1) * 4 + qq;
              *reinterpret_cast<uint4*>(rowp + ((chunk ^ (lane & 7)) * 16)) =
                  make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
            }
          } else if (valid) {
            __nv_bfloat16* dst = kReplay ? (ch < 4 ? P.h_out : P.u_out) + row * P.out_ld + c.nt * 128 + (ch & 3) * 32
                                         : P.y + row * P.out_ld + c.nt * 256 + ch * 32;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              st_global_v4(dst + qq * 8, pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          }
        }
        if (nvalid == 32) {
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_before();
        if (leader) mbar_arrive(tempty);
        else remote_arrive(map_to_rank(smem_u32(tempty), 0));
        if (nvalid == 32 && lane == 0) {
          const int y0 = static_cast<int>(row - lane);  // the slab's first row
#pragma unroll
          for (int bx = 2 * half; bx < 2 * half + 2; ++bx) {
            if (kReplay) tma_store_2d(bx < 2 ? &P.tmO0 : &P.tmO1, boxes + bx * 4096, c.nt * 128 + (bx & 1) * 64, y0);
            else tma_store_2d(&P.tmO0, boxes + bx * 4096, c.nt * 256 + bx * 64, y0);
          }
          bulk_commit();
        }
        continue;
      }
      if (kSwiglu) {
        const bool keep = P.act && valid && c.row0 + c.rows <= P.act_rows;
        // a = bf16(SiLU(h) u) of this warp's two 32-column chunks, as bf16
        // pairs (exact: a is rounded to bf16 before it is quantised), and
        // each chunk's amax; then the accumulator is released, so the next
        // tile's MMAs run while this tile's codes are formed and stored
        uint32_t apk[2][16];
        float amax[2];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * half + cc;
          uint32_t hv[32], uv[32];
          tmem_ld32(taddr + ch * 32, hv);
          tmem_ld32(taddr + 128 + ch * 32, uv);
          tmem_ld_wait();
          if (keep) {  // this row's 32 columns of h and of u, unrounded
            float* ar = P.act + row * (2 * P.out_ld) + c.nt * 128 + ch * 32;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              st_global_v4(ar + 4 * q, hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
              st_global_v4(ar + P.out_ld + 4 * q, uv[4 * q], uv[4 * q + 1], uv[4 * q + 2], uv[4 * q + 3]);
            }
          }
          float am = 0.0f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = __bfloat162float(
                __float2bfloat16_rn(silu_f(__uint_as_float(hv[2 * j])) * __uint_as_float(uv[2 * j])));
            const float a1 = __bfloat162float(
                __float2bfloat16_rn(silu_f(__uint_as_float(hv[2 * j + 1])) * __uint_as_float(uv[2 * j + 1])));
            am = fmaxf(am, fmaxf(fabsf(a0), fabsf(a1)));
            apk[cc][j] = pack_bf16x2(a0, a1);
          }
          amax[cc] = am;
        }
        tc_fence_before();
        if (leader) mbar_arrive(tempty);
        else remote_arrive(map_to_rank(smem_u32(tempty), 0));
        uint32_t words = 0;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int e = mx_exponent(amax[cc]);
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = apk[cc][2 * i], w1 = apk[cc][2 * i + 1];
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(bf16lo(w0) * inv, bf16hi(w0) * inv), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(bf16lo(w1) * inv, bf16hi(w1) * inv), __NV_SATFINITE, __NV_E4M3);
            pk[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
          }
          words |= static_cast<uint32_t>(e + 127) << (8 * cc);
          if (valid) {
            uint8_t* dst = P.aq + row * P.out_ld + c.nt * 128 + (2 * half + cc) * 32;
            st_global_v4(dst, pk[0], pk[1], pk[2], pk[3]);
            st_global_v4(dst + 16, pk[4], pk[5], pk[6], pk[7]);
          }
        }
        // this half's two bytes of the row's scale word (byte ch = block ch)
        if (valid)
          reinterpret_cast<uint16_t*>(P.asc + c.nt * P.a_ld + mx_scale_pos(mx_group_row0(c.row0, c.g) + local))[half] =
              static_cast<uint16_t>(words);
        continue;  // the accumulator was released above
      }
      tc_fence_before();
      if (leader) mbar_arrive(tempty);
      else remote_arrive(map_to_rank(smem_u32(tempty), 0));
    }
    if (kBf16Out && lane == 0) bulk_wait0();  // this warp's stores have landed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // the leader's MMAs (which read the peer's shared memory) and all remote arrivals are done
  tc_fence_after();
  if (warp == 2) tmem_dealloc2(tmem_base, 512);
}

size_t mx_smem_bytes(int G, bool staged, bool swiglu_t = false) {
  return 1024 + static_cast<size_t>(mx_stages(staged)) * mx_ksub(staged) * (CODE_BYTES + SF_BYTES) +
         (staged ? STAGING_BYTES : (swiglu_t ? XCH_BYTES : 0)) + 1024 + static_cast<size_t>(G + 1) * sizeof(int);
}

template <bool kSwiglu, bool kReplay = false, bool kT = false, bool kF32 = false, bool kRing = false>
mok_status run_mx(const MxParams& P, cudaStream_t st, int max_sms = 0) {
  constexpr bool staged = (!kSwiglu || kReplay) && !kF32 && !(kT && !kSwiglu && !kReplay);
  const size_t smem = mx_smem_bytes(P.sched.G, staged, kT && kSwiglu && !kReplay);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  auto kern = gemm_mx_pair_persistent<kSwiglu, kReplay, kT, kF32, kRing>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return MOK_ERR_CUDA;
  // the schedule counts stages of mx_ksub K blocks each
  constexpr int ksub = mx_ksub(staged);
  if (P.sched.k_blocks_fixed % ksub) return MOK_ERR_UNSUPPORTED;
  MxParams Q = P;
  Q.sched.k_blocks_fixed = P.sched.k_blocks_fixed / ksub;
  const int sms = max_sms > 0 && max_sms < num_sms() ? max_sms : num_sms();
  const int grid = sms >= 2 ? (sms / 2) * 2 : 2;
  if (!kRing) {
    kern<<<grid, THREADS, smem, st>>>(Q);
    MOK_CHECK_LAUNCH();
    return MOK_OK;
  }
  // ring producers and consumers wait on each other: all CTAs must be resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, Q) != cudaSuccess) return MOK_ERR_CUDA;
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

constexpr auto kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
constexpr auto kI32 = CU_TENSOR_MAP_DATA_TYPE_INT32;

// bf16 [rows][cols] output, boxes of 32 rows x 64 columns, 128-byte swizzle
bool out_map(CUtensorMap* m, const void* p, int64_t rows, int cols) {
  return make_tmap_2d(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rows > 0 ? rows : 1, cols,
                      static_cast<uint64_t>(cols) * 2, 32, 64, true);
}

bool code_map(CUtensorMap* m, const void* p, int64_t rows, int K, int box_rows = 128) {
  return make_tmap_2d(m, p, kU8, rows, K, static_cast<uint64_t>(K), box_rows, BKB, true);
}
// scale words [K/128][ld] as a 2D tensor of K/128 rows of ld words (ld is a
// multiple of 128), boxes of one 128-row block
bool scale_map(CUtensorMap* m, const void* p, int64_t ld, int K) {
  return make_tmap_2d(m, p, kI32, K / 128, ld, static_cast<uint64_t>(ld) * 4, 1, 128, false);
}

SchedArgs mx_sched(const int32_t* offsets, int G, int64_t m_total, int n_tiles, int k_blocks) {
  SchedArgs s;
  s.offsets = offsets;
  s.G = G;
  s.m_total = static_cast<int32_t>(m_total);
  s.n_tiles = n_tiles;
  s.m_tiles_fixed = 0;
  s.k_blocks_fixed = k_blocks;
  s.bm = 256;
  s.bk_rows = BKB;
  return s;
}

// Parameters of the up/gate pair GEMM (also the backward's replay).
mok_status upgate_mx_params(MxParams& P, const void* xq, const void* xsc, int64_t rows, const void* qg,
                            const void* sg, const void* qu, const void* su, const int32_t* offsets, int G, int D,
                            int I) {
  P.sched = mx_sched(offsets, G, rows, I / 128, D / BKB);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int64_t wrows = static_cast<int64_t>(G) * I;
  if (!code_map(&P.tmA, xq, rows, D) || !scale_map(&P.tmSA, xsc, mx_scale_ld(rows, G), D) ||
      !code_map(&P.tmB0, qg, wrows, D) || !code_map(&P.tmB1, qu, wrows, D) ||
      !scale_map(&P.tmSB0, sg, mx_scale_ld(wrows), D) || !scale_map(&P.tmSB1, su, mx_scale_ld(wrows), D))
    return MOK_ERR_CUDA;
  P.b_group_rows = I;
  P.b_tile_rows = 128;
  P.b1_off = 0;
  P.aq = nullptr;
  P.asc = nullptr;
  P.a_ld = mx_scale_ld(rows, G);
  P.y = nullptr;
  P.h_out = nullptr;
  P.u_out = nullptr;
  P.h32 = nullptr;
  P.u32 = nullptr;
  P.y32 = nullptr;
  P.act = nullptr;
  P.act_rows = 0;
  P.out_ld = I;
  return MOK_OK;
}
}  // namespace

mok_status launch_upgate_mx(const void* xq, const void* xsc, int64_t rows, const void* qg,
                            const void* sg, const void* qu, const void* su, const int32_t* offsets,
                            int G, int D, int I, void* aq, void* asc, cudaStream_t st, KeptAct kept,
                            const void* sp) {
  if (rows == 0) return MOK_OK;
  if (!offsets || G < 1) return MOK_ERR_INVALID_ARG;
  MxParams P;
  mok_status r = upgate_mx_params(P, xq, xsc, rows, qg, sg, qu, su, offsets, G, D, I);
  if (r != MOK_OK) return r;
  P.aq = static_cast<uint8_t*>(aq);
  P.asc = static_cast<uint32_t*>(asc);
  P.act = kept.act;
  P.act_rows = kept.limit();
  // fewer than 512 routed rows per group on average and the paired scale
  // blocks given: the routed rows as the MMA's N dimension (no padding rows
  // in the MMAs)
  if (sp && rows < static_cast<int64_t>(512) * G) {
    const int64_t wrows = static_cast<int64_t>(G) * I;
    if (!code_map(&P.tmU64, qu, wrows, D, 64) || !code_map(&P.tmG64, qg, wrows, D, 64) ||
        !scale_map(&P.tmSP, sp, mx_scale_ld(2 * wrows), D))
      return MOK_ERR_CUDA;
    return run_mx<true, false, true>(P, st);
  }
  return run_mx<true>(P, st);
}

mok_status launch_upgate_mx_ring(const void* x, const int32_t* table, int K, const void* qg, const void* sg,
                                 const void* qu, const void* su, const int32_t* offsets, int G, int64_t R, int D, int I,
                                 void* aq, void* asc, void* xsc, void* ring, int64_t ring_rows, int chunk_rows,
                                 int32_t* counters, cudaStream_t st, KeptAct kept) {
  if (R == 0) return MOK_OK;
  if (!offsets || G < 1 || chunk_rows < 128 || ring_rows < chunk_rows || ring_rows % chunk_rows)
    return MOK_ERR_INVALID_ARG;
  const int64_t nchunks = (R + chunk_rows - 1) / chunk_rows;
  if (nchunks > (int64_t{1} << 24)) return MOK_ERR_INVALID_ARG;
  if (cudaMemsetAsync(counters, 0, 2 * nchunks * sizeof(int32_t), st) != cudaSuccess) return MOK_ERR_CUDA;
  MxParams P;
  // tmA maps the ring (ring_rows + 128 rows of codes); tmSA the full grouped scale layout
  mok_status r = upgate_mx_params(P, ring, xsc, R, qg, sg, qu, su, offsets, G, D, I);
  if (r != MOK_OK) return r;
  if (!code_map(&P.tmA, ring, ring_rows + 128, D)) return MOK_ERR_CUDA;
  P.sched.m_outer = 1;  // rows leave the ring in order: all N tiles of an M tile before the next M tile
  P.aq = static_cast<uint8_t*>(aq);
  P.asc = static_cast<uint32_t*>(asc);
  P.act = kept.act;
  P.act_rows = kept.limit();
  P.x = static_cast<const uint4*>(x);
  P.table = table;
  P.K = K;
  P.D8 = D / 8;
  P.ring = static_cast<uint2*>(ring);
  P.xsc = static_cast<uint32_t*>(xsc);
  P.xs_ld = mx_scale_ld(R, G);
  P.ring_rows = ring_rows;
  P.chunk_rows = chunk_rows;
  P.nchunks = static_cast<int32_t>(nchunks);
  P.n_tiles = I / 128;
  P.ready = counters;
  P.done = counters + nchunks;
  return run_mx<true, false, false, false, true>(P, st);
}

mok_status launch_replay_mx(const void* xq, const void* xsc, int64_t rows, const void* qg, const void* sg,
                            const void* qu, const void* su, const int32_t* offsets, int G, int D, int I, void* h,
                            void* u, cudaStream_t st, int32_t skip_rows_below) {
  if (rows == 0) return MOK_OK;
  if (!offsets || G < 1) return MOK_ERR_INVALID_ARG;
  MxParams P;
  mok_status r = upgate_mx_params(P, xq, xsc, rows, qg, sg, qu, su, offsets, G, D, I);
  if (r != MOK_OK) return r;
  if (skip_rows_below > 0) {  // the groups the forward kept need no replay
    P.sched.row_split = skip_rows_below;
    P.sched.split_side = 2;
  }
  P.h32 = static_cast<float*>(h);
  P.u32 = static_cast<float*>(u);
  // as the down form: the routed rows as N for groups under 512 rows on average
  if (rows < static_cast<int64_t>(512) * G) return run_mx<true, true, true, true>(P, st);
  return run_mx<true, true, false, true>(P, st);
}

mok_status launch_down_mx(const void* aq, const void* asc, int64_t rows, const void* qd,
                          const void* sd, const int32_t* offsets, int G, int D, int I, void* y,
                          cudaStream_t st, bool f32_out, int max_sms) {
  if (rows == 0) return MOK_OK;
  if (!offsets || G < 1) return MOK_ERR_INVALID_ARG;
  MxParams P;
  P.sched = mx_sched(offsets, G, rows, D / 256, I / BKB);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int64_t wrows = static_cast<int64_t>(G) * D;
  if (!code_map(&P.tmA, aq, rows, I) || !scale_map(&P.tmSA, asc, mx_scale_ld(rows, G), I) ||
      !code_map(&P.tmB0, qd, wrows, I) || !scale_map(&P.tmSB0, sd, mx_scale_ld(wrows), I))
    return MOK_ERR_CUDA;
  P.tmB1 = P.tmB0;
  P.tmSB1 = P.tmSB0;
  P.b_group_rows = D;
  P.b_tile_rows = 256;
  P.b1_off = 128;
  P.aq = nullptr;
  P.asc = nullptr;
  P.act = nullptr;
  P.act_rows = 0;
  P.a_ld = 0;
  P.h_out = nullptr;
  P.u_out = nullptr;
  P.h32 = nullptr;
  P.u32 = nullptr;
  P.out_ld = D;
  const bool by_rows = rows < static_cast<int64_t>(512) * G;
  if (f32_out) {
    P.y = nullptr;
    P.y32 = static_cast<float*>(y);
    return by_rows ? run_mx<false, false, true, true>(P, st, max_sms) : run_mx<false, false, false, true>(P, st, max_sms);
  }
  P.y = static_cast<__nv_bfloat16*>(y);
  P.y32 = nullptr;
  if (!out_map(&P.tmO0, y, rows, D)) return MOK_ERR_CUDA;
  P.tmO1 = P.tmO0;
  // fewer than 512 routed rows per group on average: the routed rows as the
  // MMA's N dimension (no padding rows in the MMAs); its stages hold two K
  // blocks, so K = I must be a multiple of 256 (else the row-major form)
  if (by_rows && (I / BKB) % 2 == 0) return run_mx<false, false, true>(P, st, max_sms);
  return run_mx<false>(P, st, max_sms);
}

}  // namespace mok
