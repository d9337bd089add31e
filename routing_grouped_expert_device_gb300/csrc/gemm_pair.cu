// Forward grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// A cluster of two CTAs on two SMs computes one 256-row x 256-column tile:
// CTA rank r loads rows [128 r, 128 r + 128) of the tile's A operand and
// half of the B operand (up/gate: rank 0 the 128 W_gate rows, rank 1 the 128
// W_up rows; down: output columns [128 r, 128 r + 128)), and the leader
// (rank 0) issues M256 N256 MMAs that read both CTAs' shared memory and
// write each CTA's 128 rows of the accumulator into that CTA's TMEM.  Each
// expert's weight tile therefore crosses L2 once per 256 routed rows, and an
// SM fills 32 KB of shared memory per 64-wide K block instead of 48 KB.
//
// Barriers: both CTAs' TMA loads complete on the leader's full[stage]
// (armed by the leader for both halves); MMA completion is multicast to
// both CTAs' empty[stage] and tfull[acc]; both CTAs' epilogues arrive on the
// leader's tempty[acc].  Every wait is bounded as in gemm_core.cuh.
#include "gemm_core.cuh"
#include "kernels.h"
#include "pair.cuh"

namespace mok {
namespace {

constexpr int BOX_K = 64;   // K columns per TMA box: 128 bytes, the swizzle span
// K columns per stage (BK / BOX_K boxes per operand): three 64 KB stages
// carry as many bytes in flight as six of 32 KB and halve the MMA warp's
// per-stage waits and commits (skewed layer 3.69 -> 3.62 ms, DSV3 unchanged)
constexpr int BK = 128;
constexpr int STAGES = 3;
constexpr int BOX_BYTES = 128 * BOX_K * 2;  // one box of 128 rows
constexpr int A_BYTES = 128 * BK * 2;  // this CTA's 128 rows
constexpr int B_BYTES = 128 * BK * 2;  // this CTA's half of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_BLOCK = 32 * 128;  // one epilogue warp's staging block: 32 rows x 64 bf16
constexpr uint32_t IDESC = idesc_bf16(256, 256, false, false);

__device__ __forceinline__ void mma2(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}

struct PairParams {
  SchedArgs sched;  // bm = 256: one tile = 256 rows of one group
  int* status;
  CUtensorMap tmA;   // activations [rows][K], boxes 128 x 64
  CUtensorMap tmB0;  // B half of rank 0, boxes 128 x 64
  CUtensorMap tmB1;  // B half of rank 1
  int32_t b_group_rows, b_tile_rows, b1_off;
  __nv_bfloat16* out;
  int32_t out_ld;
  CUtensorMap tmOut;  // out as [rows][out_ld], boxes 32 rows x 64 columns, 128-byte swizzle
  // The extra group of the schedule (the shared expert): its own A, B and
  // output (B rows nt * b_tile_rows + (rank ? b1_off : 0), as above).
  CUtensorMap tmAs, tmBs0, tmBs1;
  __nv_bfloat16* out_s;
  int32_t out_ld_s;
  CUtensorMap tmOut_s;
  // Ring dispatch (kRing): tmA maps the ring, [ring_rows + 128][D]; row r
  // (expert order) sits at ring row r % ring_rows, and ring rows 0..127 are
  // repeated after the end so that no 128-row box wraps.
  const uint4* x;          // [T][D] bf16, as 16-byte vectors
  const int32_t* table;    // the plan's [R][3]: row r comes from x[table[r].src / K]
  int32_t K, D8;           // top-k; D / 8
  uint4* ring;
  int64_t ring_rows, R;
  int32_t chunk_rows, nchunks, n_tiles;
  int32_t* ready;          // [nchunks]: producer warps done with the chunk
  int32_t* done;           // [nchunks]: (row, N tile) reads of the chunk completed
  // Router scores (kSoftmax): one N tile of 256 logits per row, columns < E
  // valid; s_out [rows][E] fp32.
  float* s_out;
  int32_t E;
  // Kept activations (kSwiglu, optional): h, u fp32 of the routed rows of
  // every group whose rows end at or below act_rows, as [rows][2 * act_i]
  // (h in columns [0, act_i), u in [act_i, 2 act_i)).
  float* act;
  int32_t act_rows, act_i;
};

// ---------------------------------------------------------------------------
// Ring dispatch (Mixture-of-Kittens blog, "Scheduling"; paper note,
// "Granularity as a tunable" and "A ring buffer instead of a host
// round-trip"): producer warps gather routed rows of x into an
// expert-ordered ring in chunks of b rows and signal each finished chunk
// through a device counter; the GEMM's TMA warp waits for the chunks its
// rows lie in, and the MMA thread reports the rows it has read so that the
// slot can be refilled.  All CTAs of the launch are resident (cooperative
// launch), and every wait is bounded.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int64_t ring_slots(const PairParams& P) { return P.ring_rows / P.chunk_rows; }
__device__ __forceinline__ int chunk_row_count(const PairParams& P, int c) {
  const int64_t r0 = static_cast<int64_t>(c) * P.chunk_rows;
  const int64_t r1 = r0 + P.chunk_rows < P.R ? r0 + P.chunk_rows : P.R;
  return static_cast<int>(r1 - r0);
}

// Producer warp `pw` of `np`: rows r = c b + pw, c b + pw + np, ... of every
// chunk c in order.  Before writing chunk c it waits until chunk c - slots
// (same ring slot) has been read by all its N tiles.
__device__ void ring_produce(const PairParams& P, int pw, int np, int lane, volatile int* abort) {
  const int64_t slots = ring_slots(P);
  for (int c = 0; c < P.nchunks; ++c) {
    if (c >= slots) {
      bool ok = true;
      if (lane == 0)
        ok = wait_count(P.done + (c - slots), chunk_row_count(P, c - static_cast<int>(slots)) * P.n_tiles, abort,
                        P.status, SITE_RING_SLOT);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    }
    const int64_t r0 = static_cast<int64_t>(c) * P.chunk_rows;
    const int64_t r1 = r0 + chunk_row_count(P, c);
    for (int64_t r = r0 + pw; r < r1; r += np) {
      const int src = __ldg(P.table + r * 3) / P.K;
      const uint4* in = P.x + static_cast<int64_t>(src) * P.D8;
      const int64_t q = r % P.ring_rows;
      uint4* out = P.ring + q * P.D8;
      uint4* mirror = q < 128 ? P.ring + (P.ring_rows + q) * P.D8 : nullptr;
      int i = lane;
      for (; i + 96 < P.D8; i += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(in + i + 32 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          out[i + 32 * u] = v[u];
          if (mirror) mirror[i + 32 * u] = v[u];
        }
      }
      for (; i < P.D8; i += 32) {
        const uint4 v = __ldg(in + i);
        out[i] = v;
        if (mirror) mirror[i] = v;
      }
    }
    // the chunk's rows of this warp are written: make them visible to the
    // consumers' TMA (async proxy) reads, then count this warp in
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0) red_release_add(P.ready + c, 1);
  }
}

// Rows [max(r0, g0), min(r0 + 128, g1)) of a 128-row box that lie inside its
// group [g0, g1): their chunks, and per chunk the count of those rows.
template <class F>
__device__ __forceinline__ void for_box_chunks(const PairParams& P, int64_t r0, int64_t g0, int64_t g1, F f) {
  const int64_t v0 = r0 > g0 ? r0 : g0;
  const int64_t v1 = r0 + 128 < g1 ? r0 + 128 : g1;
  for (int64_t v = v0; v < v1;) {
    const int c = static_cast<int>(v / P.chunk_rows);
    const int64_t e = (static_cast<int64_t>(c) + 1) * P.chunk_rows < v1 ? (static_cast<int64_t>(c) + 1) * P.chunk_rows : v1;
    f(c, static_cast<int>(e - v));
    v = e;
  }
}

// Router scores epilogue: s = softmax over the row's E logits (fp32 in TMEM,
// columns 0..255 of the accumulator).  Three passes over the row: the
// maximum, the sum of exp(l - max), then exp(l - max) / sum, written as fp32.
__device__ __forceinline__ void softmax_epilogue(const PairParams& P, uint32_t taddr, int64_t row, bool valid) {
  const int E = P.E;
  float m = -INFINITY;
#pragma unroll 1
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t v[32];
    tmem_ld32(taddr + ch * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (ch * 32 + j < E) m = fmaxf(m, __uint_as_float(v[j]));
  }
  float sum = 0.0f;
#pragma unroll 1
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t v[32];
    tmem_ld32(taddr + ch * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (ch * 32 + j < E) sum += __expf(__uint_as_float(v[j]) - m);
  }
  const float inv = 1.0f / sum;
  float* orow = P.s_out + row * E;
#pragma unroll 1
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t v[32];
    tmem_ld32(taddr + ch * 32, v);
    tmem_ld_wait();
    if (valid) {
      float o[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __expf(__uint_as_float(v[j]) - m) * inv;
      if (ch * 32 + 32 <= E && (E & 3) == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(orow + ch * 32 + 4 * q) =
              make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (ch * 32 + j < E) orow[ch * 32 + j] = o[j];
      }
    }
    __syncwarp();  // converged again before the next warp-wide TMEM load
  }
}

template <bool kSwiglu, bool kRing = false, bool kSoftmax = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    gemm_pair_persistent(const __grid_constant__ PairParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi_smem = smem + STAGES * STAGE_BYTES;  // 4 staging blocks, 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_smem + 4 * EPI_BLOCK);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* total_holder = reinterpret_cast<int*>(tmem_holder + 2);
  int* tstart = reinterpret_cast<int*>(epi_smem + 4 * EPI_BLOCK + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 256);  // both CTAs' 128 epilogue threads
    }
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
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileCoord c = walk.at(tile);
        const int arow = c.row0 + c.mt * 256 + static_cast<int>(rank) * 128;
        const int brow = c.g * P.b_group_rows + c.nt * P.b_tile_rows + (rank ? P.b1_off : 0);
        const CUtensorMap* tmA = c.extra ? &P.tmAs : &P.tmA;
        const CUtensorMap* tmB = c.extra ? (rank ? &P.tmBs1 : &P.tmBs0) : (rank ? &P.tmB1 : &P.tmB0);
        int ay = arow;
        if (kRing && !c.extra) {
          // this CTA's rows of the tile must be in the ring
          for_box_chunks(P, arow, c.row0, static_cast<int64_t>(c.row0) + c.rows, [&](int ch, int) {
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
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          const uint32_t lbar = map_to_rank(smem_u32(&full[stage]), 0);
          uint8_t* st = smem + stage * STAGE_BYTES;
#pragma unroll
          for (int j = 0; j < BK / BOX_K; ++j) {
            tma_load_2d_pair(st + j * BOX_BYTES, tmA, kb * BK + j * BOX_K, ay, lbar);
            tma_load_2d_pair(st + A_BYTES + j * BOX_BYTES, tmB, kb * BK + j * BOX_K, brow, lbar);
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
    // ---------------- MMA issuer (leader only) ----------------
    if (leader) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, any = false;
      int it = 0;
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
        const TileCoord c = walk.at(tile);
        const uint32_t acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, P.status, SITE_MMA));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA));
          if (!ok) break;
          tc_fence_after();
          if (kRing && !c.extra && kb == c.kblocks - 1 && lane == 0) {
            // every load of this tile (both CTAs) has landed: its ring rows
            // are read for this N tile
            for (int h = 0; h < 2; ++h)
              for_box_chunks(P, static_cast<int64_t>(c.row0) + c.mt * 256 + h * 128, c.row0,
                             static_cast<int64_t>(c.row0) + c.rows, [&](int ch, int n) { red_release_add(P.done + ch, n); });
          }
          if (lane == 0) {
            const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b = a + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t off = (k / (BOX_K / 16)) * BOX_BYTES + (k % (BOX_K / 16)) * 32;
              mma2(d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), (kb | k) != 0);
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
        if (lane == 0) commit2(&tfull[acc], 0x3);
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
    ring_produce(P, static_cast<int>(blockIdx.x) * 2 + (warp - 2), 2 * static_cast<int>(gridDim.x), lane, abort_flag);
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, own 128 rows) ----------------
    // Each warp owns 32 rows of the tile.  Per 64 output columns it packs its
    // rows to bf16, writes them to its staging block in the 128-byte swizzle
    // of the output's tensor map (16-byte chunk c of row r at chunk c ^ (r % 8))
    // and issues one TMA store, so whole rows leave in bulk instead of
    // 16-byte pieces of 32 rows.  A 32-row slab that crosses the group's end
    // is written row by row (lanes past the end write nothing): a TMA store
    // would overwrite the next group's rows.
    const int ew = warp - 4;
    uint8_t* blk = epi_smem + ew * EPI_BLOCK;
    uint8_t* srow = blk + lane * 128;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, P.status, SITE_EPILOGUE)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(ew * 32) << 16);
      const int slab = c.mt * 256 + static_cast<int>(rank) * 128 + ew * 32;  // first row of this warp in the group
      const int nvalid = min(max(c.rows - slab, 0), 32);
      if (kSoftmax) {
        softmax_epilogue(P, taddr, static_cast<int64_t>(c.row0) + slab + lane, lane < nvalid);
        tc_fence_before();
        if (leader) mbar_arrive(&tempty[acc]);
        else remote_arrive(map_to_rank(smem_u32(&tempty[acc]), 0));
        continue;
      }
      const int y = (c.extra ? 0 : c.row0) + slab;  // its row in the output tensor
      // h, u of this group go to the kept-activation store
      const bool keep = kSwiglu && P.act && !c.extra && c.row0 + c.rows <= P.act_rows;
      const CUtensorMap* tmOut = c.extra ? &P.tmOut_s : &P.tmOut;
      __nv_bfloat16* orow = c.extra ? P.out_s + static_cast<size_t>(y + lane) * P.out_ld_s
                                    : P.out + static_cast<size_t>(y + lane) * P.out_ld;
      constexpr int kBoxes = kSwiglu ? 2 : 4;  // 64-column boxes: a 128 columns, y 256
      const int x0 = c.nt * (kSwiglu ? 128 : 256);
#pragma unroll 1
      for (int bx = 0; bx < kBoxes && nvalid > 0; ++bx) {
        uint32_t pk[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ch = 2 * bx + hh;
          if (kSwiglu) {
            uint32_t h[32], u[32];
            tmem_ld32(taddr + ch * 32, h);
            tmem_ld32(taddr + 128 + ch * 32, u);
            tmem_ld_wait();
            if (keep && lane < nvalid) {
              float* ar = P.act + static_cast<int64_t>(y + lane) * (2 * P.act_i) + c.nt * 128 + ch * 32;
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                st_global_v4(ar + 4 * q, h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                st_global_v4(ar + P.act_i + 4 * q, u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[hh * 16 + j] = pack_bf16x2(silu_f(__uint_as_float(h[2 * j])) * __uint_as_float(u[2 * j]),
                                            silu_f(__uint_as_float(h[2 * j + 1])) * __uint_as_float(u[2 * j + 1]));
          } else {
            uint32_t v[32];
            tmem_ld32(taddr + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[hh * 16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          }
        }
        if (nvalid == 32) {
          if (lane == 0) bulk_wait_read0();  // the block's previous store has read it
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(srow + ((q ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(tmOut, blk, x0 + bx * 64, y);
            bulk_commit();
          }
        } else if (lane < nvalid) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_global_v4(orow + x0 + bx * 64 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      tc_fence_before();
      if (leader) mbar_arrive(&tempty[acc]);
      else remote_arrive(map_to_rank(smem_u32(&tempty[acc]), 0));
    }
    if (lane == 0) bulk_wait0();  // every store of this warp has landed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // the leader's MMAs (which read the peer's shared memory) and all remote arrivals are done
  tc_fence_after();
  if (warp == 2) tmem_dealloc2(tmem_base, 512);
}

size_t pair_smem_bytes(int G) {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 4 * EPI_BLOCK + 1024 +
         static_cast<size_t>(G + 1) * sizeof(int);
}

// max_sms > 0: the persistent grid takes at most that many SMs (clusters
// of two), leaving the rest to kernels of other streams.
template <bool kSwiglu, bool kRing = false, bool kSoftmax = false>
mok_status run_pair(const PairParams& P, cudaStream_t st, int max_sms = 0) {
  const size_t smem = pair_smem_bytes(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  auto kern = gemm_pair_persistent<kSwiglu, kRing, kSoftmax>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  const int sms = max_sms > 0 && max_sms < num_sms() ? max_sms : num_sms();
  const int grid = sms >= 2 ? (sms / 2) * 2 : 2;
  if (!kRing) {
    kern<<<grid, 256, smem, st>>>(P);
    MOK_CHECK_LAUNCH();
    return MOK_OK;
  }
  // ring producers and consumers wait on each other: all CTAs must be resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) return MOK_ERR_CUDA;
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

SchedArgs pair_sched(const int32_t* offsets, int G, int64_t m_total, int n_tiles, int k_blocks) {
  SchedArgs s;
  s.offsets = offsets;
  s.G = offsets ? G : 1;
  s.m_total = static_cast<int32_t>(m_total);
  s.n_tiles = n_tiles;
  s.m_tiles_fixed = 0;
  s.k_blocks_fixed = k_blocks;
  s.bm = 256;
  s.bk_rows = BK;
  return s;
}

constexpr auto kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

// Output [rows][ld] bf16 for the epilogue's TMA stores (32 x 64 boxes).
bool out_map(CUtensorMap* m, const void* p, int64_t rows, int ld) {
  return make_tmap_2d(m, p, kBF16, static_cast<uint64_t>(rows > 0 ? rows : 1), ld, static_cast<uint64_t>(ld) * 2, 32,
                      64, true);
}

// Every launch needs valid output maps; with no routed rows (or no extra
// group) the unused one repeats the other.
bool set_out_maps(PairParams& P, int64_t m_total) {
  const bool routed = m_total > 0 && P.out;
  const bool extra = P.sched.extra_rows > 0 && P.out_s;
  if (routed && !out_map(&P.tmOut, P.out, m_total, P.out_ld)) return false;
  if (extra && !out_map(&P.tmOut_s, P.out_s, P.sched.extra_rows, P.out_ld_s)) return false;
  if (!routed) P.tmOut = P.tmOut_s;
  if (!extra) P.tmOut_s = P.tmOut;
  return routed || extra;
}

// ---------------------------------------------------------------------------
// Routed up/gate with the routed rows as the MMA's N dimension.
//
// The pair's tile is 128 intermediate columns i0 .. i0 + 127 of one expert
// by up to 256 of its routed rows.  The MMA's M = 256 rows are weight rows
// and N = the tile's row count rounded up to 16, so an expert with 224 rows
// costs 224 columns of MMA work where the row-major tiles above cost 256
// rows.  CTA r holds W_up rows i0 + 64 r .. + 63 as A rows 0-63 and the
// same rows of W_gate as A rows 64-127, and half of the N routed rows (the
// pair MMA reads N / 2 rows of B from each CTA).  Its accumulator lanes
// 0-63 then hold u and lanes 64-127 the matching h, one column per routed
// row.  The epilogue warps of lane quarters 0 and 1 pass u through shared
// memory to the warps of quarters 2 and 3, which form a = bf16(SiLU(h) u)
// and write [32 rows][64 columns] pieces of a with TMA stores; the
// arithmetic thus runs on the sub-partitions that do not also host the TMA
// and MMA warps (a warp's sub-partition is its index mod 4).  The four
// epilogue warps meet at named barrier 1 in the same sequence on every
// tile, and agree on an abort with a barrier reduction first.
struct PairTParams {
  SchedArgs sched;  // bm = 256 routed rows of a group, n_tiles = I / 128
  int* status;
  CUtensorMap tmG, tmU;  // W_gate, W_up as [G * I][D], boxes 64 rows x 64
  CUtensorMap tmX;       // routed rows [rows][D], boxes 128 x 64
  CUtensorMap tmOut;     // a [rows][I], boxes 32 rows x 64 columns, 128-byte swizzle
  __nv_bfloat16* out;
  int32_t I;
  float* act;            // kept h, u (as PairParams::act), or null
  int32_t act_rows;
};

constexpr int T_OUT_BYTES = 32 * 128;       // one [32 rows][64 columns] bf16 box of a
constexpr int T_XBUF_BYTES = 2 * 32 * 32 * 4;  // u of two warps for one 32-column chunk, fp32


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    gemm_pair_upgate_t(const __grid_constant__ PairTParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ostage = smem + STAGES * STAGE_BYTES;  // 1024-byte aligned
  float* xbuf = reinterpret_cast<float*>(ostage + T_OUT_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xbuf) + T_XBUF_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 256);  // both CTAs' 128 epilogue threads
    }
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
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileCoord c = walk.at(tile);
        const int wrow = c.g * P.I + c.nt * 128 + static_cast<int>(rank) * 64;  // this CTA's weight rows
        const int xrow = c.row0 + c.mt * 256 + static_cast<int>(rank) * (t_ncols(c) / 2);
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          const uint32_t lbar = map_to_rank(smem_u32(&full[stage]), 0);
          uint8_t* st = smem + stage * STAGE_BYTES;
#pragma unroll
          for (int j = 0; j < BK / BOX_K; ++j) {
            const int kx = kb * BK + j * BOX_K;
            tma_load_2d_pair(st + j * BOX_BYTES, &P.tmU, kx, wrow, lbar);
            tma_load_2d_pair(st + j * BOX_BYTES + BOX_BYTES / 2, &P.tmG, kx, wrow, lbar);
            tma_load_2d_pair(st + A_BYTES + j * BOX_BYTES, &P.tmX, kx, xrow, lbar);
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
    // ---------------- MMA issuer (leader only) ----------------
    if (leader) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, any = false;
      int it = 0;
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
        const TileCoord c = walk.at(tile);
        const uint32_t acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        const uint32_t idesc = idesc_bf16(256, t_ncols(c), false, false);
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, P.status, SITE_MMA));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b = a + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t off = (k / (BOX_K / 16)) * BOX_BYTES + (k % (BOX_K / 16)) * 32;
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                  "l"(sdesc_sw128(a + off, 16, 1024)), "l"(sdesc_sw128(b + off, 16, 1024)), "r"(idesc),
                  "r"(static_cast<uint32_t>((kb | k) != 0))
                  : "memory");
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
        if (lane == 0) commit2(&tfull[acc], 0x3);
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
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs) ----------------
    const int ew = warp - 4;  // TMEM lane quarter: 0, 1 hold u; 2, 3 the matching h
    const bool hwarp = ew >= 2;
    const int hq = ew & 1;               // which 32 of the CTA's 64 columns of a
    float* xb = xbuf + hq * 1024;        // [32 columns][32 lanes] of u for columns hq
    const bool issuer = ew == 2 && lane == 0;  // issues (and waits for) the TMA stores
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, P.status, SITE_EPILOGUE));
      ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(ew * 32) << 16);
      const int n = t_ncols(c);
      const int nrows = min(c.rows - c.mt * 256, 256);  // valid routed rows of the tile
      const int row0 = c.row0 + c.mt * 256;             // the tile's first row of a
      const int ocol = c.nt * 128 + static_cast<int>(rank) * 64;  // first column of a of this CTA
      // kept activations: lane = column ocol + 32 hq + lane of h (h warps) or
      // u (u warps), register j = row; each store writes 128 bytes of a row
      const bool keep = P.act && c.row0 + c.rows <= P.act_rows;
      float* kept = keep ? P.act + static_cast<int64_t>(row0) * (2 * P.I) + (hwarp ? 0 : P.I) + ocol + 32 * hq + lane
                         : nullptr;
#pragma unroll 1
      for (int ch = 0; ch * 32 < n; ++ch) {
        const int nv = min(nrows - ch * 32, 32);  // valid rows of the chunk (at least 1)
        uint32_t v[32];
        tmem_ld32(taddr + ch * 32, v);
        tmem_ld_wait();
        if (keep) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) kept[static_cast<int64_t>(ch * 32 + j) * (2 * P.I)] = __uint_as_float(v[j]);
        }
        if (!hwarp) {
#pragma unroll
          for (int j = 0; j < 32; ++j) xb[j * 32 + lane] = __uint_as_float(v[j]);
        } else if (issuer && nv == 32) {
          bulk_wait_read0();  // the previous store has read the staging box
        }
        named_bar(1, 128);  // u of the chunk in shared memory, the staging box free
        if (hwarp) {
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = silu_f(__uint_as_float(v[j])) * xb[j * 32 + lane];
          if (nv == 32) {
            // Row j, column 32 hq + lane of the box (128-byte swizzle: 16-byte
            // chunk q of row r at q ^ (r % 8)); lanes pair up so that each
            // store writes two neighbouring columns of one row.
            const bool odd = lane & 1;
            const int c2 = 32 * hq + (lane & ~1);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float recv = __shfl_xor_sync(0xffffffffu, odd ? a[j] : a[j + 1], 1);
              const int r = odd ? j + 1 : j;
              const uint32_t w = odd ? pack_bf16x2(recv, a[j + 1]) : pack_bf16x2(a[j], recv);
              st_shared_b32(ostage + r * 128 + (((c2 >> 3) ^ (r & 7)) << 4) + (c2 & 7) * 2, w);
            }
            fence_proxy_async_smem();
          } else {
            __nv_bfloat16* o = P.out + static_cast<size_t>(row0 + ch * 32) * P.I + ocol + 32 * hq + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv) o[static_cast<size_t>(j) * P.I] = __float2bfloat16_rn(a[j]);
          }
        }
        named_bar(1, 128);  // the box is written, u consumed
        if (issuer && nv == 32) {
          tma_store_2d(&P.tmOut, ostage, ocol, row0 + ch * 32);
          bulk_commit();
        }
      }
      tc_fence_before();
      if (leader) mbar_arrive(&tempty[acc]);
      else remote_arrive(map_to_rank(smem_u32(&tempty[acc]), 0));
    }
    if (issuer) bulk_wait0();  // the stores have landed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // the leader's MMAs (which read the peer's shared memory) and all remote arrivals are done
  tc_fence_after();
  if (warp == 2) tmem_dealloc2(tmem_base, 512);
}

size_t pair_t_smem_bytes(int G) {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + T_OUT_BYTES + T_XBUF_BYTES + 1024 +
         static_cast<size_t>(G + 1) * sizeof(int);
}

mok_status launch_upgate_pair_t(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                                const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                                cudaStream_t st, KeptAct kept) {
  PairTParams P{};
  P.sched = pair_sched(offsets, G, m_total, I / 128, D / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const uint64_t arows = a_rows > 0 ? a_rows : 1;
  const uint64_t wrows = static_cast<uint64_t>(G) * I;
  if (!make_tmap_2d(&P.tmX, A, kBF16, arows, D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmG, w_gate, kBF16, wrows, D, static_cast<uint64_t>(D) * 2, 64, BOX_K, true) ||
      !make_tmap_2d(&P.tmU, w_up, kBF16, wrows, D, static_cast<uint64_t>(D) * 2, 64, BOX_K, true) ||
      !out_map(&P.tmOut, a_out, m_total, I))
    return MOK_ERR_CUDA;
  P.out = static_cast<__nv_bfloat16*>(a_out);
  P.I = I;
  P.act = kept.act;
  P.act_rows = kept.limit();
  const size_t smem = pair_t_smem_bytes(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_pair_upgate_t, cudaFuncAttributeMaxDynamicSharedMemorySize,
                          static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  gemm_pair_upgate_t<<<(num_sms() / 2) * 2, 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

// Routed down projection with the routed rows as the MMA's N dimension
// (as the transposed up/gate above): CTA r holds rows d0 + 128 r .. + 127 of
// W_down as A and half of the tile's N routed rows of a as B; its
// accumulator lane d holds y[row][d0 + 128 r + d] for every routed row of
// the tile.  Epilogue warps of lane quarters 0, 1 and 2, 3 fill the two
// [32 rows][64 columns] boxes of each 32-row chunk, and one thread stores
// both.  The shared expert's down tiles (the schedule's extra group, its
// T rows in tiles of 256) run in the same launch.
//
// kDx: the backward's dX per route, dx = dh W_gate + du W_up, on the same
// tiles: the weight operand has the MMA's M = 256 D columns and K = 2I, the
// first I from W_gate and the rest from W_up, each stored [I][D] and so
// MN-major (128-row K boxes of 64 D columns, one 16-row K step every 2 KB,
// the two 64-column halves of a CTA's 128 D columns a box apart); B is the
// tile's routed rows of dh, then of du, K-major as a.
struct PairTDownParams {
  SchedArgs sched;  // bm = 256 routed rows, n_tiles = D / 256
  int* status;
  CUtensorMap tmW, tmA, tmOut;     // W_down [G * D][I], a [rows][I] (boxes 128 x 64), y [rows][D]
  CUtensorMap tmWs, tmAs, tmOut_s;  // the extra group: W_sd [D][I_s], a_s [T][I_s], ys [T][D]
  CUtensorMap tmW2, tmA2;          // kDx: W_up [G * I][D], du [rows][I] (tmW, tmA: W_gate, dh)
  __nv_bfloat16* out;
  __nv_bfloat16* out_s;
  int32_t D;
  int32_t I;                       // kDx: K blocks below I / BK read W_gate and dh
};

template <bool kDx>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    gemm_pair_down_t(const __grid_constant__ PairTDownParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ostage = smem + STAGES * STAGE_BYTES;  // two boxes, 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(ostage + 2 * T_OUT_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 256);  // both CTAs' 128 epilogue threads
    }
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
      const uint64_t keep_policy = policy_evict_last();     // re-read operands
      const uint64_t stream_policy = policy_evict_first();  // read-once weights
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileCoord c = walk.at(tile);
        const int wrow = c.g * P.D + c.nt * 256 + static_cast<int>(rank) * 128;  // this CTA's W_down rows
        const int xrow = c.row0 + c.mt * 256 + static_cast<int>(rank) * (t_ncols(c) / 2);
        const int dcol = c.nt * 256 + static_cast<int>(rank) * 128;  // kDx: this CTA's D columns
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          const uint32_t lbar = map_to_rank(smem_u32(&full[stage]), 0);
          uint8_t* st = smem + stage * STAGE_BYTES;
          if constexpr (kDx) {
            const bool up = kb * BK >= P.I;  // the second half of K: W_up and du
            const int k0 = up ? kb * BK - P.I : kb * BK;
#pragma unroll
            for (int j = 0; j < BK / BOX_K; ++j) {
              tma_load_2d_pair(st + j * BOX_BYTES, up ? &P.tmW2 : &P.tmW, dcol + 64 * j, c.g * P.I + k0, lbar);
              tma_load_2d_pair(st + A_BYTES + j * BOX_BYTES, up ? &P.tmA2 : &P.tmA, k0 + j * BOX_K, xrow, lbar);
            }
          } else if (c.extra) {
            // the shared expert's W_sd and a_s are re-read by all of its
            // tiles, which are spread through the launch: keep them in L2
            // while the routed weights stream through
#pragma unroll
            for (int j = 0; j < BK / BOX_K; ++j) {
              const int kx = kb * BK + j * BOX_K;
              tma_load_2d_pair_hint(st + j * BOX_BYTES, &P.tmWs, kx, wrow, lbar, keep_policy);
              tma_load_2d_pair_hint(st + A_BYTES + j * BOX_BYTES, &P.tmAs, kx, xrow, lbar, keep_policy);
            }
          } else {
#pragma unroll
            for (int j = 0; j < BK / BOX_K; ++j) {
              const int kx = kb * BK + j * BOX_K;
              tma_load_2d_pair_hint(st + j * BOX_BYTES, &P.tmW, kx, wrow, lbar, stream_policy);
              tma_load_2d_pair(st + A_BYTES + j * BOX_BYTES, &P.tmA, kx, xrow, lbar);
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
    // ---------------- MMA issuer (leader only) ----------------
    if (leader) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, any = false;
      int it = 0;
      TileWalker walk(P.sched, tstart);
      for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
        const TileCoord c = walk.at(tile);
        const uint32_t acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        const uint32_t idesc = idesc_bf16(256, t_ncols(c), kDx, false);
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, P.status, SITE_MMA));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b = a + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint32_t off = (k / (BOX_K / 16)) * BOX_BYTES + (k % (BOX_K / 16)) * 32;
              // kDx: A MN-major, K step k at 16 rows x 128 B, the 64-column halves a box apart
              const uint64_t adesc = kDx ? sdesc_sw128(a + k * 2048, BOX_BYTES, 1024) : sdesc_sw128(a + off, 16, 1024);
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                  "l"(adesc), "l"(sdesc_sw128(b + off, 16, 1024)), "r"(idesc),
                  "r"(static_cast<uint32_t>((kb | k) != 0))
                  : "memory");
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
        if (lane == 0) commit2(&tfull[acc], 0x3);
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
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs) ----------------
    const int ew = warp - 4;                     // TMEM lane quarter: columns 32 ew .. of the CTA's 128
    uint8_t* box = ostage + (ew >> 1) * T_OUT_BYTES;  // quarters 0, 1: box 0; 2, 3: box 1
    const bool issuer = ew == 2 && lane == 0;    // issues (and waits for) the TMA stores
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const TileCoord c = walk.at(tile);
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, P.status, SITE_EPILOGUE));
      ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(ew * 32) << 16);
      const int n = t_ncols(c);
      const int nrows = min(c.rows - c.mt * 256, 256);
      const int row0 = c.row0 + c.mt * 256;  // the tile's first row of y (of ys for the extra group)
      const int dcol = c.nt * 256 + static_cast<int>(rank) * 128;
      const CUtensorMap* tmOut = c.extra ? &P.tmOut_s : &P.tmOut;
      __nv_bfloat16* outp = c.extra ? P.out_s : P.out;
#pragma unroll 1
      for (int ch = 0; ch * 32 < n; ++ch) {
        const int nv = min(nrows - ch * 32, 32);  // valid rows of the chunk (at least 1)
        uint32_t v[32];
        tmem_ld32(taddr + ch * 32, v);
        tmem_ld_wait();
        if (issuer && nv == 32) bulk_wait_read0();  // the previous stores have read the boxes
        named_bar(1, 128);
        if (nv == 32) {
          // row j, column 32 (ew & 1) + lane of the box (128-byte swizzle);
          // lanes pair up so that each store writes two neighbouring columns
          const bool odd = lane & 1;
          const int c2 = 32 * (ew & 1) + (lane & ~1);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float recv = __shfl_xor_sync(0xffffffffu, __uint_as_float(odd ? v[j] : v[j + 1]), 1);
            const int r = odd ? j + 1 : j;
            const uint32_t w = odd ? pack_bf16x2(recv, __uint_as_float(v[j + 1]))
                                   : pack_bf16x2(__uint_as_float(v[j]), recv);
            st_shared_b32(box + r * 128 + (((c2 >> 3) ^ (r & 7)) << 4) + (c2 & 7) * 2, w);
          }
          fence_proxy_async_smem();
        } else {
          __nv_bfloat16* o = outp + static_cast<size_t>(row0 + ch * 32) * P.D + dcol + 32 * ew + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) o[static_cast<size_t>(j) * P.D] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
        named_bar(1, 128);  // both boxes written
        if (issuer && nv == 32) {
          tma_store_2d(tmOut, ostage, dcol, row0 + ch * 32);
          tma_store_2d(tmOut, ostage + T_OUT_BYTES, dcol + 64, row0 + ch * 32);
          bulk_commit();
        }
      }
      tc_fence_before();
      if (leader) mbar_arrive(&tempty[acc]);
      else remote_arrive(map_to_rank(smem_u32(&tempty[acc]), 0));
    }
    if (issuer) bulk_wait0();  // the stores have landed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // the leader's MMAs (which read the peer's shared memory) and all remote arrivals are done
  tc_fence_after();
  if (warp == 2) tmem_dealloc2(tmem_base, 512);
}

size_t pair_t_down_smem_bytes(int G) {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 2 * T_OUT_BYTES + 1024 +
         static_cast<size_t>(G + 1) * sizeof(int);
}

mok_status launch_down_pair_t(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets, int G,
                              int64_t m_total, int D, int I, void* y_out, cudaStream_t st,
                              const SharedOperands* sh) {
  PairTDownParams P{};
  P.sched = pair_sched(offsets, G, m_total, D / 256, I / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const uint64_t arows = a_rows > 0 ? a_rows : 1;
  if (!make_tmap_2d(&P.tmA, a, kBF16, arows, I, static_cast<uint64_t>(I) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmW, w_down, kBF16, static_cast<uint64_t>(G) * D, I, static_cast<uint64_t>(I) * 2, 128,
                    BOX_K, true))
    return MOK_ERR_CUDA;
  const bool routed = m_total > 0 && y_out;
  if (routed && !out_map(&P.tmOut, y_out, m_total, D)) return MOK_ERR_CUDA;
  P.out = static_cast<__nv_bfloat16*>(y_out);
  P.D = D;
  P.tmWs = P.tmW;
  P.tmAs = P.tmA;
  P.out_s = nullptr;
  if (sh && sh->rows > 0) {
    const int Is = sh->inner;
    if (!make_tmap_2d(&P.tmAs, sh->A, kBF16, sh->rows, Is, static_cast<uint64_t>(Is) * 2, 128, BOX_K, true) ||
        !make_tmap_2d(&P.tmWs, sh->w0, kBF16, D, Is, static_cast<uint64_t>(Is) * 2, 128, BOX_K, true) ||
        !out_map(&P.tmOut_s, sh->out, sh->rows, D))
      return MOK_ERR_CUDA;
    P.sched.extra_rows = static_cast<int32_t>(sh->rows);
    P.sched.extra_n_tiles = D / 256;
    P.sched.extra_k_blocks = Is / BK;
    P.out_s = static_cast<__nv_bfloat16*>(sh->out);
    if (!routed) P.tmOut = P.tmOut_s;
  } else {
    if (!routed) return MOK_OK;
    P.tmOut_s = P.tmOut;
  }
  const size_t smem = pair_t_down_smem_bytes(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_pair_down_t<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                          static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  gemm_pair_down_t<false><<<(num_sms() / 2) * 2, 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_dx_pair_t_impl(const void* dh, const void* du, int64_t rows, const void* w_gate, const void* w_up,
                                 const int32_t* offsets, int G, int D, int I, void* dx, cudaStream_t st, int max_sms) {
  PairTDownParams P{};
  P.sched = pair_sched(offsets, G, rows, D / 256, 2 * I / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const uint64_t wrows = static_cast<uint64_t>(G) * I;
  // dh, du K-major (128 routed rows x 64 K per box); W_gate, W_up [G I][D]
  // MN-major (128 K rows x 64 D columns per box)
  if (!make_tmap_2d(&P.tmA, dh, kBF16, rows, I, static_cast<uint64_t>(I) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmA2, du, kBF16, rows, I, static_cast<uint64_t>(I) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmW, w_gate, kBF16, wrows, D, static_cast<uint64_t>(D) * 2, BK, 64, true) ||
      !make_tmap_2d(&P.tmW2, w_up, kBF16, wrows, D, static_cast<uint64_t>(D) * 2, BK, 64, true) ||
      !out_map(&P.tmOut, dx, rows, D))
    return MOK_ERR_CUDA;
  P.out = static_cast<__nv_bfloat16*>(dx);
  P.out_s = nullptr;
  P.tmWs = P.tmW;
  P.tmAs = P.tmA;
  P.tmOut_s = P.tmOut;
  P.D = D;
  P.I = I;
  const size_t smem = pair_t_down_smem_bytes(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_pair_down_t<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  const int sms = max_sms > 0 && max_sms < num_sms() ? max_sms : num_sms();
  gemm_pair_down_t<true><<<sms >= 2 ? (sms / 2) * 2 : 2, 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

}  // namespace

mok_status launch_dx_pair_t(const void* dh, const void* du, int64_t rows, const void* w_gate, const void* w_up,
                            const int32_t* offsets, int G, int D, int I, void* dx, cudaStream_t st, int max_sms) {
  if (rows == 0) return MOK_OK;
  if ((offsets && G < 1) || D % 256 || I % BK) return MOK_ERR_INVALID_ARG;
  return launch_dx_pair_t_impl(dh, du, rows, w_gate, w_up, offsets, offsets ? G : 1, D, I, dx, st, max_sms);
}

mok_status launch_upgate_pair(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                              const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                              cudaStream_t st, const SharedOperands* sh, KeptAct kept, int max_sms) {
  if (m_total == 0 && !(sh && sh->rows)) return MOK_OK;
  // Routed rows alone, fewer than 512 per expert on average: the transposed
  // kernel, whose MMAs skip the padding rows of each expert's last tile
  // (DSV3 forward 4.57 -> 4.51 ms).  With larger groups there is little
  // padding, and the row-major kernel's lighter epilogue measured 0.3-0.6 %
  // faster (the skewed 16384-token layer).  One group (the shared expert on
  // its own stream): the transposed kernel too, whose 147 registers a thread
  // (the row-major one takes 229) leave room on every SM for the route,
  // plan and dispatch blocks that run beside it.
  if (!(sh && sh->rows) && (!offsets || routed_rows_as_n(m_total, G)))
    return launch_upgate_pair_t(A, a_rows, w_gate, w_up, offsets, G, m_total, D, I, a_out, st, kept);
  PairParams P{};
  P.sched = pair_sched(offsets, G, m_total, I / 128, D / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int groups = offsets ? G : 1;
  const uint64_t arows = a_rows > 0 ? a_rows : 1;
  if (!make_tmap_2d(&P.tmA, A, kBF16, arows, D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmB0, w_gate, kBF16, static_cast<uint64_t>(groups) * I, D, static_cast<uint64_t>(D) * 2,
                    128, BOX_K, true) ||
      !make_tmap_2d(&P.tmB1, w_up, kBF16, static_cast<uint64_t>(groups) * I, D, static_cast<uint64_t>(D) * 2,
                    128, BOX_K, true))
    return MOK_ERR_CUDA;
  P.b_group_rows = I;
  P.b_tile_rows = 128;
  P.b1_off = 0;
  P.out = static_cast<__nv_bfloat16*>(a_out);
  P.out_ld = I;
  P.tmAs = P.tmA;
  P.tmBs0 = P.tmB0;
  P.tmBs1 = P.tmB1;
  P.out_s = nullptr;
  P.out_ld_s = 0;
  if (sh && sh->rows > 0) {
    const int Is = sh->inner;
    if (!make_tmap_2d(&P.tmAs, sh->A, kBF16, sh->rows, D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true) ||
        !make_tmap_2d(&P.tmBs0, sh->w0, kBF16, Is, D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true) ||
        !make_tmap_2d(&P.tmBs1, sh->w1, kBF16, Is, D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true))
      return MOK_ERR_CUDA;
    P.sched.extra_rows = static_cast<int32_t>(sh->rows);
    P.sched.extra_n_tiles = Is / 128;
    P.sched.extra_k_blocks = D / BK;
    P.out_s = static_cast<__nv_bfloat16*>(sh->out);
    P.out_ld_s = Is;
  }
  // kept h, u: every group whose rows end at or below kept.rows (offsets
  // null: the one group of m_total rows)
  P.act = kept.act;
  P.act_rows = kept.limit();
  P.act_i = I;
  if (!set_out_maps(P, m_total)) return MOK_ERR_CUDA;
  return run_pair<true>(P, st, max_sms);
}

mok_status launch_down_pair(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets, int G,
                            int64_t m_total, int D, int I, void* y_out, cudaStream_t st,
                            const SharedOperands* sh, int max_sms) {
  if (m_total == 0 && !(sh && sh->rows)) return MOK_OK;
  // routed groups of fewer than 512 rows on average, or one group: the
  // transposed kernel (no padding rows in the MMAs, fewer registers), as
  // for the up/gate
  if (!offsets || routed_rows_as_n(m_total, G))
    return launch_down_pair_t(a, a_rows, w_down, offsets, G, m_total, D, I, y_out, st, sh);
  PairParams P{};
  P.sched = pair_sched(offsets, G, m_total, D / 256, I / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int groups = offsets ? G : 1;
  const uint64_t arows = a_rows > 0 ? a_rows : 1;
  if (!make_tmap_2d(&P.tmA, a, kBF16, arows, I, static_cast<uint64_t>(I) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmB0, w_down, kBF16, static_cast<uint64_t>(groups) * D, I, static_cast<uint64_t>(I) * 2,
                    128, BOX_K, true))
    return MOK_ERR_CUDA;
  P.tmB1 = P.tmB0;
  P.b_group_rows = D;
  P.b_tile_rows = 256;
  P.b1_off = 128;
  P.out = static_cast<__nv_bfloat16*>(y_out);
  P.out_ld = D;
  P.tmAs = P.tmA;
  P.tmBs0 = P.tmB0;
  P.tmBs1 = P.tmB0;
  P.out_s = nullptr;
  P.out_ld_s = 0;
  if (sh && sh->rows > 0) {
    const int Is = sh->inner;
    if (!make_tmap_2d(&P.tmAs, sh->A, kBF16, sh->rows, Is, static_cast<uint64_t>(Is) * 2, 128, BOX_K, true) ||
        !make_tmap_2d(&P.tmBs0, sh->w0, kBF16, D, Is, static_cast<uint64_t>(Is) * 2, 128, BOX_K, true))
      return MOK_ERR_CUDA;
    P.tmBs1 = P.tmBs0;
    P.sched.extra_rows = static_cast<int32_t>(sh->rows);
    P.sched.extra_n_tiles = D / 256;
    P.sched.extra_k_blocks = Is / BK;
    P.out_s = static_cast<__nv_bfloat16*>(sh->out);
    P.out_ld_s = D;
  }
  if (!set_out_maps(P, m_total)) return MOK_ERR_CUDA;
  return run_pair<false>(P, st, max_sms);
}

mok_status launch_upgate(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                         const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                         cudaStream_t st, int max_sms, KeptAct kept) {
  if (a_rows == 0 || m_total == 0) return MOK_OK;
  return launch_upgate_pair(A, a_rows, w_gate, w_up, offsets, G, m_total, D, I, a_out, st, nullptr, kept, max_sms);
}

mok_status launch_down(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets,
                       int G, int64_t m_total, int D, int I, void* y_out, cudaStream_t st, int max_sms) {
  return launch_down_pair(a, a_rows, w_down, offsets, G, m_total, D, I, y_out, st, nullptr, max_sms);
}

mok_status launch_router_pair(const void* x, int64_t T, const void* w_router, int E, int D, float* s_out,
                              cudaStream_t st) {
  if (T == 0) return MOK_OK;
  if (E < 1 || E > 256) return MOK_ERR_UNSUPPORTED;
  PairParams P{};
  P.sched = pair_sched(nullptr, 1, T, 1, D / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  if (!make_tmap_2d(&P.tmA, x, kBF16, static_cast<uint64_t>(T), D, static_cast<uint64_t>(D) * 2, 128, BOX_K, true) ||
      !make_tmap_2d(&P.tmB0, w_router, kBF16, static_cast<uint64_t>(E), D, static_cast<uint64_t>(D) * 2, 128, BOX_K,
                    true))
    return MOK_ERR_CUDA;
  P.tmB1 = P.tmB0;  // experts 128..255 (rows past E read as zeros, masked in the epilogue)
  P.b_group_rows = 0;
  P.b_tile_rows = 0;
  P.b1_off = 128;
  P.tmAs = P.tmA;
  P.tmBs0 = P.tmB0;
  P.tmBs1 = P.tmB0;
  P.s_out = s_out;
  P.E = E;
  return run_pair<false, false, true>(P, st);
}

mok_status launch_upgate_ring(const void* x, const int32_t* table, int K, const void* w_gate, const void* w_up,
                              const int32_t* offsets, int G, int64_t R, int D, int I, void* a_out, void* ring,
                              int64_t ring_rows, int chunk_rows, int32_t* counters, cudaStream_t st,
                              KeptAct kept) {
  if (R == 0) return MOK_OK;
  if (!offsets || chunk_rows < 128 || ring_rows < chunk_rows || ring_rows % chunk_rows) return MOK_ERR_INVALID_ARG;
  const int64_t nchunks = (R + chunk_rows - 1) / chunk_rows;
  if (nchunks > (int64_t{1} << 24)) return MOK_ERR_INVALID_ARG;
  if (cudaMemsetAsync(counters, 0, 2 * nchunks * sizeof(int32_t), st) != cudaSuccess) return MOK_ERR_CUDA;
  PairParams P{};
  P.sched = pair_sched(offsets, G, R, I / 128, D / BK);
  P.sched.m_outer = 1;  // rows leave the ring in order: all N tiles of an M tile before the next M tile
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  if (!make_tmap_2d(&P.tmA, ring, kBF16, static_cast<uint64_t>(ring_rows) + 128, D, static_cast<uint64_t>(D) * 2,
                    128, BOX_K, true) ||
      !make_tmap_2d(&P.tmB0, w_gate, kBF16, static_cast<uint64_t>(G) * I, D, static_cast<uint64_t>(D) * 2, 128, BOX_K,
                    true) ||
      !make_tmap_2d(&P.tmB1, w_up, kBF16, static_cast<uint64_t>(G) * I, D, static_cast<uint64_t>(D) * 2, 128, BOX_K,
                    true))
    return MOK_ERR_CUDA;
  P.b_group_rows = I;
  P.b_tile_rows = 128;
  P.b1_off = 0;
  P.out = static_cast<__nv_bfloat16*>(a_out);
  P.out_ld = I;
  P.tmAs = P.tmA;
  P.tmBs0 = P.tmB0;
  P.tmBs1 = P.tmB1;
  P.x = static_cast<const uint4*>(x);
  P.table = table;
  P.K = K;
  P.D8 = D / 8;
  P.ring = static_cast<uint4*>(ring);
  P.ring_rows = ring_rows;
  P.R = R;
  P.chunk_rows = chunk_rows;
  P.nchunks = static_cast<int32_t>(nchunks);
  P.n_tiles = I / 128;
  P.ready = counters;
  P.done = counters + nchunks;
  P.act = kept.act;
  P.act_rows = kept.limit();
  P.act_i = I;
  if (!set_out_maps(P, R)) return MOK_ERR_CUDA;
  return run_pair<true, true>(P, st);
}

}  // namespace mok
