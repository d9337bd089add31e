// Persistent, warp-specialised grouped GEMM skeleton for tcgen05 / TMEM.
//
// One CTA per SM walks a static tile list (tile = blockIdx.x + i*gridDim.x).
// Tiles are numbered group-major, then N tile, then M tile (M fastest), so
// the M tiles that share one weight tile run at the same time and the second
// read of that tile hits L2.
//
// Roles (256 threads):
//   warp 0      TMA producer (lane 0) -> smem ring of STAGES stages
//   warp 1      MMA issuer: the warp waits, lane 0 issues tcgen05.mma and
//               tcgen05.commit; the warp may patch a stage first (Cfg::fixup)
//   warp 2      TMEM allocator (alloc at start, dealloc at exit)
//   warp 3      builds the group -> tile table in shared memory
//   warps 4..7  epilogue: tcgen05.ld of TMEM lanes 32*(warp%4).. , math, store
// Accumulators are double buffered in TMEM when Cfg::NUM_ACC == 2, so the
// epilogue of one tile overlaps the main loop of the next.
//
// Every mbarrier wait is bounded (common.cuh); on a timeout the CTA records
// MOK_ERR_TIMEOUT, drains its own TMA loads and MMAs, frees TMEM and returns.
#pragma once

#include "common.cuh"

namespace mok {

// How tiles and K blocks follow from the group row ranges.
struct SchedArgs {
  const int32_t* offsets;  // [G+1] group row ranges; null => one group of m_total rows
  int32_t G;
  int32_t m_total;
  int32_t n_tiles;         // N tiles per group
  int32_t m_tiles_fixed;   // > 0: every group has this many M tiles; 0: ceil(M_g / bm)
  int32_t k_blocks_fixed;  // > 0: K blocks per tile; 0: ceil(M_g / bk_rows) (K runs over rows)
  int32_t bm;
  int32_t bk_rows;
  // Optional extra group (the shared expert) with its own operands: rows
  // [0, extra_rows), extra_n_tiles N tiles, extra_k_blocks K blocks.  Its
  // tiles are spread evenly through the tile order (extra_rows = 0: none).
  int32_t extra_rows = 0;
  int32_t extra_n_tiles = 0;
  int32_t extra_k_blocks = 0;
  // Order of a group's tiles: N tile outer, M tile fastest (default: the M
  // tiles that share a weight tile run together), or M tile outer (rows are
  // consumed in order, as a ring dispatch needs).
  int32_t m_outer = 0;
  // Optional split of the groups at a row limit: split_side 1 keeps only the
  // groups whose rows all lie below row_split (offsets[g + 1] <= row_split),
  // split_side 2 only the others; the rest get no tiles.  0: every group.
  int32_t row_split = 0;
  int32_t split_side = 0;
};

struct TileCoord {
  int extra;  // 1: a tile of the extra group
  int g, mt, nt;
  int row0;     // first row of the group
  int rows;     // rows of the group
  int kblocks;  // K blocks of this tile (0: no MMA, the accumulator is zero)
};

__device__ __forceinline__ int sched_m_tiles(const SchedArgs& s, int rows) {
  return s.m_tiles_fixed > 0 ? s.m_tiles_fixed : (rows + s.bm - 1) / s.bm;
}
__device__ __forceinline__ int sched_k_blocks(const SchedArgs& s, int rows) {
  return s.k_blocks_fixed > 0 ? s.k_blocks_fixed : (rows + s.bk_rows - 1) / s.bk_rows;
}

// Tiles of a group with rows [r0, r1), after the optional row split.
__device__ __forceinline__ int group_tiles(const SchedArgs& s, int r0, int r1) {
  if (s.split_side == 1 && r1 > s.row_split) return 0;
  if (s.split_side == 2 && r1 <= s.row_split) return 0;
  return sched_m_tiles(s, r1 - r0) * s.n_tiles;
}

__device__ __forceinline__ int extra_tiles(const SchedArgs& s) {
  return s.extra_rows > 0 ? ((s.extra_rows + s.bm - 1) / s.bm) * s.extra_n_tiles : 0;
}

// Warp-wide: tstart[g] = first tile of group g (exclusive scan), [G+1].
// Returns the tile count.  (Rows of a group come from s.offsets when a
// role reaches the group, so only the tile starts take shared memory.)
__device__ __forceinline__ int build_tile_table(const SchedArgs& s, int* tstart, int lane) {
  const int G = s.G;
  const int per = (G + 31) / 32;
  const int g0 = lane * per;
  int local = 0;
  for (int g = g0; g < g0 + per && g < G; ++g) {
    int r0 = s.offsets ? s.offsets[g] : 0;
    int r1 = s.offsets ? s.offsets[g + 1] : s.m_total;
    local += group_tiles(s, r0, r1);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int g = g0; g < g0 + per && g < G; ++g) {
    tstart[g] = run;
    int r0 = s.offsets ? s.offsets[g] : 0;
    int r1 = s.offsets ? s.offsets[g + 1] : s.m_total;
    run += group_tiles(s, r0, r1);
  }
  int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) tstart[G] = total;
  return total + extra_tiles(s);
}

// Tile -> coordinates for one role of a CTA.  Every role walks its tiles in
// increasing order (first + i * stride), so the group of the next tile is
// found by stepping forward from the group of the previous one, and the
// per-group quantities (rows, M tiles, K blocks) are recomputed only when the
// group changes; a tile then costs one integer division.
//
// Tile order with an extra group of S tiles among Rt grouped ones: positions
// k*p + p - 1 (k < S, p = (Rt + S) / S) hold the extra tiles, the rest the
// grouped tiles in order.
struct TileWalker {
  const SchedArgs& s;
  const int* tstart;
  int S, p, extra_mtiles;
  int g;                                    // group of the last grouped tile
  int cg, crow0, crows, cmtiles, ckblocks;  // cached quantities of group cg

  __device__ __forceinline__ TileWalker(const SchedArgs& s_, const int* tstart_)
      : s(s_), tstart(tstart_), g(0), cg(-1) {
    S = extra_tiles(s);
    p = S > 0 ? (tstart[s.G] + S) / S : 1;
    extra_mtiles = S > 0 ? (s.extra_rows + s.bm - 1) / s.bm : 1;
  }

  __device__ __forceinline__ TileCoord at(int tile) {
    TileCoord c;
    int gt = tile;
    if (S > 0) {
      const int q = tile / p;
      if (tile - q * p == p - 1 && q < S) {
        c.extra = 1;
        c.g = 0;
        c.nt = q / extra_mtiles;
        c.mt = q - c.nt * extra_mtiles;
        c.row0 = 0;
        c.rows = s.extra_rows;
        c.kblocks = s.extra_k_blocks;
        return c;
      }
      gt = tile - (q < S ? q : S);
    }
    // last group whose first tile is <= gt (steps over empty groups)
    while (g + 1 < s.G && tstart[g + 1] <= gt) ++g;
    if (g != cg) {
      cg = g;
      crow0 = s.offsets ? __ldg(s.offsets + g) : 0;
      crows = (s.offsets ? __ldg(s.offsets + g + 1) : s.m_total) - crow0;
      cmtiles = sched_m_tiles(s, crows);
      ckblocks = sched_k_blocks(s, crows);
    }
    c.extra = 0;
    c.g = g;
    c.row0 = crow0;
    c.rows = crows;
    const int local = gt - tstart[g];
    if (s.m_outer) {
      c.mt = local / s.n_tiles;
      c.nt = local - c.mt * s.n_tiles;
    } else {
      c.nt = local / cmtiles;
      c.mt = local - c.nt * cmtiles;
    }
    c.kblocks = ckblocks;
    return c;
  }
};

// Shared memory: [STAGES x STAGE_BYTES][EPI_SMEM_BYTES epilogue staging,
// 1 KB aligned][256 B barriers and flags][tile starts, G + 1 ints].
template <class Cfg>
constexpr size_t gemm_smem_bytes(int G) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(Cfg::STAGES) * Cfg::STAGE_BYTES + Cfg::EPI_SMEM_BYTES +
         256 /*barriers and flags*/ + static_cast<size_t>(G + 1) * sizeof(int);
}

// Cfg interface:
//   STAGES, STAGE_BYTES, NUM_ACC (1|2), ACC_COLS (TMEM columns per buffer),
//   full_arrivals(P) / tx_bytes(P): arrivals and TMA bytes that complete a stage,
//   TMEM_COLS (power of two >= NUM_ACC*ACC_COLS)
//   struct Params { SchedArgs sched; int* status; ... }
//   static __device__ void load(const Params&, const TileCoord&, int kb, uint8_t* stage,
//                               uint64_t* full_bar, int lane);    // all lanes of warp 0
//   static __device__ void fixup(const Params&, const TileCoord&, int kb, uint8_t* stage,
//                                int lane);                       // whole warp 1
//   static __device__ void mma(const Params&, const TileCoord&, int kb, uint8_t* stage,
//                              uint32_t d_tmem);                  // lane 0 of warp 1
//   EPI_SMEM_BYTES: shared staging for the epilogue (a quarter per epilogue warp)
//   static __device__ void epilogue(const Params&, const TileCoord&, uint32_t taddr, int ew,
//                                   int lane, bool has_acc, uint8_t* epi);  // warps 4..7
template <class Cfg>
__global__ void __launch_bounds__(256, 1) gemm_persistent(const __grid_constant__ typename Cfg::Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  static_assert((2 * Cfg::STAGES + 5) * sizeof(uint64_t) + 3 * sizeof(uint32_t) <= 256, "barrier area");
  uint8_t* epi_smem = smem + Cfg::STAGES * Cfg::STAGE_BYTES;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_smem + Cfg::EPI_SMEM_BYTES);
  uint64_t* empty = full + Cfg::STAGES;
  uint64_t* tfull = empty + Cfg::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* total_holder = reinterpret_cast<int*>(tmem_holder + 2);
  int* tstart = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + 256);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::STAGES; ++i) {
      mbar_init(&full[i], Cfg::full_arrivals(P));
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
  if (warp == 3) {
    int total = build_tile_table(P.sched, tstart, lane);
    if (lane == 0) *total_holder = total;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // Lane 0 waits for a free stage and arms its barrier; then every lane
    // may issue copies into it (Cfg::load decides which lanes do).
    uint32_t stage = 0, phase = 0;
    uint32_t issued_parity[Cfg::STAGES];
    bool issued[Cfg::STAGES];
    for (int i = 0; i < Cfg::STAGES; ++i) issued[i] = false;
    bool ok = true;
    TileWalker walk(P.sched, tstart);
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileCoord c = walk.at(tile);
      for (int kb = 0; kb < c.kblocks; ++kb) {
        bool got = false;
        if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER);
        ok = __shfl_sync(0xffffffffu, got, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], Cfg::tx_bytes(P));
        __syncwarp();
        Cfg::load(P, c, kb, smem + stage * Cfg::STAGE_BYTES, &full[stage], lane);
        issued[stage] = true;
        issued_parity[stage] = phase;
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // Let every load issued into a stage land before the CTA exits.
      for (int i = 0; i < Cfg::STAGES; ++i) {
        if (!issued[i]) continue;
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&full[i], issued_parity[i]) &&
               globaltimer() - t0 < kWaitBudgetNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    uint32_t stage = 0, phase = 0;
    bool ok = true, any = false;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const TileCoord c = walk.at(tile);
      const uint32_t acc = (Cfg::NUM_ACC == 2) ? (it & 1) : 0;
      const uint32_t acc_phase = (Cfg::NUM_ACC == 2) ? ((it >> 1) & 1) : (it & 1);
      // Waits are taken by every lane and made warp-uniform, so the warp
      // never splits around __syncwarp or the fixup.
      ok = __all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, P.status, SITE_MMA));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * Cfg::ACC_COLS;
      for (int kb = 0; kb < c.kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA));
        if (!ok) break;
        tc_fence_after();
        Cfg::fixup(P, c, kb, smem + stage * Cfg::STAGE_BYTES, lane);
        __syncwarp();
        if (lane == 0) {
          Cfg::mma(P, c, kb, smem + stage * Cfg::STAGE_BYTES, d_tmem);
          mma_commit(&empty[stage]);
          any = true;
        }
        __syncwarp();
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
    }
    any = __shfl_sync(0xffffffffu, any, 0);
    if (any) {
      // All MMAs of this CTA complete before TMEM is released.
      if (lane == 0) mma_commit(drain);
      __syncwarp();
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitBudgetNs) {
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int ew = warp - 4;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const TileCoord c = walk.at(tile);
      const uint32_t acc = (Cfg::NUM_ACC == 2) ? (it & 1) : 0;
      const uint32_t acc_phase = (Cfg::NUM_ACC == 2) ? ((it >> 1) & 1) : (it & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, P.status, SITE_EPILOGUE)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * Cfg::ACC_COLS + (static_cast<uint32_t>(ew * 32) << 16);
      Cfg::epilogue(P, c, taddr, ew, lane, c.kblocks > 0, epi_smem + ew * (Cfg::EPI_SMEM_BYTES / 4));
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    // bulk stores issued from staging must finish before shared memory goes
    if (Cfg::EPI_SMEM_BYTES > 0 && lane == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace mok
