// Backward grouped GEMMs on tcgen05 / TMEM.
//
//  dgrad+replay : per (expert, up to 160 rows, 128 cols of I) one CTA
//                 accumulates h^T = W_gate xg^T, u^T = W_up xg^T (the
//                 forward replay) and t^T = W_down^T dYg^T (W_down read
//                 MN-major) in three TMEM accumulators over K = D.  The epilogue forms, per row,
//                 a = bf16(SiLU(h) u), the router-gradient partial <t, a>
//                 (paper note "The production details": the down-projection
//                 output is never formed), da = g t,
//                 dh = bf16(da u SiLU'(h)), du = bf16(da SiLU(h)), a_g = bf16(g a).
//  dgrad, kept  : the same for the experts whose h, u the forward kept
//                 (paper note, "A ring buffer instead of a host round-trip":
//                 the backward replays only what it no longer has): only
//                 t^T = W_down^T dYg^T is accumulated (W_gate and W_up are
//                 not streamed), and the epilogue reads h, u fp32 from the
//                 kept store.
//  dx           : dx = bf16(dh W_gate + du W_up), K = 2I, weights MN-major.
//  wgrad        : dW[e] = bf16(sum over the expert's rows of P^T Q) with both
//                 operands MN-major and K running over rows; the last K block
//                 of an expert stops at its end (16-row MMA steps, the few
//                 rows past the end zeroed in A).  Clusters of two CTAs take
//                 neighbouring M tiles and share B: each loads half of it
//                 and multicasts that half into both CTAs' stages.
#include "gemm_core.cuh"
#include "kernels.h"
#include "pair.cuh"

namespace mok {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int KTILE = BM * BK * 2;  // 16 KB: 128 x 64 bf16, K-major
constexpr int MNCHUNK = 64 * 128;   // 8 KB: 64 K-rows x 64 MN elements, MN-major

// 128-byte swizzled descriptors: K-major (SBO 1024) and MN-major (LBO = one
// 64-wide MN chunk = 8 KB, SBO 1024).
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sdesc_sw128(a, 16, 1024); }
__device__ __forceinline__ uint64_t mndesc(uint32_t a) { return sdesc_sw128(a, MNCHUNK, 1024); }

// ---------------------------------------------------------------------------
// The fused epilogue of row a9 for one 32-row chunk of a dgrad tile.  Lane l
// owns I column icol = nt*128 + 32 ew + l; h[j], u[j], t[j] are row
// row0 + j's values of that column (fp32 bits).  Per row it forms
// a = bf16(SiLU(h) u), da = g t, dh = bf16(da u SiLU'(h)),
// du = bf16(da SiLU(h)), a_g = bf16(g a) (each row's 32 columns of the warp
// are one 64-byte store), and the warp's partial of the router-gradient
// inner product <t, SiLU(h) u> of each row over its 32 columns, with the
// gated activation unrounded (fp32), by a butterfly that leaves row j = l's
// sum in lane l, stored at dgp[row][nt*4 + ew].  nv: valid rows of the chunk.
template <class Params>
__device__ __forceinline__ void dgrad_chunk(const Params& P, const TileCoord& c, int64_t row0, int nv, int ew,
                                            int lane, const uint32_t* hv, const uint32_t* uv, const uint32_t* tv) {
  const int icol = c.nt * 128 + ew * 32 + lane;
  const int nI32 = P.I / 32;
  const float gl = (P.g_route && lane < nv) ? P.g_route[row0 + lane] : 1.0f;
  float dots[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float g = __shfl_sync(0xffffffffu, gl, j);
    const float h = __uint_as_float(hv[j]);
    const float u = __uint_as_float(uv[j]);
    const float t = __uint_as_float(tv[j]);
    const float sig = sigmoid_f(h);
    const float a_pre = (h * sig) * u;  // = silu_f(h) * u
    const float a = __bfloat162float(__float2bfloat16_rn(a_pre));
    dots[j] = t * a_pre;
    const float da = g * t;
    if (j < nv) {
      const size_t o = static_cast<size_t>(row0 + j) * P.I + icol;
      P.dh[o] = __float2bfloat16_rn(da * u * sig * (1.0f + h * (1.0f - sig)));
      P.du[o] = __float2bfloat16_rn(da * h * sig);
      P.ag[o] = __float2bfloat16_rn(g * a);
    }
  }
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) {
    const bool upper = (lane & sh) != 0;
#pragma unroll
    for (int j = 0; j < sh; ++j) {
      const float send = upper ? dots[j] : dots[j + sh];
      const float keep = upper ? dots[j + sh] : dots[j];
      dots[j] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
    }
  }
  if (P.dgp && lane < nv) P.dgp[(row0 + lane) * nI32 + c.nt * 4 + ew] = dots[0];
}

// ---------------------------------------------------------------------------
struct DgradCfg {
  // Transposed products: the weights are the M operand (128 I columns of
  // W_gate, W_up and W_down per tile) and the expert's rows the N operand
  // (up to 160 rows, N = rows rounded up to 16), so a ragged row count costs
  // at most 15 idle MMA columns, where 128-row tiles would run a second,
  // mostly empty tile that streams the same weights again.  The accumulators
  // are h^T, u^T, t^T: TMEM lane = I column, column = row.  32-wide K blocks
  // (64-byte swizzle) keep five 44 KB stages in flight.
  static constexpr int BKD = 32;
  static constexpr int ROWS = 160;                // rows per tile: three accumulators of 160 columns
  static constexpr int WT = 128 * BKD * 2;        // 8 KB: 128 weight rows x 32 bf16, K-major
  static constexpr int WDCHUNK = BKD * 128;       // 4 KB: 32 K rows x 64 I columns, MN-major
  static constexpr int RT = ROWS * BKD * 2;       // 10 KB: 160 rows x 32 bf16, K-major
  static constexpr int OFF_WU = WT, OFF_WD = 2 * WT, OFF_X = 2 * WT + 2 * WDCHUNK, OFF_DY = OFF_X + RT;
  static constexpr int STAGES = 5;
  static constexpr int STAGE_BYTES = OFF_DY + RT;  // 44 KB: W_gate, W_up, W_down, x, dY
  static constexpr int EPI_SMEM_BYTES = 0;
  static constexpr int NUM_ACC = 1;
  static constexpr int ACC_COLS = 3 * ROWS;  // h^T | u^T | t^T
  static constexpr uint32_t TMEM_COLS = 512;

  struct Params {
    SchedArgs sched;         // bm = ROWS
    int* status;
    CUtensorMap tmX, tmDy;   // [rows][D], K-major boxes 160 x 32, 64-byte swizzle
    CUtensorMap tmWg, tmWu;  // [G*I][D], K-major boxes 128 x 32, 64-byte swizzle
    CUtensorMap tmWd;        // [G*D][I], MN-major boxes 32 x 64, 128-byte swizzle
    int32_t I, D;
    const float* g_route;    // [rows] or null (weight 1)
    __nv_bfloat16 *dh, *du, *ag;  // [rows][I]
    float* dgp;              // [rows][I/32] or null
  };

  // K-major, 64-byte swizzle: 8-row groups of 64-byte rows 512 B apart.
  __device__ static uint64_t kdesc64(uint32_t a) {
    uint64_t d = static_cast<uint64_t>((a & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(512 >> 4) << 32;
    d |= 1ull << 46;
    d |= 4ull << 61;
    return d;
  }

  __device__ static uint32_t full_arrivals(const Params&) { return 1; }
  __device__ static uint32_t tx_bytes(const Params&) { return STAGE_BYTES; }

  __device__ static void load(const Params& P, const TileCoord& c, int kb, uint8_t* st,
                              uint64_t* bar, int lane) {
    if (lane != 0) return;
    const int k0 = kb * BKD;
    const int wrow = c.g * P.I + c.nt * 128;
    tma_load_2d(st, &P.tmWg, k0, wrow, bar);
    tma_load_2d(st + OFF_WU, &P.tmWu, k0, wrow, bar);
    const int drow = c.g * P.D + k0;
    tma_load_2d(st + OFF_WD, &P.tmWd, c.nt * 128, drow, bar);
    tma_load_2d(st + OFF_WD + WDCHUNK, &P.tmWd, c.nt * 128 + 64, drow, bar);
    const int r = c.row0 + c.mt * ROWS;
    tma_load_2d(st + OFF_X, &P.tmX, k0, r, bar);
    tma_load_2d(st + OFF_DY, &P.tmDy, k0, r, bar);
  }

  __device__ static void fixup(const Params&, const TileCoord&, int, uint8_t*, int) {}

  // Rows past the tile's end within the N rounding belong to the next group
  // (or are TMA zero fill): their accumulator columns are never read.
  __device__ static int tile_rows(const TileCoord& c) {
    const int n = c.rows - c.mt * ROWS;
    return n < ROWS ? n : ROWS;
  }

  __device__ static void mma(const Params&, const TileCoord& c, int kb, uint8_t* st, uint32_t d) {
    const uint32_t s = smem_u32(st);
    const int n = (tile_rows(c) + 15) & ~15;
    const uint32_t id_hu = idesc_bf16(128, n, false, false);
    const uint32_t id_t = idesc_bf16(128, n, true, false);
#pragma unroll
    for (int k = 0; k < BKD / 16; ++k) {
      const uint32_t acc = (kb | k) != 0;
      const uint64_t bx = kdesc64(s + OFF_X + k * 32);
      mma_bf16(d, kdesc64(s + k * 32), bx, id_hu, acc);
      mma_bf16(d + ROWS, kdesc64(s + OFF_WU + k * 32), bx, id_hu, acc);
      mma_bf16(d + 2 * ROWS, sdesc_sw128(s + OFF_WD + k * 2048, WDCHUNK, 1024), kdesc64(s + OFF_DY + k * 32),
               id_t, acc);
    }
  }

  // Lane l of warp w owns I column nt*128 + 32w + l; per chunk of 32 rows
  // it loads h, u, t of those rows and runs dgrad_chunk.
  __device__ static void epilogue(const Params& P, const TileCoord& c, uint32_t taddr, int ew,
                                  int lane, bool, uint8_t*) {
    const int nrows = tile_rows(c);
    const int64_t row0 = c.row0 + c.mt * ROWS;
#pragma unroll 1
    for (int cc = 0; cc * 32 < nrows; ++cc) {
      uint32_t hv[32], uv[32], tv[32];
      tmem_ld32(taddr + cc * 32, hv);
      tmem_ld32(taddr + ROWS + cc * 32, uv);
      tmem_ld32(taddr + 2 * ROWS + cc * 32, tv);
      tmem_ld_wait();
      dgrad_chunk(P, c, row0 + cc * 32, min(nrows - cc * 32, 32), ew, lane, hv, uv, tv);
    }
  }
};

// ---------------------------------------------------------------------------
// dgrad of the experts whose h, u the forward kept: t^T = W_down^T dYg^T
// only (TMEM lane = I column, column = row, as DgradCfg), 64-wide K blocks
// (W_down MN-major, dY K-major, both 128-byte swizzle), two accumulators so
// that a tile's epilogue overlaps the next tile's loads and MMAs.  The
// epilogue reads the kept h, u (fp32, [rows][2I]: h then u) of its rows:
// per row the warp's 32 lanes read 128 contiguous bytes of each.
struct DgradKeptCfg {
  static constexpr int BKD = 64;
  static constexpr int ROWS = 160;                // rows per tile (N = rows rounded up to 16)
  static constexpr int WDCHUNK = BKD * 128;       // 8 KB: 64 K rows x 64 I columns, MN-major
  static constexpr int RT = ROWS * BKD * 2;       // 20 KB: 160 rows x 64 bf16, K-major
  static constexpr int OFF_DY = 2 * WDCHUNK;
  static constexpr int STAGES = 5;
  static constexpr int STAGE_BYTES = OFF_DY + RT;  // 36 KB: W_down, dY
  static constexpr int EPI_SMEM_BYTES = 0;
  static constexpr int NUM_ACC = 2;
  static constexpr int ACC_COLS = ROWS;
  static constexpr uint32_t TMEM_COLS = 512;

  struct Params {
    SchedArgs sched;         // bm = ROWS; split_side 1: the kept groups only
    int* status;
    CUtensorMap tmDy;        // [rows][D], K-major boxes 160 x 64
    CUtensorMap tmWd;        // [G*D][I], MN-major boxes 64 x 64
    int32_t I, D;
    const float* g_route;    // [rows] or null (weight 1)
    const float* act;        // kept h, u [rows][2I]
    __nv_bfloat16 *dh, *du, *ag;  // [rows][I]
    float* dgp;              // [rows][I/32] or null
  };

  __device__ static uint32_t full_arrivals(const Params&) { return 1; }
  __device__ static uint32_t tx_bytes(const Params&) { return STAGE_BYTES; }

  __device__ static void load(const Params& P, const TileCoord& c, int kb, uint8_t* st,
                              uint64_t* bar, int lane) {
    if (lane != 0) return;
    const int k0 = kb * BKD;
    const int drow = c.g * P.D + k0;
    tma_load_2d(st, &P.tmWd, c.nt * 128, drow, bar);
    tma_load_2d(st + WDCHUNK, &P.tmWd, c.nt * 128 + 64, drow, bar);
    tma_load_2d(st + OFF_DY, &P.tmDy, k0, c.row0 + c.mt * ROWS, bar);
  }

  __device__ static void fixup(const Params&, const TileCoord&, int, uint8_t*, int) {}

  __device__ static int tile_rows(const TileCoord& c) {
    const int n = c.rows - c.mt * ROWS;
    return n < ROWS ? n : ROWS;
  }

  __device__ static void mma(const Params&, const TileCoord& c, int kb, uint8_t* st, uint32_t d) {
    const uint32_t s = smem_u32(st);
    const uint32_t id_t = idesc_bf16(128, (tile_rows(c) + 15) & ~15, true, false);
#pragma unroll
    for (int k = 0; k < BKD / 16; ++k)
      mma_bf16(d, sdesc_sw128(s + k * 2048, WDCHUNK, 1024), kdesc(s + OFF_DY + k * 32), id_t, (kb | k) != 0);
  }

  __device__ static void epilogue(const Params& P, const TileCoord& c, uint32_t taddr, int ew,
                                  int lane, bool, uint8_t*) {
    const int nrows = tile_rows(c);
    const int64_t row0 = c.row0 + c.mt * ROWS;
    const int64_t ld = 2 * static_cast<int64_t>(P.I);
    const float* hp = P.act + row0 * ld + c.nt * 128 + ew * 32 + lane;
#pragma unroll 1
    for (int cc = 0; cc * 32 < nrows; ++cc) {
      const int nv = min(nrows - cc * 32, 32);
      uint32_t hv[32], uv[32], tv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float* q = hp + (cc * 32 + j) * ld;
        hv[j] = j < nv ? __float_as_uint(__ldg(q)) : 0u;
        uv[j] = j < nv ? __float_as_uint(__ldg(q + P.I)) : 0u;
      }
      tmem_ld32(taddr + cc * 32, tv);
      tmem_ld_wait();
      dgrad_chunk(P, c, row0 + cc * 32, nv, ew, lane, hv, uv, tv);
    }
  }
};

// ---------------------------------------------------------------------------
struct DxCfg {
  static constexpr int STAGES = 4;
  static constexpr int STAGE_BYTES = KTILE + 4 * MNCHUNK;  // 48 KB
  static constexpr int EPI_SMEM_BYTES = 0;
  static constexpr int NUM_ACC = 2;
  static constexpr int ACC_COLS = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC = idesc_bf16(128, 256, false, true);

  struct Params {
    SchedArgs sched;
    int* status;
    CUtensorMap tmDh, tmDu;  // [rows][I], K-major boxes 128 x 64
    CUtensorMap tmWg, tmWu;  // [G*I][D], MN-major boxes 64 x 64
    int32_t I, half_kb;
    __nv_bfloat16* out;      // [rows][D]
    int32_t out_ld;
  };

  __device__ static uint32_t full_arrivals(const Params&) { return 1; }
  __device__ static uint32_t tx_bytes(const Params&) { return STAGE_BYTES; }

  __device__ static void load(const Params& P, const TileCoord& c, int kb, uint8_t* st,
                              uint64_t* bar, int lane) {
    if (lane != 0) return;
    const bool up = kb >= P.half_kb;
    const int k0 = (up ? kb - P.half_kb : kb) * BK;
    tma_load_2d(st, up ? &P.tmDu : &P.tmDh, k0, c.row0 + c.mt * BM, bar);
    const CUtensorMap* w = up ? &P.tmWu : &P.tmWg;
    const int wrow = c.g * P.I + k0;
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(st + KTILE + j * MNCHUNK, w, c.nt * 256 + 64 * j, wrow, bar);
  }

  __device__ static void fixup(const Params&, const TileCoord&, int, uint8_t*, int) {}

  __device__ static void mma(const Params&, const TileCoord&, int kb, uint8_t* st, uint32_t d) {
    const uint32_t s = smem_u32(st);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k)
      mma_bf16(d, kdesc(s + k * 32), mndesc(s + KTILE + k * 2048), IDESC, (kb | k) != 0);
  }

  __device__ static void epilogue(const Params& P, const TileCoord& c, uint32_t taddr, int ew,
                                  int lane, bool, uint8_t*) {
    const int r = ew * 32 + lane;
    const bool valid = c.mt * BM + r < c.rows;
    __nv_bfloat16* orow =
        P.out + static_cast<size_t>(c.row0 + c.mt * BM + r) * P.out_ld + c.nt * 256;
#pragma unroll 1
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t v[32];
      tmem_ld32(taddr + ch * 32, v);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4(orow + ch * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// dW[g][m][n] = sum_{p in group g} Pm[p][m] * Qn[p][n]: A = Pm^T, B = Qn^T,
// both MN-major in their [rows][...] storage.  M tile 128, N tile BN.
template <int BN>
struct WgradCfg {
  static constexpr int NB = BN / 64;  // 64-wide MN chunks of B
  static constexpr int BKW = 64;        // rows (K) per stage
  static constexpr int CH = BKW * 128;  // one 64-wide MN chunk of a stage: BKW rows of 128 B
  // Four stages (two tiles of a ~128-row expert) ahead of the MMAs: with
  // three the MMA warp waited on loads.
  static constexpr int STAGES = 4;
  static constexpr int STAGE_BYTES = (2 + NB) * CH;
  // per epilogue warp: two staging blocks of 32 rows x 64 columns of bf16,
  // 128-byte swizzled, each the source of one TMA store; chunk c of a tile
  // is written to block c % 2 while the store of chunk c - 1 reads the other
  static constexpr int EPI_SMEM_BYTES = 2 * 4 * 32 * 128;
  static_assert((BN / 64) % 2 == 0, "an even chunk count keeps the alternation across tiles");
  static constexpr int NUM_ACC = 2;
  static constexpr int ACC_COLS = BN;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t IDESC = idesc_bf16(128, BN, true, true);

  struct Params {
    SchedArgs sched;
    int* status;
    CUtensorMap tmA;  // [rows][M], MN-major boxes 64 x 64
    CUtensorMap tmB;  // [rows][N], MN-major boxes 64 x 64
    CUtensorMap tmOut;  // dW as [G*M][N], boxes 32 rows x 64 columns, 128-byte swizzle
    int32_t M, N;
    __nv_bfloat16* out;  // [G][M][N]
  };

  __device__ static uint32_t full_arrivals(const Params&) { return 1; }
  __device__ static uint32_t tx_bytes(const Params&) { return STAGE_BYTES; }

  __device__ static void load(const Params& P, const TileCoord& c, int kb, uint8_t* st,
                              uint64_t* bar, int lane) {
    if (lane != 0) return;
    const int rk = c.row0 + kb * BKW;
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_load_2d(st + j * CH, &P.tmA, c.mt * 128 + 64 * j, rk, bar);
#pragma unroll
    for (int j = 0; j < NB; ++j)
      tma_load_2d(st + (2 + j) * CH, &P.tmB, c.nt * BN + 64 * j, rk, bar);
  }

  // Rows past the group's end in its last K block belong to the next group
  // (or lie past the tensor and are zero-filled).  The MMAs of that block
  // stop at the first 16-row step at or past the end, and the rows between
  // the end and that step are zeroed in A (both 64-column chunks; lane l
  // clears 16-byte unit l % 8 of every fourth row).
  __device__ static int k_rows(const TileCoord& c, int kb) {
    const int valid = c.rows - kb * BKW;
    return valid < BKW ? valid : BKW;
  }
  __device__ static void fixup(const Params&, const TileCoord& c, int kb, uint8_t* st, int lane) {
    const int valid = k_rows(c, kb);
    const int end = (valid + 15) & ~15;
    if (valid == end) return;
    for (int r = valid + (lane >> 3); r < end; r += 4) {
      uint8_t* p = st + r * 128 + (lane & 7) * 16;
      *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(p + CH) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }

  // MN-major, 128-byte swizzle: LBO = one 64-wide MN chunk, SBO = 8 K rows
  __device__ static uint64_t desc(uint32_t a) { return sdesc_sw128(a, CH, 1024); }

  __device__ static void mma(const Params&, const TileCoord& c, int kb, uint8_t* st, uint32_t d) {
    const uint32_t s = smem_u32(st);
    const int nk = (k_rows(c, kb) + 15) / 16;
#pragma unroll
    for (int k = 0; k < BKW / 16; ++k)
      if (k < nk) mma_bf16(d, desc(s + k * 2048), desc(s + 2 * CH + k * 2048), IDESC, (kb | k) != 0);
  }

  // Each warp converts its 32 rows x 64 columns to bf16, writes them to its
  // staging block in the 128-byte swizzle the store's tensor map expects
  // (16-byte chunk c of row r at chunk c ^ (r % 8)) and issues one TMA store,
  // so every store instruction moves whole rows instead of 16 bytes of 32
  // different rows.  All wgrad tiles are full, so no row needs masking.
  __device__ static void epilogue(const Params& P, const TileCoord& c, uint32_t taddr, int ew,
                                  int lane, bool has_acc, uint8_t* epi) {
    const int y = c.g * P.M + c.mt * 128 + ew * 32;
#pragma unroll 1
    for (int cp = 0; cp < BN / 64; ++cp) {
      uint32_t pk[32];
      if (has_acc) {
        uint32_t v0[32], v1[32];
        tmem_ld32(taddr + cp * 64, v0);
        tmem_ld32(taddr + cp * 64 + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          pk[j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
          pk[16 + j] = pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = 0u;
      }
      // the store that last read this block (two chunks back) has finished
      if (lane == 0) bulk_wait_read1();
      __syncwarp();
      uint8_t* blk = epi + (cp & 1) * (32 * 128);
      uint8_t* row = blk + lane * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint4* dst = reinterpret_cast<uint4*>(row + ((ch ^ (lane & 7)) * 16));
        *dst = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&P.tmOut, blk, c.nt * BN + cp * 64, y);
        bulk_commit();
      }
    }
  }
};


// ---------------------------------------------------------------------------
// The weight gradient on clusters of two CTAs that share B.
//
// A wgrad tile writes 64 KB of dW and reads 96 KB of operand rows from L2
// (K over an expert's ~128 rows is short, so the operand reads are not
// amortised), and those L2 reads share the memory system with the dW write
// stream: the more bytes a kernel reads from L2 per byte it writes to DRAM,
// the lower its write rate.  Here the two CTAs
// of a cluster take M tiles 2p and 2p + 1 of the same (expert, N tile): each
// loads its own A chunks and one half of B (chunks rank * NB / 2 ..), the
// latter with a cluster multicast into the same stage of both CTAs, so every
// CTA requests 32 KB per 64-row stage instead of 48 KB and issues four TMA
// loads instead of six.  The MMAs stay per CTA (cta_group::1), so the rows
// past an expert's end are zeroed in each CTA's own A as before, and TMEM,
// the accumulators and the epilogue are the single-CTA kernel's.
//
// Barriers: a stage's full barrier counts its own producer's arrival and
// 48 KB (its A, its half of B, the peer's half of B); its empty barrier
// counts two arrivals, the MMA commits of both CTAs (multicast), since a
// producer refills its half of B in both CTAs.  Both CTAs walk the same
// sequence of (expert, M tile pair, N tile) units and K blocks, so their
// stage and phase counters stay in step; every wait is bounded, and the
// CTAs meet at a cluster barrier before either exits, so no multicast or
// remote arrival reaches a CTA that has left.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* m, int32_t x, int32_t y,
                                               uint64_t* bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` once this thread's
// earlier tcgen05 operations have completed (single-CTA MMAs).
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    wgrad_cluster(const __grid_constant__ typename WgradCfg<BN>::Params P) {
  using Cfg = WgradCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi_smem = smem + Cfg::STAGES * Cfg::STAGE_BYTES;
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
  const int rank = static_cast<int>(cluster_rank());
  constexpr uint16_t kBoth = 0x3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);  // the MMA commits of both CTAs
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
    const int total = build_tile_table(P.sched, tstart, lane);
    if (lane == 0) *total_holder = total;
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised before any multicast or remote commit
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;
  // this CTA's M tile of a unit: the schedule counts M tile pairs
  auto own = [rank](TileCoord c) {
    c.mt = 2 * c.mt + rank;
    return c;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    uint32_t stage = 0, phase = 0;
    uint32_t issued_parity[Cfg::STAGES];
    bool issued[Cfg::STAGES];
    for (int i = 0; i < Cfg::STAGES; ++i) issued[i] = false;
    bool ok = true;
    TileWalker walk(P.sched, tstart);
    for (int unit = cid; unit < total && ok; unit += ncl) {
      const TileCoord c = own(walk.at(unit));
      for (int kb = 0; kb < c.kblocks; ++kb) {
        bool got = false;
        if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER);
        ok = __shfl_sync(0xffffffffu, got, 0);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          const int rk = c.row0 + kb * Cfg::BKW;
#pragma unroll
          for (int j = 0; j < 2; ++j) tma_load_2d(st + j * Cfg::CH, &P.tmA, c.mt * 128 + 64 * j, rk, &full[stage]);
#pragma unroll
          for (int h = 0; h < Cfg::NB / 2; ++h) {
            const int j = rank * (Cfg::NB / 2) + h;
            tma_load_2d_mc(st + (2 + j) * Cfg::CH, &P.tmB, c.nt * BN + 64 * j, rk, &full[stage], kBoth);
          }
        }
        __syncwarp();
        issued[stage] = true;
        issued_parity[stage] = phase;
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      for (int i = 0; i < Cfg::STAGES; ++i) {
        if (!issued[i]) continue;
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&full[i], issued_parity[i]) && globaltimer() - t0 < kWaitBudgetNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    uint32_t stage = 0, phase = 0;
    bool ok = true, any = false;
    int it = 0;
    TileWalker walk(P.sched, tstart);
    for (int unit = cid; unit < total && ok; unit += ncl, ++it) {
      const TileCoord c = own(walk.at(unit));
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
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
          mma_commit_mc(&empty[stage], kBoth);  // both producers may refill the stage
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
    for (int unit = cid; unit < total; unit += ncl, ++it) {
      const TileCoord c = own(walk.at(unit));
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, P.status, SITE_EPILOGUE)))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * Cfg::ACC_COLS + (static_cast<uint32_t>(ew * 32) << 16);
      Cfg::epilogue(P, c, taddr, ew, lane, c.kblocks > 0, epi_smem + ew * (Cfg::EPI_SMEM_BYTES / 4));
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    if (lane == 0) bulk_wait0();
  }

  tc_fence_before();
  cluster_sync();  // no multicast load or remote commit still targets either CTA
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// SMs a persistent launch takes: every SM, or at most max_sms > 0 of them
// (the rest stay free for another stream's kernels).
int grid_sms(int max_sms) {
  const int n = num_sms();
  return max_sms > 0 && max_sms < n ? max_sms : n;
}

template <class Cfg>
mok_status run(const typename Cfg::Params& P, cudaStream_t st, int max_sms = 0) {
  const size_t smem = gemm_smem_bytes<Cfg>(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_persistent<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  gemm_persistent<Cfg><<<grid_sms(max_sms), 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

SchedArgs sched_rows(const int32_t* offsets, int G, int64_t m_total, int n_tiles, int k_blocks) {
  SchedArgs s;
  s.offsets = offsets;
  s.G = offsets ? G : 1;
  s.m_total = static_cast<int32_t>(m_total);
  s.n_tiles = n_tiles;
  s.m_tiles_fixed = 0;
  s.k_blocks_fixed = k_blocks;
  s.bm = BM;
  s.bk_rows = BK;
  return s;
}

constexpr auto kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

bool kmap(CUtensorMap* m, const void* p, int64_t rows, int cols) {
  return make_tmap_2d(m, p, kBF16, rows, cols, static_cast<uint64_t>(cols) * 2, 128, BK, true);
}
bool mnmap(CUtensorMap* m, const void* p, int64_t rows, int cols) {
  return make_tmap_2d(m, p, kBF16, rows, cols, static_cast<uint64_t>(cols) * 2, BK, 64, true);
}

}  // namespace

mok_status launch_bwd_dgrad(const void* xg, const void* dyg, int64_t rows, const void* w_gate,
                            const void* w_up, const void* w_down, const int32_t* offsets, int G,
                            int D, int I, const float* g_route, void* dh, void* du, void* ag,
                            float* dgp, cudaStream_t st, int32_t skip_rows_below, int max_sms) {
  if (rows == 0) return MOK_OK;
  DgradCfg::Params P;
  P.sched = sched_rows(offsets, G, rows, I / 128, D / DgradCfg::BKD);
  P.sched.bm = DgradCfg::ROWS;
  if (skip_rows_below > 0 && offsets) {  // the groups the forward kept are another launch's
    P.sched.row_split = skip_rows_below;
    P.sched.split_side = 2;
  }
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int groups = offsets ? G : 1;
  auto k64 = [](CUtensorMap* m, const void* p, int64_t r, int cols, int box_rows) {
    return make_tmap_2d_swz(m, p, kBF16, r, cols, static_cast<uint64_t>(cols) * 2, box_rows, DgradCfg::BKD,
                            CU_TENSOR_MAP_SWIZZLE_64B);
  };
  if (!k64(&P.tmX, xg, rows, D, DgradCfg::ROWS) || !k64(&P.tmDy, dyg, rows, D, DgradCfg::ROWS) ||
      !k64(&P.tmWg, w_gate, static_cast<int64_t>(groups) * I, D, 128) ||
      !k64(&P.tmWu, w_up, static_cast<int64_t>(groups) * I, D, 128) ||
      !make_tmap_2d(&P.tmWd, w_down, kBF16, static_cast<int64_t>(groups) * D, I, static_cast<uint64_t>(I) * 2,
                    DgradCfg::BKD, 64, true))
    return MOK_ERR_CUDA;
  P.I = I;
  P.D = D;
  P.g_route = g_route;
  P.dh = static_cast<__nv_bfloat16*>(dh);
  P.du = static_cast<__nv_bfloat16*>(du);
  P.ag = static_cast<__nv_bfloat16*>(ag);
  P.dgp = dgp;
  return run<DgradCfg>(P, st, max_sms);
}

mok_status launch_bwd_dgrad_kept(const void* dyg, int64_t rows, const void* w_down, const int32_t* offsets, int G,
                                 int D, int I, const float* g_route, const float* act, int32_t kept_rows, void* dh,
                                 void* du, void* ag, float* dgp, cudaStream_t st, int max_sms) {
  if (rows == 0 || kept_rows <= 0) return MOK_OK;
  DgradKeptCfg::Params P;
  P.sched = sched_rows(offsets, G, rows, I / 128, D / DgradKeptCfg::BKD);
  P.sched.bm = DgradKeptCfg::ROWS;
  P.sched.row_split = kept_rows;
  P.sched.split_side = 1;
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  if (!make_tmap_2d(&P.tmDy, dyg, kBF16, rows, D, static_cast<uint64_t>(D) * 2, DgradKeptCfg::ROWS,
                    DgradKeptCfg::BKD, true) ||
      !make_tmap_2d(&P.tmWd, w_down, kBF16, static_cast<int64_t>(G) * D, I, static_cast<uint64_t>(I) * 2,
                    DgradKeptCfg::BKD, 64, true))
    return MOK_ERR_CUDA;
  P.I = I;
  P.D = D;
  P.g_route = g_route;
  P.act = act;
  P.dh = static_cast<__nv_bfloat16*>(dh);
  P.du = static_cast<__nv_bfloat16*>(du);
  P.ag = static_cast<__nv_bfloat16*>(ag);
  P.dgp = dgp;
  return run<DgradKeptCfg>(P, st, max_sms);
}

mok_status launch_bwd_dx(const void* dh, const void* du, int64_t rows, const void* w_gate,
                         const void* w_up, const int32_t* offsets, int G, int D, int I, void* dx,
                         cudaStream_t st, int max_sms) {
  if (rows == 0) return MOK_OK;
  // fewer than 512 routed rows per group on average: the routed rows as the
  // MMA's N dimension, one tile per expert and 256 D columns (no padding
  // rows); the ungrouped rows of the shared expert too (tensor-bound there,
  // where the pair MMAs keep the tensor pipe busier than 128-row tiles)
  if ((!offsets || rows < static_cast<int64_t>(512) * G) && D % 256 == 0 && I % 128 == 0)
    return launch_dx_pair_t(dh, du, rows, w_gate, w_up, offsets, G, D, I, dx, st, max_sms);
  DxCfg::Params P;
  P.sched = sched_rows(offsets, G, rows, D / 256, 2 * (I / BK));
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int groups = offsets ? G : 1;
  if (!kmap(&P.tmDh, dh, rows, I) || !kmap(&P.tmDu, du, rows, I) ||
      !mnmap(&P.tmWg, w_gate, static_cast<int64_t>(groups) * I, D) ||
      !mnmap(&P.tmWu, w_up, static_cast<int64_t>(groups) * I, D))
    return MOK_ERR_CUDA;
  P.I = I;
  P.half_kb = I / BK;
  P.out = static_cast<__nv_bfloat16*>(dx);
  P.out_ld = D;
  return run<DxCfg>(P, st, max_sms);
}

template <int BN>
mok_status wgrad_bn(const void* pm, const void* qn, int64_t rows, const int32_t* offsets, int G,
                    int M, int N, void* dw, cudaStream_t st, int max_sms) {
  typename WgradCfg<BN>::Params P;
  SchedArgs s;
  s.offsets = offsets;
  s.G = offsets ? G : 1;
  s.m_total = static_cast<int32_t>(rows);
  s.n_tiles = N / BN;
  s.m_tiles_fixed = M / 128;
  s.k_blocks_fixed = 0;
  s.bm = BM;
  s.bk_rows = WgradCfg<BN>::BKW;
  // N tile fastest: CTAs working side by side write neighbouring column
  // pieces of the same dW rows instead of 512-byte pieces of distant rows
  s.m_outer = 1;
  P.sched = s;
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int64_t map_rows = rows > 0 ? rows : 1;
  auto mn = [](CUtensorMap* m, const void* p, int64_t rows, int cols) {
    return make_tmap_2d(m, p, kBF16, rows, cols, static_cast<uint64_t>(cols) * 2, WgradCfg<BN>::BKW, 64, true);
  };
  if (!mn(&P.tmA, pm, map_rows, M) || !mn(&P.tmB, qn, map_rows, N) ||
      !make_tmap_2d(&P.tmOut, dw, kBF16, static_cast<uint64_t>(s.G) * M, N,
                    static_cast<uint64_t>(N) * 2, 32, 64, true))
    return MOK_ERR_CUDA;
  P.M = M;
  P.N = N;
  P.out = static_cast<__nv_bfloat16*>(dw);
  const int sms = grid_sms(max_sms);
  if ((M / 128) % 2 != 0 || sms < 2) return run<WgradCfg<BN>>(P, st, max_sms);
  // clusters of two CTAs on neighbouring M tiles sharing B: the schedule
  // counts M tile pairs
  P.sched.m_tiles_fixed = M / 256;
  const size_t smem = gemm_smem_bytes<WgradCfg<BN>>(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(wgrad_cluster<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  wgrad_cluster<BN><<<(sms / 2) * 2, 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_wgrad(const void* pm, const void* qn, int64_t rows, const int32_t* offsets,
                        int G, int M, int N, void* dw, cudaStream_t st, int max_sms) {
  // 256-wide tiles unless their shared memory (which grows with the
  // number of groups) does not fit
  if (N % 256 == 0 && gemm_smem_bytes<WgradCfg<256>>(offsets ? G : 1) <= 227 * 1024)
    return wgrad_bn<256>(pm, qn, rows, offsets, G, M, N, dw, st, max_sms);
  return wgrad_bn<128>(pm, qn, rows, offsets, G, M, N, dw, st, max_sms);
}

}  // namespace mok
