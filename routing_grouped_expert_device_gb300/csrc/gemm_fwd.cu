// Forward grouped expert GEMMs on tcgen05 / TMEM (Mixture-of-Kittens blog,
// "Overlapping computation and communication in MoE": each selected expert
// runs up and gate projections, a SwiGLU, then the down projection).
//
//  up/gate : tile 128 rows x (128 gate cols | 128 up cols), K = D.  The two
//            weight tiles are stacked into one 256-row B operand, so one
//            M128 N256 MMA produces h and u side by side in TMEM; the
//            epilogue writes a = bf16(SiLU(h) * u).
//  down    : tile 128 rows x 256 output cols, K = I; y = bf16(acc).
// Operands are K-major, 128-byte swizzled, loaded by TMA in 64-wide K blocks.
#include "gemm_core.cuh"
#include "kernels.h"

namespace mok {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;

template <bool kSwiglu>
struct FwdCfg {
  static constexpr int STAGES = 4;
  static constexpr int A_BYTES = BM * BK * 2;    // 16 KB
  static constexpr int B_HALF = 128 * BK * 2;    // 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + 2 * B_HALF;
  static constexpr int EPI_SMEM_BYTES = 0;
  static constexpr int NUM_ACC = 2;
  static constexpr int ACC_COLS = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC = idesc_bf16(128, 256, false, false);

  struct Params {
    SchedArgs sched;
    int* status;
    CUtensorMap tmA;   // activations [rows][K]; with gtable: x [T][D], boxes one row high
    CUtensorMap tmB0;  // up/gate: W_gate [E*I][D]; down: W_down [E*D][I]
    CUtensorMap tmB1;  // up/gate: W_up;           down: W_down again
    int32_t b_group_rows;  // weight rows per expert (I or D)
    int32_t b_tile_rows;   // weight rows per N tile (128 or 256)
    int32_t b1_off;        // row offset of the second B half (0 or 128)
    __nv_bfloat16* out;
    int32_t out_ld;
    const int32_t* gtable;  // non-null: A row p is x[gtable[3 p] / gK] (fused dispatch)
    int32_t gK;
    const void* gx;          // x [T][D] bf16
    int64_t gld;             // x row pitch in bytes
  };

  // Fused dispatch: A arrives by cp.async (one arrival per producer lane),
  // only B by TMA.
  __device__ static uint32_t full_arrivals(const Params& P) { return P.gtable ? 33u : 1u; }
  __device__ static uint32_t tx_bytes(const Params& P) {
    return P.gtable ? static_cast<uint32_t>(2 * B_HALF) : static_cast<uint32_t>(STAGE_BYTES);
  }

  __device__ static void load(const Params& P, const TileCoord& c, int kb, uint8_t* st,
                              uint64_t* bar, int lane) {
    const int k0 = kb * BK;
    if (P.gtable) {
      // Fused dispatch (Mixture-of-Kittens blog, "Scheduling": tokens land
      // expert-contiguous with zero local copies): the producer warp copies
      // the tile's 128 token rows (64 columns each) straight from x into the
      // stage, already in the 128-byte swizzle the MMA reads.  Eight lanes
      // cover one 128-byte row, so each instruction moves 4 whole rows.
      // Rows past the expert's end read token 0; their results are dropped.
      const int p0 = c.row0 + c.mt * BM;
      const int end = c.row0 + c.rows;
      int32_t tok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + lane + 32 * j;
        tok[j] = p < end ? __ldg(P.gtable + 3 * p) / P.gK : 0;
      }
      const int chunk = lane & 7;
      const uint8_t* xb = reinterpret_cast<const uint8_t*>(P.gx) + static_cast<int64_t>(k0) * 2 + chunk * 16;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int row = 4 * i + (lane >> 3);
        const int t = __shfl_sync(0xffffffffu, tok[i >> 3], row & 31);
        cp_async16(st + row * 128 + ((chunk ^ (row & 7)) << 4), xb + static_cast<int64_t>(t) * P.gld);
      }
      cp_async_arrive(bar);
    }
    if (lane != 0) return;
    if (!P.gtable) tma_load_2d(st, &P.tmA, k0, c.row0 + c.mt * BM, bar);
    const int brow = c.g * P.b_group_rows + c.nt * P.b_tile_rows;
    tma_load_2d(st + A_BYTES, &P.tmB0, k0, brow, bar);
    tma_load_2d(st + A_BYTES + B_HALF, &P.tmB1, k0, brow + P.b1_off, bar);
  }

  // Rows copied by cp.async (generic proxy) are read by the tensor core
  // (async proxy).
  __device__ static void fixup(const Params& P, const TileCoord&, int, uint8_t*, int) {
    if (P.gtable) fence_proxy_async_smem();
  }

  __device__ static void mma(const Params&, const TileCoord&, int kb, uint8_t* st, uint32_t d) {
    const uint32_t a = smem_u32(st);
    const uint32_t b = smem_u32(st + A_BYTES);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      // 16 bf16 = 32 bytes further along K inside the 128-byte swizzle atom
      mma_bf16(d, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(b + k * 32, 16, 1024), IDESC,
               (kb | k) != 0);
    }
  }

  __device__ static void epilogue(const Params& P, const TileCoord& c, uint32_t taddr, int ew,
                                  int lane, bool, uint8_t*) {
    const int r = ew * 32 + lane;
    const bool valid = c.mt * BM + r < c.rows;
    __nv_bfloat16* orow = P.out + static_cast<size_t>(c.row0 + c.mt * BM + r) * P.out_ld;
    if (kSwiglu) {
      orow += c.nt * 128;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t h[32], u[32];
        tmem_ld32(taddr + ch * 32, h);
        tmem_ld32(taddr + 128 + ch * 32, u);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float h0 = __uint_as_float(h[2 * j]), h1 = __uint_as_float(h[2 * j + 1]);
          const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
          pk[j] = pack_bf16x2(silu_f(h0) * u0, silu_f(h1) * u1);
        }
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_global_v4(orow + ch * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                         pk[4 * q + 3]);
        }
      }
    } else {
      orow += c.nt * 256;
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
            st_global_v4(orow + ch * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                         pk[4 * q + 3]);
        }
      }
    }
  }
};

using UpGate = FwdCfg<true>;

template <class Cfg>
mok_status run(const typename Cfg::Params& P, int G, cudaStream_t st) {
  const size_t smem = gemm_smem_bytes<Cfg>(G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_persistent<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  gemm_persistent<Cfg><<<num_sms(), 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

SchedArgs fwd_sched(const int32_t* offsets, int G, int64_t m_total, int n_tiles, int k_blocks) {
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

}  // namespace

mok_status launch_upgate(const void* A, int64_t a_rows, const void* w_gate, const void* w_up,
                         const int32_t* offsets, int G, int64_t m_total, int D, int I, void* a_out,
                         cudaStream_t st, const int32_t* gather_table, int gather_k) {
  if (a_rows == 0 || m_total == 0) return MOK_OK;
  if (!gather_table) return launch_upgate_pair(A, a_rows, w_gate, w_up, offsets, G, m_total, D, I, a_out, st);
  UpGate::Params P;
  P.gtable = gather_table;
  P.gK = gather_k;
  P.gx = A;
  P.gld = static_cast<int64_t>(D) * 2;
  P.sched = fwd_sched(offsets, G, m_total, I / 128, D / BK);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int groups = offsets ? G : 1;
  const auto bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_tmap_2d(&P.tmA, A, bf16, a_rows, D, static_cast<uint64_t>(D) * 2, BM, BK, true) ||
      !make_tmap_2d(&P.tmB0, w_gate, bf16, static_cast<uint64_t>(groups) * I, D,
                    static_cast<uint64_t>(D) * 2, 128, BK, true) ||
      !make_tmap_2d(&P.tmB1, w_up, bf16, static_cast<uint64_t>(groups) * I, D,
                    static_cast<uint64_t>(D) * 2, 128, BK, true))
    return MOK_ERR_CUDA;
  P.b_group_rows = I;
  P.b_tile_rows = 128;
  P.b1_off = 0;
  P.out = static_cast<__nv_bfloat16*>(a_out);
  P.out_ld = I;
  return run<UpGate>(P, P.sched.G, st);
}

mok_status launch_down(const void* a, int64_t a_rows, const void* w_down, const int32_t* offsets,
                       int G, int64_t m_total, int D, int I, void* y_out, cudaStream_t st) {
  return launch_down_pair(a, a_rows, w_down, offsets, G, m_total, D, I, y_out, st);
}

}  // namespace mok
