// MXFP8 grouped expert GEMMs (Mixture-of-Kittens paper note, "The
// production details": MXFP8 with quantisation fused into the dispatch, the
// grouped GEMMs and the gated activation).
//
// Operands are E4M3 codes with one E8M0 scale per 1x32 block along K.  Scale
// storage of a [rows][K] tensor: int32 words sc[K/128][ld] (ld = rows rounded
// up to 4); word (g, r) holds the 4 block scales of row r for K columns
// [128 g, 128 g + 128), byte b for block 4 g + b.
//
// Per stage (128 K columns = 4 MMAs of K 32) the TMA producer loads the A and
// B code tiles (128-byte swizzle) and the tile's scale words.  The epilogue
// warps, idle during the main loop (one TMEM accumulator), copy the scale
// words into a TMEM ring with tcgen05.st, in the layout the block-scaled MMA
// reads for M = 128 and one scale per 32 K:
//   A row m : TMEM lane m,                     column sfa + m/32, byte = MMA k
//   B row n : lanes 32 q + n%32, every quarter q, column sfb + n/32, byte = MMA k
// then arrive on sf_ready[stage]; the MMA thread issues the 4 block-scaled
// MMAs of the stage.
//
// up/gate : tile 128 rows x (128 gate | 128 up); the epilogue forms
//           a = bf16(SiLU(h) u) and quantises it to E4M3 per 32 columns (one
//           TMEM load of 32 columns is one block).
// down    : tile 128 rows x 256 columns; y = bf16(acc).
#include <cuda_fp8.h>

#include "gemm_core.cuh"
#include "kernels.h"

namespace mok {
namespace {

constexpr int BM = 128;
constexpr int BKB = 128;                      // K columns (bytes) per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;             // 16 KB
constexpr int B_HALF = 128 * BKB;             // 16 KB
constexpr int SA_OFF = A_BYTES + 2 * B_HALF;  // raw A scale words (132 used)
constexpr int SB_OFF = SA_OFF + 1024;         // raw B scale words (256)
constexpr int STAGE_BYTES = SB_OFF + 1024;    // 50 KB
constexpr int SA_WORDS = 132;                 // 128 rows + up to 3 words of misalignment
constexpr uint32_t TX_BYTES = A_BYTES + 2 * B_HALF + SA_WORDS * 4 + 256 * 4;
constexpr uint32_t ACC_COLS = 256;
constexpr uint32_t SF_COLS = 12;  // per stage: 4 (A) + 8 (B)

// Block-scaled instruction descriptor, kind::mxf8f6f4: B scale id (bits 4-5),
// A and B format E4M3 = 0 (7-9, 10-12), both K-major, N >> 3 (17-22), scale
// format UE8M0 (23), M >> 4 (24-28), A scale id (29-30).
__device__ __forceinline__ uint32_t idesc_mx(int N, uint32_t sf_id) {
  return (sf_id << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Smallest e with amax <= 448 * 2^e (same rule as the quantiser in
// elementwise.cu): amax = 1.f * 2^E and 448 = 1.75 * 2^8.
__device__ __forceinline__ int mx_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int eb = static_cast<int>((b >> 23) & 0xFFu);
  if (eb == 0) return -127;
  const int e = eb - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

struct MxParams {
  SchedArgs sched;
  int* status;
  CUtensorMap tmA;    // codes [rows][K] u8, box 128 x 128
  CUtensorMap tmSA;   // scale words [K/128][ld] i32, box 132 x 1
  CUtensorMap tmB0;   // codes [G*NB][K], box 128 x 128
  CUtensorMap tmB1;
  CUtensorMap tmSB0;  // scale words of B0 [K/128][G*NB] i32, box 128 x 1
  CUtensorMap tmSB1;  // scale words of B1
  int32_t b_group_rows, b_tile_rows, b1_off;
  uint8_t* aq;        // up/gate: a codes [rows][I]
  uint32_t* asc;      // up/gate: a scale words [I/128][a_ld]
  int32_t a_ld;
  __nv_bfloat16* y;   // down: y [rows][D]
  int32_t out_ld;
};

template <bool kSwiglu>
__global__ void __launch_bounds__(256, 1) gemm_mx_persistent(const __grid_constant__ MxParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* sfready = empty + STAGES;
  uint64_t* tfull = sfready + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* total_holder = reinterpret_cast<int*>(tmem_holder + 2);
  int* tstart = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);
  int* rstart = tstart + (P.sched.G + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sfready[i], 128);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_holder, 512);
  if (warp == 3) {
    const int total = build_tile_table(P.sched, tstart, rstart, lane);
    if (lane == 0) *total_holder = total;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_parity[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileCoord c = decode_tile(P.sched, tstart, rstart, tile);
        const int r0 = c.row0 + c.mt * BM;
        const int brow = c.g * P.b_group_rows + c.nt * P.b_tile_rows;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.status, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], TX_BYTES);
          tma_load_2d(st, &P.tmA, kb * BKB, r0, &full[stage]);
          tma_load_2d(st + A_BYTES, &P.tmB0, kb * BKB, brow, &full[stage]);
          tma_load_2d(st + A_BYTES + B_HALF, &P.tmB1, kb * BKB, brow + P.b1_off, &full[stage]);
          // A's scale words start at row r0, which need not sit on a 16-byte
          // boundary: fetch from r0 rounded down to 4 words, index from the
          // remainder.
          tma_load_2d(st + SA_OFF, &P.tmSA, r0 & ~3, kb, &full[stage]);
          tma_load_2d(st + SB_OFF, &P.tmSB0, brow, kb, &full[stage]);
          tma_load_2d(st + SB_OFF + 512, &P.tmSB1, brow + P.b1_off, kb, &full[stage]);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int i = 0; i < STAGES; ++i) {
          if (!issued[i]) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(&full[i], issued_parity[i]) && globaltimer() - t0 < kWaitBudgetNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    uint32_t stage = 0, phase = 0;
    bool ok = true, any = false;
    int it = 0;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const TileCoord c = decode_tile(P.sched, tstart, rstart, tile);
      ok = __all_sync(0xffffffffu, mbar_wait(tempty, (it & 1) ^ 1, abort_flag, P.status, SITE_MMA));
      if (!ok) break;
      tc_fence_after();
      for (int kb = 0; kb < c.kblocks; ++kb) {
        const bool got = mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_MMA) &&
                         mbar_wait(&sfready[stage], phase, abort_flag, P.status, SITE_MMA);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
          const uint32_t sfa = tmem_base + ACC_COLS + stage * SF_COLS;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mx(tmem_base, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(b + k * 32, 16, 1024),
                   idesc_mx(256, k), sfa, sfa + 4, (kb | k) != 0);
          mma_commit(&empty[stage]);
          any = true;
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(tfull);
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
    // ---------------- scales into TMEM, then the epilogue ----------------
    const int q = warp - 4;  // TMEM lane quarter of this warp
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t stage = 0, phase = 0;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const TileCoord c = decode_tile(P.sched, tstart, rstart, tile);
      const int r0 = c.row0 + c.mt * BM;
      for (int kb = 0; kb < c.kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, P.status, SITE_EPILOGUE));
        if (!ok) break;
        const uint8_t* st = smem + stage * STAGE_BYTES;
        const uint32_t* sa = reinterpret_cast<const uint32_t*>(st + SA_OFF) + (r0 & 3);
        const uint32_t* sb = reinterpret_cast<const uint32_t*>(st + SB_OFF);
        const uint32_t sf = tmem_base + lane_off + ACC_COLS + stage * SF_COLS;
        tmem_st1(sf + q, sa[q * 32 + lane]);
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = sb[j * 32 + lane];
        tmem_st8(sf + 4, v);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sfready[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(tfull, it & 1, abort_flag, P.status, SITE_EPILOGUE));
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_off;
      const int r = q * 32 + lane;
      const bool valid = c.mt * BM + r < c.rows;
      const int64_t row = r0 + r;
      if (kSwiglu) {
        uint32_t words = 0;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t hv[32], uv[32];
          tmem_ld32(taddr + ch * 32, hv);
          tmem_ld32(taddr + 128 + ch * 32, uv);
          tmem_ld_wait();
          float av[32];
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            av[j] = __bfloat162float(
                __float2bfloat16_rn(silu_f(__uint_as_float(hv[j])) * __uint_as_float(uv[j])));
            amax = fmaxf(amax, fabsf(av[j]));
          }
          const int e = mx_exp(amax);
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(av[4 * i] * inv, av[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(av[4 * i + 2] * inv, av[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
            pk[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
          }
          words |= static_cast<uint32_t>(e + 127) << (8 * ch);
          if (valid) {
            uint8_t* dst = P.aq + row * P.out_ld + c.nt * 128 + ch * 32;
            st_global_v4(dst, pk[0], pk[1], pk[2], pk[3]);
            st_global_v4(dst + 16, pk[4], pk[5], pk[6], pk[7]);
          }
        }
        if (valid) P.asc[static_cast<int64_t>(c.nt) * P.a_ld + row] = words;
      } else {
        __nv_bfloat16* orow = P.y + row * P.out_ld + c.nt * 256;
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          if (valid) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              st_global_v4(orow + ch * 32 + qq * 8, pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, 512);
}

size_t mx_smem_bytes(int G) {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256 + static_cast<size_t>(2 * (G + 1)) * sizeof(int);
}

template <bool kSwiglu>
mok_status run_mx(const MxParams& P, cudaStream_t st) {
  const size_t smem = mx_smem_bytes(P.sched.G);
  if (smem > 227 * 1024) return MOK_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gemm_mx_persistent<kSwiglu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOK_ERR_CUDA;
  gemm_mx_persistent<kSwiglu><<<num_sms(), 256, smem, st>>>(P);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

constexpr auto kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
constexpr auto kI32 = CU_TENSOR_MAP_DATA_TYPE_INT32;

bool code_map(CUtensorMap* m, const void* p, int64_t rows, int K) {
  return make_tmap_2d(m, p, kU8, rows, K, static_cast<uint64_t>(K), 128, BKB, true);
}
// scale words [K/128][ld] (ld = rows rounded up to 4 words, so that the row
// pitch is a multiple of 16 bytes) as a 2D tensor of K/128 rows of `rows` words
bool scale_map(CUtensorMap* m, const void* p, int64_t rows, int K, uint32_t box) {
  return make_tmap_2d(m, p, kI32, K / 128, rows, static_cast<uint64_t>(mx_scale_ld(rows)) * 4, 1, box,
                      false);
}

SchedArgs mx_sched(const int32_t* offsets, int G, int64_t m_total, int n_tiles, int k_blocks) {
  SchedArgs s;
  s.offsets = offsets;
  s.G = offsets ? G : 1;
  s.m_total = static_cast<int32_t>(m_total);
  s.n_tiles = n_tiles;
  s.m_tiles_fixed = 0;
  s.k_blocks_fixed = k_blocks;
  s.bm = BM;
  s.bk_rows = BKB;
  return s;
}

}  // namespace

mok_status launch_upgate_mx(const void* xq, const void* xsc, int64_t rows, const void* qg,
                            const void* sg, const void* qu, const void* su, const int32_t* offsets,
                            int G, int D, int I, void* aq, void* asc, cudaStream_t st) {
  if (rows == 0) return MOK_OK;
  MxParams P;
  P.sched = mx_sched(offsets, G, rows, I / 128, D / BKB);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int64_t wrows = static_cast<int64_t>(offsets ? G : 1) * I;
  if (!code_map(&P.tmA, xq, rows, D) || !scale_map(&P.tmSA, xsc, rows, D, SA_WORDS) ||
      !code_map(&P.tmB0, qg, wrows, D) || !code_map(&P.tmB1, qu, wrows, D) ||
      !scale_map(&P.tmSB0, sg, wrows, D, 128) || !scale_map(&P.tmSB1, su, wrows, D, 128))
    return MOK_ERR_CUDA;
  P.b_group_rows = I;
  P.b_tile_rows = 128;
  P.b1_off = 0;
  P.aq = static_cast<uint8_t*>(aq);
  P.asc = static_cast<uint32_t*>(asc);
  P.a_ld = static_cast<int32_t>(mx_scale_ld(rows));
  P.y = nullptr;
  P.out_ld = I;
  return run_mx<true>(P, st);
}

mok_status launch_down_mx(const void* aq, const void* asc, int64_t rows, const void* qd,
                          const void* sd, const int32_t* offsets, int G, int D, int I, void* y,
                          cudaStream_t st) {
  if (rows == 0) return MOK_OK;
  MxParams P;
  P.sched = mx_sched(offsets, G, rows, D / 256, I / BKB);
  P.status = status_ptr();
  if (!P.status) return MOK_ERR_CUDA;
  const int64_t wrows = static_cast<int64_t>(offsets ? G : 1) * D;
  if (!code_map(&P.tmA, aq, rows, I) || !scale_map(&P.tmSA, asc, rows, I, SA_WORDS) ||
      !code_map(&P.tmB0, qd, wrows, I) || !scale_map(&P.tmSB0, sd, wrows, I, 128))
    return MOK_ERR_CUDA;
  P.tmB1 = P.tmB0;
  P.tmSB1 = P.tmSB0;
  P.b_group_rows = D;
  P.b_tile_rows = 256;
  P.b1_off = 128;
  P.aq = nullptr;
  P.asc = nullptr;
  P.a_ld = 0;
  P.y = static_cast<__nv_bfloat16*>(y);
  P.out_ld = D;
  return run_mx<false>(P, st);
}

}  // namespace mok
