// Memory-bound kernels: gather (dispatch), MXFP8 quantisation and the
// fixed-order weighted combine.  All accesses are 16-byte vectors.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "mx_quant.cuh"

namespace mok {
namespace {

// One warp per row: lane l holds 16 consecutive values (two 16-byte
// vectors), so a 1x32 block is 2 lanes (its amax: one xor shuffle), one pass
// of the warp covers 512 columns, four 128-column scale groups, and every
// code store is 16 bytes; loads and code stores are contiguous across the
// warp.  Each group's 4 scale bytes are gathered into one 32-bit word
// (layout in kernels.h).  route_dst == nullptr: row r is stored at row r,
// plain layout (the quantiser).  Else (the dispatch with fused
// quantisation) the rows are tokens: token t is quantised once and stored
// at each of its K positions p = route_dst[t K + k] (lane k holds p and its
// scale position, K <= 32), with the grouped scale layout of expert
// table[p].e.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ src,
                                                         const int32_t* __restrict__ route_dst,
                                                         const int32_t* __restrict__ table,
                                                         const int32_t* __restrict__ offsets, int K,
                                                         int64_t rows, int64_t cols, int64_t ld,
                                                         uint4* __restrict__ q,
                                                         uint32_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int c8 = static_cast<int>(cols / 8);  // 16-byte vectors per row (a multiple of 16)
  const int c16 = c8 / 2;                     // 16-byte code vectors per row
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows;
       row += nwarps) {
    int ndst = 1;
    int64_t dst = row, dpos = mx_scale_pos(row);
    if (route_dst) {
      ndst = K;
      if (lane < K) {
        dst = __ldg(route_dst + row * K + lane);
        const int e = __ldg(table + dst * 3 + 1);
        const int64_t off = __ldg(offsets + e);
        dpos = mx_scale_pos(mx_group_row0(off, e) + (dst - off));
      }
    }
    const uint4* in = src + row * c8;
#pragma unroll 1
    for (int v0 = 0; v0 < c8; v0 += 128) {  // 2 passes of 512 columns in flight
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int vi = v0 + 64 * u + 2 * lane;  // even; vi < c8 implies vi + 1 < c8
        v[2 * u] = vi < c8 ? ld_nc_v4(in + vi) : make_uint4(0, 0, 0, 0);
        v[2 * u + 1] = vi < c8 ? ld_nc_v4(in + vi + 1) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int vi = v0 + 64 * u + 2 * lane;
        if (v0 + 64 * u >= c8) break;  // warp-uniform
        const uint32_t w[8] = {v[2 * u].x, v[2 * u].y, v[2 * u].z, v[2 * u].w,
                               v[2 * u + 1].x, v[2 * u + 1].y, v[2 * u + 1].z, v[2 * u + 1].w};
        float f[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[2 * j] = bf16lo(w[j]);
          f[2 * j + 1] = bf16hi(w[j]);
        }
        int e;
        const uint4 codes = mx_codes16(f, e);
        const uint32_t word = mx_word8(e, lane);
#pragma unroll 1
        for (int k = 0; k < ndst; ++k) {
          const int64_t p = __shfl_sync(0xffffffffu, dst, k);
          const int64_t pos = __shfl_sync(0xffffffffu, dpos, k);
          if (vi < c8) q[p * c16 + vi / 2] = codes;
          if ((lane & 7) == 0 && vi < c8) scale[static_cast<int64_t>(vi / 16) * ld + pos] = word;
        }
      }
    }
  }
}

// Activation gradient of the MXFP8 backward (paper note, "The production
// details": MXFP8 with quantisation fused into the gated activation; the
// router-gradient inner product).  One warp per routed row p, 8 columns per
// lane: from fp32 h, u (the replay's, or for rows of a group that ends at or
// below kept_rows the forward's kept store act [R][2I]) and t = dY W_down
// it forms
// a = bf16(SiLU(h) u), da = g t, dh = bf16(da u SiLU'(h)), du = bf16(da SiLU(h)),
// a_g = bf16(g a) (bf16 [R][I], for the weight gradients), the E4M3 codes of
// [dh | du] [R][2I] with their scale words in the grouped layout of expert
// table[p].e (for dX), and dgp[p] = <t, SiLU(h) u> with the activation
// unrounded (per-lane sums in column order, then a fixed butterfly over the
// lanes).  g_route null: weight 1.
__global__ void __launch_bounds__(256) act_grad_mx_kernel(
    const float4* __restrict__ h, const float4* __restrict__ u, const float4* __restrict__ t,
    const float* __restrict__ g_route, const int32_t* __restrict__ table, const int32_t* __restrict__ offsets,
    int64_t R, int I, int64_t ld, uint4* __restrict__ dh, uint4* __restrict__ du, uint4* __restrict__ ag,
    uint2* __restrict__ dhu_q, uint32_t* __restrict__ dhu_sc, float* __restrict__ dgp,
    const float4* __restrict__ act, int32_t kept_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int I8 = I / 8;
  for (int64_t p = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; p < R; p += nwarps) {
    const int e = __ldg(table + p * 3 + 1);
    const int64_t off = __ldg(offsets + e);
    const int64_t pos = mx_scale_pos(mx_group_row0(off, e) + (p - off));
    // h, u of this row: the kept store (float4 units: h at p*2*I8*2, u I/4 later) or the replay's
    const bool kept = act && __ldg(offsets + e + 1) <= kept_rows;
    const float4* hsrc = kept ? act + p * (4 * I8) : h + p * (2 * I8);
    const float4* usrc = kept ? act + p * (4 * I8) + 2 * I8 : u + p * (2 * I8);
    const float g = g_route ? g_route[p] : 1.0f;
    float dot = 0.0f;
#pragma unroll 1
    for (int v0 = 0; v0 < I8; v0 += 32) {
      const int vi = v0 + lane;
      const bool in = vi < I8;  // warp-uniform per 16 lanes: I is a multiple of 128
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      const int64_t at = (p * I8 + vi) * 2;  // two float4 per 8 columns
      const float4 h0 = in ? hsrc[2 * vi] : z, h1 = in ? hsrc[2 * vi + 1] : z, u0 = in ? usrc[2 * vi] : z,
                   u1 = in ? usrc[2 * vi + 1] : z, t0 = in ? t[at] : z, t1 = in ? t[at + 1] : z;
      const float hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      const float uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      const float tw[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      float dhf[8], duf[8];
      uint32_t pdh[4], pdu[4], pag[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float agv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float hf = hw[2 * j + q], uf = uw[2 * j + q], tf = tw[2 * j + q];
          const float sig = sigmoid_f(hf);
          const float a_pre = (hf * sig) * uf;  // = silu_f(h) * u
          const float a = __bfloat162float(__float2bfloat16_rn(a_pre));
          dot = __fmaf_rn(tf, a_pre, dot);  // the router gradient takes the unrounded activation
          const float da = g * tf;
          dhf[2 * j + q] = __bfloat162float(__float2bfloat16_rn(da * uf * sig * (1.0f + hf * (1.0f - sig))));
          duf[2 * j + q] = __bfloat162float(__float2bfloat16_rn(da * hf * sig));
          agv[q] = g * a;
        }
        pdh[j] = pack_bf16x2(dhf[2 * j], dhf[2 * j + 1]);
        pdu[j] = pack_bf16x2(duf[2 * j], duf[2 * j + 1]);
        pag[j] = pack_bf16x2(agv[0], agv[1]);
      }
      if (in) {
        dh[p * I8 + vi] = make_uint4(pdh[0], pdh[1], pdh[2], pdh[3]);
        du[p * I8 + vi] = make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]);
        ag[p * I8 + vi] = make_uint4(pag[0], pag[1], pag[2], pag[3]);
      }
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        int ex;
        const uint2 codes = mx_codes8(part ? duf : dhf, ex);
        const uint32_t word = mx_word16(ex, lane);
        const int col8 = part * I8 + vi;  // 8-column unit within [dh | du]
        if (in) dhu_q[p * (2 * I8) + col8] = codes;
        if (in && (lane & 15) == 0) dhu_sc[static_cast<int64_t>(col8 / 16) * ld + pos] = word;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) dgp[p] = dot;
  }
}

// Paired scale blocks for the MXFP8 up/gate with the routed rows as N: the
// virtual row v = 128 b + m of block b = e (I / 64) + s is W_up row
// e I + 64 s + m (m < 64) or W_gate row e I + 64 s + m - 64, so that one
// 512-byte block holds the scales of a CTA's A operand (64 W_up rows, then
// the same W_gate rows) in the order the block-scaled MMA reads them.  For
// every 128-column group k of K: dst[k][pos(v)] = src[k][pos(row)].
__global__ void __launch_bounds__(256) pair_scales_kernel(const uint32_t* __restrict__ sg,
                                                          const uint32_t* __restrict__ su, int64_t ld_src,
                                                          int64_t ld_dst, int64_t vrows, int I, int kgroups,
                                                          uint32_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < vrows; v += stride) {
    const int64_t b = v >> 7;
    const int m = static_cast<int>(v & 127);
    const int64_t slices = I / 64;
    const int64_t r = (b / slices) * I + 64 * (b % slices) + (m & 63);
    const uint32_t* src = m < 64 ? su : sg;
    const int64_t ps = mx_scale_pos(r), pd = mx_scale_pos(v);
    for (int k = 0; k < kgroups; ++k) dst[k * ld_dst + pd] = src[k * ld_src + ps];
  }
}

// MXFP8 codes of transposed weights: output row (g, n) holds the M values
// src[g][m][n] (src bf16 [G][M][N]), quantised along m in 1x32 blocks:
// codes at q[(g N + n) * out_cols + col0 + m], scale words in the plain
// layout of G*N rows and out_cols columns.  A CTA moves a 128 (m) x 64 (n)
// tile through shared memory; each warp then quantises 8 output rows, lane
// l holding m = 4l .. 4l + 3 (a 32-block is 8 lanes, one scale word per row).
__global__ void __launch_bounds__(256) quant_cols_kernel(const uint4* __restrict__ src, int M, int N,
                                                         uint32_t* __restrict__ q, uint32_t* __restrict__ scale,
                                                         int out_cols, int col0, int64_t ld) {
  __shared__ uint16_t tile[128][66];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t gn0 = static_cast<int64_t>(blockIdx.x) * 64;  // first output row (g N + n0)
  const int64_t g = gn0 / N;
  const int n0 = static_cast<int>(gn0 - g * N);
  const int m0 = blockIdx.y * 128;
  const int N8 = N / 8;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = threadIdx.x / 8 + 32 * i, seg = threadIdx.x % 8;
    const uint4 v = src[(g * M + m0 + row) * N8 + n0 / 8 + seg];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      tile[row][seg * 8 + 2 * j] = static_cast<uint16_t>(w[j] & 0xFFFFu);
      tile[row][seg * 8 + 2 * j + 1] = static_cast<uint16_t>(w[j] >> 16);
    }
  }
  __syncthreads();
#pragma unroll 1
  for (int r = 0; r < 8; ++r) {
    const int n = warp * 8 + r;
    float f[4];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[i] = __uint_as_float(static_cast<uint32_t>(tile[4 * lane + i][n]) << 16);
      amax = fmaxf(amax, fabsf(f[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int e = mx_exponent(amax);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(f[0] * inv, f[1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(f[2] * inv, f[3] * inv), __NV_SATFINITE, __NV_E4M3);
    const int64_t orow = gn0 + n;
    q[(orow * out_cols + col0 + m0) / 4 + lane] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    const uint32_t byte = static_cast<uint32_t>(e + 127);
    const uint32_t word = __shfl_sync(0xffffffffu, byte, 0) | (__shfl_sync(0xffffffffu, byte, 8) << 8) |
                          (__shfl_sync(0xffffffffu, byte, 16) << 16) | (__shfl_sync(0xffffffffu, byte, 24) << 24);
    if (lane == 0) scale[static_cast<int64_t>((col0 + m0) / 128) * ld + mx_scale_pos(orow)] = word;
  }
}

// Fixed-order combine (paper note, "The production details": a fixed
// reduction order makes the layer bitwise deterministic).  One CTA per token;
// fp32 accumulation base -> k = 0 .. K-1, one rounding to bf16 at the end.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ rows,
                                                      const uint4* __restrict__ base,
                                                      const float* __restrict__ w,
                                                      const int32_t* __restrict__ route_dst, int T,
                                                      int K, int D8, uint4* __restrict__ out) {
  __shared__ int dst[32];
  __shared__ float wk[32];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < K) {
      dst[threadIdx.x] = route_dst[static_cast<int64_t>(t) * K + threadIdx.x];
      wk[threadIdx.x] = w ? w[static_cast<int64_t>(t) * K + threadIdx.x] : 1.0f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D8; i += blockDim.x) {
      float acc[8];
      if (base) {
        const uint4 b = ld_nc_v4(base + static_cast<int64_t>(t) * D8 + i);
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = bf16lo(bw[j]);
          acc[2 * j + 1] = bf16hi(bw[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      }
      for (int k = 0; k < K; ++k) {
        const uint4 v = ld_nc_v4(rows + static_cast<int64_t>(dst[k]) * D8 + i);
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
        const float gk = wk[k];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = __fmaf_rn(gk, bf16lo(vw[j]), acc[2 * j]);
          acc[2 * j + 1] = __fmaf_rn(gk, bf16hi(vw[j]), acc[2 * j + 1]);
        }
      }
      out[static_cast<int64_t>(t) * D8 + i] =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
    __syncthreads();
  }
}

// Router-weight gradient (g_k = s_k / den, den the fp32 sum of the top-k s
// in k order): dg_k = sum of the route's partials in order,
// ds[t, topk_k] = (dg_k - sum_k' g_k' dg_k') / den, zero elsewhere.
// One warp per token.
__global__ void __launch_bounds__(256) router_grad_kernel(
    const float* __restrict__ dgp, int nI, const int32_t* __restrict__ route_dst,
    const int32_t* __restrict__ topk, const float* __restrict__ g, const float* __restrict__ s,
    int T, int E, int K, float* __restrict__ ds, float* __restrict__ dg_out) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float dgk = 0.0f, gk = 0.0f, sk = 0.0f;
    int ek = 0;
    if (lane < K) {
      const int64_t r = static_cast<int64_t>(t) * K + lane;
      const int64_t dst = route_dst[r];
      for (int j = 0; j < nI; ++j) dgk = __fadd_rn(dgk, dgp[dst * nI + j]);
      gk = g[r];
      ek = topk[r];
      sk = s[static_cast<int64_t>(t) * E + ek];
    }
    float den = __shfl_sync(0xffffffffu, sk, 0);
    float dot = __fmul_rn(__shfl_sync(0xffffffffu, gk, 0), __shfl_sync(0xffffffffu, dgk, 0));
    for (int k = 1; k < K; ++k) {
      den = __fadd_rn(den, __shfl_sync(0xffffffffu, sk, k));
      dot = __fadd_rn(dot, __fmul_rn(__shfl_sync(0xffffffffu, gk, k), __shfl_sync(0xffffffffu, dgk, k)));
    }
    float* row = ds + static_cast<int64_t>(t) * E;
    for (int e = lane; e < E; e += 32) row[e] = 0.0f;
    __syncwarp();
    if (lane < K) {
      row[ek] = __fdiv_rn(__fsub_rn(dgk, dot), den);
      if (dg_out) dg_out[static_cast<int64_t>(t) * K + lane] = dgk;
    }
    __syncwarp();
  }
}

// Dispatch (Mixture-of-Kittens blog, "Scheduling": rows land
// expert-contiguous) by bulk copies, the TMA copy engine moving the bytes
// instead of vector loads and stores by threads: a warp per CTA moves one
// piece of P bytes of one token's row at a time, a bulk load into P bytes of
// shared memory and then K bulk stores from there, one per route (lane k
// stores to p = route_dst[t K + k]).  Each row is read once however many
// routes it has.  A CTA needs one warp, a few registers and P + 8 bytes of
// shared memory, so several fit beside a persistent GEMM that holds most of
// an SM (the shared expert's up/gate in the first dispatch window), where a
// warp-per-token dispatch got only the registers the GEMM leaves (DSV3
// forward 4.52-4.55 -> 4.49-4.50 ms).  Units (token, piece) are taken in
// token order; the next piece is loaded once every store of the current one
// has read the buffer.  Waits are bounded.  When g_route is non-null also
// g_route[p] = g[t K + k].
__global__ void __launch_bounds__(32) dispatch_bulk_kernel(const uint8_t* __restrict__ x,
                                                           const int32_t* __restrict__ route_dst, int T, int K,
                                                           int row_bytes, int pieces, uint8_t* __restrict__ xg,
                                                           const float* __restrict__ g, float* __restrict__ g_route,
                                                           int* status) {
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int lane = threadIdx.x;
  const int piece = row_bytes / pieces;
  if (lane == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  uint32_t phase = 0;
  const int64_t units = static_cast<int64_t>(T) * pieces;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int t = static_cast<int>(u / pieces);
    const int off = static_cast<int>(u - static_cast<int64_t>(t) * pieces) * piece;
    // (clamped to the R rows: a plan that reported a bad route leaves no store outside xg)
    const int dst = lane < K ? min(max(__ldg(route_dst + static_cast<int64_t>(t) * K + lane), 0), T * K - 1) : 0;
    if (g_route && off == 0 && lane < K) g_route[dst] = __ldg(g + static_cast<int64_t>(t) * K + lane);
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar, piece);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(buf)),
          "l"(x + static_cast<int64_t>(t) * row_bytes + off), "r"(piece), "r"(smem_u32(&bar))
          : "memory");
    }
    const bool ok = mbar_wait(&bar, phase, reinterpret_cast<volatile int*>(&abort_flag), status, SITE_PRODUCER);
    if (!__all_sync(0xffffffffu, ok)) {
      // the wait ran out (status set): give the load one more budget to
      // land before the CTA's shared memory is released
      if (lane == 0) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&bar, phase) && globaltimer() - t0 < kWaitBudgetNs) {
        }
      }
      __syncwarp();
      return;
    }
    phase ^= 1;
    if (lane < K) {
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       xg + static_cast<int64_t>(dst) * row_bytes + off),
                   "r"(smem_u32(buf)), "r"(piece)
                   : "memory");
      bulk_commit();
      bulk_wait_read0();  // the buffer is free again once every store has read it
    }
    __syncwarp();
  }
  if (lane < K) bulk_wait0();  // the stores have landed before the CTA exits
}

int grid_for(int64_t work_items, int per_block) {
  int64_t b = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (b > cap) b = cap;
  return b < 1 ? 1 : static_cast<int>(b);
}

}  // namespace

mok_status launch_dispatch_bf16(const void* x, const int32_t* route_dst, int T, int K, int D, void* xg,
                                const float* g, float* g_route, cudaStream_t st) {
  if (T == 0) return MOK_OK;
  if (K > 32) return MOK_ERR_UNSUPPORTED;
  // pieces of at most 4 KB that split the row evenly in 512-byte units
  const int row_bytes = D * 2;
  const int units = row_bytes / 512;  // D % 256 == 0
  int pieces = 1;
  while (units % pieces || 512 * (units / pieces) > 4096) ++pieces;
  int* status = status_ptr();
  if (!status) return MOK_ERR_CUDA;
  const int64_t n = static_cast<int64_t>(T) * pieces;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  const int grid = static_cast<int>(n < cap ? n : cap);
  dispatch_bulk_kernel<<<grid, 32, row_bytes / pieces, st>>>(static_cast<const uint8_t*>(x), route_dst, T, K,
                                                            row_bytes, pieces, static_cast<uint8_t*>(xg), g,
                                                            g_route, status);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_dispatch_mxfp8(const void* x, const int32_t* route_dst, const int32_t* table,
                                 const int32_t* offsets, int T, int K, int D, int E, void* xg_q, uint8_t* xg_scale,
                                 cudaStream_t st) {
  if (T == 0) return MOK_OK;
  if (K > 32) return MOK_ERR_UNSUPPORTED;
  const int64_t R = static_cast<int64_t>(T) * K;
  quant_rows_kernel<<<grid_for(T, 8), 256, 0, st>>>(static_cast<const uint4*>(x), route_dst, table, offsets, K, T,
                                                    D, mx_scale_ld(R, E), static_cast<uint4*>(xg_q),
                                                    reinterpret_cast<uint32_t*>(xg_scale));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_quantize_mxfp8(const void* src, int64_t rows, int64_t cols, void* q,
                                 uint8_t* scale, cudaStream_t st) {
  if (rows == 0) return MOK_OK;
  quant_rows_kernel<<<grid_for(rows, 8), 256, 0, st>>>(static_cast<const uint4*>(src), nullptr, nullptr, nullptr, 1,
                                                       rows, cols, mx_scale_ld(rows), static_cast<uint4*>(q),
                                                       reinterpret_cast<uint32_t*>(scale));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_pair_scales(const void* sg, const void* su, int G, int I, int D, void* sp, cudaStream_t st) {
  if (G == 0) return MOK_OK;
  if (I % 128 || D % 128) return MOK_ERR_UNSUPPORTED;
  const int64_t vrows = 2 * static_cast<int64_t>(G) * I;
  pair_scales_kernel<<<grid_for(vrows, 256), 256, 0, st>>>(
      static_cast<const uint32_t*>(sg), static_cast<const uint32_t*>(su), mx_scale_ld(static_cast<int64_t>(G) * I),
      mx_scale_ld(vrows), vrows, I, D / 128, static_cast<uint32_t*>(sp));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_act_grad_mx(const void* h, const void* u, const void* t, const float* g_route,
                              const int32_t* table, const int32_t* offsets, int64_t R, int I, int E, void* dh,
                              void* du, void* ag, void* dhu_q, uint8_t* dhu_sc, float* dgp, cudaStream_t st,
                              KeptAct kept) {
  if (R == 0) return MOK_OK;
  if (I % 128) return MOK_ERR_UNSUPPORTED;
  act_grad_mx_kernel<<<grid_for(R, 8), 256, 0, st>>>(
      static_cast<const float4*>(h), static_cast<const float4*>(u), static_cast<const float4*>(t), g_route, table,
      offsets, R, I, mx_scale_ld(R, E), static_cast<uint4*>(dh), static_cast<uint4*>(du), static_cast<uint4*>(ag),
      static_cast<uint2*>(dhu_q), reinterpret_cast<uint32_t*>(dhu_sc), dgp,
      reinterpret_cast<const float4*>(kept.act), kept.limit());
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_quantize_cols_mxfp8(const void* src, int G, int M, int N, void* q, uint8_t* scale, int out_cols,
                                      int col0, cudaStream_t st) {
  if (G == 0) return MOK_OK;
  if (M % 128 || N % 64 || col0 % 128 || out_cols % 128 || col0 + M > out_cols) return MOK_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(G) * N / 64), static_cast<unsigned>(M / 128));
  quant_cols_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), M, N, static_cast<uint32_t*>(q),
                                          reinterpret_cast<uint32_t*>(scale), out_cols, col0,
                                          mx_scale_ld(static_cast<int64_t>(G) * N));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_router_grad(const float* dgp, int nI, const int32_t* route_dst,
                              const int32_t* topk, const float* g, const float* s, int T, int E,
                              int K, float* ds, float* dg, cudaStream_t st) {
  if (T == 0) return MOK_OK;
  router_grad_kernel<<<grid_for(T, 8), 256, 0, st>>>(dgp, nI, route_dst, topk, g, s, T, E, K, ds,
                                                      dg);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_combine(const void* rows, const void* base, const float* w,
                          const int32_t* route_dst, int T, int K, int D, void* out,
                          cudaStream_t st) {
  if (T == 0) return MOK_OK;
  int blocks = T;
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  const int D8 = D / 8;
  const int threads = D8 >= 256 ? 256 : ((D8 + 31) / 32) * 32;
  combine_kernel<<<blocks, threads, 0, st>>>(static_cast<const uint4*>(rows),
                                             static_cast<const uint4*>(base), w, route_dst, T, K,
                                             D8, static_cast<uint4*>(out));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

}  // namespace mok
