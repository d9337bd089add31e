// Memory-bound kernels: gather (dispatch), MXFP8 quantisation and the
// fixed-order weighted combine.  All accesses are 16-byte vectors.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace mok {
namespace {

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Dispatch (Mixture-of-Kittens blog, "Scheduling": rows land
// expert-contiguous).  One warp per token: its row is read once, 4 vectors
// per lane in flight, and stored at each of its K positions in expert order,
// p = route_dst[t K + k] (lane k holds p, K <= 32).  Reading each row once
// instead of once per route keeps x's K re-reads off DRAM while the K D-wide
// copies stream out.  When g_route is non-null also g_route[p] = g[t K + k].
__global__ void __launch_bounds__(256) dispatch_bf16_kernel(const uint4* __restrict__ x,
                                                            const int32_t* __restrict__ route_dst,
                                                            int T, int K, int D8,
                                                            uint4* __restrict__ xg,
                                                            const float* __restrict__ g,
                                                            float* __restrict__ g_route) {
  const int lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>((static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5);
  for (int t = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5); t < T;
       t += nwarps) {
    const int64_t r0 = static_cast<int64_t>(t) * K;
    const int dst = lane < K ? __ldg(route_dst + r0 + lane) : 0;
    if (g_route && lane < K) g_route[dst] = g[r0 + lane];
    const uint4* in = x + static_cast<int64_t>(t) * D8;
#pragma unroll 1
    for (int i0 = 0; i0 < D8; i0 += 128) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + 32 * u + lane;
        v[u] = i < D8 ? ld_nc_v4(in + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        uint4* out = xg + static_cast<int64_t>(__shfl_sync(0xffffffffu, dst, k)) * D8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < D8) out[i] = v[u];
        }
      }
    }
  }
}

// Smallest e with amax <= 448 * 2^e for a finite amax >= 0: with
// amax = 1.f * 2^E, 448 = 1.75 * 2^8, e = E - 8 if 1.f <= 1.75 else E - 7.
// Zero and subnormal amax give the E8M0 minimum, -127.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int eb = static_cast<int>((b >> 23) & 0xFFu);
  if (eb == 0) return -127;
  const int e = eb - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// One warp per row: lane l holds 8 consecutive values (16 bytes), so a
// 1x32 block is 4 lanes (its amax: two xor shuffles) and one pass of the warp
// covers 256 columns, two 128-column scale groups; loads and code stores are
// contiguous across the warp.  Each group's 4 scale bytes are gathered into
// one 32-bit word (layout in kernels.h).  route_dst == nullptr: row r is
// stored at row r, plain layout (the quantiser).  Else (the dispatch with
// fused quantisation) the rows are tokens: token t is quantised once and
// stored at each of its K positions p = route_dst[t K + k] (lane k holds p
// and its scale position, K <= 32), with the grouped scale layout of expert
// table[p].e.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ src,
                                                         const int32_t* __restrict__ route_dst,
                                                         const int32_t* __restrict__ table,
                                                         const int32_t* __restrict__ offsets, int K,
                                                         int64_t rows, int64_t cols, int64_t ld,
                                                         uint2* __restrict__ q,
                                                         uint32_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int c8 = static_cast<int>(cols / 8);  // 16-byte vectors per row
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
    for (int v0 = 0; v0 < c8; v0 += 128) {  // 4 passes of 256 columns in flight
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vi = v0 + 32 * u + lane;
        v[u] = vi < c8 ? ld_nc_v4(in + vi) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vi = v0 + 32 * u + lane;
        if (v0 + 32 * u >= c8) break;  // warp-uniform: cols is a multiple of 128 (16 vectors)
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[2 * j] = bf16lo(w[j]);
          f[2 * j + 1] = bf16hi(w[j]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = mx_exponent(amax);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
        uint32_t packed[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2(f[4 * j] * inv, f[4 * j + 1] * inv), __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
              make_float2(f[4 * j + 2] * inv, f[4 * j + 3] * inv), __NV_SATFINITE, __NV_E4M3);
          packed[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        // scale word of the 128-column group of lanes 16h .. 16h + 15: byte b
        // from lane 16h + 4b
        const uint32_t byte = static_cast<uint32_t>(e + 127);
        const int base = lane & 16;
        const uint32_t word = __shfl_sync(0xffffffffu, byte, base) |
                              (__shfl_sync(0xffffffffu, byte, base + 4) << 8) |
                              (__shfl_sync(0xffffffffu, byte, base + 8) << 16) |
                              (__shfl_sync(0xffffffffu, byte, base + 12) << 24);
#pragma unroll 1
        for (int k = 0; k < ndst; ++k) {
          const int64_t p = __shfl_sync(0xffffffffu, dst, k);
          const int64_t pos = __shfl_sync(0xffffffffu, dpos, k);
          if (vi < c8) q[p * c8 + vi] = make_uint2(packed[0], packed[1]);
          if ((lane & 15) == 0 && vi < c8) scale[static_cast<int64_t>(vi / 16) * ld + pos] = word;
        }
      }
    }
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
  dispatch_bf16_kernel<<<grid_for(T, 8), 256, 0, st>>>(static_cast<const uint4*>(x), route_dst, T, K, D / 8,
                                                        static_cast<uint4*>(xg), g, g_route);
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
                                                    D, mx_scale_ld(R, E), static_cast<uint2*>(xg_q),
                                                    reinterpret_cast<uint32_t*>(xg_scale));
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_quantize_mxfp8(const void* src, int64_t rows, int64_t cols, void* q,
                                 uint8_t* scale, cudaStream_t st) {
  if (rows == 0) return MOK_OK;
  quant_rows_kernel<<<grid_for(rows, 8), 256, 0, st>>>(static_cast<const uint4*>(src), nullptr, nullptr, nullptr, 1,
                                                       rows, cols, mx_scale_ld(rows), static_cast<uint2*>(q),
                                                       reinterpret_cast<uint32_t*>(scale));
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
