// Top-K routing and the device-side plan (Mixture-of-Kittens blog,
// "Overlapping computation and communication in MoE" for the router weights
// g, "Scheduling" for the pull schedule: counts, exclusive-scan offsets and a
// table indexed by destination slot; one source rank on one GPU).
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace mok {
namespace {

// ---------------------------------------------------------------------------
// route: one warp per token.  Lane l holds scores e = j*32 + l.  K rounds of
// a warp arg-max (larger score first, lower index on ties) pick the experts
// in descending order; den is summed in k order and g = s / den (IEEE).
// ---------------------------------------------------------------------------
template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ s, int T, int E, int K,
                                                    int32_t* __restrict__ topk,
                                                    float* __restrict__ g) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    const float* row = s + static_cast<size_t>(t) * E;
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = j * 32 + lane;
      v[j] = e < E ? __ldg(row + e) : 0.0f;
    }
    uint32_t taken = 0;
    float my_v = 0.0f;
    int my_i = 0;
    for (int k = 0; k < K; ++k) {
      float bv = 0.0f;
      int bi = INT_MAX;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = j * 32 + lane;
        if (e < E && !((taken >> j) & 1u) && (bi == INT_MAX || v[j] > bv)) {
          bv = v[j];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const bool take = (oi != INT_MAX) && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi));
        if (take) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == k) {
        my_v = bv;
        my_i = bi;
      }
    }
    float den = __shfl_sync(0xffffffffu, my_v, 0);
    for (int k = 1; k < K; ++k) den = __fadd_rn(den, __shfl_sync(0xffffffffu, my_v, k));
    if (lane < K) {
      topk[static_cast<size_t>(t) * K + lane] = my_i;
      g[static_cast<size_t>(t) * K + lane] = __fdiv_rn(my_v, den);
    }
  }
}

// ---------------------------------------------------------------------------
// plan: routes are cut into chunks of kPlanChunk consecutive route ids, one
// chunk per CTA and kPlanChunk/kPlanWarps routes per warp.
//   count : per-chunk histogram hist[chunk][e]
//   scan  : counts, offsets, and hist[chunk][e] <- offsets[e] + routes of e
//           in earlier chunks (the chunk's first slot for expert e)
//   place : per warp, the slot of each route = chunk base + routes of e in
//           earlier warps of the chunk + rank among equal experts of the
//           same 32-route batch (match.any) + earlier batches of the warp.
// Every step keeps (t, k) order inside an expert, so the result is the
// stable counting sort the pull schedule reduces to with one source rank.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;

__device__ __forceinline__ void warp_histogram(const int32_t* __restrict__ topk, int64_t r0,
                                               int64_t r1, int E, int* hist_row, int* status) {
  const int lane = threadIdx.x & 31;
  for (int64_t base = r0; base < r1; base += 32) {
    const int64_t r = base + lane;
    const bool in = r < r1;
    int e = in ? __ldg(topk + r) : -1;
    const bool ok = in && e >= 0 && e < E;
    if (in && !ok) report(status, MOK_ERR_BAD_ROUTE);
    if (!ok) e = -1 - lane;  // distinct sentinel per lane, never counted
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (ok && (__ffs(peers) - 1) == lane) hist_row[e] += __popc(peers);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(const int32_t* __restrict__ topk,
                                                                  int64_t R, int E, int chunk,
                                                                  int* __restrict__ hist,
                                                                  int* status) {
  extern __shared__ int sh[];  // [kPlanWarps][E]
  for (int i = threadIdx.x; i < kPlanWarps * E; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int per_warp = chunk / kPlanWarps;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * chunk + static_cast<int64_t>(warp) * per_warp;
  const int64_t r1 = r0 + per_warp < R ? r0 + per_warp : R;
  if (r0 < R) warp_histogram(topk, r0, r1, E, sh + warp * E, status);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < kPlanWarps; ++w) c += sh[w * E + e];
    hist[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

// One CTA of up to 1024 threads; thread e owns expert e.
__global__ void __launch_bounds__(1024) plan_scan_kernel(int* __restrict__ hist, int nchunks, int E,
                                                         int64_t R, int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    // eight independent loads in flight, then their running sum
    for (int c0 = 0; c0 < nchunks; c0 += 8) {
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = c0 + u < nchunks ? hist[static_cast<size_t>(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < nchunks) hist[static_cast<size_t>(c0 + u) * E + e] = run;
        run += h[u];
      }
    }
  }
  // exclusive scan of run over e
  const int lane = e & 31, w = e >> 5;
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int t = lane < nw ? warp_tot[lane] : 0;
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += v;
    }
    warp_tot[lane] = ti - t;
  }
  __syncthreads();
  const int excl = warp_tot[w] + incl - run;
  if (e < E) {
    counts[e] = run;
    offsets[e] = excl;
    for (int c = 0; c < nchunks; ++c) hist[static_cast<size_t>(c) * E + e] += excl;  // independent updates
  }
  if (e == 0) offsets[E] = static_cast<int32_t>(R);
}

__global__ void __launch_bounds__(kPlanThreads) plan_place_kernel(const int32_t* __restrict__ topk,
                                                                  int64_t R, int E, int chunk,
                                                                  const int* __restrict__ base,
                                                                  int32_t* __restrict__ table,
                                                                  int32_t* __restrict__ route_dst) {
  extern __shared__ int sh[];  // [kPlanWarps][E]: per-warp histogram, then per-warp cursor
  for (int i = threadIdx.x; i < kPlanWarps * E; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_warp = chunk / kPlanWarps;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * chunk + static_cast<int64_t>(warp) * per_warp;
  const int64_t r1 = r0 + per_warp < R ? r0 + per_warp : R;
  if (r0 < R) warp_histogram(topk, r0, r1, E, sh + warp * E, nullptr);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[static_cast<size_t>(blockIdx.x) * E + e];
    for (int w = 0; w < kPlanWarps; ++w) {
      const int h = sh[w * E + e];
      sh[w * E + e] = run;
      run += h;
    }
  }
  __syncthreads();
  int* cur = sh + warp * E;
  for (int64_t b = r0; b < r1; b += 32) {
    const int64_t r = b + lane;
    const bool in = r < r1;
    int e = in ? __ldg(topk + r) : -1;
    const bool ok = in && e >= 0 && e < E;
    if (!ok) e = -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (ok) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int dst = cur[e] + rank;
      table[static_cast<size_t>(dst) * 3 + 0] = static_cast<int32_t>(r);
      table[static_cast<size_t>(dst) * 3 + 1] = e;
      table[static_cast<size_t>(dst) * 3 + 2] = dst;
      route_dst[r] = dst;
    }
    __syncwarp();
    if (ok && (__ffs(peers) - 1) == lane) cur[e] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// The pull schedule with several source ranks (blog, "Scheduling"; paper
// note, "Pull dispatch, push combine": slots of a local expert ordered by
// per-source ordinal, then source rank), on one GPU: the T tokens form
// `ranks` contiguous virtual source ranks of T / ranks tokens.  Starting from
// the one-rank plan, route (t, k) of expert e, rank r = t / (T / ranks) and
// ordinal o among the routes of (e, r) gets slot
// offsets[e] + sum_r' min(M[e][r'], o) + |{r' < r : M[e][r'] > o}|.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) plan_rank_count_kernel(const int32_t* __restrict__ topk, int64_t R, int K,
                                                              int per_rank, int ranks, int* __restrict__ M) {
  for (int64_t src = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; src < R;
       src += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = __ldg(topk + src);
    const int r = static_cast<int>((src / K) / per_rank);
    atomicAdd(M + static_cast<int64_t>(e) * ranks + r, 1);  // integer counts: order-independent
  }
}

// one thread per expert: exclusive prefix of M[e][.] over ranks
__global__ void plan_rank_prefix_kernel(const int* __restrict__ M, int E, int ranks, int* __restrict__ pre) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int run = 0;
  for (int r = 0; r < ranks; ++r) {
    pre[static_cast<int64_t>(e) * ranks + r] = run;
    run += M[static_cast<int64_t>(e) * ranks + r];
  }
}

__global__ void __launch_bounds__(256) plan_rank_place_kernel(const int32_t* __restrict__ topk, int64_t R, int K,
                                                              int per_rank, int ranks, const int* __restrict__ M,
                                                              const int* __restrict__ pre,
                                                              const int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ table,
                                                              int32_t* __restrict__ route_dst) {
  for (int64_t src = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; src < R;
       src += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = __ldg(topk + src);
    const int r = static_cast<int>((src / K) / per_rank);
    const int* Me = M + static_cast<int64_t>(e) * ranks;
    // the one-rank slot is the route's ordinal within its expert
    const int o = route_dst[src] - offsets[e] - pre[static_cast<int64_t>(e) * ranks + r];
    int p = 0;
    for (int q = 0; q < ranks; ++q) {
      const int m = Me[q];
      p += m < o ? m : o;
      if (q < r && m > o) ++p;
    }
    const int dst = offsets[e] + p;
    table[static_cast<int64_t>(dst) * 3 + 0] = static_cast<int32_t>(src);
    table[static_cast<int64_t>(dst) * 3 + 1] = e;
    table[static_cast<int64_t>(dst) * 3 + 2] = dst;
    route_dst[src] = dst;
  }
}

}  // namespace

int plan_chunks(int64_t R) { return static_cast<int>((R + kPlanChunk - 1) / kPlanChunk); }

size_t plan_scratch_bytes(int64_t R, int E) {
  return static_cast<size_t>(plan_chunks(R > 0 ? R : 1)) * static_cast<size_t>(E) * sizeof(int);
}

mok_status launch_route(const float* s, int T, int E, int K, int32_t* topk, float* g,
                        cudaStream_t st) {
  if (T == 0) return MOK_OK;
  const int threads = 256;
  const int warps_needed = T;
  int blocks = (warps_needed + (threads / 32) - 1) / (threads / 32);
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) route_kernel<1><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  else if (vpl <= 2) route_kernel<2><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  else if (vpl <= 4) route_kernel<4><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  else if (vpl <= 8) route_kernel<8><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  else if (vpl <= 16) route_kernel<16><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  else route_kernel<32><<<blocks, threads, 0, st>>>(s, T, E, K, topk, g);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

mok_status launch_plan(const int32_t* topk, int64_t R, int E, int32_t* counts, int32_t* offsets,
                       int32_t* table, int32_t* route_dst, int* hist, cudaStream_t st) {
  int* status = status_ptr();
  if (!status) return MOK_ERR_CUDA;
  const int nchunks = plan_chunks(R > 0 ? R : 1);
  const size_t sh = static_cast<size_t>(kPlanWarps) * E * sizeof(int);
  if (sh > 48 * 1024) {
    if (cudaFuncSetAttribute(plan_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sh)) != cudaSuccess ||
        cudaFuncSetAttribute(plan_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sh)) != cudaSuccess)
      return MOK_ERR_CUDA;
  }
  plan_count_kernel<<<nchunks, kPlanThreads, sh, st>>>(topk, R, E, kPlanChunk, hist, status);
  MOK_CHECK_LAUNCH();
  const int scan_threads = ((E + 31) / 32) * 32;
  plan_scan_kernel<<<1, scan_threads, 0, st>>>(hist, nchunks, E, R, counts, offsets);
  MOK_CHECK_LAUNCH();
  if (R > 0) {
    plan_place_kernel<<<nchunks, kPlanThreads, sh, st>>>(topk, R, E, kPlanChunk, hist, table,
                                                         route_dst);
    MOK_CHECK_LAUNCH();
  }
  return MOK_OK;
}

size_t plan_ranks_scratch_bytes(int64_t R, int E, int ranks) {
  return plan_scratch_bytes(R, E) + 2 * static_cast<size_t>(E) * ranks * sizeof(int);
}

mok_status launch_plan_ranks(const int32_t* topk, int64_t T, int K, int E, int ranks, int32_t* counts,
                             int32_t* offsets, int32_t* table, int32_t* route_dst, int* scratch,
                             cudaStream_t st) {
  const int64_t R = T * K;
  mok_status r = launch_plan(topk, R, E, counts, offsets, table, route_dst, scratch, st);
  if (r != MOK_OK || ranks == 1 || R == 0) return r;
  int* M = scratch + plan_scratch_bytes(R, E) / sizeof(int);
  int* pre = M + static_cast<int64_t>(E) * ranks;
  const int per_rank = static_cast<int>(T / ranks);
  if (cudaMemsetAsync(M, 0, static_cast<size_t>(E) * ranks * sizeof(int), st) != cudaSuccess) return MOK_ERR_CUDA;
  const int blocks = static_cast<int>((R + 255) / 256 < num_sms() * 8 ? (R + 255) / 256 : num_sms() * 8);
  plan_rank_count_kernel<<<blocks, 256, 0, st>>>(topk, R, K, per_rank, ranks, M);
  MOK_CHECK_LAUNCH();
  plan_rank_prefix_kernel<<<(E + 255) / 256, 256, 0, st>>>(M, E, ranks, pre);
  MOK_CHECK_LAUNCH();
  plan_rank_place_kernel<<<blocks, 256, 0, st>>>(topk, R, K, per_rank, ranks, M, pre, offsets, table, route_dst);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}

}  // namespace mok

extern "C" mok_status mok_route(const float* s, int32_t T, int32_t E, int32_t K, int32_t* topk_idx,
                                float* g, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOK_ERR_INVALID_ARG;
  if (T > 0 && (!s || !topk_idx || !g)) return MOK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K >= (int64_t(1) << 31)) return MOK_ERR_UNSUPPORTED;
  return mok::launch_route(s, T, E, K, topk_idx, g, static_cast<cudaStream_t>(stream));
}

extern "C" mok_status mok_plan(const int32_t* topk_idx, int32_t T, int32_t E, int32_t K,
                               int32_t* counts, int32_t* offsets, int32_t* table,
                               int32_t* route_dst, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOK_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(T) * K;
  if (R >= (int64_t(1) << 31)) return MOK_ERR_UNSUPPORTED;
  if (!counts || !offsets || !ws) return MOK_ERR_INVALID_ARG;
  if (R > 0 && (!topk_idx || !table || !route_dst)) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < mok::plan_scratch_bytes(R, E)) return MOK_ERR_WORKSPACE;
  return mok::launch_plan(topk_idx, R, E, counts, offsets, table, route_dst, static_cast<int*>(ws),
                          static_cast<cudaStream_t>(stream));
}

extern "C" size_t mok_plan_ranks_workspace_bytes(int32_t T, int32_t E, int32_t K, int32_t ranks) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E || ranks < 1 || (ranks > 1 && T % ranks)) return 0;
  return mok::plan_ranks_scratch_bytes(static_cast<int64_t>(T) * K, E, ranks);
}

extern "C" mok_status mok_plan_ranks(const int32_t* topk_idx, int32_t T, int32_t E, int32_t K, int32_t ranks,
                                     int32_t* counts, int32_t* offsets, int32_t* table, int32_t* route_dst,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E || ranks < 1 || ranks > 4096) return MOK_ERR_INVALID_ARG;
  if (ranks > 1 && T % ranks) return MOK_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(T) * K;
  if (R >= (int64_t(1) << 31)) return MOK_ERR_UNSUPPORTED;
  if (!counts || !offsets || !ws) return MOK_ERR_INVALID_ARG;
  if (R > 0 && (!topk_idx || !table || !route_dst)) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < mok::plan_ranks_scratch_bytes(R, E, ranks)) return MOK_ERR_WORKSPACE;
  return mok::launch_plan_ranks(topk_idx, T, K, E, ranks, counts, offsets, table, route_dst, static_cast<int*>(ws),
                                static_cast<cudaStream_t>(stream));
}
