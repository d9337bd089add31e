// mok_plan_static: the device plan without caller-provided scratch.
//
// mok_plan needs a few tens of kilobytes of device scratch for its per-chunk
// expert histograms, which the caller passes in as `ws`.  Some callers have
// no way to hand over device memory: their device memory is owned by another
// allocator (a framework's caching allocator, or a fixed arena carved up at
// start-up) that they may not call into from where the plan is built, or the
// code path is not allowed to allocate at all.  For them this entry point
// keeps the scratch in a fixed array that lives in this library's device
// image.  It allocates nothing.
//
// The array is `static __device__`, so every GPU that loads the library holds
// kStaticPlanScratchInts * 4 bytes (1 MiB) until the process exits.  In host
// code the name g_plan_scratch is only a host-side stand-in: the kernels get
// its device address, looked up with cudaGetSymbolAddress once per device
// and context (again after a cudaDeviceReset, whose new context reloads the
// module and may place the array elsewhere).
#include "common.cuh"
#include "kernels.h"

namespace {

// Histogram entries available: plan_chunks(R) * E must not exceed this.
constexpr int kStaticPlanScratchInts = 1 << 18;

static __device__ __align__(256) int g_plan_scratch[kStaticPlanScratchInts];

mok::SymbolCache g_scratch_cache;

// Device address of g_plan_scratch on the current device (with that device
// current): looked up on the first call in each context, then cached.
mok_status scratch_address(int** out) {
  *out = static_cast<int*>(mok::symbol_address(g_plan_scratch, g_scratch_cache));
  return *out ? MOK_OK : MOK_ERR_CUDA;
}

}  // namespace

extern "C" mok_status mok_plan_static(const int32_t* topk_idx, int32_t T, int32_t E, int32_t K,
                                      int32_t* counts, int32_t* offsets, int32_t* table,
                                      int32_t* route_dst, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOK_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(T) * K;
  if (R >= (int64_t(1) << 31)) return MOK_ERR_UNSUPPORTED;
  // The count kernel writes every histogram entry it later reads, so the
  // array needs no clearing between calls.
  if (static_cast<int64_t>(mok::plan_chunks(R > 0 ? R : 1)) * E > kStaticPlanScratchInts)
    return MOK_ERR_WORKSPACE;
  if (!counts || !offsets) return MOK_ERR_INVALID_ARG;
  if (R > 0 && (!topk_idx || !table || !route_dst)) return MOK_ERR_INVALID_ARG;
  int* scratch = nullptr;
  const mok_status st = scratch_address(&scratch);
  if (st != MOK_OK) return st;
  return mok::launch_plan(topk_idx, R, E, counts, offsets, table, route_dst, scratch,
                          static_cast<cudaStream_t>(stream));
}
