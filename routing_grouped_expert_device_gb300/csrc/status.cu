// Device status word, tensor-map encoding and small host utilities.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// One status word per device that loads the library.  Kernels receive its
// address; mok_get_error() reads and clears it.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
mok::SymbolCache g_status_cache;
int g_num_sms[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

template <class F>
bool driver_fn(const char* name, int version, F* out) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  *out = reinterpret_cast<F>(fn);
  return true;
}

// Id of the context current on this thread (unique for the life of the
// process; a context made after cudaDeviceReset gets a new one).  Called
// with g_mu held.
bool current_context_id(unsigned long long* id) {
  if (!g_ctx_current && !driver_fn("cuCtxGetCurrent", 4000, &g_ctx_current)) return false;
  if (!g_ctx_id && !driver_fn("cuCtxGetId", 12000, &g_ctx_id)) return false;
  CUcontext c = nullptr;
  if (g_ctx_current(&c) != CUDA_SUCCESS || !c) return false;
  return g_ctx_id(c, id) == CUDA_SUCCESS;
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

}  // namespace

namespace mok {

void* symbol_address(const void* symbol, SymbolCache& cache) {
  int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);
  if (!known || !cache.addr[d] || cache.ctx[d] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
    // the lookup made the device's context current if none was
    if (!known && !current_context_id(&ctx)) ctx = 0;
    cache.addr[d] = p;
    cache.ctx[d] = ctx;
  }
  return cache.addr[d];
}

int* status_ptr() { return static_cast<int*>(symbol_address(&g_status_word, g_status_cache)); }

int num_sms() {
  int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_num_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_num_sms[d] = n > 0 ? n : 1;
  }
  return g_num_sms[d];
}

bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t rows,
                  uint64_t cols, uint64_t pitch_bytes, uint32_t box_rows, uint32_t box_cols,
                  bool swizzle128) {
  return make_tmap_2d_swz(m, base, dt, rows, cols, pitch_bytes, box_rows, box_cols,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_tmap_2d_swz(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t rows,
                      uint64_t cols, uint64_t pitch_bytes, uint32_t box_rows, uint32_t box_cols,
                      CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mok

extern "C" mok_status mok_get_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOK_ERR_CUDA;
  int* p = mok::status_ptr();
  if (!p) return MOK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOK_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOK_ERR_CUDA;
  }
  return static_cast<mok_status>(v & 0xFF);
}

extern "C" const char* mok_status_string(mok_status s) {
  switch (s) {
    case MOK_OK: return "ok";
    case MOK_ERR_INVALID_ARG: return "invalid argument";
    case MOK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOK_ERR_WORKSPACE: return "workspace too small";
    case MOK_ERR_CUDA: return "CUDA runtime or launch error";
    case MOK_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOK_ERR_BAD_ROUTE: return "expert index out of range";
  }
  return "unknown status";
}
