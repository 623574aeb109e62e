// awq_search_noalloc: the alpha-grid search with its scratch in a fixed
// device array of this library instead of a caller-provided workspace, for
// callers that cannot allocate device memory (declared in include/awq.h).
//
// The array is a file-scope __device__ variable.  On the host its name is
// only a stand-in for the symbol, not a device address, so the host looks
// the address up with cudaGetSymbolAddress, once per device with that
// device current, and hands the result to the ordinary search path as its
// workspace.  That path clears every workspace word that must start at
// zero on each call, so stale contents of an earlier call do not matter.
#include <mutex>

#include "awq.h"
#include "awq_internal.h"

namespace awq {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[AWQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (cached), or
// nullptr with *err set when the lookup fails.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace awq

extern "C" int awq_search_noalloc(const void* W, const void* X, int dtype, int64_t out,
                                  int64_t in, int64_t N, const double* sx, int bits, int group,
                                  int sym, int grid, double* err, int32_t* best, float* s_best,
                                  int32_t* dev_status, awq_stream_t stream) {
  const size_t need = awq_search_workspace_min_bytes(dtype, out, in, N, group, grid);
  if (need == 0) return AWQ_ERR_INVALID_ARG;               // sizes the search rejects anyway
  if (need > AWQ_NOALLOC_SCRATCH_BYTES) return AWQ_ERR_UNSUPPORTED;  // beyond the fixed array
  cudaError_t e = cudaSuccess;
  void* ws = awq::scratch_on_current_device(&e);
  if (ws == nullptr) return AWQ_ERR_CUDA;
  return awq_search_ex(W, X, dtype, out, in, N, sx, bits, group, sym, grid, ws,
                       AWQ_NOALLOC_SCRATCH_BYTES, err, best, s_best, dev_status, stream, nullptr);
}
