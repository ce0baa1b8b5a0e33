// tp_colsum_noalloc: the column-sum reduction (bias gradients) for callers
// that cannot allocate device memory.
//
// tp_colsum needs a caller-provided workspace for its per-chunk partial sums.
// Some callers have no way to provide one: code that is not allowed to call
// cudaMalloc (it synchronises the device and can stall every other stream of
// a latency-bound service), code whose device memory is entirely held by
// another allocator's pool, or plugin-style code that receives only its input
// and output pointers.  This entry point takes the same inputs and outputs and
// keeps its scratch in a fixed-size array that lives in this library's device
// image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kColsumNoallocMaxFloats * 4 bytes (4 MiB) until the process
// exits.  In host code the array's name is only a host-side stand-in: its
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, on the first call made on that device, and passed to
// the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "trace.h"

namespace tp {
namespace {

constexpr size_t kColsumNoallocMaxFloats = size_t(1) << 20;  // 4 MiB of fp32 partial sums

__device__ __align__(256) float g_colsum_noalloc_scratch[kColsumNoallocMaxFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
float* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_colsum_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace tp

extern "C" tp_status tp_colsum_noalloc(const tp_bf16* G, int64_t rows, int64_t cols, float* out, int accumulate,
                                       tp_stream stream) {
  TP_TRACE();
  using namespace tp;
  if (rows < 0 || cols < 0) return TP_ERR_INVALID_ARG;
  if (cols == 0) return TP_OK;
  // The partial sums need colsum_ws_floats(rows, cols) floats; beyond the array's size the call is refused.
  if (colsum_ws_floats(rows, cols) > kColsumNoallocMaxFloats) return TP_ERR_SHAPE;
  if (!G || !out) return TP_ERR_INVALID_ARG;
  TP_RETURN_IF(ready());
  float* scratch = scratch_for_current_device();
  if (!scratch) return TP_ERR_CUDA;
  // Every chunk's partial sums are written before they are read, so the
  // previous call's contents never leak into this one.
  return run_colsum(G, rows, cols, cols, out, accumulate, scratch, kColsumNoallocMaxFloats,
                    reinterpret_cast<cudaStream_t>(stream));
}
