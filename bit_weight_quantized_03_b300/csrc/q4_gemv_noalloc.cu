// q4_gemv_noalloc.cu -- the batch-1 / small-batch GEMV for callers that cannot
// allocate device memory.
//
// q4_gemv takes its split-K scratch (row-group arrival counters and partial
// row sums) from a workspace the caller allocates.  Some callers cannot make
// that allocation: a host that embeds this library inside another runtime's
// fixed memory pool and forbids cudaMalloc, a real-time audio loop that must
// not allocate (or risk an implicit device synchronisation) once streaming has
// started, or a plugin that is only ever handed input and output buffers.
// q4_gemv_noalloc gives them the same product with the scratch taken from one
// fixed array compiled into this file.
//
// The array lives in device memory of every GPU that loads the library, until
// the process exits.  Its device address is looked up once per device, with
// that device current, on the first call made there; do that first call
// before any stream capture.  All calls share the array: the part a call uses
// is cleared on the stream at the start of the call, and calls whose
// executions overlap on the GPU (different streams) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/q4.h"
#include "q4_internal.h"

namespace {

constexpr size_t kScratchBytes = Q4_GEMV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_gemv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_dev_addr[kMaxDevices] = {};

// Device address of g_gemv_scratch on the current device.  In host code the
// name g_gemv_scratch is only a host-side stand-in for the symbol, never an
// address a kernel may be given.
q4_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_dev_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress((void**)&ptr, g_gemv_scratch);
    if (e != cudaSuccess || ptr == nullptr) return Q4_ERR_CUDA;
    g_scratch_dev_addr[dev] = ptr;
  }
  *out = g_scratch_dev_addr[dev];
  return Q4_OK;
}

}  // namespace

extern "C" q4_status q4_gemv_noalloc(const void* W, int64_t n, int64_t k, const float* x,
                                     int64_t m, int64_t ldx, float* y, int64_t ldy,
                                     int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  // Cheap checks first, so that bad arguments are reported without touching
  // the device; q4_gemv repeats every check before it launches.
  if (W == nullptr || x == nullptr || y == nullptr || n <= 0 || k <= 0 || m <= 0)
    return Q4_ERR_INVALID_ARG;
  if (k % Q4_BLOCK_ELEMS != 0 || m > Q4_GEMV_MAX_M) return Q4_ERR_UNSUPPORTED_SHAPE;
  const size_t need = q4_gemv_workspace_bytes(n, k, m);
  if (need > kScratchBytes) return Q4_ERR_UNSUPPORTED_SHAPE;
  void* scratch = nullptr;
  if (need > 0) {
    const q4_status st = scratch_address(&scratch);
    if (st != Q4_OK) return st;
    // The arrival counters must start at zero whatever an earlier call left.
    if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess)
      return Q4_ERR_CUDA;
  }
  return q4_gemv(W, n, k, x, m, ldx, y, ldy, scratch, need, status_dev, flags, s);
}
