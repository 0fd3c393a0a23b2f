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
// the process exits.  Its device address is looked up once per CUDA context
// (normally once per device), with that context current, on the first call
// made there; do that first call before any stream capture.  All calls share
// the array: the part a call uses is cleared on the stream at the start of the
// call, and calls whose executions overlap on the GPU (different streams) race
// on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/q4.h"
#include "q4_internal.h"

namespace {

constexpr size_t kScratchBytes = Q4_GEMV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_gemv_scratch[kScratchBytes];

// Device address of g_gemv_scratch per CUDA context.  A context is named by
// its process-unique ID (cuCtxGetId), not by the device ordinal: after a
// cudaDeviceReset the device gets a new primary context, the module is loaded
// again and the array may sit at a new address, which a per-ordinal cache
// would miss.
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch_cache[kMaxContexts] = {};
int g_scratch_used = 0;

// The two driver calls used to name the current context, fetched from the
// driver at run time like every driver call of this library (no link-time
// dependency on libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_fns_once;

bool context_fns() {
  std::call_once(g_ctx_fns_once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return g_ctx_get_current != nullptr && g_ctx_get_id != nullptr;
}

// In host code the name g_gemv_scratch is only a host-side stand-in for the
// symbol, never an address a kernel may be given: the address comes from
// cudaGetSymbolAddress with the caller's context current.
q4_status scratch_address(void** out) {
  if (!context_fns()) return Q4_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return Q4_ERR_CUDA;
  if (ctx == nullptr) {
    // No context is current yet (the runtime creates the primary context
    // lazily): the symbol lookup below creates it.
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gemv_scratch) != cudaSuccess || ptr == nullptr)
      return Q4_ERR_CUDA;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return Q4_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return Q4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  for (int i = 0; i < g_scratch_used; ++i)
    if (g_scratch_cache[i].ctx_id == id) {
      *out = g_scratch_cache[i].addr;
      return Q4_OK;
    }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_gemv_scratch);
  if (e != cudaSuccess || ptr == nullptr) return Q4_ERR_CUDA;
  // Cache it; when the table is full the oldest entry makes room (a lookup
  // that misses only costs another cudaGetSymbolAddress).
  if (g_scratch_used == kMaxContexts) {
    for (int i = 1; i < kMaxContexts; ++i) g_scratch_cache[i - 1] = g_scratch_cache[i];
    --g_scratch_used;
  }
  g_scratch_cache[g_scratch_used++] = {id, ptr};
  *out = ptr;
  return Q4_OK;
}

}  // namespace

extern "C" q4_status q4_gemv_noalloc(const void* W, int64_t n, int64_t k, const float* x,
                                     int64_t m, int64_t ldx, float* y, int64_t ldy,
                                     int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  // Every argument rule of q4_gemv first, so that a refused call puts nothing
  // on the stream (and no memset node into a stream capture).
  q4_status st = q4::gemv_check_args(W, n, k, x, m, ldx, y, ldy);
  if (st != Q4_OK) return st;
  const size_t need = q4_gemv_workspace_bytes(n, k, m);
  if (need > kScratchBytes) return Q4_ERR_UNSUPPORTED_SHAPE;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != Q4_OK) return st;
    // The arrival counters must start at zero whatever an earlier call left
    // (a call that ended with a device error may leave partial sums behind).
    if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess)
      return Q4_ERR_CUDA;
  }
  return q4_gemv(W, n, k, x, m, ldx, y, ldy, scratch, need, status_dev, flags, s);
}
