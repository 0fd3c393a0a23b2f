// q4_api.cu -- the extern "C" entry points declared in include/q4.h: argument
// and alignment checks (nothing is launched when they fail), workspace sizing,
// the batch-size crossover of q4_linear, and the kernel launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/q4.h"
#include "q4_internal.h"

namespace q4 {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cached[dev] = v;
  }
  return cached[dev];
}

}  // namespace q4

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline q4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA; }

// Largest product sizes the kernels index with their 64-bit offsets; far above
// anything that fits in device memory, so these only catch garbage arguments.
constexpr int64_t kMaxDim = int64_t(1) << 40;

q4_status check_matrix(const void* W, int64_t n, int64_t k) {
  if (W == nullptr || n <= 0 || k <= 0 || n > kMaxDim || k > kMaxDim) return Q4_ERR_INVALID_ARG;
  if (k % Q4_BLOCK_ELEMS != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W, 16)) return Q4_ERR_MISALIGNED;
  return Q4_OK;
}

// Every argument rule of q4_gemm that the host can check (the workspace aside).
q4_status gemm_check_args(const void* W, int64_t n, int64_t k, const void* X, int64_t m,
                          int64_t ldx, const void* Y, q4_dtype y_dtype, int64_t ldy) {
  q4_status st = check_matrix(W, n, k);
  if (st != Q4_OK) return st;
  if (X == nullptr || Y == nullptr || m <= 0 || m > kMaxDim || ldx < k || ldy < n)
    return Q4_ERR_INVALID_ARG;
  if (y_dtype != Q4_F32 && y_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  if (k % 256 != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(X, 16) || ldx % 8 != 0) return Q4_ERR_MISALIGNED;
  if (!aligned(Y, y_dtype == Q4_F32 ? 4 : 2)) return Q4_ERR_MISALIGNED;
  return Q4_OK;
}

}  // namespace

namespace q4 {

q4_status gemv_check_args(const void* W, int64_t n, int64_t k, const float* x, int64_t m,
                          int64_t ldx, const float* y, int64_t ldy) {
  q4_status st = check_matrix(W, n, k);
  if (st != Q4_OK) return st;
  if (x == nullptr || y == nullptr || m <= 0 || ldx < k || ldy < n) return Q4_ERR_INVALID_ARG;
  if (m > Q4_GEMV_MAX_M) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || ldx % 4 != 0 || !aligned(y, 4)) return Q4_ERR_MISALIGNED;
  return Q4_OK;
}

}  // namespace q4

extern "C" {

const char* q4_version(void) { return "q4-b300 0.1 (sm_103a)"; }

const char* q4_status_string(q4_status st) {
  switch (st) {
    case Q4_OK: return "ok";
    case Q4_ERR_INVALID_ARG: return "invalid argument";
    case Q4_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case Q4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case Q4_ERR_NONFINITE: return "non-finite input or binary16 scale overflow";
    case Q4_ERR_ID_OUT_OF_RANGE: return "token id out of range";
    case Q4_ERR_TIMEOUT: return "bounded wait in a kernel ran out";
    case Q4_ERR_CUDA: return "CUDA error";
    case Q4_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

q4_status q4_quantize(const float* w, int64_t n, int64_t k, void* blocks, int32_t* status_dev,
                      q4_stream_t s) {
  if (w == nullptr || blocks == nullptr || n <= 0 || k <= 0 || n > kMaxDim || k > kMaxDim)
    return Q4_ERR_INVALID_ARG;
  if (k % Q4_BLOCK_ELEMS != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(blocks, 16)) return Q4_ERR_MISALIGNED;
  return from_cuda(q4::quantize_launch(w, n, k, static_cast<uint8_t*>(blocks), status_dev,
                                       reinterpret_cast<cudaStream_t>(s)));
}

q4_status q4_dequant_rows(const void* blocks, int64_t row0, int64_t n_rows, int64_t k, void* out,
                          q4_dtype out_dtype, q4_stream_t s) {
  q4_status st = check_matrix(blocks, n_rows, k);
  if (st != Q4_OK) return st;
  if (out == nullptr || row0 < 0 || row0 > kMaxDim) return Q4_ERR_INVALID_ARG;
  if (out_dtype != Q4_F32 && out_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  if (!aligned(out, 16)) return Q4_ERR_MISALIGNED;
  return from_cuda(q4::dequant_rows_launch(static_cast<const uint8_t*>(blocks), row0, n_rows, k,
                                           out, out_dtype == Q4_BF16,
                                           reinterpret_cast<cudaStream_t>(s)));
}

size_t q4_gemv_workspace_bytes(int64_t n, int64_t k, int64_t m) {
  if (n <= 0 || k <= 0 || k % Q4_BLOCK_ELEMS || m <= 0 || m > Q4_GEMV_MAX_M) return 0;
  return q4::gemv_plan(n, k, m).ws_bytes;
}

q4_status q4_gemv(const void* W, int64_t n, int64_t k, const float* x, int64_t m, int64_t ldx,
                  float* y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* status_dev,
                  uint32_t flags, q4_stream_t s) {
  q4_status st = q4::gemv_check_args(W, n, k, x, m, ldx, y, ldy);
  if (st != Q4_OK) return st;
  const q4::GemvPlan plan = q4::gemv_plan(n, k, m);
  if (plan.ws_bytes > 0 && (workspace == nullptr || ws_bytes < plan.ws_bytes))
    return Q4_ERR_WORKSPACE;
  if (plan.ws_bytes > 0 && !aligned(workspace, 16)) return Q4_ERR_MISALIGNED;
  return from_cuda(q4::gemv_launch(plan, static_cast<const uint8_t*>(W), n, k, x, m, ldx, y, ldy,
                                   workspace, status_dev, flags, reinterpret_cast<cudaStream_t>(s)));
}

q4_status q4_gemv_prefetch(const void* W, int64_t n, int64_t k, const float* x, int64_t m,
                           int64_t ldx, float* y, int64_t ldy, void* workspace, size_t ws_bytes,
                           int32_t* status_dev, uint32_t flags, const void* prefetch,
                           size_t prefetch_bytes, q4_stream_t s) {
  q4_status st = q4::gemv_check_args(W, n, k, x, m, ldx, y, ldy);
  if (st != Q4_OK) return st;
  if (prefetch_bytes != 0 && prefetch == nullptr) return Q4_ERR_INVALID_ARG;
  if (prefetch_bytes != 0 && (!aligned(prefetch, 16) || prefetch_bytes % 16 != 0))
    return Q4_ERR_MISALIGNED;
  const q4::GemvPlan plan = q4::gemv_plan(n, k, m);
  if (plan.ws_bytes > 0 && (workspace == nullptr || ws_bytes < plan.ws_bytes))
    return Q4_ERR_WORKSPACE;
  if (plan.ws_bytes > 0 && !aligned(workspace, 16)) return Q4_ERR_MISALIGNED;
  return from_cuda(q4::gemv_launch(plan, static_cast<const uint8_t*>(W), n, k, x, m, ldx, y, ldy,
                                   workspace, status_dev, flags, reinterpret_cast<cudaStream_t>(s),
                                   prefetch, prefetch_bytes));
}

size_t q4_gemm_workspace_bytes(int64_t n, int64_t k, int64_t m) {
  if (n <= 0 || k <= 0 || k % 256 || m <= 0) return 0;
  return q4::gemm_plan(n, k, m).ws_bytes;
}

q4_status q4_gemm(const void* W, int64_t n, int64_t k, const void* X, int64_t m, int64_t ldx,
                  void* Y, q4_dtype y_dtype, int64_t ldy, void* workspace, size_t ws_bytes,
                  int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  q4_status st = gemm_check_args(W, n, k, X, m, ldx, Y, y_dtype, ldy);
  if (st != Q4_OK) return st;
  const q4::GemmPlan plan = q4::gemm_plan(n, k, m);
  if (plan.ws_bytes > 0 && (workspace == nullptr || ws_bytes < plan.ws_bytes))
    return Q4_ERR_WORKSPACE;
  if (plan.ws_bytes > 0 && !aligned(workspace, 16)) return Q4_ERR_MISALIGNED;
  cudaError_t e = q4::gemm_launch(plan, static_cast<const uint8_t*>(W), n, k, X, m, ldx, Y,
                                  y_dtype == Q4_BF16, ldy, workspace, status_dev, flags,
                                  reinterpret_cast<cudaStream_t>(s));
  if (e == cudaErrorNotSupported) return Q4_ERR_UNSUPPORTED_SHAPE;
  return from_cuda(e);
}

q4_status q4_embed_gather(const void* table, int64_t vocab, int64_t k, const int32_t* ids,
                          int64_t n_ids, float* out, int32_t* status_dev, q4_stream_t s) {
  q4_status st = check_matrix(table, vocab, k);
  if (st != Q4_OK) return st;
  if (ids == nullptr || out == nullptr || n_ids <= 0 || n_ids > kMaxDim) return Q4_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(out, 16)) return Q4_ERR_MISALIGNED;
  return from_cuda(q4::embed_gather_launch(static_cast<const uint8_t*>(table), vocab, k, ids, n_ids,
                                           out, status_dev, reinterpret_cast<cudaStream_t>(s)));
}

}  // extern "C"

namespace {

// Validates a chain and fills the kernel parameters (except the pointers that
// come from the workspace).  Returns the workspace the chain needs in *ws.
q4_status plan_chain(const q4_gemv_stage* st, int32_t ns, q4::ChainParams* cp, size_t* ws) {
  if (st == nullptr || ns < 1 || ns > Q4_CHAIN_MAX_STAGES || ns > q4::kMaxChain)
    return Q4_ERR_INVALID_ARG;
  const int ctas = q4::sm_count();
  const int64_t kmax = q4::gemv_chain_max_k();
  int64_t max_pn = 0;
  for (int32_t s = 0; s < ns; ++s) {
    const q4_gemv_stage& a = st[s];
    q4_status e = check_matrix(a.W, a.n, a.k);
    if (e != Q4_OK) return e;
    if (a.x == nullptr || a.y == nullptr) return Q4_ERR_INVALID_ARG;
    if (a.k % 256 != 0 || a.k > kmax || a.n % 4 != 0 || a.n > (int64_t(1) << 30))
      return Q4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(a.x, 16) || !aligned(a.y, 4)) return Q4_ERR_MISALIGNED;
    const int64_t groups = (a.n + 31) / 32, nsb = a.k / 256;
    const int p = q4::gemv_chain_split(groups, nsb, ctas);
    if (p == 0) return Q4_ERR_UNSUPPORTED_SHAPE;
    max_pn = std::max<int64_t>(max_pn, p * a.n);
    // Links behave as if run one after another.  x_s overlapping the previous
    // link's y is taken from that link's partial sums (the buffer itself is
    // written while link s starts), so it must lie inside it, on a multiple
    // of 4 floats; any other x is read from memory as it stands then.
    int32_t x_off = -1;
    if (s > 0) {
      const uintptr_t xb = reinterpret_cast<uintptr_t>(a.x), xe = xb + 4 * a.k;
      const uintptr_t yb = reinterpret_cast<uintptr_t>(st[s - 1].y), ye = yb + 4 * st[s - 1].n;
      if (xb < ye && yb < xe) {
        if (xb < yb || xe > ye || (xb - yb) % 16 != 0) return Q4_ERR_INVALID_ARG;
        x_off = static_cast<int32_t>((xb - yb) / 4);
      }
    }
    if (cp != nullptr) {
      q4::ChainStage& c = cp->st[s];
      c.x = a.x;
      c.y = a.y;
      c.n = static_cast<int32_t>(a.n);
      c.nsb = static_cast<int32_t>(nsb);
      c.groups = static_cast<int32_t>(groups);
      c.P = p;
      c.x_off = x_off;
      c.reserved = 0;
      const uint64_t rowbytes = static_cast<uint64_t>(a.k / 32 * Q4_BLOCK_BYTES);
      if (!q4::encode_tmap_2d(&cp->tmap[s], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, rowbytes,
                              static_cast<uint64_t>(a.n), rowbytes, 144, 32,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q4_ERR_CUDA;
    }
  }
  const size_t part = (static_cast<size_t>(max_pn) * 4 + 255) / 256 * 256;
  *ws = 256 + 2 * part;
  if (cp != nullptr) cp->n_stages = ns;
  return Q4_OK;
}

}  // namespace

extern "C" {

size_t q4_gemv_chain_workspace_bytes(const q4_gemv_stage* stages, int32_t n_stages) {
  size_t ws = 0;
  return plan_chain(stages, n_stages, nullptr, &ws) == Q4_OK ? ws : 0;
}

q4_status q4_gemv_chain(const q4_gemv_stage* stages, int32_t n_stages, void* workspace,
                        size_t ws_bytes, int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  static thread_local q4::ChainParams cp;  // ~21 KB: kept off the stack
  size_t need = 0;
  q4_status st = plan_chain(stages, n_stages, &cp, &need);
  if (st != Q4_OK) return st;
  if (workspace == nullptr || ws_bytes < need) return Q4_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return Q4_ERR_MISALIGNED;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t part = (need - 256) / 2;
  cp.done = reinterpret_cast<int32_t*>(w);
  cp.part[0] = reinterpret_cast<float*>(w + 256);
  cp.part[1] = reinterpret_cast<float*>(w + 256 + part);
  cp.status = status_dev;
  cp.flags = flags;
  return from_cuda(q4::gemv_chain_launch(cp, reinterpret_cast<cudaStream_t>(s)));
}

int64_t q4_linear_crossover_m(int64_t n, int64_t k) {
  // The tensor-core path needs k % 256 == 0.
  if (n <= 0 || k <= 0 || k % 256 != 0) return Q4_GEMV_MAX_M;
  // Largest batch still sent to the fp32 GEMV, measured on B300 per decoder
  // and encoder shape (L2-cold weight copies, CUDA graphs): the smallest M in
  // {1..6, 8, 12, 16} at which the bf16 tensor-core GEMM beat the GEMV, less
  // one step.  The GEMV reads the weights once per 4 rows of x, so its time
  // steps up after M = 4, 8, ...; the GEMM's stays ~flat over this range.
  struct Entry {
    int64_t n, k, m;
  };
  static const Entry kTable[] = {
      {4096, 3072, 4}, {1024, 3072, 6}, {3072, 4096, 4}, {9216, 3072, 4}, {3072, 9216, 4},
      {3840, 1280, 8}, {1280, 1280, 6}, {5120, 1280, 8}, {1280, 5120, 6},
  };
  // exact shape, else the entry nearest in weight count (log scale)
  const double size = static_cast<double>(n) * static_cast<double>(k);
  const Entry* best = &kTable[0];
  double best_d = 1e300;
  for (const Entry& e : kTable) {
    if (e.n == n && e.k == k) return e.m;
    const double r = size / (static_cast<double>(e.n) * static_cast<double>(e.k));
    const double d = r > 1.0 ? r : 1.0 / r;
    if (d < best_d) {
      best_d = d;
      best = &e;
    }
  }
  return best->m;
}

size_t q4_linear_workspace_bytes(int64_t n, int64_t k, int64_t m, q4_dtype x_dtype) {
  if (n <= 0 || k <= 0 || k % Q4_BLOCK_ELEMS || m <= 0) return 0;
  if (x_dtype == Q4_F32 && m <= q4_linear_crossover_m(n, k)) return q4_gemv_workspace_bytes(n, k, m);
  size_t bytes = q4_gemm_workspace_bytes(n, k, m);
  if (x_dtype == Q4_F32) bytes = (bytes + 255) / 256 * 256 + static_cast<size_t>(m) * k * 2;
  return bytes;
}

q4_status q4_linear(const void* W, int64_t n, int64_t k, const void* X, q4_dtype x_dtype, int64_t m,
                    int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                    int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  q4_status st = check_matrix(W, n, k);
  if (st != Q4_OK) return st;
  if (X == nullptr || Y == nullptr || m <= 0 || ldx < k || ldy < n) return Q4_ERR_INVALID_ARG;
  if (x_dtype != Q4_F32 && x_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  if (x_dtype == Q4_F32 && m <= q4_linear_crossover_m(n, k))
    return q4_gemv(W, n, k, static_cast<const float*>(X), m, ldx, Y, ldy, workspace, ws_bytes,
                   status_dev, flags, s);
  if (x_dtype == Q4_BF16)
    return q4_gemm(W, n, k, X, m, ldx, Y, Q4_F32, ldy, workspace, ws_bytes, status_dev, flags, s);
  // fp32 activations on the tensor-core path: round them to bf16 into the
  // workspace first.  Every rule q4_gemm will apply to that call is checked
  // here, before the conversion is launched, so that a refused call launches
  // nothing and leaves the workspace as it was.
  if (!aligned(X, 16) || ldx % 4 != 0) return Q4_ERR_MISALIGNED;
  const size_t gemm_ws = (q4_gemm_workspace_bytes(n, k, m) + 255) / 256 * 256;
  void* xb = workspace == nullptr ? nullptr : static_cast<uint8_t*>(workspace) + gemm_ws;
  st = gemm_check_args(W, n, k, X, m, k, Y, Q4_F32, ldy);
  if (st != Q4_OK) return st;
  const size_t need = q4_linear_workspace_bytes(n, k, m, x_dtype);
  if (workspace == nullptr || ws_bytes < need) return Q4_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return Q4_ERR_MISALIGNED;
  cudaError_t e = q4::f32_to_bf16_launch(static_cast<const float*>(X), m, k, ldx, xb, k,
                                         reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return Q4_ERR_CUDA;
  q4_status st2 = q4_gemm(W, n, k, xb, m, k, Y, Q4_F32, ldy, workspace, gemm_ws, status_dev,
                          flags & ~Q4_FLAG_PDL, s);
  if (st2 != Q4_OK) return st2;
  // hand the workspace back all-zero, as every call promises
  return from_cuda(cudaMemsetAsync(xb, 0, static_cast<size_t>(m) * k * 2,
                                   reinterpret_cast<cudaStream_t>(s)));
}

}  // extern "C"
