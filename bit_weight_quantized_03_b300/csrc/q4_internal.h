// q4_internal.h -- declarations shared between the C-ABI host code (q4_api.cu)
// and the kernel files.  Not part of the public interface (that is include/q4.h).
#pragma once

#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/q4.h"

namespace q4 {

// Wall-clock limit of every bounded wait inside a kernel (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// Internal flag: tests make one bounded wait run out on purpose (see
// gemv_launch); never set by the public API.
constexpr uint32_t kFlagTestStallOneWait = 1u << 30;

// --------------------------------------------------------------- elementwise
cudaError_t dequant_rows_launch(const uint8_t* blocks, int64_t row0, int64_t n_rows, int64_t k,
                                void* out, bool out_bf16, cudaStream_t s);
cudaError_t embed_gather_launch(const uint8_t* table, int64_t vocab, int64_t k, const int32_t* ids,
                                int64_t n_ids, float* out, int32_t* status, cudaStream_t s);
cudaError_t quantize_launch(const float* w, int64_t n, int64_t k, uint8_t* blocks,
                            int32_t* status, cudaStream_t s);
cudaError_t f32_to_bf16_launch(const float* x, int64_t m, int64_t k, int64_t ldx, void* out,
                               int64_t ldo, cudaStream_t s);

// --------------------------------------------------------------- GEMV
// The host-side argument rules of q4_gemv (matrix, x, y, m, leading
// dimensions, alignment); Q4_OK or the status q4_gemv would return.
q4_status gemv_check_args(const void* W, int64_t n, int64_t k, const float* x, int64_t m,
                          int64_t ldx, const float* y, int64_t ldy);

struct GemvPlan {
  bool fast;          // streamed kernel (k % 256 == 0) vs the generic one
  bool b1;            // batch-1 streamed kernel (q4_gemv_b1.cu)
  bool bm;            // 2..16 rows of x through the batched tile kernel, <= 4 per launch
  int64_t units;      // (32-row group, 256-wide k slice) pairs
  int64_t warps;      // workers the units are split over
  int64_t groups;     // 32-row groups
  size_t ws_bytes;    // workspace the plan needs
};
GemvPlan gemv_plan(int64_t n, int64_t k, int64_t m);
// pf, pf_bytes: a region (16-byte aligned, a multiple of 16 bytes) to prefetch
// into L2 while the product runs; taken by the batch-1 path, ignored elsewhere.
cudaError_t gemv_launch(const GemvPlan& plan, const uint8_t* W, int64_t n, int64_t k,
                        const float* x, int64_t m, int64_t ldx, float* y, int64_t ldy,
                        void* workspace, int32_t* status, uint32_t flags, cudaStream_t s,
                        const void* pf = nullptr, uint64_t pf_bytes = 0);

// Rows of x one batched tile launch carries (q4_gemv_b1.cu).
constexpr int64_t kMaxBatchRows = 4;

int64_t gemv_b1_warps(int64_t units);
int64_t gemv_bm_warps(int64_t units);
bool gemv_bm_supports(int64_t k, int64_t mb);
cudaError_t gemv_bm_launch(const uint8_t* W, int64_t n, int64_t k, const float* x, int64_t mb,
                           int64_t ldx, float* y, int64_t ldy, int32_t* counters,
                           float* partials, int64_t units, int32_t* status, uint32_t flags,
                           cudaStream_t s);
bool gemv_b1_supports(int64_t k);
cudaError_t gemv_b1_launch(const uint8_t* W, int64_t n, int64_t k, const float* x, float* y,
                           int32_t* counters, float* partials, int64_t units, int64_t warps,
                           int32_t* status, uint32_t flags, cudaStream_t s,
                           const void* pf = nullptr, uint64_t pf_bytes = 0);

// --------------------------------------------------------------- GEMV chain
constexpr int kMaxChain = 128;      // links per launch
constexpr int kMaxChainItems = 8;   // (row group, K-split) items per CTA per link

struct ChainStage {
  const float* x;       // external input (x_off < 0)
  float* y;             // output, written once the next link starts
  int32_t n, nsb;       // rows, 256-wide slices of k
  int32_t groups, P;    // 32-row groups, K-splits
  int32_t x_off;        // >= 0: x = y of the previous link from this element
  int32_t reserved;
};

struct ChainParams {
  CUtensorMap tmap[kMaxChain];  // per link: the packed matrix, box 144 B x 32 rows
  ChainStage st[kMaxChain];
  int32_t n_stages;
  int32_t* done;                // barrier counter (workspace, zero between launches)
  float* part[2];               // per-link partial sums [P][n], alternating buffers
  int32_t* status;
  uint32_t flags;
};

int64_t gemv_chain_max_k();
int gemv_chain_split(int64_t groups, int64_t nsb, int ctas);  // 0: too many rows
cudaError_t gemv_chain_launch(ChainParams& params, cudaStream_t s);

// --------------------------------------------------------------- GEMM (tcgen05)
struct GemmPlan {
  int64_t n_tiles, m_tiles, splits;
  int block_n;        // tokens per tile (MMA N)
  size_t ws_bytes;
};
GemmPlan gemm_plan(int64_t n, int64_t k, int64_t m);
cudaError_t gemm_launch(const GemmPlan& plan, const uint8_t* W, int64_t n, int64_t k,
                        const void* X, int64_t m, int64_t ldx, void* Y, bool y_bf16,
                        int64_t ldy, void* workspace, int32_t* status, uint32_t flags,
                        cudaStream_t s);

int sm_count();

// 2-D TMA tensor map (cached by address/sizes/strides/box).  false on failure.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                    uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle);

}  // namespace q4
