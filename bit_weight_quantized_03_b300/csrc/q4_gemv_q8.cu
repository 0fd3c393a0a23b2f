// q4_gemv_q8.cu -- the Q4 x Q8 integer path of the batch-1 product.
//
// GGUF Q4_0 (GeekNews, es.news.hada.io/topic?id=26595, "Arquitectura") is
// usually paired with an integer dot product: the activation is quantized per
// 32-element block to int8 with one scale, and each block contributes
//   d_w * d_x * sum_j (q_w,j - 8) * q_x,j
// with the inner sum in exact integer arithmetic.  The pages give no detail;
// this library's reading: amax = max |x_j| per block, d_x = amax / 127 (fp32,
// IEEE division), q_x,j = x_j / d_x (IEEE division) rounded to the nearest
// integer with halves away from zero; amax == 0 gives d_x = +0 and codes 0; a
// block with a NaN or an infinity gives d_x = NaN and codes 0.
//
// Kernel: every CTA first quantizes x into shared memory (one warp per block:
// a warp max and a warp sum of the codes), then its warps take rows.  When a
// row is a whole number of 16-byte words (k % 256 == 0) a warp brings its
// next row into shared memory with one bulk copy while it works on the
// current one; otherwise it reads the row from global memory directly.  A
// lane takes blocks lane, lane + 32, ... of a row: it reads the 18-byte block
// as nine 2-byte words (the block is 2-byte aligned), splits the 16 code bytes
// into the low nibbles (elements 0..15) and the high nibbles (16..31) with
// one AND and one shift-AND per word, and feeds them to DP4A against the int8
// codes of x.  With the codes
// taken unsigned (0..15), the -8 offset is one multiply by the block's code
// sum of x.  The block term is added in fp32 as (d_w * d_x) * isum; a warp
// adds its lanes' row sums in a fixed order, so results do not depend on
// timing.
#include <cuda_runtime.h>

#include "../../include/q4.h"
#include "q4_device.cuh"

namespace q4 {
namespace {

constexpr int kQ8Warps = 8;
constexpr int kQ8Threads = kQ8Warps * 32;
constexpr int kQ8MaxK = 12288;
constexpr int kQ8CtasPerSm = 3;
constexpr int kQ8Unroll = 4;       // blocks per lane in flight

struct Q8Args {
  const uint8_t* W;
  const float* x;
  float* y;
  int32_t* status;
  int32_t n, k;
};

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(const uint8_t* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}

// The block term of block b (nine 2-byte words h[]) against the staged x.
__device__ __forceinline__ float q8_block(const uint32_t (&h)[9], const int8_t* qx, const float* dx,
                                          const int* sx, int b) {
  const int4 xlo = *reinterpret_cast<const int4*>(qx + 32 * b);       // elements 0..15
  const int4 xhi = *reinterpret_cast<const int4*>(qx + 32 * b + 16);  // elements 16..31
  const int xl[4] = {xlo.x, xlo.y, xlo.z, xlo.w};
  const int xh[4] = {xhi.x, xhi.y, xhi.z, xhi.w};
  int isum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = h[1 + 2 * i] | (h[2 + 2 * i] << 16);  // code bytes 4i..4i+3
    isum = __dp4a(static_cast<int>(w & 0x0F0F0F0Fu), xl[i], isum);
    isum = __dp4a(static_cast<int>((w >> 4) & 0x0F0F0F0Fu), xh[i], isum);
  }
  isum -= 8 * sx[b];
  return half_bits_to_float(h[0]) * dx[b] * static_cast<float>(isum);
}

template <bool kBulk, int S>
__global__ void __launch_bounds__(kQ8Threads, kQ8CtasPerSm) gemv_q8_kernel(const Q8Args a) {
  __shared__ __align__(16) int8_t qx[kQ8MaxK];
  __shared__ float dx[kQ8MaxK / 32];
  __shared__ int sx[kQ8MaxK / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = a.k / 32;

  // ---- x -> int8 codes, per-block scale and code sum (one warp per block;
  // a warp loads four blocks of x before it reduces any)
  for (int b0 = warp; b0 < nb; b0 += 4 * kQ8Warps) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + u * kQ8Warps;
      v[u] = b < nb ? a.x[32 * b + lane] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = b0 + u * kQ8Warps;
      if (b >= nb) break;
      const bool finite = __all_sync(0xffffffffu, isfinite(v[u]));
      float amax = fabsf(v[u]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      float d = amax / 127.0f;
      int c = 0;
      if (!finite) {
        d = __uint_as_float(0x7FC00000u);
      } else if (d != 0.0f) {
        float t = roundf(v[u] / d);  // halves away from zero
        t = fminf(fmaxf(t, -127.0f), 127.0f);
        c = static_cast<int>(t);
      }
      int sc = c;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
      qx[32 * b + lane] = static_cast<int8_t>(c);
      if (lane == 0) {
        dx[b] = d;
        sx[b] = sc;
      }
    }
  }
  __syncthreads();

  // ---- rows: warp w of CTA c takes rows w + W c, + W C, ...
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kQ8Warps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQ8Warps;
  const int64_t row_bytes = static_cast<int64_t>(nb) * kBlockBytes;
  if constexpr (kBulk) {
    // S row buffers per warp, each filled by one bulk copy
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ __align__(8) uint64_t rbar[kQ8Warps][S];
    uint8_t* const buf0 = rows_smem + static_cast<size_t>(warp) * S * row_bytes;
    const uint32_t bar0 = smem_u32(&rbar[warp][0]);
    if (lane == 0)
      for (int j = 0; j < S; ++j) mbar_init(bar0 + 8 * j, 1);
    fence_mbarrier_init();
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t r, int slot) {
      if (lane == 0 && r < a.n) {
        mbar_arrive_expect_tx(bar0 + 8 * slot, static_cast<uint32_t>(row_bytes));
        bulk_g2s(smem_u32(buf0 + slot * row_bytes), a.W + r * row_bytes,
                 static_cast<uint32_t>(row_bytes), bar0 + 8 * slot, pol);
      }
    };
    for (int j = 0; j < S; ++j) issue(gw + j * nwarps, j);
    int i = 0;
    bool ok = true;
    for (int64_t r = gw; r < a.n; r += nwarps, ++i) {
      const int slot = i % S;
      const bool landed = mbar_wait(bar0 + 8 * slot, (i / S) & 1);
      if (!__all_sync(0xffffffffu, landed)) {
        ok = false;
        break;
      }
      const uint8_t* row = buf0 + slot * row_bytes;
      float acc = 0.f;
      for (int b = lane; b < nb; b += 32) {
        const uint8_t* blk = row + b * kBlockBytes;
        uint32_t h[9];
#pragma unroll
        for (int j = 0; j < 9; ++j) h[j] = lds_u16(blk + 2 * j);
        acc += q8_block(h, qx, dx, sx, b);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) a.y[r] = acc;
      __syncwarp();
      fence_proxy_async_smem();  // this slot's reads come before the copy that reuses it
      issue(r + S * nwarps, slot);
    }
    if (!ok && lane == 0) report(a.status, 6 /* Q4_ERR_TIMEOUT */);
    // copies still in flight land before the warp exits
    const int i_end = i + S;
    for (int64_t r = gw + static_cast<int64_t>(i) * nwarps; r < a.n && i < i_end;
         r += nwarps, ++i)
      mbar_wait(bar0 + 8 * (i % S), (i / S) & 1);
  } else {
    // a lane reads kQ8Unroll blocks of its row from global memory before it
    // uses any, so that enough bytes are in flight per SM
    for (int64_t r = gw; r < a.n; r += nwarps) {
      const uint8_t* row = a.W + r * row_bytes;
      float acc = 0.f;
      for (int b0 = lane; b0 < nb; b0 += 32 * kQ8Unroll) {
        uint32_t h[kQ8Unroll][9];
#pragma unroll
        for (int u = 0; u < kQ8Unroll; ++u) {
          const int b = b0 + 32 * u;
          if (b < nb) {
            const uint8_t* blk = row + static_cast<int64_t>(b) * kBlockBytes;
#pragma unroll
            for (int j = 0; j < 9; ++j) h[u][j] = ldg_u16(blk + 2 * j);
          }
        }
#pragma unroll
        for (int u = 0; u < kQ8Unroll; ++u) {
          const int b = b0 + 32 * u;
          if (b >= nb) break;
          acc += q8_block(h[u], qx, dx, sx, b);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) a.y[r] = acc;
    }
  }
}

}  // namespace
}  // namespace q4

extern "C" q4_status q4_gemv_q8(const void* W, int64_t n, int64_t k, const float* x, float* y,
                                q4_stream_t s) {
  if (W == nullptr || x == nullptr || y == nullptr || n <= 0 || k <= 0 ||
      n > (int64_t(1) << 31) - 1)
    return Q4_ERR_INVALID_ARG;
  if (k % 32 != 0 || k > q4::kQ8MaxK) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || reinterpret_cast<uintptr_t>(x) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(y) % 4 != 0)
    return Q4_ERR_MISALIGNED;
  q4::Q8Args a{static_cast<const uint8_t*>(W), x, y, nullptr, static_cast<int32_t>(n),
               static_cast<int32_t>(k)};
  const int64_t rows_per_cta = q4::kQ8Warps;
  int64_t ctas = (n + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = static_cast<int64_t>(q4::sm_count()) * q4::kQ8CtasPerSm;
  if (ctas > cap) ctas = cap;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  if (k % 256 == 0) {
    // whole 16-byte rows in dynamic shared memory: four row buffers per warp
    // while three CTAs still fit an SM (k <= 3072), else two
    const size_t row_bytes = static_cast<size_t>(k / 32) * q4::kBlockBytes;
    const bool four = k <= 3072;
    const size_t smem = static_cast<size_t>(q4::kQ8Warps) * (four ? 4 : 2) * row_bytes;
    static bool configured[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
    if (!configured[dev]) {
      const size_t most2 = static_cast<size_t>(q4::kQ8Warps) * 2 * (q4::kQ8MaxK / 32) *
                           q4::kBlockBytes;
      const size_t most4 = static_cast<size_t>(q4::kQ8Warps) * 4 * (3072 / 32) * q4::kBlockBytes;
      if (cudaFuncSetAttribute(q4::gemv_q8_kernel<true, 2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(most2)) != cudaSuccess ||
          cudaFuncSetAttribute(q4::gemv_q8_kernel<true, 4>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(most4)) != cudaSuccess)
        return Q4_ERR_CUDA;
      configured[dev] = true;
    }
    if (four)
      q4::gemv_q8_kernel<true, 4><<<static_cast<unsigned>(ctas), q4::kQ8Threads, smem, cs>>>(a);
    else
      q4::gemv_q8_kernel<true, 2><<<static_cast<unsigned>(ctas), q4::kQ8Threads, smem, cs>>>(a);
  } else {
    q4::gemv_q8_kernel<false, 1><<<static_cast<unsigned>(ctas), q4::kQ8Threads, 0, cs>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}
