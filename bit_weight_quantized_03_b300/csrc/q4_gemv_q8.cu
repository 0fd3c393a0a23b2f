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
// a warp max and a warp sum of the codes), then its warps take rows.  A lane
// takes blocks lane, lane + 32, ... of a row: it reads the 18-byte block as
// nine 2-byte words (the block is 2-byte aligned; a warp's reads are 576
// contiguous bytes), splits the 16 code bytes into the low nibbles (elements
// 0..15) and the high nibbles (16..31) with one AND and one shift-AND per
// word, and feeds them to DP4A against the int8 codes of x.  With the codes
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
  int32_t n, k;
};

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

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

  // ---- rows: warp w of CTA c takes rows w + W c, + W C, ...; a lane reads
  // kQ8Unroll blocks of its row before it uses any, so that enough bytes are
  // in flight per SM
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kQ8Warps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQ8Warps;
  for (int64_t r = gw; r < a.n; r += nwarps) {
    const uint8_t* row = a.W + r * nb * static_cast<int64_t>(kBlockBytes);
    float acc = 0.f;
    for (int b0 = lane; b0 < nb; b0 += 32 * kQ8Unroll) {
      uint32_t h[kQ8Unroll][9];
#pragma unroll
      for (int u = 0; u < kQ8Unroll; ++u) {
        const int b = b0 + 32 * u;
        if (b < nb) {
          const uint8_t* blk = row + static_cast<int64_t>(b) * kBlockBytes;
#pragma unroll
          for (int i = 0; i < 9; ++i) h[u][i] = ldg_u16(blk + 2 * i);
        }
      }
#pragma unroll
      for (int u = 0; u < kQ8Unroll; ++u) {
        const int b = b0 + 32 * u;
        if (b >= nb) break;
        const int4 xlo = *reinterpret_cast<const int4*>(qx + 32 * b);       // elements 0..15
        const int4 xhi = *reinterpret_cast<const int4*>(qx + 32 * b + 16);  // elements 16..31
        const int xl[4] = {xlo.x, xlo.y, xlo.z, xlo.w};
        const int xh[4] = {xhi.x, xhi.y, xhi.z, xhi.w};
        int isum = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w = h[u][1 + 2 * i] | (h[u][2 + 2 * i] << 16);  // code bytes 4i..4i+3
          isum = __dp4a(static_cast<int>(w & 0x0F0F0F0Fu), xl[i], isum);
          isum = __dp4a(static_cast<int>((w >> 4) & 0x0F0F0F0Fu), xh[i], isum);
        }
        isum -= 8 * sx[b];
        const float dw = half_bits_to_float(h[u][0]);
        acc = fmaf(dw * dx[b], static_cast<float>(isum), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.y[r] = acc;
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
  q4::Q8Args a{static_cast<const uint8_t*>(W), x, y, static_cast<int32_t>(n),
               static_cast<int32_t>(k)};
  const int64_t rows_per_cta = q4::kQ8Warps;
  int64_t ctas = (n + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = static_cast<int64_t>(q4::sm_count()) * q4::kQ8CtasPerSm;
  if (ctas > cap) ctas = cap;
  q4::gemv_q8_kernel<<<static_cast<unsigned>(ctas), q4::kQ8Threads, 0,
                       reinterpret_cast<cudaStream_t>(s)>>>(a);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}
