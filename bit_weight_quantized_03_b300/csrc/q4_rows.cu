// q4_rows.cu -- row-wise Q4_0 kernels: decode rows (dequant), embedding-row
// gather, quantize, and the fp32 -> bf16 activation cast used by q4_linear.
//
// The gather restates "Q4 embeddings on the GPU + row lookup" from the GeekNews
// write-up (es.news.hada.io/topic?id=26595, "Soluciones técnicas"); there the
// lookup runs on the host, here it is a device kernel so a decode step never
// leaves the GPU.
//
// These kernels are bound by HBM writes (12 KB of fp32 out per 1.7 KB of blocks
// in for a 3072-wide row): each CTA stages a row segment of packed blocks in
// shared memory with 16-byte loads, then every thread emits whole 16-byte
// output chunks so consecutive threads write consecutive addresses, with
// streaming (evict-first) stores.
#include "q4_device.cuh"

namespace q4 {
namespace {

constexpr int kRowThreads = 256;
constexpr int kSegBlocks = 256;  // blocks per staged segment (4608 B)

// Decodes output rows of a Q4_0 matrix.  Output row r reads source row
// ids ? ids[r] : row0 + r.  OUT_BF16 selects the output type.
template <bool OUT_BF16>
__global__ void __launch_bounds__(kRowThreads) rows_decode_kernel(
    const uint8_t* __restrict__ blocks, int64_t row0, const int32_t* __restrict__ ids,
    int64_t vocab, int64_t n_out, int64_t nb, void* __restrict__ out, int32_t* status) {
  __shared__ __align__(16) uint8_t seg[kSegBlocks * kBlockBytes];
  const int64_t rowbytes = nb * kBlockBytes;
  const int64_t k = nb * kBlockElems;
  for (int64_t r = blockIdx.x; r < n_out; r += gridDim.x) {
    int64_t src;
    bool valid = true;
    if (ids != nullptr) {
      src = ids[r];
      if (src < 0 || src >= vocab) valid = false;
    } else {
      src = row0 + r;
    }
    if (!valid) {
      if (threadIdx.x == 0) report(status, 5 /* Q4_ERR_ID_OUT_OF_RANGE */);
      if constexpr (OUT_BF16) {
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + r * k);
        for (int64_t c = threadIdx.x; c < k / 8; c += blockDim.x) o[c] = make_uint4(0, 0, 0, 0);
      } else {
        float* o = static_cast<float*>(out) + r * k;
        for (int64_t c = threadIdx.x; c < k / 4; c += blockDim.x)
          stg_cs_f4(o + 4 * c, make_float4(0.f, 0.f, 0.f, 0.f));
      }
      continue;
    }
    const uint8_t* row = blocks + src * rowbytes;
    for (int64_t b0 = 0; b0 < nb; b0 += kSegBlocks) {
      const int sb = static_cast<int>(nb - b0 < kSegBlocks ? nb - b0 : kSegBlocks);
      const uint8_t* g = row + b0 * kBlockBytes;
      const int bytes = sb * kBlockBytes;
      __syncthreads();  // previous segment fully consumed
      if ((reinterpret_cast<uintptr_t>(g) & 15) == 0 && (bytes & 15) == 0) {
        for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x)
          reinterpret_cast<uint4*>(seg)[i] = __ldcs(reinterpret_cast<const uint4*>(g) + i);
      } else {  // rows are always 2-byte aligned
        for (int i = threadIdx.x; i < bytes / 2; i += blockDim.x)
          reinterpret_cast<uint16_t*>(seg)[i] = reinterpret_cast<const uint16_t*>(g)[i];
      }
      __syncthreads();
      if constexpr (OUT_BF16) {
        // 8 outputs per thread: chunk c covers weights 8*(c%4) .. +7 of block c/4.
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + r * k + b0 * kBlockElems;
        for (int c = threadIdx.x; c < sb * 4; c += blockDim.x) {
          const uint8_t* blk = seg + (c >> 2) * kBlockBytes;
          const int e0 = (c & 3) * 8;
          const float d = half_bits_to_float(blk[0] | (blk[1] << 8));
          const int shift = e0 < 16 ? 0 : 4;
          const uint8_t* qs = blk + 2 + (e0 & 15);
          __align__(16) __nv_bfloat162 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float w0 = static_cast<float>(static_cast<int>((qs[2 * i] >> shift) & 15) - 8) * d;
            const float w1 =
                static_cast<float>(static_cast<int>((qs[2 * i + 1] >> shift) & 15) - 8) * d;
            v[i] = __floats2bfloat162_rn(w0, w1);
          }
          reinterpret_cast<uint4*>(o)[c] = *reinterpret_cast<uint4*>(v);
        }
      } else {
        // 4 outputs per thread: chunk c covers weights 4*(c%8) .. +3 of block c/8.
        float* o = static_cast<float*>(out) + r * k + b0 * kBlockElems;
        for (int c = threadIdx.x; c < sb * 8; c += blockDim.x) {
          const uint8_t* blk = seg + (c >> 3) * kBlockBytes;
          const int e0 = (c & 7) * 4;
          const float d = half_bits_to_float(blk[0] | (blk[1] << 8));
          const int shift = e0 < 16 ? 0 : 4;
          const uint8_t* qs = blk + 2 + (e0 & 15);
          float4 v;
          v.x = static_cast<float>(static_cast<int>((qs[0] >> shift) & 15) - 8) * d;
          v.y = static_cast<float>(static_cast<int>((qs[1] >> shift) & 15) - 8) * d;
          v.z = static_cast<float>(static_cast<int>((qs[2] >> shift) & 15) - 8) * d;
          v.w = static_cast<float>(static_cast<int>((qs[3] >> shift) & 15) - 8) * d;
          stg_cs_f4(o + 4 * c, v);
        }
      }
    }
  }
}

// One thread per block of 32 weights.  Bit-exact restatement of the quantizer
// reading (see include/q4.h): IEEE fp32 division and add (no contraction),
// binary16 round-to-nearest-even for the scale.
__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ w,
                                                       int64_t total_blocks,
                                                       uint8_t* __restrict__ blocks,
                                                       int32_t* status) {
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total_blocks;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float x[32];
    const float4* src = reinterpret_cast<const float4*>(w + g * kBlockElems);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = __ldcs(src + i);
      x[4 * i + 0] = v.x;
      x[4 * i + 1] = v.y;
      x[4 * i + 2] = v.z;
      x[4 * i + 3] = v.w;
    }
    bool bad = false;
    int im = 0;
    float amax = fabsf(x[0]);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (!isfinite(x[i])) bad = true;
      if (i > 0 && fabsf(x[i]) > amax) {
        amax = fabsf(x[i]);
        im = i;
      }
    }
    float m = x[0];
#pragma unroll
    for (int i = 1; i < 32; ++i)
      if (i == im) m = x[i];
    uint32_t dbits = 0;
    if (!bad && amax != 0.0f) {
      const float d32 = __fdiv_rn(m, -8.0f);
      dbits = __half_as_ushort(__float2half_rn(d32));
      if ((dbits & 0x7C00u) == 0x7C00u) bad = true;
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(blocks + g * kBlockBytes);
    if (bad) {
      report(status, 4 /* Q4_ERR_NONFINITE */);
      dst[0] = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[1 + j] = 0x8888;
      continue;
    }
    const float dd = half_bits_to_float(dbits);
    uint32_t q[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (dd == 0.0f) {
        q[i] = 8;
      } else {
        const float t = __fdiv_rn(x[i], dd);
        const float u = __fadd_rn(t, 8.5f);
        float fq = floorf(u);
        fq = fminf(fmaxf(fq, 0.0f), 15.0f);
        q[i] = static_cast<uint32_t>(fq);
      }
    }
    dst[0] = static_cast<uint16_t>(dbits);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b0 = q[2 * j] | (q[2 * j + 16] << 4);
      const uint32_t b1 = q[2 * j + 1] | (q[2 * j + 17] << 4);
      dst[1 + j] = static_cast<uint16_t>(b0 | (b1 << 8));
    }
  }
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ x, int64_t m,
                                                          int64_t k, int64_t ldx,
                                                          __nv_bfloat16* __restrict__ o,
                                                          int64_t ldo) {
  const int64_t per_row = k / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < m * per_row;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, c = (i % per_row) * 4;
    const float4 v = *reinterpret_cast<const float4*>(x + r * ldx + c);
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&a);
    packed.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(o + r * ldo + c) = packed;
  }
}

int grid_for(int64_t work, int per_sm) {
  const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  return static_cast<int>(work < cap ? (work > 0 ? work : 1) : cap);
}

}  // namespace

cudaError_t dequant_rows_launch(const uint8_t* blocks, int64_t row0, int64_t n_rows, int64_t k,
                                void* out, bool out_bf16, cudaStream_t s) {
  const int grid = grid_for(n_rows, 8);
  if (out_bf16)
    rows_decode_kernel<true><<<grid, kRowThreads, 0, s>>>(blocks, row0, nullptr, 0, n_rows, k / 32,
                                                          out, nullptr);
  else
    rows_decode_kernel<false><<<grid, kRowThreads, 0, s>>>(blocks, row0, nullptr, 0, n_rows,
                                                           k / 32, out, nullptr);
  return cudaGetLastError();
}

cudaError_t embed_gather_launch(const uint8_t* table, int64_t vocab, int64_t k, const int32_t* ids,
                                int64_t n_ids, float* out, int32_t* status, cudaStream_t s) {
  const int grid = grid_for(n_ids, 8);
  rows_decode_kernel<false><<<grid, kRowThreads, 0, s>>>(table, 0, ids, vocab, n_ids, k / 32, out,
                                                         status);
  return cudaGetLastError();
}

cudaError_t quantize_launch(const float* w, int64_t n, int64_t k, uint8_t* blocks,
                            int32_t* status, cudaStream_t s) {
  const int64_t total = n * (k / 32);
  const int grid = grid_for((total + 255) / 256, 16);
  quantize_kernel<<<grid, 256, 0, s>>>(w, total, blocks, status);
  return cudaGetLastError();
}

cudaError_t f32_to_bf16_launch(const float* x, int64_t m, int64_t k, int64_t ldx, void* out,
                               int64_t ldo, cudaStream_t s) {
  const int grid = grid_for((m * k / 4 + 255) / 256, 8);
  f32_to_bf16_kernel<<<grid, 256, 0, s>>>(x, m, k, ldx, static_cast<__nv_bfloat16*>(out), ldo);
  return cudaGetLastError();
}

}  // namespace q4
