// q4r_tile.cuh -- the repacked Q4_0 tile and its batch-1 tensor-core dot product.
//
// GGUF Q4_0 (the weight format of the quantized path in the GeekNews write-up
// es.news.hada.io/topic?id=26595, "Arquitectura") stores 18-byte blocks: a
// binary16 scale d and 16 bytes of 4-bit codes, w = (q - 8) * d.  Streaming
// those blocks row by row leaves every block at an odd 2-byte offset and the
// codes in an order no arithmetic unit wants.  The repacked layout keeps every
// byte of the blocks but moves them into the operand order of the tensor
// cores' 16 x 16 (f16) A fragment:
//
//   * rows are taken in groups of 16 and k in slices of 256 (8 blocks); the
//     16 x 256 tile (G, t) is 2304 contiguous bytes at (G * k/256 + t) * 2304,
//     so a run of tiles is one contiguous byte range;
//   * scales (bytes 0..255): the 32-bit word at 32g + 4b holds the binary16 d
//     of block b of row g (low half) and of row g + 8 (high half);
//   * codes (bytes 256..2303): the tile's columns form 16 steps of 16; lane
//     L = 4g + t of step s owns the 32-bit word at 256 + 512 (s/4) + 16L +
//     4 (s%4).  Its nibble m holds row g + 8 (m & 1) at column
//     16s + 2t + 8 ((m >> 1) & 1) + (m >> 2), so a lane's four words for steps
//     4j..4j+3 are one 16-byte load, and a warp's loads are 512 consecutive
//     bytes;
//   * rows past n in the last group are padding with d = +0 and codes 8.
//
// Decode: with the word w, (w & 0x000F000F) | 0x64006400 is the binary16 pair
// (1024 + q_a, 1024 + q_b) for the nibbles at bits 0 and 16, and
// (w & 0x00F000F0) | 0x64006400 is (1024 + 16 q_c, 1024 + 16 q_d) for those at
// bits 4 and 20; one packed f16 subtract (- 1032), resp. one packed f16 FMA
// (x 1/16, - 72), turns them into (q - 8) exactly.  The same on w >> 8 gives
// the other four nibbles.  These four registers are exactly the A fragment of
// mma.m16n8k16 (rows g and g + 8, columns 2t, 2t+1 and 2t+8, 2t+9).
//
// B: the activation x enters the tensor core as binary16, so it is carried as
// an exact-to-2^-22 pair hi + lo in columns 0 and 1 of B (columns 2..7 repeat
// them and are not read), after scaling each 256-element slice of x by a power of two that puts
// its largest magnitude in [2^14, 2^15): rows g / g+8 of the result then sit in
// the lanes t = 0 as D columns 0 (hi part) and 1 (lo part).  Per block the
// fp32 fragment sums are multiplied by d, per tile by the slice's inverse
// scale.
#pragma once

#include "q4_device.cuh"

namespace q4 {
namespace rt {

constexpr int kRows = 16;            // rows per tile
constexpr int kCols = 256;           // columns (8 blocks) per tile
constexpr int kTileBytes = 2304;     // 16 rows x 8 blocks x 18 bytes
constexpr int kScaleBytes = 256;     // 8 row pairs x 8 blocks x 2 binary16
constexpr int kStepBytes = 512;      // code bytes of four steps (32 lanes x 16)
constexpr int kXStepBytes = 64;      // staged x of one 16-column step

// Staged x: per step s, 64 bytes: for column n = 0 (hi) / 1 (lo) and lane
// quad t, two words {x[16s+2t], x[16s+2t+1]} and {x[16s+2t+8], x[16s+2t+9]}
// (binary16 pairs, lower column in the low half) at s*64 + (4n + t)*8.  So the
// eight lanes 0..7 of a warp fetch their B fragment of a step with one 8-byte
// load each at s*64 + lane*8.
__host__ __device__ constexpr int64_t x16_bytes(int64_t k) { return k / 16 * kXStepBytes; }
// Byte offset of the word holding column pair (i, i+1) (i even) of step s in
// column n.
__device__ __forceinline__ int x16_word(int s, int n, int i) {
  return s * kXStepBytes + (4 * n + ((i & 7) >> 1)) * 8 + ((i >> 3) << 2);
}

// Power-of-two scale for a slice whose largest magnitude is amax: s puts amax
// in [2^14, 2^15) (clamped to 2^-126 .. 2^126); returns s and 1/s, both exact.
__device__ __forceinline__ void slice_scale(float amax, float& s, float& inv) {
  const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
  int se = 268 - ef;  // biased exponent of 2^(14 - (ef - 127))
  se = amax == 0.f ? 127 : (se < 1 ? 1 : (se > 253 ? 253 : se));
  s = __uint_as_float(static_cast<uint32_t>(se) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(254 - se) << 23);
}

// hi + lo of v (already scaled): hi = f16(v), lo = f16(v - hi).
__device__ __forceinline__ void split_hi_lo(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

__device__ __forceinline__ uint32_t lop3_magic(uint32_t w, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(0x64006400u));
  return r;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ __half2 bits_h2(uint32_t u) {
  return *reinterpret_cast<__half2*>(&u);
}

// D (+)= A B for one m16n8k16 step, f16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The A fragment (q - 8 as f16) of one step word.
__device__ __forceinline__ void decode_step(uint32_t w, uint32_t (&a)[4]) {
  const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));   // 1032
  const __half2 k16 = __half2half2(__ushort_as_half(0x2C00));     // 1/16
  const __half2 km72 = __half2half2(__ushort_as_half(0xD480));    // -72
  const uint32_t t = w >> 8;
  a[0] = h2_bits(__hsub2(bits_h2(lop3_magic(w, 0x000F000Fu)), k1032));
  a[1] = h2_bits(__hfma2(bits_h2(lop3_magic(w, 0x00F000F0u)), k16, km72));
  a[2] = h2_bits(__hsub2(bits_h2(lop3_magic(t, 0x000F000Fu)), k1032));
  a[3] = h2_bits(__hfma2(bits_h2(lop3_magic(t, 0x00F000F0u)), k16, km72));
}

// One tile for this warp: y[0] += row g's and y[1] += row g+8's dot product
// with the tile's 256 columns of x (meaningful in lanes with lane % 4 == 0;
// the other lanes accumulate copies of other columns).  tile: the landed tile; xs: the staged x
// of the tile's slice (16 steps); xinv: the slice's inverse scale.
__device__ __forceinline__ void tile_dot(const uint8_t* tile, const uint8_t* xs, float xinv,
                                         int lane, float (&y)[2]) {
  const int g = lane >> 2;
  const uint4 sa = *reinterpret_cast<const uint4*>(tile + 32 * g);
  const uint4 sb = *reinterpret_cast<const uint4*>(tile + 32 * g + 16);
  const uint32_t sw[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
  float yt[2] = {0.f, 0.f};
  const uint8_t* codes = tile + kScaleBytes + 16 * lane;
  // lane 4n + t (n = 0, 1) carries B column n; lanes 8.. read the same words
  const uint8_t* xb = xs + 8 * (lane & 7);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 w4 = *reinterpret_cast<const uint4*>(codes + kStepBytes * j);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // block 2j + h = steps 4j + 2h, 4j + 2h + 1
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int s = 4 * j + 2 * h + u;
        const uint2 b = *reinterpret_cast<const uint2*>(xb + s * kXStepBytes);
        uint32_t a[4];
        decode_step(w[2 * h + u], a);
        mma_f16(d, a, b.x, b.y);
      }
      const int blk = 2 * j + h;
      yt[0] = fmaf(d[0] + d[1], half_bits_to_float(sw[blk]), yt[0]);
      yt[1] = fmaf(d[2] + d[3], half_bits_to_float(sw[blk] >> 16), yt[1]);
    }
  }
  y[0] = fmaf(yt[0], xinv, y[0]);
  y[1] = fmaf(yt[1], xinv, y[1]);
}

}  // namespace rt
}  // namespace q4
