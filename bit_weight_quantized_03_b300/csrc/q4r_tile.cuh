// q4r_tile.cuh -- the repacked Q4_0 tile and its batch-1 dot product.
//
// GGUF Q4_0 (the weight format of the quantized path in the GeekNews write-up
// es.news.hada.io/topic?id=26595, "Arquitectura") stores 18-byte blocks: a
// binary16 scale d and 16 bytes of 4-bit codes, w = (q - 8) * d.  Streaming
// those blocks row by row leaves every block at an odd 2-byte offset, so a
// GPU reads them in 4-byte pieces and re-aligns them in registers.  The
// repacked layout below keeps every byte of the blocks but moves them so that
// each lane of a warp finds its data in whole 16-byte and 8-byte words:
//
//   * rows are taken in groups of 16 and k in slices of 256 (8 blocks); the
//     16 x 256 tile (group g, slice t) is 2304 contiguous bytes at
//     (g * k/256 + t) * 2304, so a run of tiles is one contiguous byte range;
//   * lane L = 8h + b (h = 0..3, b = 0..7) owns rows 4h + j (j = 0..3) of
//     block b of the slice: their four scales are the 8 bytes at 8L
//     (binary16, little-endian, row 4h + j at 8L + 2j) and row 4h + j's codes
//     are the 16 bytes at 256 + 512j + 16L;
//   * those 16 bytes are four little-endian 32-bit words; nibble m of word u
//     holds element 16 (u / 2) + 2m + (u % 2).  So nibble m of the word pair
//     (2w, 2w + 1), read as one 64-bit value, holds the adjacent elements
//     16w + 2m and 16w + 2m + 1: the bit operations that decode a pair act on
//     a 64-bit register pair directly and their result feeds one packed
//     fp32x2 subtract and one packed FMA with no moves in between;
//   * rows past n in the last group are padding with d = +0 and codes 8.
//
// The eight lanes that share h read the same rows and blocks b = 0..7; the
// four lanes that share b read the same 32 activations.  x is staged in
// shared memory with 16 bytes of padding after every 32 floats, so the eight
// blocks' activations sit in eight different bank quads and a 16-byte load by
// the whole warp is served in one pass; the warp's code loads are 512
// consecutive bytes.
#pragma once

#include "q4_device.cuh"

namespace q4 {
namespace rt {

constexpr int kRows = 16;            // rows per tile
constexpr int kCols = 256;           // columns (8 blocks) per tile
constexpr int kTileBytes = 2304;     // 16 rows x 8 blocks x 18 bytes
constexpr int kScaleBytes = 256;     // 32 lanes x 4 binary16 scales
constexpr int kCodeRowBytes = 512;   // 32 lanes x 16 bytes, one per row j

// x in shared memory: element e at float index e + 4 * (e / 32).
__host__ __device__ constexpr int64_t xpad_floats(int64_t k) { return k + k / 32 * 4; }
__device__ __forceinline__ int xpad(int e) { return e + ((e >> 5) << 2); }

// Decode constants, each in both halves of a 64-bit value: the exponent bits
// of 2^(23 - p) for p = 0, 4, 8, 12, 16 (a nibble at bit p OR-ed with them
// reads as the float 2^(23-p) + q) and the bias 2^(23-p) + 8.  Written through
// an opaque move so that the OR takes them from registers.
struct PairConsts {
  unsigned long long bits[5];
  unsigned long long bias[5];
};

__device__ __forceinline__ PairConsts make_pair_consts() {
  PairConsts c;
  const uint32_t b[5] = {NibbleMagic<0>::kBits, NibbleMagic<4>::kBits, NibbleMagic<8>::kBits,
                         NibbleMagic<12>::kBits, NibbleMagic<16>::kBits};
  const float f[5] = {NibbleMagic<0>::kBias, NibbleMagic<4>::kBias, NibbleMagic<8>::kBias,
                      NibbleMagic<12>::kBias, NibbleMagic<16>::kBias};
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const uint32_t bb = opaque(b[i]), fb = opaque(__float_as_uint(f[i]));
    c.bits[i] = (static_cast<unsigned long long>(bb) << 32) | bb;
    c.bias[i] = (static_cast<unsigned long long>(fb) << 32) | fb;
  }
  return c;
}

// (q - 8) of the nibbles at bit P of both halves of v, exact, as an fp32 pair:
// a 64-bit AND and OR (one LOP3 per half) and one packed subtract.
template <int P>
__device__ __forceinline__ unsigned long long qm8_pair(unsigned long long v, unsigned long long bits,
                                                       unsigned long long bias) {
  static_assert(P >= 0 && P <= 16 && P % 4 == 0, "nibble must sit in the significand");
  constexpr unsigned long long kMask = static_cast<unsigned long long>(0xFu << P) * 0x100000001ull;
  unsigned long long r;
  asm("{\n\t"
      "and.b64 %0, %1, %2;\n\t"
      "or.b64 %0, %0, %3;\n\t"
      "sub.rn.f32x2 %0, %0, %4;\n\t}"
      : "=l"(r)
      : "l"(v), "n"(kMask), "l"(bits), "l"(bias));
  return r;
}

// sum over the 16 elements of word pair v (its nibble m = elements 2m, 2m+1 of
// the half-block) of (q - 8) * x, accumulated into acc as an fp32 pair; xb[m]
// holds the activation pair of nibble m.  Nibbles 5..7 (bits 20..31 of each
// word) are read after one 64-bit shift by 12, which moves each word's top
// three nibbles to bits 8..19 (bits shifted in from the high word land above
// bit 19 and are masked off).
__device__ __forceinline__ unsigned long long pair_dot(unsigned long long v,
                                                       const unsigned long long* xb,
                                                       const PairConsts& c, unsigned long long acc,
                                                       bool first) {
  const unsigned long long t = v >> 12;
  const unsigned long long a0 = qm8_pair<0>(v, c.bits[0], c.bias[0]);
  acc = first ? fmul2(a0, xb[0]) : ffma2(a0, xb[0], acc);
  acc = ffma2(qm8_pair<4>(v, c.bits[1], c.bias[1]), xb[1], acc);
  acc = ffma2(qm8_pair<8>(v, c.bits[2], c.bias[2]), xb[2], acc);
  acc = ffma2(qm8_pair<12>(v, c.bits[3], c.bias[3]), xb[3], acc);
  acc = ffma2(qm8_pair<16>(v, c.bits[4], c.bias[4]), xb[4], acc);
  acc = ffma2(qm8_pair<8>(t, c.bits[2], c.bias[2]), xb[5], acc);
  acc = ffma2(qm8_pair<12>(t, c.bits[3], c.bias[3]), xb[6], acc);
  acc = ffma2(qm8_pair<16>(t, c.bits[4], c.bias[4]), xb[7], acc);
  return acc;
}

// One tile for this lane: yv[j] += d_j * sum_e (q_je - 8) x_e over block b of
// rows 4h + j.  tile = shared address of the landed tile, xs = shared address
// of the padded x, t = the tile's slice of k.
__device__ __forceinline__ void tile_dot(uint32_t tile, uint32_t xs, int t, int lane,
                                         const PairConsts& c, float (&yv)[4]) {
  const int b = lane & 7;
  unsigned long long xb[16];
  const uint32_t xa = xs + 4 * xpad(t * kCols + 32 * b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];"
                 : "=l"(xb[2 * i]), "=l"(xb[2 * i + 1])
                 : "r"(xa + 16 * i));
  }
  uint32_t s01, s23;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(s01), "=r"(s23) : "r"(tile + 8 * lane));
  const float d[4] = {half_bits_to_float(s01), half_bits_to_float(s01 >> 16),
                      half_bits_to_float(s23), half_bits_to_float(s23 >> 16)};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    unsigned long long v0, v1;  // words (0, 1): elements 0..15; words (2, 3): 16..31
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];"
                 : "=l"(v0), "=l"(v1)
                 : "r"(tile + kScaleBytes + kCodeRowBytes * j + 16 * lane));
    unsigned long long acc = pair_dot(v0, xb, c, 0ull, true);
    acc = pair_dot(v1, xb + 8, c, acc, false);
    const f2 a = unpack2(acc);
    yv[j] = fmaf(a.x + a.y, d[j], yv[j]);
  }
}

}  // namespace rt
}  // namespace q4
