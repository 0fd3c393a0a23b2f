// q4_gemv_tile.cuh -- the batch-1 work unit shared by the single-GEMV kernel
// (q4_gemv_b1.cu) and the chained decode-step kernel (q4_gemv_chain.cu).
//
// A unit is 32 weight rows x 256 weights (8 Q4_0 blocks = 144 contiguous bytes
// per row), landed in shared memory by one 2-D TMA tile with rows 144 B apart.
// Lane l works on block pair j = l % 4 (weights 64j .. 64j+63 of the unit) of
// rows l/4 + 8i, i = 0..3; it reads its activations from a copy of x staged in
// shared memory with 16 bytes of padding after every 64 floats (the four
// block pairs a warp reads at once then sit in different banks), and the
// 36 bytes of a block pair start on a 4-byte boundary, so the lanes' 32-bit
// loads of the weights hit 32 distinct banks.
//
// Decode: a nibble at bit p <= 16 of a 32-bit word becomes the float
// 2^(23-p) + q with one LOP3 (the one ALU operation per weight); the nibbles at
// bits 20..31 are first moved down by 12 bits with an integer multiply-high
// (FMA pipe).  One packed fp32x2 subtract gives (q - 8) exactly for two weights
// and one packed fp32x2 FMA multiplies them by the adjacent activation pair.
// Per block the 32 products are summed and scaled by d once.
#pragma once

#include "q4_device.cuh"

namespace q4 {
namespace tile {

// x is staged once per CTA in shared memory, with 16 bytes of padding after
// every 64 floats, so that the four block pairs a warp reads at once (256 B
// apart in x) fall into different banks.
__host__ __device__ constexpr int64_t xpad_floats(int64_t k) { return k + k / 64 * 4; }
__device__ __forceinline__ int xpad_index(int e) { return e + (e >> 6) * 4; }

// Dot product of block BLK (0 or 1) of a 36-byte block pair r[9] (only the
// words of that block are read) with its 16 activation pairs xb: returns sum_e (q_e - 8) * x_e as an fp32
// pair (even and odd elements) and the block's scale in d.
//   BLK 0: d = low half of r[0]; qs[0..1] high half of r[0], qs[2..13] in
//          r[1..3], qs[14..15] low half of r[4].
//   BLK 1: d = high half of r[4]; qs[0..15] in r[5..8].
// Byte c of qs holds element c (low nibble) and element c + 16 (high nibble).
template <int BLK>
__device__ __forceinline__ unsigned long long block_dot(const uint32_t (&r)[9],
                                                        const unsigned long long (&xb)[16],
                                                        const DecodeConsts& c, float& d) {
  unsigned long long acc;
  if constexpr (BLK == 0) {
    d = half_bits_to_float(r[0]);
    {
      const uint32_t w = r[0], t = shr12(w);
      acc = fmul2(qm8<16, 12>(w, t, c), xb[0]);          // elements 0, 1
      acc = ffma2(qm8<8, 16>(t, t, c), xb[8], acc);      // 16, 17
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint32_t w = r[1 + i], t = shr12(w);      // qs[2+4i .. 5+4i]
      acc = ffma2(qm8<0, 8>(w, w, c), xb[1 + 2 * i], acc);    // 2+4i, 3+4i
      acc = ffma2(qm8<16, 12>(w, t, c), xb[2 + 2 * i], acc);  // 4+4i, 5+4i
      acc = ffma2(qm8<4, 12>(w, w, c), xb[9 + 2 * i], acc);   // 18+4i, 19+4i
      acc = ffma2(qm8<8, 16>(t, t, c), xb[10 + 2 * i], acc);  // 20+4i, 21+4i
    }
    {
      const uint32_t w = r[4];
      acc = ffma2(qm8<0, 8>(w, w, c), xb[7], acc);   // 14, 15
      acc = ffma2(qm8<4, 12>(w, w, c), xb[15], acc); // 30, 31
    }
  } else {
    d = half_bits_to_float(r[4] >> 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = r[5 + i], t = shr12(w);      // qs[4i .. 4i+3]
      const unsigned long long a = qm8<0, 8>(w, w, c);   // 4i, 4i+1
      acc = i == 0 ? fmul2(a, xb[0]) : ffma2(a, xb[2 * i], acc);
      acc = ffma2(qm8<16, 12>(w, t, c), xb[2 * i + 1], acc);  // 4i+2, 4i+3
      acc = ffma2(qm8<4, 12>(w, w, c), xb[8 + 2 * i], acc);   // 4i+16, 4i+17
      acc = ffma2(qm8<8, 16>(t, t, c), xb[9 + 2 * i], acc);   // 4i+18, 4i+19
    }
  }
  return acc;
}

// The same decode as block_dot without the products: dq[t] holds (q - 8) of
// the element pair that block_dot multiplies by its activation pair xb[t], so
// one decoded block can serve several rows of x.
template <int BLK>
__device__ __forceinline__ void block_decode(const uint32_t (&r)[9], const DecodeConsts& c,
                                             unsigned long long (&dq)[16], float& d) {
  if constexpr (BLK == 0) {
    d = half_bits_to_float(r[0]);
    {
      const uint32_t w = r[0], t = shr12(w);
      dq[0] = qm8<16, 12>(w, t, c);  // elements 0, 1
      dq[8] = qm8<8, 16>(t, t, c);   // 16, 17
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint32_t w = r[1 + i], t = shr12(w);  // qs[2+4i .. 5+4i]
      dq[1 + 2 * i] = qm8<0, 8>(w, w, c);        // 2+4i, 3+4i
      dq[2 + 2 * i] = qm8<16, 12>(w, t, c);      // 4+4i, 5+4i
      dq[9 + 2 * i] = qm8<4, 12>(w, w, c);       // 18+4i, 19+4i
      dq[10 + 2 * i] = qm8<8, 16>(t, t, c);      // 20+4i, 21+4i
    }
    {
      const uint32_t w = r[4];
      dq[7] = qm8<0, 8>(w, w, c);    // 14, 15
      dq[15] = qm8<4, 12>(w, w, c);  // 30, 31
    }
  } else {
    d = half_bits_to_float(r[4] >> 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = r[5 + i], t = shr12(w);  // qs[4i .. 4i+3]
      dq[2 * i] = qm8<0, 8>(w, w, c);            // 4i, 4i+1
      dq[2 * i + 1] = qm8<16, 12>(w, t, c);      // 4i+2, 4i+3
      dq[8 + 2 * i] = qm8<4, 12>(w, w, c);       // 4i+16, 4i+17
      dq[9 + 2 * i] = qm8<8, 16>(t, t, c);       // 4i+18, 4i+19
    }
  }
}

__device__ __forceinline__ void lds_v2u64(uint32_t addr, unsigned long long& a,
                                          unsigned long long& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Accumulates one unit into yv[i] (row rr + 8i of the group) for this lane:
// slot = shared address of the landed 32 x 144-byte tile, xs = the padded x
// copy, sb = the unit's 256-wide slice of k.
__device__ __forceinline__ void unit_dot(uint32_t slot, uint32_t xs, int sb, int j, int rr,
                                         const DecodeConsts& dc, float (&yv)[4]) {
  const uint32_t src = slot + rr * kSuperBytes + 36 * j;
  const int xe = sb * kSuperElems + 64 * j;  // first element of the pair
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    unsigned long long xb[16];
    const uint32_t xa = xs + 4 * xpad_index(xe + 32 * b);
#pragma unroll
    for (int i = 0; i < 8; ++i) lds_v2u64(xa + 16 * i, xb[2 * i], xb[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t r[9];
#pragma unroll
      for (int w = 0; w < 5; ++w) r[4 * b + w] = lds32(src + i * 8 * kSuperBytes + 4 * (4 * b + w));
      float d;
      const f2 a = unpack2(b == 0 ? block_dot<0>(r, xb, dc, d) : block_dot<1>(r, xb, dc, d));
      yv[i] = fmaf(a.x + a.y, d, yv[i]);
    }
  }
}

// unit_dot for MB rows of x at once (MB small): every block of the lane's four
// weight rows is decoded once and multiplied by the MB activation rows, which
// are staged xrow bytes apart in shared memory; yv[m][i] accumulates row rr + 8i
// of the group for activation row m.
template <int MB>
__device__ __forceinline__ void unit_dot_m(uint32_t slot, uint32_t xs, uint32_t xrow, int sb,
                                           int j, int rr, const DecodeConsts& dc,
                                           float (&yv)[MB][4]) {
  const uint32_t src = slot + rr * kSuperBytes + 36 * j;
  const int xe = sb * kSuperElems + 64 * j;  // first element of the pair
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t xa = xs + 4 * xpad_index(xe + 32 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t r[9];
#pragma unroll
      for (int w = 0; w < 5; ++w) r[4 * b + w] = lds32(src + i * 8 * kSuperBytes + 4 * (4 * b + w));
      unsigned long long dq[16];
      float d;
      if (b == 0)
        block_decode<0>(r, dc, dq, d);
      else
        block_decode<1>(r, dc, dq, d);
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        unsigned long long xb[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) lds_v2u64(xa + m * xrow + 16 * q, xb[2 * q], xb[2 * q + 1]);
        unsigned long long acc = fmul2(dq[0], xb[0]);
#pragma unroll
        for (int t = 1; t < 16; ++t) acc = ffma2(dq[t], xb[t], acc);
        const f2 a = unpack2(acc);
        yv[m][i] = fmaf(a.x + a.y, d, yv[m][i]);
      }
    }
  }
}

}  // namespace tile
}  // namespace q4
