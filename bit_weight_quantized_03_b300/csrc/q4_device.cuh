// q4_device.cuh -- device-side helpers shared by the Q4_0 kernels (sm_103a).
//
// Q4_0 block (GGUF Q4_0, the weight format of the quantized path in the GeekNews
// write-up es.news.hada.io/topic?id=26595, "Arquitectura"): 18 bytes = binary16
// scale d (little-endian) + qs[16]; weight j is the low nibble of qs[j], weight
// j+16 its high nibble; w = (q - 8) * d.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_internal.h"

namespace q4 {

constexpr int kBlockElems = 32;
constexpr int kBlockBytes = 18;
constexpr int kSuperElems = 256;  // 8 blocks: the smallest 16-byte-aligned run of blocks
constexpr int kSuperBytes = 144;  // 8 * 18 = 9 * 16

// Device-side error report: first error wins.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// ----------------------------------------------------------------------------
// Exact nibble -> float decode without integer-to-float conversion.
//
// For a nibble q sitting at bits [p, p+4) of a 32-bit word (p <= 16), OR-ing
// the bits of 2^(23-p) into the masked word gives the float 2^(23-p) + q
// exactly (the nibble lands in the significand at weight 1).  Subtracting
// 2^(23-p) + 8 then yields (q - 8) exactly.  One LOP3 per weight.
template <int P>
struct NibbleMagic {
  static_assert(P >= 0 && P <= 16 && P % 4 == 0, "nibble must sit in the significand");
  static constexpr uint32_t kMask = 0xFu << P;
  static constexpr uint32_t kBits = static_cast<uint32_t>(127 + 23 - P) << 23;  // 2^(23-P)
  static constexpr float kBias = static_cast<float>(1u << (23 - P)) + 8.0f;     // 2^(23-P) + 8
};

template <int P>
__device__ __forceinline__ float nibble_magic(uint32_t word) {
  return __uint_as_float((word & NibbleMagic<P>::kMask) | NibbleMagic<P>::kBits);
}

// ----------------------------------------------------------------------------
// Packed fp32x2 arithmetic (sm_100 family).
struct f2 {
  float x, y;
};

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ f2 unpack2(unsigned long long v) {
  f2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long fsub2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ----------------------------------------------------------------------------
// Single-LOP3 nibble decode shared by the GEMV and GEMM kernels.

// w >> 12 computed as the high word of w * 2^20: an integer multiply, issued
// to the FMA pipe instead of the (busier) ALU pipe.
__device__ __forceinline__ uint32_t shr12(uint32_t w) { return __umulhi(w, 1u << 20); }

// Loop-invariant decode constants, kept in registers: the exponent bits of
// 2^(23-p) for the five nibble positions p = 0, 4, 8, 12, 16, and the packed
// (2^(23-pa) + 8, 2^(23-pb) + 8) bias pairs of the four position pairs used.
// Written through an opaque move so that each magic OR stays one LOP3 (mask as
// the immediate, bits from the register) instead of an AND plus an OR.
struct DecodeConsts {
  uint32_t bits[5];
  unsigned long long bias_16_12, bias_8_16, bias_0_8, bias_4_12;
};

__device__ __forceinline__ uint32_t opaque(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ DecodeConsts make_consts() {
  DecodeConsts c;
  c.bits[0] = opaque(NibbleMagic<0>::kBits);
  c.bits[1] = opaque(NibbleMagic<4>::kBits);
  c.bits[2] = opaque(NibbleMagic<8>::kBits);
  c.bits[3] = opaque(NibbleMagic<12>::kBits);
  c.bits[4] = opaque(NibbleMagic<16>::kBits);
  auto bias = [](float a, float b) {
    return pack2(__uint_as_float(opaque(__float_as_uint(a))),
                 __uint_as_float(opaque(__float_as_uint(b))));
  };
  c.bias_16_12 = bias(NibbleMagic<16>::kBias, NibbleMagic<12>::kBias);
  c.bias_8_16 = bias(NibbleMagic<8>::kBias, NibbleMagic<16>::kBias);
  c.bias_0_8 = bias(NibbleMagic<0>::kBias, NibbleMagic<8>::kBias);
  c.bias_4_12 = bias(NibbleMagic<4>::kBias, NibbleMagic<12>::kBias);
  return c;
}

template <int P>
__device__ __forceinline__ uint32_t pos_bits(const DecodeConsts& c) {
  return c.bits[P / 4];
}

template <int PA, int PB>
__device__ __forceinline__ unsigned long long pair_bias(const DecodeConsts& c) {
  if constexpr (PA == 16 && PB == 12) return c.bias_16_12;
  else if constexpr (PA == 8 && PB == 16) return c.bias_8_16;
  else if constexpr (PA == 0 && PB == 8) return c.bias_0_8;
  else return c.bias_4_12;
}

// (q - 8) for the weight pair whose nibbles sit at bit PA of wa and PB of wb:
// two LOP3 ((w & 0xF << p) | bits(2^(23-p))) and one packed fp32x2 subtract.
template <int PA, int PB>
__device__ __forceinline__ unsigned long long qm8(uint32_t wa, uint32_t wb,
                                                  const DecodeConsts& c) {
  static_assert((PA == 16 && PB == 12) || (PA == 8 && PB == 16) || (PA == 0 && PB == 8) ||
                    (PA == 4 && PB == 12),
                "position pair without a bias constant");
  unsigned long long r;
  asm("{\n\t.reg .b32 lo, hi;\n\t"
      "lop3.b32 lo, %1, %3, %4, 0xEA;\n\t"
      "lop3.b32 hi, %2, %5, %6, 0xEA;\n\t"
      "mov.b64 %0, {lo, hi};\n\t"
      "sub.rn.f32x2 %0, %0, %7;\n\t}"
      : "=l"(r)
      : "r"(wa), "r"(wb), "n"(NibbleMagic<PA>::kMask), "r"(pos_bits<PA>(c)),
        "n"(NibbleMagic<PB>::kMask), "r"(pos_bits<PB>(c)), "l"(pair_bias<PA, PB>(c)));
  return r;
}

// ----------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk copies (PTX ISA: mbarrier,
// cp.async.bulk).  Every wait is bounded by a wall-clock limit read from
// %globaltimer; on expiry the caller gets `false` and reports Q4_ERR_TIMEOUT.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false after about
// kWaitLimitNs of wall-clock time, or at once if *abort became non-zero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D TMA tile load global -> shared with an L2 cache-policy hint.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, int32_t c0,
                                                 int32_t c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch controls (no-ops when the launch did not enable PDL).
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 ldg_nc_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void stg_cs_f4(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

}  // namespace q4
