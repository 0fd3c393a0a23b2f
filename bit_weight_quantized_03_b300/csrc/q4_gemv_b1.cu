// q4_gemv_b1.cu -- fused Q4_0 dequant-GEMV at batch 1 (one token per decode step):
//   y[r] = sum_j ((q[r][j] - 8) * d[r][j/32]) * x[j],  fp32 accumulation.
//
// This is the per-token product of every decoder linear and of the output head
// in the Voxtral Mini 4B Realtime port (GeekNews, es.news.hada.io/topic?id=26595,
// "Arquitectura": 26-layer decoder, hidden 3072, GQA 32Q/8KV, GGUF Q4_0
// weights through custom GPU shaders).  Each weight is read once and used
// once, so the kernel has to decode Q4_0 as fast as HBM delivers it: at the
// measured ~6.5 TB/s that is ~38 weights per SM clock, against an integer ALU
// pipe that retires 64 lane-operations per SM clock.  The design therefore
// spends one ALU operation per weight and keeps everything else on the FMA
// pipe or out of the loop:
//
//   * Work unit = 32 rows x 256 weights (8 blocks = 144 contiguous bytes per
//     row).  Units are ordered row-group major; every warp takes one contiguous
//     range of them ("stream-K"), so each warp gets the same number +-1.
//   * Each warp streams its units through its own ring of shared-memory slots,
//     one 2-D TMA tile (144 B x 32 rows, evict-first) per unit.  The ring is
//     filled before waiting on the previous kernel (programmatic dependent
//     launch), so weight reads overlap the previous layer's tail.
//   * Lane l works on block pair j = l % 4 (weights 64j .. 64j+63 of the unit)
//     of rows l/4, l/4 + 8, l/4 + 16, l/4 + 24.  Its 64 activations are loaded
//     once per unit into registers as fp32 pairs and serve all four rows; the
//     36 bytes of a block pair start on a 4-byte boundary, and the lanes' 32-bit
//     shared loads hit 32 distinct banks.
//   * Decode: a nibble at bit p <= 16 of a 32-bit word becomes the float
//     2^(23-p) + q with one AND/OR (LOP3, the one ALU operation per weight);
//     the nibbles at bits 20..31 are first moved down by 12 bits with an
//     integer multiply-high (FMA pipe).  One packed fp32x2 subtract gives
//     (q - 8) exactly for two weights, one packed fp32x2 FMA multiplies them by
//     the adjacent activation pair.  Per block the 32 products are summed and
//     scaled by d once.
//   * Row groups split between warps are finished deterministically: partial
//     row sums go to the workspace, the last warp to arrive (atomic counter)
//     adds them in warp order, zeroes them and resets the counter.
#include "q4_gemv_tile.cuh"

namespace q4 {
namespace {

using tile::unit_dot;
using tile::xpad_floats;
using tile::xpad_index;

constexpr int kWarps = 16;                    // warps per CTA, one CTA per SM
constexpr int kStages = 2;                    // ring slots per warp
constexpr int kSlotBytes = 32 * kSuperBytes;  // 32 rows x 144 B
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kMaxSmem = 226 * 1024;  // dynamic part; the static barriers need the rest

struct B1Params {
  const uint8_t* W;
  int64_t n, nsb;
  const float* x;
  float* y;
  int32_t* counters;  // [groups]
  float* partials;    // [warps][2][32]
  int64_t units, warps;
  int32_t* status;
  uint32_t flags;
};

__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// First unit of warp i when `units` units are cut into `warps` contiguous
// ranges [units*i/warps, units*(i+1)/warps), and the warp that owns unit u.
__device__ __forceinline__ int64_t range_start(int64_t i, int64_t units, int64_t warps) {
  return units * i / warps;
}
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t units, int64_t warps) {
  return ((u + 1) * warps - 1) / units;
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    gemv_b1_kernel(const __grid_constant__ CUtensorMap tmap, const B1Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ __align__(8) uint64_t never[kWarps];  // test hook: nothing ever arrives here
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Warps are dealt to CTAs round-robin so that small matrices still spread
  // over every SM.
  const int64_t wid = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x;
  const bool active = wid < p.warps;
  const uint32_t xs = smem_u32(smem);
  const int64_t xpad = xpad_floats(p.nsb * kSuperElems);
  const uint32_t ring = xs + static_cast<uint32_t>((xpad * 4 + 127) / 128 * 128);
  const uint32_t slots = ring + warp * (kStages * kSlotBytes);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);
  const uint32_t never_bar = smem_u32(&never[warp]);
  const uint64_t pol = l2_evict_first_policy();
  const bool stall_test = (p.flags & kFlagTestStallOneWait) != 0 && wid == 0;

  int64_t u0 = 0, nunits = 0, g_first = 0;
  int64_t ig = 0, isb = 0, issued = 0;
  int islot = 0;
  if (active) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
      mbar_init(never_bar, 1);
      fence_mbarrier_init();
    }
    __syncwarp();
    u0 = range_start(wid, p.units, p.warps);
    nunits = range_start(wid + 1, p.units, p.warps) - u0;  // >= 1
    g_first = u0 / p.nsb;
    ig = g_first;
    isb = u0 - g_first * p.nsb;
  }
  // Producer side: the next unit to load, walked without divisions.
  auto issue_next = [&]() {
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * islot;
      mbar_arrive_expect_tx(bar, kSlotBytes);
      tma_load_2d_hint(slots + islot * kSlotBytes, &tmap, static_cast<int32_t>(isb * kSuperBytes),
                       static_cast<int32_t>(ig * 32), bar, pol);
    }
    ++issued;
    if (++isb == p.nsb) {
      isb = 0;
      ++ig;
    }
    if (++islot == kStages) islot = 0;
  };
  pdl_allow_dependents();
  pdl_wait_prior_grid();  // x, y and the workspace are now safe to touch

  // Stage x (all of it) into shared memory with the padded layout.  Its loads
  // are issued before the weight stream starts, so that they are not queued
  // behind the first units' tile loads.
  {
    constexpr int kXRegs = 5;  // covers k <= 5 * 4 * 512 = 10240 in one pass
    const int k4 = static_cast<int>(p.nsb * (kSuperElems / 4));
    const float4* xg = reinterpret_cast<const float4*>(p.x);
    float4 xv[kXRegs];
#pragma unroll
    for (int t = 0; t < kXRegs; ++t) {
      const int i = static_cast<int>(threadIdx.x) + t * kWarps * 32;
      if (i < k4) xv[t] = __ldg(xg + i);
    }
    while (issued < nunits && issued < kStages) issue_next();
    auto put = [&](int i, const float4& v) {
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(xs + 4 * xpad_index(4 * i)),
                   "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                   : "memory");
    };
#pragma unroll
    for (int t = 0; t < kXRegs; ++t) {
      const int i = static_cast<int>(threadIdx.x) + t * kWarps * 32;
      if (i < k4) put(i, xv[t]);
    }
    for (int i = static_cast<int>(threadIdx.x) + kXRegs * kWarps * 32; i < k4; i += kWarps * 32)
      put(i, __ldg(xg + i));
  }
  __syncthreads();
  if (!active) return;

  const DecodeConsts dc = make_consts();
  const int j = lane & 3;    // block pair within the unit
  const int rr = lane >> 2;  // rows rr, rr + 8, rr + 16, rr + 24 of the group
  float yv[4] = {0.f, 0.f, 0.f, 0.f};

  // Consumer side: unit `done` of the range is (g, sb) in ring slot `slot`.
  int64_t g = g_first, sb = u0 - g_first * p.nsb, done = 0;
  int slot = 0;
  uint32_t parity = 0;
  bool ok = true;
  for (; done < nunits; ++done) {
    // every lane waits; the verdict is made warp-uniform before any __syncwarp.
    // The test hook waits on a barrier that nothing arrives on, so that wait
    // runs out after kWaitLimitNs.
    const bool landed = (stall_test && done == 0) ? mbar_wait(never_bar, 0)
                                                   : mbar_wait(bar0 + 8 * slot, parity);
    if (!__all_sync(0xffffffffu, landed)) {
      ok = false;
      break;
    }
    unit_dot(slots + slot * kSlotBytes, xs, static_cast<int>(sb), j, rr, dc, yv);
    __syncwarp();
    fence_proxy_async_smem();
    if (issued < nunits) issue_next();
    if (sb == p.nsb - 1 || done == nunits - 1) {
      // Row group g is done for this warp: the four lanes of a quad hold the
      // four block-pair sums of the same rows; add them (fixed order).
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] = yv[i];
        v[i] += __shfl_xor_sync(0xffffffffu, v[i], 1);
        v[i] += __shfl_xor_sync(0xffffffffu, v[i], 2);
        yv[i] = 0.f;
      }
      const int64_t gu0 = g * p.nsb, gu1 = gu0 + p.nsb;
      if (gu0 >= u0 && gu1 <= u0 + nunits) {
        if (j == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t row = g * 32 + rr + 8 * i;
            if (row < p.n) p.y[row] = v[i];
          }
        }
      } else {
        // Partial slot 0 holds a warp's first row group, slot 1 its last.
        float* mine = p.partials + (wid * 2 + (g == g_first ? 0 : 1)) * 32;
        if (j == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) __stcg(mine + rr + 8 * i, v[i]);
        }
        __syncwarp();  // the lanes' partials are ordered before lane 0's release
        const int64_t i0 = owner_of(gu0, p.units, p.warps);
        const int64_t i1 = owner_of(gu1 - 1, p.units, p.warps);
        int last = 0;
        // acq_rel: releases this warp's partials; the last arrival acquires all
        if (lane == 0) last = atomic_add_acq_rel_gpu(&p.counters[g], 1) == static_cast<int>(i1 - i0);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          // Owner i0 may have started in an earlier group (then this group is
          // its slot 1); every later owner starts inside this group (slot 0).
          const int64_t i0_slot = range_start(i0, p.units, p.warps) < gu0 ? 1 : 0;
          const int np = static_cast<int>(i1 - i0 + 1);
          float s = 0.f;
          for (int b = 0; b < np; b += 8) {
            float pv[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int64_t i = i0 + b + t;
              const int64_t sl = (t == 0 && b == 0) ? i0_slot : 0;
              pv[t] = (b + t < np) ? __ldcg(p.partials + (i * 2 + sl) * 32 + lane) : 0.f;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (b + t < np) s += pv[t];  // warp order: deterministic
          }
          for (int b = 0; b < np; ++b) {  // the workspace goes back to all-zero
            const int64_t sl = b == 0 ? i0_slot : 0;
            __stcg(p.partials + ((i0 + b) * 2 + sl) * 32 + lane, 0.f);
          }
          const int64_t row = g * 32 + lane;
          if (row < p.n) p.y[row] = s;
          if (lane == 0) p.counters[g] = 0;
        }
      }
    }
    if (++sb == p.nsb) {
      sb = 0;
      ++g;
    }
    if (++slot == kStages) {
      slot = 0;
      parity ^= 1u;
    }
  }

  if (!ok) {
    if (lane == 0) report(p.status, 6 /* Q4_ERR_TIMEOUT */);
    // Let every copy this warp still has in flight (unit `done`'s included)
    // land before the CTA exits; each of these waits is bounded too.
    for (int64_t v = done; v < issued; ++v)
      mbar_wait(bar0 + 8 * static_cast<uint32_t>(v % kStages),
                static_cast<uint32_t>((v / kStages) & 1));
  }
}

}  // namespace

int64_t gemv_b1_warps(int64_t units) {
  const int64_t target = static_cast<int64_t>(sm_count()) * kWarps;
  return units < target ? units : target;
}

bool gemv_b1_supports(int64_t k) {
  const int64_t xbytes = (xpad_floats(k) * 4 + 127) / 128 * 128;
  return xbytes + kRingBytes <= kMaxSmem;
}

cudaError_t gemv_b1_launch(const uint8_t* W, int64_t n, int64_t k, const float* x, float* y,
                           int32_t* counters, float* partials, int64_t units, int64_t warps,
                           int32_t* status, uint32_t flags, cudaStream_t s) {
  const int64_t rowbytes = k / 32 * kBlockBytes;
  CUtensorMap tmap;
  if (!encode_tmap_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, static_cast<uint64_t>(rowbytes),
                      static_cast<uint64_t>(n), static_cast<uint64_t>(rowbytes), kSuperBytes, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemv_b1_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  B1Params p;
  p.W = W;
  p.n = n;
  p.nsb = k / kSuperElems;
  p.x = x;
  p.y = y;
  p.counters = counters;
  p.partials = partials;
  p.units = units;
  p.warps = warps;
  p.status = status;
  p.flags = flags;
  cudaLaunchConfig_t cfg = {};
  const int64_t sms = sm_count();
  cfg.gridDim = dim3(static_cast<unsigned>(warps < sms ? warps : sms));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes =
      static_cast<unsigned>((xpad_floats(k) * 4 + 127) / 128 * 128 + kRingBytes);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (flags & 1u) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_b1_kernel, tmap, p);
}

}  // namespace q4
