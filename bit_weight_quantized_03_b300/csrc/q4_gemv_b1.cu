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
//     one 2-D TMA tile (144 B x 32 rows, evict-first) per unit.
//   * Two shapes of CTA.  Alone on the GPU, 16 warps per CTA and one CTA per
//     SM; x is staged first and the ring filled behind it.  In a chain of
//     dependent launches (programmatic dependent launch), 8 warps per CTA and
//     at most ~113 KB of shared memory, so that the next product's CTA fits on
//     the same SM beside the running one: it fills its ring (the weights do
//     not depend on the previous product) and then waits, and when the
//     previous product completes its first tiles are already on chip.  Above
//     64 MB of weights the prefetch is too small a share and the solo shape
//     is used even in a chain.
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
//   * Row groups split between warps are finished without atomics.  Each warp
//     walks its range from the last unit down, so of the warps sharing a row
//     group, the one that owns the group's last unit (its "reducer") reaches
//     the group at the very end of its walk, and every other owner reaches it
//     first.  Those store their 32 row sums as tagged 64-bit words (value and
//     a presence tag in one single-copy-atomic store: no fence is needed, and
//     the warp is free at once); the reducer, by then normally finding every
//     word present, polls for any missing one (bounded wait), adds them in
//     warp order (deterministic), clears them and writes y.  A warp publishes
//     before it ever waits, and warps are numbered CTA by CTA, so a reducer
//     waits only for its own CTA or CTAs placed before it; the wait is bounded
//     all the same (Q4_ERR_TIMEOUT after about a second, never a hang).
#include "q4_gemv_tile.cuh"

namespace q4 {
namespace {

using tile::unit_dot;
using tile::unit_dot_m;
using tile::xpad_floats;
using tile::xpad_index;

constexpr int kStages = 2;                    // ring slots per warp
constexpr int kSlotBytes = 32 * kSuperBytes;  // 32 rows x 144 B
// Alone: 16 warps, one CTA per SM, up to 226 KB dynamic shared memory (the
// static barriers take the rest of the 227 KB a CTA may hold).
constexpr int kSoloWarps = 16;
constexpr int kSoloMaxSmem = 226 * 1024;
// In a chain: 8 warps, and two CTAs must fit in one SM's 228 KB (each CTA
// also costs 1 KB of reserved shared memory and its static barriers).
constexpr int kPairWarps = 8;
constexpr int kPairMaxSmem = 115200;
constexpr uint64_t kPairMaxWeightBytes = 64ull << 20;
constexpr int ring_bytes(int warps) { return warps * kStages * kSlotBytes; }

struct B1Params {
  const uint8_t* W;
  int64_t n, nsb;
  const float* x;      // [MB][ldx] (MB = rows of x per launch, 1..4)
  float* y;            // [MB][ldy]
  int64_t ldx, ldy;
  int32_t* counters;   // [groups], unused here (left zero)
  uint64_t* partials;  // [warps][MB][32] tagged row sums, zero when empty
  int64_t units, warps;
  int32_t* status;
  uint32_t flags;
  const uint8_t* pf;   // region prefetched into L2 (the next product's weights), or null
  uint64_t pf_bytes;   // a multiple of 16
};

// A partial row sum as one 64-bit word: the float's bits below a presence tag.
constexpr uint64_t kPresent = 1ull << 32;

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// First unit of warp i when `units` units are cut into `warps` contiguous
// ranges [units*i/warps, units*(i+1)/warps), and the warp that owns unit u.
__device__ __forceinline__ int64_t range_start(int64_t i, int64_t units, int64_t warps) {
  return units * i / warps;
}
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t units, int64_t warps) {
  return ((u + 1) * warps - 1) / units;
}

constexpr int64_t xrow_bytes(int64_t k) { return (xpad_floats(k) * 4 + 127) / 128 * 128; }

// kWarps warps per CTA; kEarlyRing: fill the ring before waiting on the
// previous kernel (the chain shape) rather than after staging x; MB rows of x
// (each unit is decoded once and applied to all of them).
template <int kWarps, bool kEarlyRing, int MB>
__device__ __forceinline__ void gemv_tile_body(const CUtensorMap& tmap, const B1Params& p) {
  constexpr int kRingBytes = ring_bytes(kWarps);
  static_assert(kRingBytes > 0 && MB >= 1 && MB <= 4, "shape");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ __align__(8) uint64_t never[kWarps];  // test hook: nothing ever arrives here
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Warps are numbered CTA by CTA, so a reducer (below) only ever waits for
  // warps of its own CTA or of CTAs with a lower index, which were placed on
  // the GPU before it.
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const bool active = wid < p.warps;
  const uint32_t xs = smem_u32(smem);
  const uint32_t xrow = static_cast<uint32_t>(xrow_bytes(p.nsb * kSuperElems));
  const uint32_t ring = xs + MB * xrow;
  const uint32_t slots = ring + warp * (kStages * kSlotBytes);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);
  const uint32_t never_bar = smem_u32(&never[warp]);
  const uint64_t pol = l2_evict_first_policy();
  const bool stall_test = (p.flags & kFlagTestStallOneWait) != 0 && wid == 0;

  // The warp's range is [u0, u0 + nunits); it is walked from its last unit down.
  int64_t u0 = 0, nunits = 0, g_top = 0, sb_top = 0;
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
    const int64_t u_last = u0 + nunits - 1;
    g_top = u_last / p.nsb;
    sb_top = u_last - g_top * p.nsb;
    ig = g_top;
    isb = sb_top;
  }
  // Producer side: the next unit to load, walked down without divisions.
  auto issue_next = [&]() {
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * islot;
      mbar_arrive_expect_tx(bar, kSlotBytes);
      tma_load_2d_hint(slots + islot * kSlotBytes, &tmap, static_cast<int32_t>(isb * kSuperBytes),
                       static_cast<int32_t>(ig * 32), bar, pol);
    }
    ++issued;
    if (isb-- == 0) {
      isb = p.nsb - 1;
      --ig;
    }
    if (++islot == kStages) islot = 0;
  };
  pdl_allow_dependents();
  // L2 prefetch of the region handed in (in a decode step, the weights of the
  // product after this one), split over the CTAs in 32 KB bulk prefetches: it
  // keeps HBM busy through this product's hand-offs.
  if (p.pf_bytes != 0 && threadIdx.x == 0) {
    const uint64_t share = ((p.pf_bytes + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
    const uint64_t lo = share * blockIdx.x;
    const uint64_t hi = lo + share < p.pf_bytes ? lo + share : p.pf_bytes;
    for (uint64_t o = lo; o < hi; o += 32768) {
      const uint32_t sz = static_cast<uint32_t>(hi - o < 32768 ? hi - o : 32768);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.pf + o), "r"(sz)
                   : "memory");
    }
  }
  // The weights never depend on the previous kernel: in the chain shape the
  // ring is filled while that kernel still runs.
  if (kEarlyRing)
    while (issued < nunits && issued < kStages) issue_next();
  pdl_wait_prior_grid();  // x, y and the workspace are now safe to touch

  // Stage x (all of it) into shared memory with the padded layout.  Its loads
  // are issued before the weight stream starts, so that they are not queued
  // behind the first units' tile loads.
  if constexpr (MB == 1) {
    constexpr int kXRegs = 5;  // covers k <= 5 * 4 * 512 = 10240 in one pass
    const int k4 = static_cast<int>(p.nsb * (kSuperElems / 4));
    const float4* xg = reinterpret_cast<const float4*>(p.x);
    float4 xv[kXRegs];
#pragma unroll
    for (int t = 0; t < kXRegs; ++t) {
      const int i = static_cast<int>(threadIdx.x) + t * kWarps * 32;
      if (i < k4) xv[t] = __ldg(xg + i);
    }
    if (!kEarlyRing)
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
  } else {
    const int k4 = static_cast<int>(p.nsb * (kSuperElems / 4));
    if (!kEarlyRing)
      while (issued < nunits && issued < kStages) issue_next();
    for (int i = static_cast<int>(threadIdx.x); i < MB * k4; i += kWarps * 32) {
      const int m = i / k4, c = i - m * k4;
      const float4 v = __ldg(reinterpret_cast<const float4*>(p.x + m * p.ldx) + c);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(xs + m * xrow +
                                                                     4 * xpad_index(4 * c)),
                   "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                   : "memory");
    }
  }
  __syncthreads();
  if (!active) return;

  const DecodeConsts dc = make_consts();
  const int j = lane & 3;    // block pair within the unit
  const int rr = lane >> 2;  // rows rr, rr + 8, rr + 16, rr + 24 of the group
  float yv[MB][4];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) yv[m][i] = 0.f;

  // Consumer side: unit `done` of the walk is (g, sb) in ring slot `slot`.
  int64_t g = g_top, sb = sb_top, done = 0;
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
    if constexpr (MB == 1)
      unit_dot(slots + slot * kSlotBytes, xs, static_cast<int>(sb), j, rr, dc, yv[0]);
    else
      unit_dot_m<MB>(slots + slot * kSlotBytes, xs, xrow, static_cast<int>(sb), j, rr, dc, yv);
    __syncwarp();
    fence_proxy_async_smem();
    if (issued < nunits) issue_next();
    if (sb == 0 || done == nunits - 1) {
      // Row group g is done for this warp: the four lanes of a quad hold the
      // four block-pair sums of the same rows; add them (fixed order).
      float v[MB][4];
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[m][i] = yv[m][i];
          v[m][i] += __shfl_xor_sync(0xffffffffu, v[m][i], 1);
          v[m][i] += __shfl_xor_sync(0xffffffffu, v[m][i], 2);
          yv[m][i] = 0.f;
        }
      const int64_t gu0 = g * p.nsb, gu1 = gu0 + p.nsb;
      if (gu0 >= u0 && gu1 <= u0 + nunits) {
        if (j == 0) {
#pragma unroll
          for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int64_t row = g * 32 + rr + 8 * i;
              if (row < p.n) p.y[m * p.ldy + row] = v[m][i];
            }
        }
      } else {
        // Lane l takes row l's sums: rows rr + 8i sit in quad rr (lane 4rr).
        float mine[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          mine[m] = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float t = __shfl_sync(0xffffffffu, v[m][i], 4 * (lane & 7));
            if ((lane >> 3) == i) mine[m] = t;
          }
        }
        if (u0 + nunits < gu1) {
          // not the reducer: publish and move on
#pragma unroll
          for (int m = 0; m < MB; ++m)
            st_relaxed_u64(p.partials + (wid * MB + m) * 32 + lane,
                           kPresent | __float_as_uint(mine[m]));
        } else {
          // reducer (owns unit gu1 - 1): owners i0 .. wid - 1 published MB
          // words each, owner-major, so they form one run of `items` words.
          const int64_t i0 = owner_of(gu0, p.units, p.warps);
          const int64_t items = (wid - i0) * MB;
          uint64_t* const run = p.partials + i0 * MB * 32 + lane;
          float s[MB];
#pragma unroll
          for (int m = 0; m < MB; ++m) s[m] = 0.f;
          const uint64_t t0 = global_timer_ns();
          for (int64_t b = 0; b < items; b += 8) {
            // Poll a batch of up to 8 words: every pass re-reads all the words
            // still missing at once, so late owners cost one round trip together.
            uint64_t pv[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) pv[t] = 0;
            while (true) {
#pragma unroll
              for (int t = 0; t < 8; ++t)
                if (b + t < items && !(pv[t] & kPresent)) pv[t] = ld_relaxed_u64(run + (b + t) * 32);
              bool all = true;
#pragma unroll
              for (int t = 0; t < 8; ++t) all = all && (b + t >= items || (pv[t] & kPresent));
              if (all) break;
              if (global_timer_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
              }
            }
            const int m0 = static_cast<int>(b % MB);
#pragma unroll
            for (int t = 0; t < 8; ++t) {  // owner order within each row of x: deterministic
              if (b + t >= items) continue;
              const float val = __uint_as_float(static_cast<uint32_t>(pv[t]));
              const int mt = (m0 + t) % MB;
#pragma unroll
              for (int m = 0; m < MB; ++m)
                if (mt == m) s[m] += val;
            }
          }
          for (int64_t b = 0; b < items; ++b)  // the workspace goes back to all-zero
            st_relaxed_u64(run + b * 32, 0ull);
          const int64_t row = g * 32 + lane;
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            s[m] += mine[m];
            if (row < p.n) p.y[m * p.ldy + row] = s[m];
          }
          if (!__all_sync(0xffffffffu, ok)) ok = false;
        }
      }
    }
    if (sb-- == 0) {
      sb = p.nsb - 1;
      --g;
    }
    if (++slot == kStages) {
      slot = 0;
      parity ^= 1u;
    }
    if (!ok) {
      ++done;  // this unit's copy has been consumed
      break;
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

template <int kWarps, bool kEarlyRing>
__global__ void __launch_bounds__(kWarps * 32, 16 / kWarps)
    gemv_b1_kernel(const __grid_constant__ CUtensorMap tmap, const B1Params p) {
  gemv_tile_body<kWarps, kEarlyRing, 1>(tmap, p);
}

// 2..4 rows of x (batched decode): 8 warps, registers uncapped.
template <int MB, bool kEarlyRing>
__global__ void __launch_bounds__(kPairWarps * 32, 1)
    gemv_bm_kernel(const __grid_constant__ CUtensorMap tmap, const B1Params p) {
  gemv_tile_body<kPairWarps, kEarlyRing, MB>(tmap, p);
}

size_t b1_smem_bytes(int64_t k, int warps, int mb = 1) {
  return static_cast<size_t>(mb * xrow_bytes(k) + ring_bytes(warps));
}

// Launches one of the kernels above (W warps per CTA) once its attributes are
// set on the current device.
template <int W, typename Kernel>
cudaError_t launch_tiles(Kernel kernel, bool (&configured)[64], const CUtensorMap& tmap,
                         const B1Params& p, size_t smem, int max_smem, bool pdl, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    // All of the SM's unified L1/shared storage as shared memory, so that a
    // second CTA can be placed beside a running one without a reconfiguration.
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  const int64_t sms = sm_count();
  const int64_t ctas = (p.warps + W - 1) / W;  // <= sms: warps <= sms * W
  cfg.gridDim = dim3(static_cast<unsigned>(ctas < sms ? ctas : sms));
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = static_cast<unsigned>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, tmap, p);
}

template <int W, bool E>
cudaError_t launch_shape(const CUtensorMap& tmap, const B1Params& p, size_t smem, int max_smem,
                         bool pdl, cudaStream_t s) {
  static bool configured[64] = {false};
  return launch_tiles<W>(gemv_b1_kernel<W, E>, configured, tmap, p, smem, max_smem, pdl, s);
}

template <int MB, bool E>
cudaError_t launch_batched(const CUtensorMap& tmap, const B1Params& p, size_t smem, bool pdl,
                           cudaStream_t s) {
  static bool configured[64] = {false};
  return launch_tiles<kPairWarps>(gemv_bm_kernel<MB, E>, configured, tmap, p, smem,
                                  kSoloMaxSmem, pdl, s);
}

bool make_tmap(CUtensorMap* tmap, const uint8_t* W, int64_t n, int64_t k) {
  const int64_t rowbytes = k / 32 * kBlockBytes;
  return encode_tmap_2d(tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, static_cast<uint64_t>(rowbytes),
                        static_cast<uint64_t>(n), static_cast<uint64_t>(rowbytes), kSuperBytes,
                        32, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

// Warps of the solo shape; the chain shape uses no more (the workspace is
// sized from this count).
int64_t gemv_b1_warps(int64_t units) {
  const int64_t target = static_cast<int64_t>(sm_count()) * kSoloWarps;
  return units < target ? units : target;
}

bool gemv_b1_supports(int64_t k) { return b1_smem_bytes(k, kSoloWarps) <= kSoloMaxSmem; }

cudaError_t gemv_b1_launch(const uint8_t* W, int64_t n, int64_t k, const float* x, float* y,
                           int32_t* counters, float* partials, int64_t units, int64_t warps,
                           int32_t* status, uint32_t flags, cudaStream_t s, const void* pf,
                           uint64_t pf_bytes) {
  const int64_t rowbytes = k / 32 * kBlockBytes;
  CUtensorMap tmap;
  if (!make_tmap(&tmap, W, n, k)) return cudaErrorInvalidValue;
  const bool pdl = (flags & 1u) != 0;
  B1Params p;
  p.W = W;
  p.n = n;
  p.nsb = k / kSuperElems;
  p.x = x;
  p.y = y;
  p.ldx = k;
  p.ldy = n;
  p.counters = counters;
  p.partials = reinterpret_cast<uint64_t*>(partials);
  p.units = units;
  p.status = status;
  p.flags = flags;
  p.pf = static_cast<const uint8_t*>(pf);
  p.pf_bytes = pf_bytes;
  const size_t pair_smem = b1_smem_bytes(k, kPairWarps);
  // The chain shape pays while the next product's ring fill is a real share of
  // that product: for the 7-32 MB decoder products it takes ~13 % off a decode
  // step, for the 226 MB output head the solo shape is faster (53 vs 56 us).
  const bool pair_worth =
      static_cast<uint64_t>(n) * static_cast<uint64_t>(rowbytes) <= kPairMaxWeightBytes;
  if (pdl && pair_worth && pair_smem <= static_cast<size_t>(kPairMaxSmem)) {
    const int64_t target = static_cast<int64_t>(sm_count()) * kPairWarps;
    p.warps = units < target ? units : target;  // <= warps: the workspace holds its partials
    return launch_shape<kPairWarps, true>(tmap, p, pair_smem, kPairMaxSmem, pdl, s);
  }
  p.warps = warps;
  return launch_shape<kSoloWarps, false>(tmap, p, b1_smem_bytes(k, kSoloWarps), kSoloMaxSmem,
                                          pdl, s);
}

bool gemv_bm_supports(int64_t k, int64_t mb) {
  return mb >= 2 && mb <= kMaxBatchRows &&
         b1_smem_bytes(k, kPairWarps, static_cast<int>(mb)) <= kSoloMaxSmem;
}

int64_t gemv_bm_warps(int64_t units) {
  const int64_t target = static_cast<int64_t>(sm_count()) * kPairWarps;
  return units < target ? units : target;
}

cudaError_t gemv_bm_launch(const uint8_t* W, int64_t n, int64_t k, const float* x, int64_t mb,
                           int64_t ldx, float* y, int64_t ldy, int32_t* counters,
                           float* partials, int64_t units, int32_t* status, uint32_t flags,
                           cudaStream_t s) {
  if (!gemv_bm_supports(k, mb)) return cudaErrorInvalidValue;
  CUtensorMap tmap;
  if (!make_tmap(&tmap, W, n, k)) return cudaErrorInvalidValue;
  const bool pdl = (flags & 1u) != 0;
  B1Params p;
  p.W = W;
  p.n = n;
  p.nsb = k / kSuperElems;
  p.x = x;
  p.y = y;
  p.ldx = ldx;
  p.ldy = ldy;
  p.counters = counters;
  p.partials = reinterpret_cast<uint64_t*>(partials);
  p.units = units;
  p.warps = gemv_bm_warps(units);
  p.status = status;
  p.flags = flags;
  p.pf = nullptr;
  p.pf_bytes = 0;
  const size_t smem = b1_smem_bytes(k, kPairWarps, static_cast<int>(mb));
  switch (mb) {
    case 2: return pdl ? launch_batched<2, true>(tmap, p, smem, pdl, s)
                       : launch_batched<2, false>(tmap, p, smem, pdl, s);
    case 3: return pdl ? launch_batched<3, true>(tmap, p, smem, pdl, s)
                       : launch_batched<3, false>(tmap, p, smem, pdl, s);
    default: return pdl ? launch_batched<4, true>(tmap, p, smem, pdl, s)
                        : launch_batched<4, false>(tmap, p, smem, pdl, s);
  }
}

}  // namespace q4
