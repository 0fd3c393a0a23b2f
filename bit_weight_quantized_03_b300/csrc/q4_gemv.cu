// q4_gemv.cu -- fused Q4_0 dequant-GEMV for batch-1 (and small-batch) decode:
//   y[i][r] = sum_j ((q[r][j] - 8) * d[r][j/32]) * x[i][j],  fp32 accumulation.
//
// This is the per-token product of every decoder linear of the Voxtral Mini 4B
// Realtime port (GeekNews, es.news.hada.io/topic?id=26595, "Arquitectura":
// 26-layer decoder, hidden 3072, GQA 32Q/8KV; Q4 GGUF weights multiplied by
// custom GPU shaders).  At one token per step the weights are read once and
// used once, so the product is bound by HBM bandwidth; the design keeps the
// weight stream in flight and the per-weight instruction count low.
//
// Dispatch (gemv_launch): k % 256 == 0 goes to the tile kernels of
// q4_gemv_b1.cu -- one row of x to the batch-1 kernel, 2..16 rows to launches of
// up to 4 rows of the batched tile kernel (each unit decoded once for all of
// its rows).  The streamed kernel below serves the rows those cannot take (x
// too wide for shared memory); the generic kernel any k % 32 == 0.
//
// Streamed kernel (k % 256 == 0):
//   * Work unit = 32 rows x 256 weights (8 blocks = 144 contiguous, 16-byte
//     aligned bytes per row).  Units are ordered row-group major and every warp
//     takes one contiguous range of them ("stream-K"), so every warp gets the
//     same number of units +-1 whatever the shape.
//   * Each warp streams its units through its own ring of shared-memory slots:
//     one 2-D TMA tile load per unit (box 144 B x 32 rows over the packed
//     matrix, evict-first L2 hint), completion counted on the slot's mbarrier.
//     (Thirty-two 144-byte bulk copies per unit instead were bound by the copy
//     engine's per-request cost.)  Slot rows are 144 B apart (9 x 16 B, odd), so
//     each lane's 16-byte shared loads of its row are bank-conflict free.  The
//     ring is filled before waiting on the previous kernel (programmatic
//     dependent launch), so weight reads overlap the previous layer's tail.
//   * Decode: a nibble sitting at bit p <= 16 of a 32-bit word becomes the float
//     2^(23-p) + q with one AND/OR (LOP3); one packed subtract gives (q - 8)
//     exactly for two weights.  Weights are paired with the adjacent activation
//     pair (x[j], x[j+1]) so the products are packed fp32x2 FMAs.  Per block
//     the 32 products are summed, then scaled by d once.
//   * Row groups split between warps are finished deterministically: each warp
//     writes its partial row sums to the workspace, and the last warp to arrive
//     (atomic counter) adds the partials in warp order, then zeroes them and
//     resets the counter, so the whole workspace is zero again after the call.
//
// Generic kernel (any k % 32 == 0): one warp per row, lanes stride over blocks.
#include "q4_device.cuh"

namespace q4 {
namespace {

// ---------------------------------------------------------------- generic

template <int M>
__global__ void __launch_bounds__(256) gemv_generic_kernel(const uint8_t* __restrict__ W,
                                                           int64_t n, int64_t nb,
                                                           const float* __restrict__ x,
                                                           int64_t ldx, float* __restrict__ y,
                                                           int64_t ldy) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  if (row >= n) return;
  const uint8_t* wr = W + row * nb * kBlockBytes;
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.f;
  for (int64_t b = lane; b < nb; b += 32) {
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(wr + b * kBlockBytes);
    const float d = half_bits_to_float(blk[0]);
    float w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t two = blk[1 + j];  // qs[2j] | qs[2j+1] << 8
      w[2 * j] = static_cast<float>(static_cast<int>(two & 15) - 8) * d;
      w[2 * j + 1] = static_cast<float>(static_cast<int>((two >> 8) & 15) - 8) * d;
      w[2 * j + 16] = static_cast<float>(static_cast<int>((two >> 4) & 15) - 8) * d;
      w[2 * j + 17] = static_cast<float>(static_cast<int>((two >> 12) & 15) - 8) * d;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4* xb = reinterpret_cast<const float4*>(x + m * ldx + b * kBlockElems);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(xb + i);
        acc[m] = fmaf(w[4 * i + 0], v.x, acc[m]);
        acc[m] = fmaf(w[4 * i + 1], v.y, acc[m]);
        acc[m] = fmaf(w[4 * i + 2], v.z, acc[m]);
        acc[m] = fmaf(w[4 * i + 3], v.w, acc[m]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) y[m * ldy + row] = v;
  }
}

// ---------------------------------------------------------------- streamed

constexpr int kWarps = 4;                      // independent warps per CTA
constexpr int kStages = 4;                     // ring slots per warp
constexpr int kSlotBytes = 32 * kSuperBytes;   // 32 rows x 144 B
constexpr int kSmemBytes = kWarps * kStages * kSlotBytes;

struct StreamParams {
  const uint8_t* W;
  int64_t n, nsb, rowbytes;
  const float* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  int32_t* counters;  // [groups]
  float* partials;    // [warps][2][M][32]
  int64_t units, warps, groups;
  int32_t* status;
  uint32_t flags;
};

// Warp that owns unit u when `units` units are cut into `warps` contiguous
// ranges [units*i/warps, units*(i+1)/warps).
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t units, int64_t warps) {
  return ((u + 1) * warps - 1) / units;
}

__device__ __forceinline__ unsigned long long bias_pair(float a, float b) { return pack2(a, b); }

// (q - 8) for the weight pair whose nibbles sit at bits (PA of wa, PB of wb).
template <int PA, int PB>
__device__ __forceinline__ unsigned long long wpair(uint32_t wa, uint32_t wb) {
  return fsub2(pack2(nibble_magic<PA>(wa), nibble_magic<PB>(wb)),
               bias_pair(NibbleMagic<PA>::kBias, NibbleMagic<PB>::kBias));
}

// Decodes block BLK (0..7) of a 144-byte run held in r[36] into 16 pairs of
// (q - 8): wp[e/2] = (w[e], w[e+1]) for e even.  Returns the block's scale.
template <int BLK>
__device__ __forceinline__ float decode_pairs(const uint32_t (&r)[36], unsigned long long (&wp)[16]) {
  constexpr int ob = 18 * BLK;  // byte offset of the block
  constexpr int wd = ob / 4;
  constexpr bool d_high = ((ob / 2) & 1) != 0;
  const float d = half_bits_to_float(d_high ? (r[wd] >> 16) : r[wd]);
  if constexpr ((BLK & 1) == 1) {
    // qs starts 4-byte aligned: word i holds qs[4i .. 4i+3]
    constexpr int w0 = (ob + 2) / 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = r[w0 + i], t = w >> 12;
      wp[2 * i] = wpair<0, 8>(w, w);             // elements 4i, 4i+1
      wp[2 * i + 1] = wpair<16, 12>(w, t);       // 4i+2, 4i+3
      wp[8 + 2 * i] = wpair<4, 12>(w, w);        // 4i+16, 4i+17
      wp[8 + 2 * i + 1] = wpair<8, 16>(t, t);    // 4i+18, 4i+19
    }
  } else {
    // qs starts 2 bytes into a word: qs[0..1] in the high half of word ob/4,
    // qs[2..13] in the next three words, qs[14..15] in the low half after them
    constexpr int w0 = ob / 4;
    {
      const uint32_t w = r[w0], t = w >> 12;
      wp[0] = wpair<16, 12>(w, t);  // elements 0, 1
      wp[8] = wpair<8, 16>(t, t);   // 16, 17
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint32_t w = r[w0 + 1 + i], t = w >> 12;  // qs[2+4i .. 5+4i]
      wp[1 + 2 * i] = wpair<0, 8>(w, w);      // 2+4i, 3+4i
      wp[2 + 2 * i] = wpair<16, 12>(w, t);    // 4+4i, 5+4i
      wp[9 + 2 * i] = wpair<4, 12>(w, w);     // 18+4i, 19+4i
      wp[10 + 2 * i] = wpair<8, 16>(t, t);    // 20+4i, 21+4i
    }
    {
      const uint32_t w = r[w0 + 4];
      wp[7] = wpair<0, 8>(w, w);    // 14, 15
      wp[15] = wpair<4, 12>(w, w);  // 30, 31
    }
  }
  return d;
}

// Accumulates block BLK of the run against x (pointer to x[0][k of block 0]).
template <int BLK, int M>
__device__ __forceinline__ void block_fma(const uint32_t (&r)[36], const float* __restrict__ xrun,
                                          int64_t ldx, unsigned long long (&y2)[M]) {
  unsigned long long wp[16];
  const float d = decode_pairs<BLK>(r, wp);
  const unsigned long long d2 = pack2(d, d);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float4* xb = reinterpret_cast<const float4*>(xrun + m * ldx + BLK * kBlockElems);
    unsigned long long acc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = __ldg(xb + i);
      const unsigned long long x01 = pack2(v.x, v.y), x23 = pack2(v.z, v.w);
      // pairs 2i, 2i+1 cover elements 4i..4i+3 of the block
      if (i == 0)
        acc = fmul2(wp[0], x01);
      else
        acc = ffma2(wp[2 * i], x01, acc);
      acc = ffma2(wp[2 * i + 1], x23, acc);
    }
    y2[m] = ffma2(acc, d2, y2[m]);
  }
}

template <int M>
__global__ void __launch_bounds__(kWarps * 32)
    gemv_stream_kernel(const __grid_constant__ CUtensorMap tmap, const StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ __align__(8) uint64_t never[kWarps];  // test hook: nothing ever arrives here
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (wid >= p.warps) {
    pdl_allow_dependents();
    return;
  }
  const uint32_t slots = smem_u32(smem) + warp * (kStages * kSlotBytes);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);
  const uint32_t never_bar = smem_u32(&never[warp]);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init(never_bar, 1);
    fence_mbarrier_init();
  }
  __syncwarp();

  const int64_t u0 = p.units * wid / p.warps;
  const int64_t u1 = p.units * (wid + 1) / p.warps;
  const uint64_t pol = l2_evict_first_policy();
  const bool stall_test = (p.flags & kFlagTestStallOneWait) != 0 && wid == 0;

  // Issue the TMA load of unit u into its ring slot (lane 0).  Rows past n
  // arrive zero-filled; the full box is always counted.
  auto issue = [&](int64_t u) {
    if (lane == 0) {
      const int64_t g = u / p.nsb, sb = u - g * p.nsb;
      const int slot = static_cast<int>((u - u0) % kStages);
      const uint32_t bar = bar0 + 8 * slot;
      mbar_arrive_expect_tx(bar, kSlotBytes);
      tma_load_2d_hint(slots + slot * kSlotBytes, &tmap, static_cast<int32_t>(sb * kSuperBytes),
                       static_cast<int32_t>(g * 32), bar, pol);
    }
  };

  int64_t issued = u0;
  for (; issued < u1 && issued < u0 + kStages; ++issued) issue(issued);

  pdl_allow_dependents();
  pdl_wait_prior_grid();  // x, y and the workspace are now safe to touch

  const int64_t g_first = u0 / p.nsb;
  unsigned long long y2[M];
#pragma unroll
  for (int m = 0; m < M; ++m) y2[m] = 0;

  bool ok = true;
  int64_t u = u0;
  for (; u < u1; ++u) {
    const int slot = static_cast<int>((u - u0) % kStages);
    const uint32_t parity = static_cast<uint32_t>(((u - u0) / kStages) & 1);
    // every lane waits; the verdict is made warp-uniform before any __syncwarp.
    // The test hook waits on a barrier that nothing arrives on, so that wait
    // runs out after kWaitLimitNs.
    const bool landed = (stall_test && u == u0) ? mbar_wait(never_bar, 0)
                                                 : mbar_wait(bar0 + 8 * slot, parity);
    if (!__all_sync(0xffffffffu, landed)) {
      ok = false;
      break;
    }
    uint32_t r[36];
    const uint32_t src = slots + slot * kSlotBytes + lane * kSuperBytes;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint4 v = lds128(src + 16 * i);
      r[4 * i + 0] = v.x;
      r[4 * i + 1] = v.y;
      r[4 * i + 2] = v.z;
      r[4 * i + 3] = v.w;
    }
    __syncwarp();
    fence_proxy_async_smem();
    if (issued < u1) issue(issued++);

    const int64_t g = u / p.nsb, sb = u - g * p.nsb;
    const float* xrun = p.x + sb * kSuperElems;
    block_fma<0, M>(r, xrun, p.ldx, y2);
    block_fma<1, M>(r, xrun, p.ldx, y2);
    block_fma<2, M>(r, xrun, p.ldx, y2);
    block_fma<3, M>(r, xrun, p.ldx, y2);
    block_fma<4, M>(r, xrun, p.ldx, y2);
    block_fma<5, M>(r, xrun, p.ldx, y2);
    block_fma<6, M>(r, xrun, p.ldx, y2);
    block_fma<7, M>(r, xrun, p.ldx, y2);

    if (sb == p.nsb - 1 || u == u1 - 1) {
      // Row group g is done for this warp: finish it or hand in a partial.
      const int64_t row = g * 32 + lane;
      const int64_t gu0 = g * p.nsb, gu1 = gu0 + p.nsb;
      float v[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const f2 t = unpack2(y2[m]);
        v[m] = t.x + t.y;
        y2[m] = 0;
      }
      if (gu0 >= u0 && gu1 <= u1) {
        if (row < p.n) {
#pragma unroll
          for (int m = 0; m < M; ++m) p.y[m * p.ldy + row] = v[m];
        }
      } else {
        const int slot_id = g == g_first ? 0 : 1;
        float* mine = p.partials + ((wid * 2 + slot_id) * M) * 32;
#pragma unroll
        for (int m = 0; m < M; ++m) __stcg(mine + m * 32 + lane, v[m]);
        __threadfence();
        __syncwarp();
        const int64_t i0 = owner_of(gu0, p.units, p.warps);
        const int64_t i1 = owner_of(gu1 - 1, p.units, p.warps);
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.counters[g], 1) == static_cast<int>(i1 - i0);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          float s[M];
#pragma unroll
          for (int m = 0; m < M; ++m) s[m] = 0.f;
          for (int64_t i = i0; i <= i1; ++i) {
            const int64_t gi_first = (p.units * i / p.warps) / p.nsb;
            const int sid = g == gi_first ? 0 : 1;
            float* part = p.partials + ((i * 2 + sid) * M) * 32;
#pragma unroll
            for (int m = 0; m < M; ++m) {
              s[m] += __ldcg(part + m * 32 + lane);
              __stcg(part + m * 32 + lane, 0.f);  // the workspace goes back to all-zero
            }
          }
          if (row < p.n) {
#pragma unroll
            for (int m = 0; m < M; ++m) p.y[m * p.ldy + row] = s[m];
          }
          if (lane == 0) p.counters[g] = 0;
        }
      }
    }
  }

  if (!ok) {
    if (lane == 0) report(p.status, 6 /* Q4_ERR_TIMEOUT */);
    // Let every copy this warp still has in flight (unit u's included) land
    // before the CTA exits; each of these waits is bounded too.
    for (int64_t v = u; v < issued; ++v) {
      const int slot = static_cast<int>((v - u0) % kStages);
      const uint32_t parity = static_cast<uint32_t>(((v - u0) / kStages) & 1);
      mbar_wait(bar0 + 8 * slot, parity);
    }
  }
}

constexpr int kCtasPerSm = 2;

template <int M>
cudaError_t launch_stream(const StreamParams& sp, int64_t grid, bool pdl, cudaStream_t s) {
  CUtensorMap tmap;
  if (!encode_tmap_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, sp.W,
                      static_cast<uint64_t>(sp.rowbytes), static_cast<uint64_t>(sp.n),
                      static_cast<uint64_t>(sp.rowbytes), kSuperBytes, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<M>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<M>, tmap, sp);
}

template <int M>
cudaError_t launch_generic(const uint8_t* W, int64_t n, int64_t nb, const float* x, int64_t ldx,
                           float* y, int64_t ldy, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_generic_kernel<M>, W, n, nb, x, ldx, y, ldy);
}

template <int M>
cudaError_t dispatch(const GemvPlan& plan, const uint8_t* W, int64_t n, int64_t k, const float* x,
                     int64_t ldx, float* y, int64_t ldy, void* ws, int32_t* status,
                     uint32_t flags, bool pdl, cudaStream_t s) {
  if (!plan.fast) return launch_generic<M>(W, n, k / 32, x, ldx, y, ldy, pdl, s);
  StreamParams sp;
  sp.W = W;
  sp.n = n;
  sp.nsb = k / kSuperElems;
  sp.rowbytes = k / 32 * kBlockBytes;
  sp.x = x;
  sp.ldx = ldx;
  sp.y = y;
  sp.ldy = ldy;
  sp.counters = static_cast<int32_t*>(ws);
  const size_t cnt_bytes = (static_cast<size_t>(plan.groups) * 4 + 255) / 256 * 256;
  sp.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cnt_bytes);
  sp.units = plan.units;
  sp.warps = plan.warps;
  sp.groups = plan.groups;
  sp.status = status;
  sp.flags = flags;
  return launch_stream<M>(sp, (plan.warps + kWarps - 1) / kWarps, pdl, s);
}

}  // namespace

GemvPlan gemv_plan(int64_t n, int64_t k, int64_t m) {
  GemvPlan p = {};
  p.fast = (k % kSuperElems) == 0;
  p.groups = (n + 31) / 32;
  if (!p.fast) return p;
  p.units = p.groups * (k / kSuperElems);
  p.b1 = (m == 1) && gemv_b1_supports(k);
  // 2..16 rows: launches of up to kMaxBatchRows rows of the batched tile
  // kernel (a single leftover row goes to the batch-1 kernel)
  p.bm = (m >= 2) && gemv_bm_supports(k, 2) && gemv_b1_supports(k);
  const int64_t target = static_cast<int64_t>(sm_count()) * kCtasPerSm * kWarps;
  p.warps = p.b1 ? gemv_b1_warps(p.units) : (p.units < target ? p.units : target);
  const size_t cnt_bytes = (static_cast<size_t>(p.groups) * 4 + 255) / 256 * 256;
  size_t part = static_cast<size_t>(p.warps) * 2 * static_cast<size_t>(m) * 32 * 4;
  if (p.bm) {  // [warps][rows of the launch][32] tagged words of 8 bytes
    part = std::max(part, static_cast<size_t>(gemv_bm_warps(p.units)) * kMaxBatchRows * 32 * 8);
    part = std::max(part, static_cast<size_t>(gemv_b1_warps(p.units)) * 32 * 8);
  }
  p.ws_bytes = cnt_bytes + part;
  return p;
}

cudaError_t gemv_launch(const GemvPlan& plan, const uint8_t* W, int64_t n, int64_t k,
                        const float* x, int64_t m, int64_t ldx, float* y, int64_t ldy,
                        void* workspace, int32_t* status, uint32_t flags, cudaStream_t s,
                        const void* pf, uint64_t pf_bytes) {
  const bool pdl = (flags & 1u) != 0;
  if (plan.fast && plan.b1 && m == 1) {
    const size_t cnt_bytes = (static_cast<size_t>(plan.groups) * 4 + 255) / 256 * 256;
    return gemv_b1_launch(W, n, k, x, y, static_cast<int32_t*>(workspace),
                          reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + cnt_bytes),
                          plan.units, plan.warps, status, flags, s, pf, pf_bytes);
  }
  if (plan.fast && plan.bm && m >= 2) {
    // Launches of up to kMaxBatchRows rows (fewer where x would not fit in
    // shared memory), in order on the stream; each leaves the workspace zero
    // for the next, and under PDL a launch touches it only after the wait.
    const size_t cnt_bytes = (static_cast<size_t>(plan.groups) * 4 + 255) / 256 * 256;
    int32_t* counters = static_cast<int32_t*>(workspace);
    float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + cnt_bytes);
    for (int64_t r0 = 0; r0 < m;) {
      const int64_t rem = m - r0;
      cudaError_t e;
      int64_t c = 1;
      if (rem == 1) {
        e = gemv_b1_launch(W, n, k, x + r0 * ldx, y + r0 * ldy, counters, partials, plan.units,
                           gemv_b1_warps(plan.units), status, flags, s);
      } else {
        c = std::min(rem, kMaxBatchRows);
        while (c > 2 && !gemv_bm_supports(k, c)) --c;
        e = gemv_bm_launch(W, n, k, x + r0 * ldx, c, ldx, y + r0 * ldy, ldy, counters, partials,
                           plan.units, status, flags, s);
      }
      if (e != cudaSuccess) return e;
      r0 += c;
    }
    return cudaSuccess;
  }
  switch (m) {
#define Q4_GEMV_CASE(MM) \
  case MM:               \
    return dispatch<MM>(plan, W, n, k, x, ldx, y, ldy, workspace, status, flags, pdl, s);
    Q4_GEMV_CASE(1)
    Q4_GEMV_CASE(2)
    Q4_GEMV_CASE(3)
    Q4_GEMV_CASE(4)
    Q4_GEMV_CASE(5)
    Q4_GEMV_CASE(6)
    Q4_GEMV_CASE(7)
    Q4_GEMV_CASE(8)
#undef Q4_GEMV_CASE
    default:
      break;
  }
  // 9..16: two passes of up to 8 rows of x each
  const int64_t m0 = 8;
  cudaError_t e = gemv_launch(plan, W, n, k, x, m0, ldx, y, ldy, workspace, status, flags, s);
  if (e != cudaSuccess) return e;
  return gemv_launch(plan, W, n, k, x + m0 * ldx, m - m0, ldx, y + m0 * ldy, ldy, workspace,
                     status, flags, s);
}

}  // namespace q4
