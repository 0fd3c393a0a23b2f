// q4_gemm.cu -- Q4_0 dequant -> bf16 tensor-core GEMM for the audio encoder and
// prefill:  Y[t][r] = sum_j bf16((q[r][j] - 8) * d[r][j/32]) * X[t][j]  (fp32 acc).
//
// The encoder of the Voxtral Mini 4B Realtime port is 32 layers of 1280-wide
// linears run over every audio frame (GeekNews, es.news.hada.io/topic?id=26595,
// "Arquitectura"), so with hundreds to thousands of frames the product is a
// dense contraction and belongs on the tcgen05 tensor cores.
//
// One CTA computes a 128 (weight rows) x BN (tokens) tile over the whole k:
//   warp 0   TMA producer: packed Q4 rows (2-D map over the bytes, box 144 B x
//            128 rows = 256 weights per row) and bf16 X tiles (box 64 x BN,
//            128-byte swizzle), each into a ring guarded by mbarriers.
//   warp 1   owns the tensor memory and issues tcgen05.mma (kind::f16, bf16 in,
//            fp32 accumulate in TMEM) from one thread; tcgen05.commit releases
//            the ring slots.
//   warps 2-5  dequantize: thread t decodes row t of the packed tile to exact
//            fp32 (q - 8) * d, rounds to bf16 and writes the K-major 128-byte-
//            swizzled operand layout the MMA descriptor expects; then they run
//            the epilogue (tcgen05.ld 32x32b, fp32 or bf16 stores).
// The weight tile is the MMA's M side (128 rows) and the tokens its N side, so
// one dequantization serves BN tokens.  Every wait is bounded; on expiry the
// CTA reports Q4_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include "q4_device.cuh"

namespace q4 {
namespace {

constexpr int kThreads = 192;
constexpr int kTileRows = 128;       // weight rows per tile (MMA M)
constexpr int kKStep = 64;           // weights per MMA stage (128 B of bf16 per row)
constexpr int kStagesX = 4;
constexpr int kStagesA = 3;
constexpr int kStagesW = 2;
constexpr int kPackedStageBytes = kTileRows * kSuperBytes;  // 18432
constexpr int kATileBytes = kTileRows * 128;                // 16384

template <int BN>
struct Smem {
  static constexpr int kXTileBytes = BN * 128;
  static constexpr int kX = 0;
  static constexpr int kA = kX + kStagesX * kXTileBytes;
  static constexpr int kW = kA + kStagesA * kATileBytes;
  static constexpr int kBars = kW + kStagesW * kPackedStageBytes;
  // barriers: x_full, x_empty, a_full, a_empty, w_full, w_empty, d_full, drain
  static constexpr int kNumBars = 2 * kStagesX + 2 * kStagesA + 2 * kStagesW + 2;
  static constexpr int kMisc = kBars + 8 * kNumBars;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared-memory matrix descriptor (tcgen05): K-major, 128-byte swizzle, 8-row
// core groups 1024 B apart.  start = byte address >> 4 (bits 0-13), leading
// byte offset field 1 (unused for swizzled K-major), stride byte offset 1024 B
// >> 4 (bits 32-45), fixed 0b001 at bits 46-48, swizzle mode 2 at bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits
// 7-9 and 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ------------------------------------------------------------ dequant helpers

template <int PA, int PB>
__device__ __forceinline__ uint32_t wq_bf16x2(uint32_t wa, uint32_t wb, float d) {
  // exact (q - 8) for the two nibbles, times d (exact in fp32), rounded to bf16
  const unsigned long long qm8 =
      fsub2(pack2(nibble_magic<PA>(wa), nibble_magic<PB>(wb)),
            pack2(NibbleMagic<PA>::kBias, NibbleMagic<PB>::kBias));
  const f2 w = unpack2(fmul2(qm8, pack2(d, d)));
  return bf16x2_rn(w.x, w.y);
}

// Decodes block BLK (0..7) of a 144-byte run r[36] into 16 bf16x2 words:
// out[e/2] = (w[e], w[e+1]) for e even.
template <int BLK>
__device__ __forceinline__ void decode_block_bf16(const uint32_t (&r)[36], uint32_t (&o)[16]) {
  constexpr int ob = 18 * BLK;
  constexpr int wd = ob / 4;
  constexpr bool d_high = ((ob / 2) & 1) != 0;
  const float d = half_bits_to_float(d_high ? (r[wd] >> 16) : r[wd]);
  if constexpr ((BLK & 1) == 1) {
    constexpr int w0 = (ob + 2) / 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = r[w0 + i], t = w >> 12;
      o[2 * i] = wq_bf16x2<0, 8>(w, w, d);
      o[2 * i + 1] = wq_bf16x2<16, 12>(w, t, d);
      o[8 + 2 * i] = wq_bf16x2<4, 12>(w, w, d);
      o[8 + 2 * i + 1] = wq_bf16x2<8, 16>(t, t, d);
    }
  } else {
    constexpr int w0 = ob / 4;
    {
      const uint32_t w = r[w0], t = w >> 12;
      o[0] = wq_bf16x2<16, 12>(w, t, d);
      o[8] = wq_bf16x2<8, 16>(t, t, d);
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint32_t w = r[w0 + 1 + i], t = w >> 12;
      o[1 + 2 * i] = wq_bf16x2<0, 8>(w, w, d);
      o[2 + 2 * i] = wq_bf16x2<16, 12>(w, t, d);
      o[9 + 2 * i] = wq_bf16x2<4, 12>(w, w, d);
      o[10 + 2 * i] = wq_bf16x2<8, 16>(t, t, d);
    }
    {
      const uint32_t w = r[w0 + 4];
      o[7] = wq_bf16x2<0, 8>(w, w, d);
      o[15] = wq_bf16x2<4, 12>(w, w, d);
    }
  }
}

// Writes the 64 weights (blocks B0, B0+1 of the run) of row `row` into an A
// tile: 8 chunks of 16 B, chunk c at row*128 + ((c ^ (row & 7)) * 16).
template <int B0>
__device__ __forceinline__ void write_a_kstep(const uint32_t (&r)[36], uint32_t a_tile, int row) {
  uint32_t o0[16], o1[16];
  decode_block_bf16<B0>(r, o0);
  decode_block_bf16<B0 + 1>(r, o1);
  const uint32_t base = a_tile + row * 128;
  const int sw = row & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    sts128(base + ((c ^ sw) << 4), o0[4 * c], o0[4 * c + 1], o0[4 * c + 2], o0[4 * c + 3]);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    sts128(base + (((c + 4) ^ sw) << 4), o1[4 * c], o1[4 * c + 1], o1[4 * c + 2], o1[4 * c + 3]);
}

struct GemmArgs {
  int64_t n, k, m, ldy;
  void* y;
  int32_t* status;
  int y_bf16;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
  using L = Smem<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t xs = base + L::kX, as = base + L::kA, wsm = base + L::kW;
  const uint32_t bars = base + L::kBars;
  const uint32_t x_full = bars, x_empty = x_full + 8 * kStagesX;
  const uint32_t a_full = x_empty + 8 * kStagesX, a_empty = a_full + 8 * kStagesA;
  const uint32_t w_full = a_empty + 8 * kStagesA, w_empty = w_full + 8 * kStagesW;
  const uint32_t d_full = w_empty + 8 * kStagesW, drain = d_full + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTileRows;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BN;
  const int ksteps = static_cast<int>(args.k / kKStep);
  constexpr uint32_t kTmemCols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesX; ++s) {
      mbar_init(x_full + 8 * s, 1);
      mbar_init(x_empty + 8 * s, 1);
    }
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(a_full + 8 * s, 4);
      mbar_init(a_empty + 8 * s, 1);
    }
    for (int s = 0; s < kStagesW; ++s) {
      mbar_init(w_full + 8 * s, 1);
      mbar_init(w_empty + 8 * s, 4);
    }
    mbar_init(d_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(base + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_allow_dependents();
  pdl_wait_prior_grid();

  auto fail = [&]() {
    if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) report(args.status, 6);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- producer
    int issued_x = 0, issued_w = 0;
    bool ok = true;
    for (int ks = 0; ks < ksteps && ok; ++ks) {
      if ((ks & 3) == 0) {
        const int j = ks >> 2, s = j % kStagesW;
        if (!mbar_wait(w_empty + 8 * s, ((j / kStagesW) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(w_full + 8 * s, kPackedStageBytes);
        tma_load_2d(wsm + s * kPackedStageBytes, &tmap_w, j * kSuperBytes,
                    static_cast<int32_t>(n0), w_full + 8 * s);
        ++issued_w;
      }
      const int s = ks % kStagesX;
      if (!mbar_wait(x_empty + 8 * s, ((ks / kStagesX) & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(x_full + 8 * s, L::kXTileBytes);
      tma_load_2d(xs + s * L::kXTileBytes, &tmap_x, ks * kKStep, static_cast<int32_t>(m0),
                  x_full + 8 * s);
      ++issued_x;
    }
    if (!ok) {
      fail();
      // let issued copies land before the CTA can exit
      for (int i = issued_x - kStagesX > 0 ? issued_x - kStagesX : 0; i < issued_x; ++i)
        mbar_wait(x_full + 8 * (i % kStagesX), (i / kStagesX) & 1);
      for (int i = issued_w - kStagesW > 0 ? issued_w - kStagesW : 0; i < issued_w; ++i)
        mbar_wait(w_full + 8 * (i % kStagesW), (i / kStagesW) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kTileRows, BN);
    bool ok = true, any = false;
    for (int ks = 0; ks < ksteps; ++ks) {
      const int sa = ks % kStagesA, sx = ks % kStagesX;
      if (!mbar_wait(a_full + 8 * sa, (ks / kStagesA) & 1, abort_flag) ||
          !mbar_wait(x_full + 8 * sx, (ks / kStagesX) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t adesc = sw128_desc(as + sa * kATileBytes);
      const uint64_t bdesc = sw128_desc(xs + sx * L::kXTileBytes);
#pragma unroll
      for (int kk = 0; kk < kKStep / 16; ++kk)
        umma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (ks | kk) != 0);
      any = true;
      umma_commit(x_empty + 8 * sx);
      umma_commit(a_empty + 8 * sa);
    }
    if (ok) {
      umma_commit(d_full);
    } else {
      fail();
    }
    if (any) {  // every MMA has finished reading shared memory before exit
      umma_commit(drain);
      mbar_wait(drain, 0);
    }
  } else if (warp >= 2) {
    // ---------------- dequantize, then epilogue
    const int row = threadIdx.x - 64;  // 0..127
    bool ok = true;
    for (int j = 0; j < ksteps / 4 && ok; ++j) {
      const int s = j % kStagesW;
      const bool landed = mbar_wait(w_full + 8 * s, (j / kStagesW) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform verdict
        ok = false;
        break;
      }
      uint32_t r[36];
      const uint32_t src = wsm + s * kPackedStageBytes + row * kSuperBytes;
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const uint4 v = lds128(src + 16 * i);
        r[4 * i + 0] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(w_empty + 8 * s);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int ks = 4 * j + kk, sa = ks % kStagesA;
        const bool free_slot = mbar_wait(a_empty + 8 * sa, ((ks / kStagesA) & 1) ^ 1, abort_flag);
        if (!__all_sync(0xffffffffu, free_slot)) {
          ok = false;
          break;
        }
        const uint32_t a_tile = as + sa * kATileBytes;
        if (kk == 0) write_a_kstep<0>(r, a_tile, row);
        if (kk == 1) write_a_kstep<2>(r, a_tile, row);
        if (kk == 2) write_a_kstep<4>(r, a_tile, row);
        if (kk == 3) write_a_kstep<6>(r, a_tile, row);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full + 8 * sa);
      }
    }
    if (!ok) fail();
    const bool done = ok && mbar_wait(d_full, 0, abort_flag);
    if (__all_sync(0xffffffffu, done)) {
      tc_fence_after();
      const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
      const int64_t grow = n0 + 32 * quarter + lane;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + c0, v);
        tmem_ld_wait();
        if (grow < args.n) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t t = m0 + c0 + j;
            if (t < args.m) {
              if (args.y_bf16)
                static_cast<__nv_bfloat16*>(args.y)[t * args.ldy + grow] =
                    __float2bfloat16_rn(__uint_as_float(v[j]));
              else
                static_cast<float*>(args.y)[t * args.ldy + grow] = __uint_as_float(v[j]);
            }
          }
        }
      }
    } else if (ok) {
      fail();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ host side

int pick_bn(int64_t m) {
  if (m <= 16) return 16;
  if (m <= 32) return 32;
  if (m <= 64) return 64;
  if (m <= 128) return 128;
  if (m <= 192) return 192;
  if (m <= 256) return 256;
  const int64_t t192 = (m + 191) / 192 * 192, t256 = (m + 255) / 256 * 256;
  return t192 < t256 ? 192 : 256;
}

template <int BN>
cudaError_t launch_bn(const uint8_t* W, int64_t n, int64_t k, const void* X, int64_t m,
                      int64_t ldx, void* Y, bool y_bf16, int64_t ldy, int32_t* status,
                      bool pdl, cudaStream_t s) {
  CUtensorMap tw, tx;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, W,
                      static_cast<uint64_t>(k / 32 * kBlockBytes), static_cast<uint64_t>(n),
                      static_cast<uint64_t>(k / 32 * kBlockBytes), kSuperBytes, kTileRows,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(k),
                      static_cast<uint64_t>(m), static_cast<uint64_t>(ldx * 2), kKStep,
                      static_cast<uint32_t>(BN), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Smem<BN>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  GemmArgs a;
  a.n = n;
  a.k = k;
  a.m = m;
  a.ldy = ldy;
  a.y = Y;
  a.status = status;
  a.y_bf16 = y_bf16 ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + kTileRows - 1) / kTileRows),
                     static_cast<unsigned>((m + BN - 1) / BN));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<BN>::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN>, tw, tx, a);
}

}  // namespace

GemmPlan gemm_plan(int64_t n, int64_t k, int64_t m) {
  GemmPlan p = {};
  p.block_n = pick_bn(m);
  p.n_tiles = (n + kTileRows - 1) / kTileRows;
  p.m_tiles = (m + p.block_n - 1) / p.block_n;
  p.splits = 1;
  p.ws_bytes = 0;
  (void)k;
  return p;
}

cudaError_t gemm_launch(const GemmPlan& plan, const uint8_t* W, int64_t n, int64_t k,
                        const void* X, int64_t m, int64_t ldx, void* Y, bool y_bf16,
                        int64_t ldy, void* workspace, int32_t* status, uint32_t flags,
                        cudaStream_t s) {
  (void)workspace;
  const bool pdl = (flags & 1u) != 0;
  if (plan.m_tiles > 65535) return cudaErrorNotSupported;
  switch (plan.block_n) {
    case 16: return launch_bn<16>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
    case 32: return launch_bn<32>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
    case 64: return launch_bn<64>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
    case 128: return launch_bn<128>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
    case 192: return launch_bn<192>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
    case 256: return launch_bn<256>(W, n, k, X, m, ldx, Y, y_bf16, ldy, status, pdl, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace q4
