// q4_gemm.cu -- Q4_0 dequant -> bf16 tensor-core GEMM for the audio encoder and
// prefill:  Y[t][r] = sum_j bf16((q[r][j] - 8) * d[r][j/32]) * X[t][j]  (fp32 acc).
//
// The encoder of the Voxtral Mini 4B Realtime port is 32 layers of 1280-wide
// linears run over every audio frame (GeekNews, es.news.hada.io/topic?id=26595,
// "Arquitectura"), so with hundreds to thousands of frames the product is a
// dense contraction and belongs on the tcgen05 tensor cores.
//
// Persistent kernel, one CTA per SM, each CTA looping over output tiles of
// 128 weight rows (MMA M) x BN tokens (MMA N, a multiple of 32 up to 224,
// picked per shape so that the tiles fill the SMs in whole waves):
//   warp 0     TMA producer: packed Q4 rows (2-D map over the bytes, box
//              144 B x 128 rows = 256 weights per row) and bf16 X tiles (box
//              64 x BN, 128-byte swizzle, two per barrier), each into a ring of
//              mbarrier-guarded shared-memory stages.
//   warp 1     allocates all 512 TMEM columns and issues tcgen05.mma
//              (kind::f16: A = the dequantized weights, read from TMEM; B = the
//              X tile, read from shared memory; fp32 accumulator in TMEM) from
//              one thread; tcgen05.commit releases the stages.
//   warps 2-9  dequantize: thread t of a warp in TMEM lane quarter q decodes row
//              32q + t to exact fp32 (q - 8) * d, rounds to bf16 and writes the
//              64 weights of a k-step to its TMEM lane with one tcgen05.st.
//              Warps 2-5 produce the even k-steps, warps 6-9 the odd ones, into
//              two TMEM A stages.
//   warps 10-13  epilogue: tcgen05.ld of the finished accumulator, fp32 or bf16
//              stores (consecutive rows per warp store).
// Keeping A in TMEM leaves shared memory to the X operand only, whose traffic
// (64 tokens-bytes in, the same out per 64 k) is what bounds a 128-row MMA.
// Two accumulators (columns [0, 224) and [224, 448)) let the epilogue of one
// tile overlap the main loop of the next; the A stages sit at columns 448 and
// 480.  Every wait is bounded; on expiry the CTA reports Q4_ERR_TIMEOUT, lets
// its copies and MMAs drain, frees TMEM and exits.
#include <type_traits>

#include "q4_device.cuh"

namespace q4 {
namespace {

constexpr int kThreads = 14 * 32;
constexpr int kTileRows = 128;  // weight rows per tile (MMA M)
constexpr int kKStep = 64;      // weights per k-step (128 B of bf16 per row)
constexpr int kStagesW = 2;
constexpr int kPackedStageBytes = kTileRows * kSuperBytes;  // 18432
constexpr int kMaxBN = 224;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulator b at acc_col(b), A stage p at a_col(p).
__host__ __device__ constexpr uint32_t acc_col(int b) { return static_cast<uint32_t>(b) * 224u; }
__host__ __device__ constexpr uint32_t a_col(int p) { return 448u + 32u * static_cast<uint32_t>(p); }
constexpr int kAStages = 2;  // one 64-weight k-step (32 columns) each
constexpr int kMaxXStages = 8;
constexpr int kSmemBudget = 226 * 1024;
constexpr int kBarBytes = 1024;  // barriers and flags, after the rings

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
// D (TMEM) [+]= A (TMEM) x B (shared-memory descriptor)
__device__ __forceinline__ void umma_ts_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
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

// Weights (q-8)*d of a pair, exact in fp32, rounded to bf16 and packed.
template <int PA, int PB>
__device__ __forceinline__ uint32_t wq_bf16x2(uint32_t wa, uint32_t wb, const DecodeConsts& c,
                                              unsigned long long d2) {
  const f2 w = unpack2(fmul2(qm8<PA, PB>(wa, wb, c), d2));
  return bf16x2_rn(w.x, w.y);
}

// Decodes block BLK (0..7) of a 144-byte run r[36] into 16 bf16x2 words:
// o[e/2] = (w[e], w[e+1]) for e even.  Byte c of qs holds element c (low
// nibble) and element c + 16 (high nibble).
template <int BLK>
__device__ __forceinline__ void decode_block_bf16(const uint32_t (&r)[36], const DecodeConsts& c,
                                                  uint32_t* o) {
  constexpr int ob = 18 * BLK;  // byte offset of the block in the run
  constexpr int wd = ob / 4;
  constexpr bool d_high = ((ob / 2) & 1) != 0;
  const float d = half_bits_to_float(d_high ? (r[wd] >> 16) : r[wd]);
  const unsigned long long d2 = pack2(d, d);
  if constexpr ((BLK & 1) == 1) {
    // qs starts 4-byte aligned: word i holds qs[4i .. 4i+3]
    constexpr int w0 = (ob + 2) / 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = r[w0 + i], t = shr12(w);
      o[2 * i] = wq_bf16x2<0, 8>(w, w, c, d2);           // elements 4i, 4i+1
      o[2 * i + 1] = wq_bf16x2<16, 12>(w, t, c, d2);     // 4i+2, 4i+3
      o[8 + 2 * i] = wq_bf16x2<4, 12>(w, w, c, d2);      // 4i+16, 4i+17
      o[8 + 2 * i + 1] = wq_bf16x2<8, 16>(t, t, c, d2);  // 4i+18, 4i+19
    }
  } else {
    // qs starts 2 bytes into a word: qs[0..1] in the high half of word ob/4,
    // qs[2..13] in the next three words, qs[14..15] in the low half after them
    constexpr int w0 = ob / 4;
    {
      const uint32_t w = r[w0], t = shr12(w);
      o[0] = wq_bf16x2<16, 12>(w, t, c, d2);  // elements 0, 1
      o[8] = wq_bf16x2<8, 16>(t, t, c, d2);   // 16, 17
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint32_t w = r[w0 + 1 + i], t = shr12(w);  // qs[2+4i .. 5+4i]
      o[1 + 2 * i] = wq_bf16x2<0, 8>(w, w, c, d2);     // 2+4i, 3+4i
      o[2 + 2 * i] = wq_bf16x2<16, 12>(w, t, c, d2);   // 4+4i, 5+4i
      o[9 + 2 * i] = wq_bf16x2<4, 12>(w, w, c, d2);    // 18+4i, 19+4i
      o[10 + 2 * i] = wq_bf16x2<8, 16>(t, t, c, d2);   // 20+4i, 21+4i
    }
    {
      const uint32_t w = r[w0 + 4];
      o[7] = wq_bf16x2<0, 8>(w, w, c, d2);   // 14, 15
      o[15] = wq_bf16x2<4, 12>(w, w, c, d2); // 30, 31
    }
  }
}

struct GemmArgs {
  int64_t n, k, m, ldy;
  void* y;
  int32_t* status;
  int y_bf16;
  int bn;         // tokens per tile (multiple of 32, <= kMaxBN)
  int n_tiles;    // tiles along the weight rows
  int tiles;      // n_tiles x token tiles
  int x_stages;   // X ring depth
  int splits;     // K-splits per tile (work items = tiles x splits)
  int32_t* counters;  // [tiles] arrivals per tile (splits > 1), zero between calls
  float* partials;    // [splits][m][n] fp32 (splits > 1)
};

// Work item w: tile w / splits, K-split w % splits, which covers 256-wide
// weight stages [j0, j1).
struct Item {
  int tile, split, j0, j1;
};
__device__ __forceinline__ Item item_of(int w, int splits, int wstages) {
  Item it;
  it.tile = w / splits;
  it.split = w - it.tile * splits;
  it.j0 = wstages * it.split / splits;
  it.j1 = wstages * (it.split + 1) / splits;
  return it;
}

struct Bars {
  uint32_t w_full, w_empty, x_full, x_empty, a_full, a_empty, acc_full, acc_empty, drain;
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int nx = args.x_stages;
  // X tiles move in pairs (two 64-wide k-steps, one full and one empty
  // barrier per pair): the MMA thread waits for X and releases it once per two
  // k-steps.
  const int nxp = nx / 2;
  const uint32_t x_tile_bytes = static_cast<uint32_t>(args.bn) * 128u;
  const uint32_t xs = base;                                    // X ring
  const uint32_t wsm = xs + static_cast<uint32_t>(nx) * x_tile_bytes;  // packed W ring
  const uint32_t bar_base = wsm + kStagesW * kPackedStageBytes;
  Bars B;
  B.w_full = bar_base;
  B.w_empty = B.w_full + 8 * kStagesW;
  B.x_full = B.w_empty + 8 * kStagesW;
  B.x_empty = B.x_full + 8 * kMaxXStages;
  B.a_full = B.x_empty + 8 * kMaxXStages;
  B.a_empty = B.a_full + 8 * kAStages;
  B.acc_full = B.a_empty + 8 * kAStages;
  B.acc_empty = B.acc_full + 16;
  B.drain = B.acc_empty + 16;
  const uint32_t misc = B.drain + 8;  // tmem slot, abort flag, last-split flag
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + (misc - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (misc - base) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = static_cast<int>(args.k / kKStep);
  const int wstages = ksteps / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesW; ++s) {
      mbar_init(B.w_full + 8 * s, 1);
      mbar_init(B.w_empty + 8 * s, 8);
    }
    for (int s = 0; s < nx; ++s) {
      mbar_init(B.x_full + 8 * s, 1);
      mbar_init(B.x_empty + 8 * s, 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(B.a_full + 8 * s, 4);
      mbar_init(B.a_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(B.acc_full + 8 * s, 1);
      mbar_init(B.acc_empty + 8 * s, 4);
    }
    mbar_init(B.drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(misc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int cta = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);

  pdl_allow_dependents();
  pdl_wait_prior_grid();

  auto fail = [&]() {
    if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) report(args.status, 6);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      // X ring slot and phase as running counters: a division by the runtime
      // ring depth per k-step sits on this thread's critical path.
      int wj = 0, xk = 0, xslot = 0;
      uint32_t xph = 0;
      bool ok = true;
      for (int w = cta; w < args.tiles * args.splits && ok; w += ncta) {
        const Item it = item_of(w, args.splits, wstages);
        const int32_t n0 = (it.tile % args.n_tiles) * kTileRows;
        const int32_t m0 = (it.tile / args.n_tiles) * args.bn;
        for (int j = it.j0; j < it.j1 && ok; ++j) {
          const int s = wj % kStagesW;
          if (!mbar_wait(B.w_empty + 8 * s, ((wj / kStagesW) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B.w_full + 8 * s, kPackedStageBytes);
          tma_load_2d(wsm + s * kPackedStageBytes, &tmap_w, j * kSuperBytes, n0, B.w_full + 8 * s);
          ++wj;
          for (int pp = 0; pp < 2; ++pp) {
            if (!mbar_wait(B.x_empty + 8 * xslot, xph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(B.x_full + 8 * xslot, 2 * x_tile_bytes);
            const uint32_t dst = xs + static_cast<uint32_t>(xslot) * 2u * x_tile_bytes;
            tma_load_2d(dst, &tmap_x, (4 * j + 2 * pp) * kKStep, m0, B.x_full + 8 * xslot);
            tma_load_2d(dst + x_tile_bytes, &tmap_x, (4 * j + 2 * pp + 1) * kKStep, m0,
                        B.x_full + 8 * xslot);
            xk += 2;
            if (++xslot == nxp) {
              xslot = 0;
              xph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        fail();
        // let the copies still in flight land before the CTA can exit
        for (int i = wj - kStagesW > 0 ? wj - kStagesW : 0; i < wj; ++i)
          mbar_wait(B.w_full + 8 * (i % kStagesW), (i / kStagesW) & 1);
        for (int i = xk / 2 - nxp > 0 ? xk / 2 - nxp : 0; i < xk / 2; ++i)
          mbar_wait(B.x_full + 8 * (i % nxp), (i / nxp) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      // This one thread paces the tensor pipe: its per-k-step work is kept to
      // waits, MMAs and commits (ring slots and phases as running counters,
      // the X descriptor advanced by adding a stage's address units), and the
      // loop takes the two k-steps of an X pair (A stages 0 and 1) together.
      const uint32_t idesc = idesc_bf16(kTileRows, args.bn);
      const uint64_t xdesc0 = sw128_desc(xs);
      const uint32_t xdesc_step = x_tile_bytes >> 4;  // descriptor address field in 16 B
      int iter = 0, xslot = 0;
      uint32_t xph = 0;  // phase of the X slot's next fill
      uint32_t aph = 0;  // bit p: phase of A stage p's next fill
      bool ok = true, any = false;
      for (int w = cta; w < args.tiles * args.splits && ok; w += ncta, ++iter) {
        const Item it = item_of(w, args.splits, wstages);
        const int b = iter & 1;
        if (!mbar_wait(B.acc_empty + 8 * b, ((iter >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem + acc_col(b);
        const int ks0 = 4 * it.j0, ks1 = 4 * it.j1;
        for (int ks = ks0; ks < ks1; ks += 2) {
          if (!mbar_wait(B.a_full, aph & 1u, abort_flag) ||
              !mbar_wait(B.x_full + 8 * xslot, xph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc =
              xdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(xslot) * 2u * xdesc_step);
#pragma unroll
          for (int kk = 0; kk < kKStep / 16; ++kk)
            umma_ts_bf16(d_acc, tmem + a_col(0) + 8 * kk, bdesc + 2 * kk, idesc,
                         (ks != ks0 || kk != 0) ? 1u : 0u);
          any = true;
          umma_commit(B.a_empty);
          if (!mbar_wait(B.a_full + 8, (aph >> 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKStep / 16; ++kk)
            umma_ts_bf16(d_acc, tmem + a_col(1) + 8 * kk, bdesc + xdesc_step + 2 * kk, idesc, 1u);
          umma_commit(B.x_empty + 8 * xslot);
          umma_commit(B.a_empty + 8);
          aph ^= 3u;
          if (++xslot == nxp) {
            xslot = 0;
            xph ^= 1u;
          }
        }
        if (ok) umma_commit(B.acc_full + 8 * b);
      }
      if (!ok) fail();
      if (any) {  // every MMA has finished with TMEM and shared memory before exit
        umma_commit(B.drain);
        mbar_wait(B.drain, 0);
      }
    }
  } else if (warp < 10) {
    // ---------------- dequantize into the TMEM A stages
    const int q = warp & 3;         // TMEM lane quarter
    const int p = (warp - 2) >> 2;  // 0: even k-steps, 1: odd k-steps
    const int row = 32 * q + lane;  // tile row = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const DecodeConsts dc = make_consts();
    int wj = 0, a_use = 0;  // a_use: productions into A stage p so far
    bool ok = true;
    for (int w = cta; w < args.tiles * args.splits && ok; w += ncta) {
      const Item it = item_of(w, args.splits, wstages);
      for (int j = it.j0; j < it.j1 && ok; ++j) {
        const int s = wj % kStagesW;
        const bool landed = mbar_wait(B.w_full + 8 * s, (wj / kStagesW) & 1, abort_flag);
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
        if (lane == 0) mbar_arrive(B.w_empty + 8 * s);
        ++wj;
        // k-steps 4j + p and 4j + p + 2 (blocks 2p, 2p + 1 and 2p + 4, 2p + 5 of
        // the run) go to A stage p
        // The k-step is decoded before waiting for its A stage, so that only
        // the TMEM store sits between the MMA that frees the stage and the
        // MMA that reads it next.
        auto one_kstep = [&](auto kk_tag) -> bool {
          constexpr int KK = decltype(kk_tag)::value;
          uint32_t o[32];
          decode_block_bf16<2 * KK>(r, dc, o);
          decode_block_bf16<2 * KK + 1>(r, dc, o + 16);
          const bool free_stage = mbar_wait(B.a_empty + 8 * p, (a_use & 1) ^ 1, abort_flag);
          if (!__all_sync(0xffffffffu, free_stage)) return false;
          tc_fence_after();
          tmem_st32(lane_addr + a_col(p), o);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(B.a_full + 8 * p);
          ++a_use;
          return true;
        };
        if (p == 0)
          ok = one_kstep(std::integral_constant<int, 0>{}) &&
               one_kstep(std::integral_constant<int, 2>{});
        else
          ok = one_kstep(std::integral_constant<int, 1>{}) &&
               one_kstep(std::integral_constant<int, 3>{});
      }
    }
    if (!ok) fail();
  } else {
    // ---------------- epilogue
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int iter = 0;
    bool ok = true;
    volatile int* last_flag = abort_flag + 1;  // set by the epilogue's counter thread
    for (int w = cta; w < args.tiles * args.splits && ok; w += ncta, ++iter) {
      const Item it = item_of(w, args.splits, wstages);
      const int t = it.tile;
      const int b = iter & 1;
      const int64_t n0 = static_cast<int64_t>(t % args.n_tiles) * kTileRows;
      const int64_t m0 = static_cast<int64_t>(t / args.n_tiles) * args.bn;
      const bool done = mbar_wait(B.acc_full + 8 * b, (iter >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, done)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t grow = n0 + 32 * q + lane;
      const bool split = args.splits > 1;
      // 4-byte stores of bf16 pairs need an even row stride and a 4-byte base
      const bool pair_stores =
          (reinterpret_cast<uintptr_t>(args.y) & 3u) == 0 && (args.ldy & 1) == 0;
#pragma unroll 1
      for (int c0 = 0; c0 < args.bn; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + acc_col(b) + c0, v);
        tmem_ld_wait();
        if (c0 + 32 >= args.bn) {  // the accumulator can be reused once it is read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(B.acc_empty + 8 * b);
        }
        const int64_t tleft = args.m - (m0 + c0);
        const int cnt = tleft < 32 ? static_cast<int>(tleft) : 32;
        if (!split && args.y_bf16 && pair_stores) {
          // bf16 Y: lanes 2i and 2i + 1 (rows r0, r0 + 1) swap one value per
          // token pair, so each lane stores one 4-byte bf16 pair: the even
          // lane rows (r0, r0 + 1) of token j, the odd lane those of token
          // j + 1.  Warp-uniform branch: every lane takes part in the shuffle.
          const bool odd = (lane & 1) != 0;
          const int64_t r0 = grow - (odd ? 1 : 0);
          __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(args.y);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float own_j = __uint_as_float(v[j]), own_j1 = __uint_as_float(v[j + 1]);
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? own_j : own_j1, 1);
            const int tj = odd ? j + 1 : j;
            if (tj < cnt && r0 < args.n) {
              const float lo = odd ? recv : own_j;   // row r0
              const float hi = odd ? own_j1 : recv;  // row r0 + 1
              __nv_bfloat16* p = yb + (m0 + c0 + tj) * args.ldy + r0;
              if (r0 + 1 < args.n)
                *reinterpret_cast<uint32_t*>(p) = bf16x2_rn(lo, hi);
              else
                *p = __float2bfloat16_rn(lo);
            }
          }
        } else if (grow < args.n) {
          if (split) {  // this K-split's partial tile, fp32
            float* pp = args.partials + (static_cast<int64_t>(it.split) * args.m + m0 + c0) *
                                            args.n + grow;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < cnt) __stcg(pp + j * args.n, __uint_as_float(v[j]));
          } else if (args.y_bf16) {
            __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(args.y) + (m0 + c0) * args.ldy + grow;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < cnt) yp[j * args.ldy] = __float2bfloat16_rn(__uint_as_float(v[j]));
          } else {
            float* yp = static_cast<float*>(args.y) + (m0 + c0) * args.ldy + grow;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < cnt) yp[j * args.ldy] = __uint_as_float(v[j]);
          }
        }
      }
      if (split) {
        // The last K-split of the tile to arrive adds the partials in split
        // order (deterministic), writes Y and puts the counter back to zero.
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the 4 epilogue warps
        if (warp == 10 && lane == 0) {
          __threadfence();
          const int old = atomicAdd(args.counters + t, 1);
          *last_flag = old == args.splits - 1;
          if (old == args.splits - 1) args.counters[t] = 0;
          __threadfence();
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*last_flag && grow < args.n) {
          const int64_t tleft = args.m - m0;
          const int cnt = tleft < args.bn ? static_cast<int>(tleft) : args.bn;
          const int64_t split_stride = args.m * args.n;
          // 16 tokens x 2 splits = 32 independent loads in flight per pass; the
          // partials are still added in split order (deterministic)
          constexpr int kT = 16;
          for (int c = 0; c < cnt; c += kT) {
            float acc[kT];
#pragma unroll
            for (int u = 0; u < kT; ++u) acc[u] = 0.f;
            const float* pp = args.partials + (m0 + c) * args.n + grow;
            for (int sp = 0; sp < args.splits; sp += 2) {
              const bool two = sp + 1 < args.splits;
              float v0[kT], v1[kT];
#pragma unroll
              for (int u = 0; u < kT; ++u) {
                v0[u] = c + u < cnt ? __ldcg(pp + sp * split_stride + u * args.n) : 0.f;
                v1[u] = (two && c + u < cnt) ? __ldcg(pp + (sp + 1) * split_stride + u * args.n)
                                              : 0.f;
              }
#pragma unroll
              for (int u = 0; u < kT; ++u) {
                acc[u] += v0[u];
                if (two) acc[u] += v1[u];
              }
            }
            // the workspace goes back to all-zero, as every call leaves it
            for (int sp = 0; sp < args.splits; ++sp) {
#pragma unroll
              for (int u = 0; u < kT; ++u)
                if (c + u < cnt) __stcg(const_cast<float*>(pp) + sp * split_stride + u * args.n, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kT; ++u) {
              if (c + u >= cnt) break;
              const int64_t tok = m0 + c + u;
              if (args.y_bf16)
                static_cast<__nv_bfloat16*>(args.y)[tok * args.ldy + grow] =
                    __float2bfloat16_rn(acc[u]);
              else
                static_cast<float*>(args.y)[tok * args.ldy + grow] = acc[u];
            }
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // last_flag is reused next item
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ host side

// X ring depth in 64-wide tiles: an even number (the tiles move in pairs), at
// least 6 for every BN <= 224.
int x_stages_for(int bn) {
  const int avail = kSmemBudget - 1024 /* alignment */ - kStagesW * kPackedStageBytes - kBarBytes;
  int s = avail / (bn * 128);
  s = s > kMaxXStages ? kMaxXStages : s;
  return s & ~1;
}

}  // namespace

GemmPlan gemm_plan(int64_t n, int64_t k, int64_t m) {
  GemmPlan p = {};
  p.n_tiles = (n + kTileRows - 1) / kTileRows;
  const int64_t g = sm_count();
  // Pick the token-tile width that finishes in the fewest tile-widths of time:
  // each tile costs about max(BN, 80) + 32 token-columns (the dequantization
  // of 128 x K weights bounds narrow tiles; 32 covers the per-tile overhead),
  // and tiles run in waves of one per SM.
  int64_t best_cost = -1;
  for (int bn = 32; bn <= kMaxBN; bn += 32) {
    const int64_t mt = (m + bn - 1) / bn;
    const int64_t tiles = p.n_tiles * mt;
    const int64_t waves = (tiles + g - 1) / g;
    const int64_t cost = waves * ((bn > 80 ? bn : 80) + 32);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      p.block_n = bn;
      p.m_tiles = mt;
    }
    if (bn >= m) break;
  }
  // Too few tiles for the SMs (small M): split K, in 256-weight stages, so that
  // tiles x splits fill about one wave; partial tiles are added in the epilogue.
  // The split is not free: partials out, a counter, the last split's
  // reduction and the clearing of the workspace, none of it overlapped.  For
  // 64-token tiles that costs ~9-10 us, the time of ~24 of the CTA's 64-wide
  // k-steps, and it grows with the tile width: split only when it removes more
  // than 24 * BN / 64 k-steps from every CTA (on B300: 1280 x 1280 at M = 375
  // runs in 13.9 us whole and 19.5 us split in two; 1280 x 5120 in 39.3 us
  // whole and 31.6 us split in two; at M = 8, 32-token tiles, 1280 x 1280 split
  // in five and 9216 x 3072 in two are faster than whole).
  p.splits = 1;
  const int64_t tiles = p.n_tiles * p.m_tiles, wstages = k / 256;
  if (tiles * 2 <= g) {
    int64_t sp = g / tiles;
    if (sp > wstages) sp = wstages;
    if (sp > 16) sp = 16;
    const int64_t ksteps = k / kKStep;
    if (sp > 1 && ksteps * (sp - 1) * 64 > 24 * p.block_n * sp) p.splits = sp;
  }
  p.ws_bytes = 0;
  if (p.splits > 1) {
    const size_t cnt = (static_cast<size_t>(tiles) * 4 + 255) / 256 * 256;
    p.ws_bytes = cnt + static_cast<size_t>(p.splits) * m * n * 4;
  }
  return p;
}

cudaError_t gemm_launch(const GemmPlan& plan, const uint8_t* W, int64_t n, int64_t k,
                        const void* X, int64_t m, int64_t ldx, void* Y, bool y_bf16,
                        int64_t ldy, void* workspace, int32_t* status, uint32_t flags,
                        cudaStream_t s) {
  const int64_t tiles = plan.n_tiles * plan.m_tiles;
  if (tiles > (int64_t(1) << 30)) return cudaErrorNotSupported;
  const int bn = plan.block_n;
  CUtensorMap tw, tx;
  if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, W,
                      static_cast<uint64_t>(k / 32 * kBlockBytes), static_cast<uint64_t>(n),
                      static_cast<uint64_t>(k / 32 * kBlockBytes), kSuperBytes, kTileRows,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(k),
                      static_cast<uint64_t>(m), static_cast<uint64_t>(ldx * 2), kKStep,
                      static_cast<uint32_t>(bn), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
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
  a.bn = bn;
  a.n_tiles = static_cast<int>(plan.n_tiles);
  a.tiles = static_cast<int>(tiles);
  a.x_stages = x_stages_for(bn);
  a.splits = static_cast<int>(plan.splits);
  a.counters = nullptr;
  a.partials = nullptr;
  if (plan.splits > 1) {
    const size_t cnt = (static_cast<size_t>(tiles) * 4 + 255) / 256 * 256;
    a.counters = static_cast<int32_t*>(workspace);
    a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + cnt);
  }
  const int64_t g = sm_count();
  cudaLaunchConfig_t cfg = {};
  const int64_t items = tiles * plan.splits;
  cfg.gridDim = dim3(static_cast<unsigned>(items < g ? items : g));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBudget;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (flags & 1u) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, tw, tx, a);
}

}  // namespace q4
