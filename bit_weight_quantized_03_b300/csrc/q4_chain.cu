// q4_chain.cu -- the repacked Q4_0 layout (q4_repack) and the decode-step
// chain kernel behind q4_chain / q4_gemv_r.
//
// One decode step of the Voxtral Mini 4B Realtime port (GeekNews,
// es.news.hada.io/topic?id=26595, "Arquitectura": a 26-layer decoder, hidden
// 3072, GQA 32Q/8KV, GGUF Q4_0 weights) is a chain of batch-1 products, each
// reading the previous one's output: per layer qkv, wo (+ the residual), the
// gated FFN pair w1/w3 and w2 (+ the residual), and at the end the output head,
// whose largest logit is the next token.  Every product streams its weights
// from HBM once; the products are short (1-5 us of weight traffic each), so
// what a step costs beyond the weight traffic is the hand-off between
// products, of which there are 104 per step.
//
// Design (one cooperative launch, one 16-warp CTA per SM):
//   * Weights are read in the repacked 16-row x 256-column tiles
//     (q4r_tile.cuh) and multiplied on the tensor cores (mma.m16n8k16, f16
//     operands decoded exactly from the codes, fp32 accumulation).  Link s's
//     T tiles are cut into contiguous CTA ranges, each CTA range into 16
//     contiguous warp ranges.  Each warp streams its own tiles, two per bulk
//     copy, through a ring of two slots and runs ahead into later links while
//     it waits, so the weight stream does not stop at a hand-off.
//   * A warp sums its tiles' row products per 16-row group; at the end of a
//     link the CTA adds its warps' group sums in warp order and publishes one
//     partial per (group, CTA) into a slot of 16 floats in the workspace.  The
//     first owner of a group (the CTA holding its first tile) adds the
//     residual.  A group is split between at most a few CTAs.
//   * A link's input is read from the slots of the link that produced it: an
//     element is the sum of its group's partials in CTA order (so the result
//     does not depend on timing).  A slot word holds a NaN pattern that
//     arithmetic never produces until its value is written, and a reader
//     checks the values themselves; each CTA also counts itself done on a
//     per-link counter after publishing, and one thread per reader CTA waits
//     for that count before the CTA reads, so that the slots are not polled by
//     every thread while the producers still compute.  The workspace keeps two
//     sets of slots used by alternate launches; each launch puts the set the
//     next launch will use back to that pattern, and the last CTA to finish
//     puts the counters back to zero.
//   * The staged input is split for the tensor cores: each 256-element slice
//     is scaled by a power of two that puts its largest magnitude in
//     [2^14, 2^15) and carried as a binary16 pair hi + lo (relative error
//     below 2^-22); the slice's inverse scale is applied to each tile's fp32
//     sums.
//   * An output with the argmax op is reduced without writing it: each CTA
//     takes the largest of the rows it finishes, and CTA 0 reduces the CTAs'
//     records at the end of the launch.
//   * Every wait is bounded (about a second) and reports Q4_ERR_TIMEOUT.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/q4.h"
#include "q4r_tile.cuh"

namespace q4 {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;            // ring slots per warp (a power of two)
constexpr int kChunk = 2;            // tiles per bulk copy
constexpr int kChunkBytes = kChunk * rt::kTileBytes;
constexpr int kWarpGroups = 8;       // 16-row groups one warp may touch in one link
constexpr int kCtaGroups = 64;       // groups one CTA may first-own in a link with a residual
constexpr int kMaxLinks = Q4_CHAIN_MAX_LINKS;
constexpr int kMaxK = 12288;
constexpr int kStageQuads = 2;       // element quads per thread and staging pass: a warp
                                     // stages one 256-element slice
constexpr int kSlotFloats = 16;      // one 16-row group partial
constexpr uint32_t kEmpty = 0x7FBADBADu;  // NaN pattern that no arithmetic produces
constexpr int kHeaderBytes = 4096;
// header words (uint32): epoch, finished-CTA counter, abort flag, reset barrier,
// clean extent of buffer 0 / 1 (floats), the one-product kernel's ticket, each
// on its own 64-byte line; one done-CTA counter per link; from byte 1024 the
// one-product kernel's argmax records (2 words per CTA)
constexpr int kHdrEpoch = 0, kHdrFinished = 16, kHdrAbort = 32, kHdrBarrier = 48;
constexpr int kHdrClean0 = 64, kHdrClean1 = 80, kHdrTicket = 96, kHdrCount = 128;
constexpr int kHdrRecords = 256, kMaxCtas = (kHeaderBytes / 4 - kHdrRecords) / 2;
static_assert(kHdrCount + kMaxLinks <= kHdrRecords, "header");

// floor(n / d) for 32-bit n by a multiply-high and a shift (constants made on
// the host), then checked exactly.
struct Div {
  uint32_t m, s, d;
};

__device__ __forceinline__ uint32_t divq(uint32_t n, const Div& v) {
  uint32_t q =
      static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(v.m, n)) + n) >> v.s);
  if (static_cast<uint64_t>(q) * v.d > n) --q;
  else if (static_cast<uint64_t>(q + 1) * v.d <= n) ++q;
  return q;
}

struct ChainLink {
  const uint8_t* R;
  float* y;
  int32_t* argmax;
  const float* ext[2];   // x, residual read from memory (src_link < 0)
  int32_t src_link[2];   // earlier link whose output is read, or -1
  int32_t src_off[2];    // first element of the source
  int32_t n, k, nsb, groups, tiles;
  int32_t unit;          // tiles per partition unit: nsb (group-aligned) or 1
  uint32_t ops;
  uint32_t slot0;        // first slot of this link in a slot set
  uint32_t rec0;         // first argmax record (2 floats per CTA) in a slot set
  Div divU;              // division by the number of units (tiles / unit)
  Div divNsb;            // division by nsb
};

struct ChainArgs {
  ChainLink L[kMaxLinks];
  int32_t n_links, kmax;
  float* set[2];         // the two slot sets
  uint32_t set_floats;   // floats per set this chain uses
  uint32_t* hdr;
  int32_t* status;
  uint32_t flags;
  Div divC;              // division by the grid size
};

enum : uint32_t { kOpSwiglu = Q4_OP_SWIGLU, kOpResidual = Q4_OP_RESIDUAL, kOpArgmax = Q4_OP_ARGMAX };

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const float* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_f32(float* p, float v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(__float_as_uint(v)) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool empty4(const uint4& v) {
  return v.x == kEmpty || v.y == kEmpty || v.z == kEmpty || v.w == kEmpty;
}
__device__ __forceinline__ float4 as_f4(const uint4& v) {
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                     __uint_as_float(v.w));
}
__device__ __forceinline__ void add4(float4& a, const uint4& v) {
  a.x += __uint_as_float(v.x);
  a.y += __uint_as_float(v.y);
  a.z += __uint_as_float(v.z);
  a.w += __uint_as_float(v.w);
}

// Per-link data that a CTA reads in its loops, copied from the kernel
// parameters into shared memory when the launch starts (parameter reads with
// a link index that varies are constant-cache loads that miss).  A link's work
// is cut into units of `unit` tiles (a whole 16-row group, or one tile); CTA c
// holds units [U c / C, U (c+1) / C), i.e. tiles [ca, cb).
struct SLink {
  const uint8_t* R;
  float* y;
  int32_t* argmax;
  const float* ext[2];
  int32_t src_link[2], src_off[2];
  uint32_t slot0;      // this link's first slot in a slot set
  uint32_t rec0;       // its first argmax record
  int32_t ca, cb;      // this CTA's tiles
  int32_t nsb, n, k;
  int32_t unit, units;
  int32_t g0c, gcount; // this CTA's first 16-row group and its number of groups
  Div divU;
  Div divNsb;          // division by nsb
  uint32_t ops;
};

// CTAs holding the first and last tile of 16-row group g.
__device__ __forceinline__ void group_owners(const SLink& S, int g, uint32_t C, int& clo,
                                             int& chi) {
  if (S.unit == S.nsb) {
    clo = chi = static_cast<int>(divq(static_cast<uint32_t>(g + 1) * C - 1u, S.divU));
  } else {
    clo = static_cast<int>(divq(static_cast<uint32_t>(g * S.nsb + 1) * C - 1u, S.divU));
    chi = static_cast<int>(divq(static_cast<uint32_t>((g + 1) * S.nsb) * C - 1u, S.divU));
  }
}

// Warp w's share [a, b) of a CTA's tiles [ca, cb) when NW warps split them.
template <int NW>
__device__ __forceinline__ void warp_range(int ca, int cb, int w, int& a, int& b) {
  a = ca + (cb - ca) * w / NW;
  b = ca + (cb - ca) * (w + 1) / NW;
}

// What a thread carries around for bounded waits.
struct Ctx {
  uint32_t c, C;
  uint64_t t0;         // start of the current bounded wait
  int* s_abort;        // shared abort flag of the CTA
  uint32_t* hdr;
  int32_t* status;
};

__device__ __noinline__ void fail(Ctx& x) {
  if (atomicExch(x.s_abort, 1) == 0) {
    report(x.status, 6 /* Q4_ERR_TIMEOUT */);
    if (x.hdr != nullptr) atomicExch(x.hdr + kHdrAbort, 1u);
  }
}

// True while the bounded wait that started at x.t0 may continue.
__device__ __forceinline__ bool keep_waiting(Ctx& x, int& spins) {
  if (spins >= 8) __nanosleep(64);
  if ((++spins & 15) != 0) return true;
  if (*reinterpret_cast<volatile int*>(x.s_abort)) return false;
  if ((x.hdr != nullptr && ld_relaxed_u32(x.hdr + kHdrAbort) != 0u) ||
      global_timer_ns() - x.t0 > kWaitLimitNs) {
    fail(x);
    return false;
  }
  return true;
}

// Thread 0 waits until every CTA has counted itself done with link s (bounded);
// the CTA then reads that link's slots.  Called by all threads (barrier).
__device__ __forceinline__ void wait_link_done(Ctx& x, int s, int tid) {
  if (s >= 0 && tid == 0) {
    const uint32_t* cnt = x.hdr + kHdrCount + s;
    if (ld_relaxed_u32(cnt) < x.C) {
      x.t0 = global_timer_ns();
      int sp = 0;
      while (ld_relaxed_u32(cnt) < x.C)
        if (!keep_waiting(x, sp)) break;
    }
  }
  __syncthreads();
}

// An element quad a thread reads before a link: the first of np partials of an
// earlier link's output (slots kSlotFloats apart, summed in CTA order), or a
// plain vector in memory (np == 0); np < 0: nothing to read.  Its address is
// worked out before the thread waits for the producing link, so that only the
// loads remain once that link is done.
struct Ent {
  const float* p;
  int np;
};

// Elements [row, row + 4) of a source: an earlier link's output (src >= 0)
// or memory at ext.
__device__ __forceinline__ Ent make_entry(const SLink* sl, float* set_base, const float* ext,
                                          int src, int row, uint32_t C) {
  Ent en;
  if (src < 0) {
    en.p = ext + row;
    en.np = 0;
    return en;
  }
  const SLink& T = sl[src];
  const int shift = (T.ops & kOpSwiglu) ? 3 : 4;
  const int g = row >> shift;
  int clo, chi;
  group_owners(T, g, C, clo, chi);
  en.p = set_base + static_cast<size_t>(T.slot0 + g + clo) * kSlotFloats +
         (row & ((1 << shift) - 1));
  en.np = chi - clo + 1;
  return en;
}

// Loads W entries (the first two partials of every entry in one pass,
// re-read while a value still holds the empty pattern; further partials one
// after another).  false on abort.
template <int W>
__device__ __forceinline__ bool load_entries(const Ent (&en)[W], Ctx& x, float4 (&out)[W]) {
  uint4 v0[W], v1[W];
  bool d0[W], d1[W];
#pragma unroll
  for (int m = 0; m < W; ++m) {
    d0[m] = en[m].np <= 0;
    d1[m] = en[m].np <= 1;
    if (en[m].np == 0) out[m] = __ldcg(reinterpret_cast<const float4*>(en[m].p));
  }
  x.t0 = global_timer_ns();
  int spins = 0;
  while (true) {
#pragma unroll
    for (int m = 0; m < W; ++m) {
      if (!d0[m]) v0[m] = ld_relaxed_v4(en[m].p);
      if (!d1[m]) v1[m] = ld_relaxed_v4(en[m].p + kSlotFloats);
    }
    bool all = true;
#pragma unroll
    for (int m = 0; m < W; ++m) {
      if (!d0[m]) d0[m] = !empty4(v0[m]);
      if (!d1[m]) d1[m] = !empty4(v1[m]);
      all = all && d0[m] && d1[m];
    }
    if (all) break;
    if (!keep_waiting(x, spins)) return false;
  }
#pragma unroll
  for (int m = 0; m < W; ++m) {
    if (en[m].np < 1) continue;
    float4 s = as_f4(v0[m]);
    if (en[m].np > 1) add4(s, v1[m]);
    for (int cc = 2; cc < en[m].np; ++cc) {
      const float* p = en[m].p + static_cast<size_t>(cc) * kSlotFloats;
      uint4 u;
      x.t0 = global_timer_ns();
      int sp = 0;
      while (true) {
        u = ld_relaxed_v4(p);
        if (!empty4(u)) break;
        if (!keep_waiting(x, sp)) return false;
      }
      add4(s, u);
    }
    out[m] = s;
  }
  return true;
}

// The element quad that lane `lane` of warp `warp` stages as its m-th in pass
// `pass`: warp w stages slice 16 pass + w, two quads per lane.
template <int NW>
__device__ __forceinline__ int stage_quad(int pass, int warp, int lane, int m) {
  return 64 * (pass * NW + warp) + 32 * m + lane;
}

// The x entries of staging pass `pass`.
template <int NW>
__device__ __forceinline__ void x_entries(const SLink* sl, float* set_base, const SLink& S,
                                          int pass, int tid, uint32_t C,
                                          Ent (&en)[kStageQuads + 1]) {
  const int quads = S.k / 4;
#pragma unroll
  for (int m = 0; m < kStageQuads; ++m) {
    const int q = stage_quad<NW>(pass, tid >> 5, tid & 31, m);
    en[m].np = -1;
    if (q < quads) en[m] = make_entry(sl, set_base, S.ext[0], S.src_link[0], S.src_off[0] + 4 * q, C);
  }
}

__device__ __forceinline__ float silu_gate(float a, float b) { return a / (1.0f + __expf(-a)) * b; }

// Staged x for the tensor cores: every 256-element slice (one warp's two
// quads per lane) scaled by a power of two and split into binary16 hi + lo
// (q4r_tile.cuh layout), its inverse scale in xinv[slice].  A warp's quads
// are all valid or all past k (k % 256 == 0).
template <int NW>
__device__ __forceinline__ void convert_x(const float4 (&v)[kStageQuads + 1],
                                          const Ent (&en)[kStageQuads + 1], int pass, int tid,
                                          uint8_t* x16, float* xinv) {
  const int warp = tid >> 5, lane = tid & 31;
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < kStageQuads; ++m)
    if (en[m].np >= 0)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[m].x), fabsf(v[m].y)),
                               fmaxf(fabsf(v[m].z), fabsf(v[m].w))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float sc, inv;
  rt::slice_scale(amax, sc, inv);
#pragma unroll
  for (int m = 0; m < kStageQuads; ++m) {
    if (en[m].np < 0) continue;
    const int e = 4 * stage_quad<NW>(pass, warp, lane, m);
    __half h[4], l[4];
    rt::split_hi_lo(v[m].x * sc, h[0], l[0]);
    rt::split_hi_lo(v[m].y * sc, h[1], l[1]);
    rt::split_hi_lo(v[m].z * sc, h[2], l[2]);
    rt::split_hi_lo(v[m].w * sc, h[3], l[3]);
    const int s = e >> 4, i0 = e & 15;
    *reinterpret_cast<__half2*>(x16 + rt::x16_word(s, 0, i0)) = __halves2half2(h[0], h[1]);
    *reinterpret_cast<__half2*>(x16 + rt::x16_word(s, 0, i0 + 2)) = __halves2half2(h[2], h[3]);
    *reinterpret_cast<__half2*>(x16 + rt::x16_word(s, 1, i0)) = __halves2half2(l[0], l[1]);
    *reinterpret_cast<__half2*>(x16 + rt::x16_word(s, 1, i0 + 2)) = __halves2half2(l[2], l[3]);
    if (m == 0 && lane == 0) xinv[e >> 8] = inv;
  }
}

// Argmax candidates: larger value wins, then the lower index; NaN never wins.
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v != v) return;
  if (bi < 0 || v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}
__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi >= 0) better(bv, bi, ov, oi);
  }
}

// A warp's weight stream: its tiles of every link in order, in chunks of up to
// kChunk tiles (a warp range is cut into chunks from its start), kSlots chunks
// in flight through its ring.  `left` tiles remain in link ps, the next one at
// psrc.
struct TileStream {
  int ps, left, issued, consumed;
  const uint8_t* psrc;
};

template <int NW>
__device__ __forceinline__ void stream_enter(const SLink* sl, TileStream& ts, int warp) {
  const SLink& L = sl[ts.ps];
  int a, b;
  warp_range<NW>(L.ca, L.cb, warp, a, b);
  ts.left = b - a;
  ts.psrc = L.R + static_cast<size_t>(a) * rt::kTileBytes;
}

template <int NW>
__device__ __forceinline__ void stream_settle(const SLink* sl, int n_links, TileStream& ts,
                                              int warp) {
  while (ts.ps < n_links && ts.left == 0)
    if (++ts.ps < n_links) stream_enter<NW>(sl, ts, warp);
}

template <int NW>
__device__ __forceinline__ void stream_issue(const SLink* sl, int n_links, TileStream& ts,
                                             int warp, int lane, uint32_t ring, uint32_t bar0,
                                             uint64_t pol) {
  if (ts.ps >= n_links) return;
  const int nt = ts.left < kChunk ? ts.left : kChunk;
  if (lane == 0) {
    const uint32_t slot = static_cast<uint32_t>(ts.issued) & (kSlots - 1);
    mbar_arrive_expect_tx(bar0 + 8 * slot, nt * rt::kTileBytes);
    bulk_g2s(ring + slot * kChunkBytes, ts.psrc, nt * rt::kTileBytes, bar0 + 8 * slot, pol);
  }
  ++ts.issued;
  ts.psrc += nt * rt::kTileBytes;
  ts.left -= nt;
  if (ts.left == 0) stream_settle<NW>(sl, n_links, ts, warp);
}

// This warp's tiles [wa, wb) of the current link (g0w = wa / nsb): each
// 16-row group's row products end in Pw[group - g0w][row].  Kept out of line
// so that the decode loop is register-allocated on its own (inlined, the
// staging code's live values cost it spills).
template <int NW>
__device__ __noinline__ bool run_tiles(const SLink* sl, int n_links, TileStream& tsr, Ctx& x,
                                          int warp, int lane, const uint8_t* ring_p,
                                          uint32_t ring, uint32_t bar0, const uint8_t* x16,
                                          const float* xinv, int wa, int wb, int g0w, int nsb,
                                          float (*Pw)[kSlotFloats]) {
  TileStream ts = tsr;
  const uint64_t pol = l2_evict_first_policy();
  int cur = -1;
  float y[2] = {0.f, 0.f};
  auto flush = [&](int g) {
    if ((lane & 3) == 0) {
      Pw[g - g0w][lane >> 2] = y[0];
      Pw[g - g0w][(lane >> 2) + 8] = y[1];
    }
    y[0] = y[1] = 0.f;
  };
  bool ok = true;
  int g = g0w, t = wa - g0w * nsb;
  for (int i = wa; i < wb; i += kChunk) {
    const int nt = wb - i < kChunk ? wb - i : kChunk;
    const uint32_t slot = static_cast<uint32_t>(ts.consumed) & (kSlots - 1);
    const uint32_t parity = static_cast<uint32_t>(ts.consumed / kSlots) & 1u;
    const bool landed = mbar_wait(bar0 + 8 * slot, parity, x.s_abort);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) fail(x);
      ok = false;
      break;
    }
    const uint8_t* chunk = ring_p + slot * kChunkBytes;
#pragma unroll
    for (int p = 0; p < kChunk; ++p) {
      if (p < nt) {
        if (g != cur) {
          if (cur >= 0) flush(cur);
          cur = g;
        }
        rt::tile_dot(chunk + p * rt::kTileBytes, x16 + t * (16 * rt::kXStepBytes), xinv[t], lane,
                     y);
        if (++t == nsb) {
          t = 0;
          ++g;
        }
      }
    }
    __syncwarp();
    fence_proxy_async_smem();
    ++ts.consumed;
    stream_issue<NW>(sl, n_links, ts, warp, lane, ring, bar0, pol);
  }
  if (ok && cur >= 0) flush(cur);
  tsr = ts;
  return ok;
}

__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ ChainArgs A) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kWarps][kSlots];
  __shared__ __align__(8) uint64_t never_bar;
  __shared__ __align__(16) float P[kWarps][kWarpGroups][kSlotFloats];
  __shared__ __align__(16) float sres[kCtaGroups][kSlotFloats];
  __shared__ __align__(16) SLink s_links[kMaxLinks];
  __shared__ int s_wa[kWarps], s_wb[kWarps];
  __shared__ int2 s_wg[kWarps];  // first and last group of each warp range (empty: 1, 0)
  __shared__ float sown[kSlotFloats];
  __shared__ float s_bv[kWarps];
  __shared__ int s_bi[kWarps];
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Ctx x;
  x.c = blockIdx.x;
  x.C = gridDim.x;
  x.s_abort = &s_abort;
  x.hdr = A.hdr;
  x.status = A.status;
  const int n_links = A.n_links;
  // dynamic shared memory: ring | staged x | inverse slice scales
  uint8_t* const ring_p = smem + warp * kSlots * kChunkBytes;
  const uint32_t ring = smem_u32(ring_p);
  uint8_t* const x16 = smem + kWarps * kSlots * kChunkBytes;
  float* const xinv = reinterpret_cast<float*>(x16 + rt::x16_bytes(A.kmax));
  const uint32_t bar0 = smem_u32(&full_bar[warp][0]);
  const uint64_t pol = l2_evict_first_policy();

  // the header's words are loaded together, first, so that their latency
  // overlaps the set-up and the first weight copies below (nothing before the
  // slot-set reset depends on them)
  const uint32_t epoch = ld_relaxed_u32(A.hdr + kHdrEpoch);
  const uint32_t clean0 = ld_relaxed_u32(A.hdr + kHdrClean0);
  const uint32_t clean1 = ld_relaxed_u32(A.hdr + kHdrClean1);
  if (tid == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&never_bar), 1);
  }
  if (lane == 0)
    for (int i = 0; i < kSlots; ++i) mbar_init(bar0 + 8 * i, 1);
  for (int s = tid; s < n_links; s += kThreads) {
    const ChainLink& L = A.L[s];
    SLink& S = s_links[s];
    const uint32_t units = static_cast<uint32_t>(L.tiles / L.unit);
    S.R = L.R;
    S.y = L.y;
    S.argmax = L.argmax;
    for (int j = 0; j < 2; ++j) {
      S.ext[j] = L.ext[j];
      S.src_link[j] = L.src_link[j];
      S.src_off[j] = L.src_off[j];
    }
    S.k = L.k;
    S.rec0 = L.rec0;
    S.slot0 = L.slot0;
    S.ca = L.unit * static_cast<int>(divq(units * x.c, A.divC));
    S.cb = L.unit * static_cast<int>(divq(units * (x.c + 1), A.divC));
    S.nsb = L.nsb;
    S.n = L.n;
    S.unit = L.unit;
    S.units = static_cast<int>(units);
    S.divU = L.divU;
    S.divNsb = L.divNsb;
    S.ops = L.ops;
    S.g0c = static_cast<int>(divq(static_cast<uint32_t>(S.ca), L.divNsb));
    S.gcount = S.ca < S.cb
                   ? static_cast<int>(divq(static_cast<uint32_t>(S.cb - 1), L.divNsb)) - S.g0c + 1
                   : 0;
  }
  fence_mbarrier_init();
  __syncthreads();

  // ---- this warp's weight stream: the first kSlots chunks go out now
  TileStream ts;
  ts.ps = 0;
  ts.issued = 0;
  ts.consumed = 0;
  stream_enter<kWarps>(s_links, ts, warp);
  stream_settle<kWarps>(s_links, n_links, ts, warp);
  for (int i = 0; i < kSlots; ++i)
    stream_issue<kWarps>(s_links, n_links, ts, warp, lane, ring, bar0, pol);

  // ---- slot sets: a fresh workspace (or one last used with a smaller chain)
  // gets both sets reset before anyone publishes; otherwise the set of the
  // next launch is reset while this one runs.
  const int set = static_cast<int>(epoch & 1u);
  const uint32_t clean_mine = set ? clean1 : clean0;
  float* const set_base = A.set[set];
  {
    const bool fresh = epoch == 0u || clean_mine < A.set_floats;
    const uint32_t total = A.set_floats / 4;  // float4s per set
    const uint32_t q0 = divq(total * x.c, A.divC), q1 = divq(total * (x.c + 1), A.divC);
    const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
    for (int st = 0; st < 2; ++st) {
      if (st == set && !fresh) continue;
      uint4* p = reinterpret_cast<uint4*>(A.set[st]);
      for (uint32_t i = q0 + tid; i < q1; i += kThreads) p[i] = e4;
    }
    if (fresh) {
      // every CTA's reset of this launch's set lands before anything is published
      __syncthreads();
      if (tid == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(A.hdr + kHdrBarrier) : "memory");
        x.t0 = global_timer_ns();
        int sp = 0;
        while (ld_acquire_u32(A.hdr + kHdrBarrier) < x.C)
          if (!keep_waiting(x, sp)) break;
      }
      __syncthreads();
    }
  }

  // Test hook: one bounded wait that nothing ends (thread 0 of CTA 0, which
  // every launch has), so the call reports Q4_ERR_TIMEOUT.
  if ((A.flags & kFlagTestStallOneWait) != 0 && x.c == 0 && tid == 0)
    if (!mbar_wait(smem_u32(&never_bar), 0, &s_abort)) fail(x);
  float bv = 0.f;  // argmax candidate of this thread
  int bi = -1;
  // Every decision taken on the abort flag is made uniform by a barrier that
  // ORs it over the CTA, so that no warp or CTA splits around a collective.
  volatile int* abort_flag = &s_abort;
  bool stop = __syncthreads_or(*abort_flag) != 0;

  for (int s = 0; s <= n_links && !stop; ++s) {
    const bool last = s == n_links;
    // ---------------- before waiting on other CTAs: this link's warp ranges
    // and the addresses of everything it reads
    bool finish_prev = false;  // this CTA first-owns a split group of link s-1
    if (s > 0) {
      const SLink& S1 = s_links[s - 1];
      if (S1.gcount > 0 && (S1.y != nullptr || (S1.ops & kOpArgmax))) {
        const int g = S1.g0c + S1.gcount - 1;
        finish_prev = g * S1.nsb >= S1.ca && (g + 1) * S1.nsb > S1.cb;
      }
    }
    int need = finish_prev ? s - 1 : -1;
    Ent en[kStageQuads + 1];  // x quads of the first staging pass, then a residual quad
#pragma unroll
    for (int m = 0; m <= kStageQuads; ++m) en[m].np = -1;
    if (!last) {
      const SLink& S = s_links[s];
      need = max(need, S.src_link[0]);
      if (S.ops & kOpResidual) need = max(need, S.src_link[1]);
      if (lane == 0) {
        int a, b;
        warp_range<kWarps>(S.ca, S.cb, warp, a, b);
        s_wa[warp] = a;
        s_wb[warp] = b;
        s_wg[warp] = a < b ? make_int2(static_cast<int>(divq(static_cast<uint32_t>(a), S.divNsb)),
                                       static_cast<int>(divq(static_cast<uint32_t>(b - 1), S.divNsb)))
                           : make_int2(1, 0);
      }
      if (S.gcount > 0) {
        x_entries<kWarps>(s_links, set_base, S, 0, tid, x.C, en);
        // the residual rows of the groups this CTA holds the first tile of
        if ((S.ops & kOpResidual) && tid < S.gcount * 4) {
          const int g = S.g0c + tid / 4, row = 16 * g + 4 * (tid & 3);
          if (g * S.nsb >= S.ca && row < S.n)
            en[kStageQuads] = make_entry(s_links, set_base, S.ext[1], S.src_link[1],
                                         S.src_off[1] + row, x.C);
        }
      }
    }
    wait_link_done(x, need, tid);

    // ---------------- finish link s-1: the CTA's split first-owned group
    if (s > 0 && warp == kWarps - 1) {
      const SLink& S1 = s_links[s - 1];
      float fv = 0.f;
      int fi = -1;
      if (finish_prev && lane < kSlotFloats) {
        const int g = S1.g0c + S1.gcount - 1;
        int clo, chi;
        group_owners(S1, g, x.C, clo, chi);
        float v = sown[lane];
        bool ok = true;
        for (int cc = clo + 1; cc <= chi && ok; ++cc) {
          const uint32_t* q = reinterpret_cast<const uint32_t*>(
              set_base + static_cast<size_t>(S1.slot0 + g + cc) * kSlotFloats + lane);
          x.t0 = global_timer_ns();
          int sp = 0;
          uint32_t u;
          while ((u = ld_relaxed_u32(q)) == kEmpty)
            if (!keep_waiting(x, sp)) {
              ok = false;
              break;
            }
          v += __uint_as_float(u);
        }
        const int row = 16 * g + lane;
        if (ok && row < S1.n) {
          if (S1.y != nullptr) S1.y[row] = v;
          better(fv, fi, v, row);
        }
      }
      if (S1.ops & kOpArgmax) {
        // this CTA's record: its fully held rows (from the publish step) and
        // the split group finished here, reduced in a fixed order
        warp_best(fv, fi);
        if (lane == 0) {
          float v = fv;
          int i = fi;
          for (int w = 0; w < kWarps; ++w)
            if (s_bi[w] >= 0) better(v, i, s_bv[w], s_bi[w]);
          float* rec = set_base + S1.rec0 + 2 * x.c;
          st_relaxed_f32(rec, i >= 0 ? v : 0.f);
          st_relaxed_f32(rec + 1, __int_as_float(i));
        }
      }
    }
    if (last) break;
    const SLink& S = s_links[s];
    const int ca = S.ca, cb = S.cb, g0c = S.g0c, gcount = S.gcount;

    // ---------------- stage x_s (and the residual rows this CTA adds)
    if (!*abort_flag && gcount > 0) {
      float4 v[kStageQuads + 1];
      bool ok = load_entries(en, x, v);
      if (ok) {
        convert_x<kWarps>(v, en, 0, tid, x16, xinv);
        if (en[kStageQuads].np >= 0)
          *reinterpret_cast<float4*>(&sres[tid / 4][4 * (tid & 3)]) = v[kStageQuads];
      }
      for (int pass = 1; ok && pass * kWarps * 256 < S.k; ++pass) {
        x_entries<kWarps>(s_links, set_base, S, pass, tid, x.C, en);
        en[kStageQuads].np = -1;
        ok = load_entries(en, x, v);
        if (ok) convert_x<kWarps>(v, en, pass, tid, x16, xinv);
      }
    }
    stop = __syncthreads_or(*abort_flag) != 0;
    if (stop) break;

    // ---------------- this warp's tiles of link s
    run_tiles<kWarps>(s_links, n_links, ts, x, warp, lane, ring_p, ring, bar0, x16, xinv,
                      s_wa[warp], s_wb[warp], s_wg[warp].x, S.nsb, P[warp]);
    stop = __syncthreads_or(*abort_flag) != 0;
    if (stop) break;

    // ---------------- publish: one partial per (group, CTA); y and argmax
    // candidates for the groups held whole
    bi = -1;
    if (ca == cb && tid < kSlotFloats) {
      // A CTA without tiles in this link sits at tile ca, inside the group
      // ca / nsb when the link has fewer tiles than SMs; readers of that group
      // count it among the group's CTAs, so it publishes zeros there.  Its
      // slot index ca / nsb + c is still unique.
      st_relaxed_f32(set_base + static_cast<size_t>(S.slot0 + g0c + x.c) * kSlotFloats + tid,
                     0.f);
    }
    if (gcount > 0 && (S.ops & kOpSwiglu)) {
      // gated link (whole groups): 8 values per group, a * sigmoid(a) * b
      float* const y = S.y;
      for (int idx = tid; idx < gcount * 8; idx += kThreads) {
        const int gl = idx >> 3, j = idx & 7, g = g0c + gl;
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int2 r = s_wg[w];
          if (g >= r.x && g <= r.y) {
            a += P[w][g - r.x][j];
            b += P[w][g - r.x][j + 8];
          }
        }
        const float v = silu_gate(a, b);
        st_relaxed_f32(set_base + static_cast<size_t>(S.slot0 + g + x.c) * kSlotFloats + j, v);
        if (y != nullptr && 8 * g + j < S.n / 2) y[8 * g + j] = v;
      }
    } else if (gcount > 0) {
      float* const y = S.y;
      for (int idx = tid; idx < gcount * kSlotFloats; idx += kThreads) {
        const int gl = idx >> 4, row16 = idx & 15, g = g0c + gl;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int2 r = s_wg[w];
          if (g >= r.x && g <= r.y) sum += P[w][g - r.x][row16];
        }
        // this CTA holds the group's first tile / all of its tiles
        const bool first = g * S.nsb >= ca;
        const bool whole = first && (g + 1) * S.nsb <= cb;
        if (first && (S.ops & kOpResidual)) sum += sres[gl][row16];
        st_relaxed_f32(set_base + static_cast<size_t>(S.slot0 + g + x.c) * kSlotFloats + row16,
                       sum);
        const int row = 16 * g + row16;
        if (whole) {
          if (row < S.n) {
            if (y != nullptr) y[row] = sum;
            better(bv, bi, sum, row);
          }
        } else if (first) {
          sown[row16] = sum;
        }
      }
    }
    if (S.ops & kOpArgmax) {
      warp_best(bv, bi);
      if (lane == 0) {
        s_bv[warp] = bv;
        s_bi[warp] = bi;
      }
    }
    stop = __syncthreads_or(*abort_flag) != 0;
    // this CTA is done with link s: its slot stores are issued (the readers
    // check the values, the count only tells them when to look)
    if (!stop && tid == 0) red_relaxed_add(A.hdr + kHdrCount + s, 1u);
  }

  // ---------------- argmax over the CTAs' records (CTA 0), then the epoch
  stop = __syncthreads_or(*abort_flag) != 0;
  if (!stop && x.c == 0 && warp == 0) {
    for (int s = 0; s < n_links; ++s) {
      const SLink& L = s_links[s];
      if (!(L.ops & kOpArgmax)) continue;
      const uint32_t* rec = reinterpret_cast<const uint32_t*>(set_base + L.rec0);
      float v = 0.f;
      int i = -1;
      bool ok = true;
      for (uint32_t cc = lane; cc < x.C; cc += 32) {
        x.t0 = global_timer_ns();
        int sp = 0;
        uint32_t rv, ri;
        while (true) {
          rv = ld_relaxed_u32(rec + 2 * cc);
          ri = ld_relaxed_u32(rec + 2 * cc + 1);
          if (rv != kEmpty && ri != kEmpty) break;
          if (!keep_waiting(x, sp)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (static_cast<int>(ri) >= 0) better(v, i, __uint_as_float(rv), static_cast<int>(ri));
      }
      warp_best(v, i);
      const bool all_ok = __all_sync(0xffffffffu, ok);  // every lane votes
      if (lane == 0 && all_ok) {
        L.argmax[0] = i;
        L.argmax[1] = __float_as_int(i >= 0 ? v : __uint_as_float(0x7FC00000u));
      }
    }
  }
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    // the last CTA to finish records that the next set is clean, puts the
    // link counters back to zero and moves the epoch
    const uint32_t prev = atomicAdd(A.hdr + kHdrFinished, 1u);
    if (prev == x.C - 1) {
      // every other CTA is done with the header: plain stores, nothing waits
      for (int s = 0; s < n_links; ++s) st_relaxed_u32(A.hdr + kHdrCount + s, 0u);
      st_relaxed_u32(A.hdr + kHdrFinished, 0u);
      st_relaxed_u32(A.hdr + kHdrBarrier, 0u);
      st_relaxed_u32(A.hdr + (set ? kHdrClean0 : kHdrClean1), A.set_floats);
      st_relaxed_u32(A.hdr + kHdrEpoch, epoch + 1u);
    }
  }
  // copies this warp still has in flight land before the CTA exits
  for (int q = ts.consumed; q < ts.issued; ++q)
    mbar_wait(bar0 + 8 * static_cast<uint32_t>(q % kSlots),
              static_cast<uint32_t>((q / kSlots) & 1));
}


// ------------------------------------------------------------------ one product
// A chain of one link needs no hand-off: CTA c takes whole 16-row groups
// [G c / C, G (c+1) / C) (for the 131072-row output head the busiest CTA
// holds 1.2 % more than the average), so every output is finished inside one
// CTA, and the launch is an ordinary one.  Only the argmax crosses CTAs: each
// CTA writes a record, takes a ticket, and the CTA with the last ticket reduces
// the records (nothing waits).
struct SingleArgs {
  const uint8_t* R;
  const float* x;         // k elements (offset applied)
  const float* residual;  // n elements, or nullptr
  float* y;               // or nullptr
  int32_t* argmax;        // or nullptr
  uint32_t* hdr;          // workspace header (ticket, records)
  int32_t* status;
  int32_t n, k, nsb, groups;
  uint32_t ops, flags;
};

// NW = 16: one CTA per SM (a call alone).  NW = 8: half the warps and shared
// memory, so that under programmatic dependent launch the next call's CTA fits
// beside this one, fills its ring and only then waits for this call to end.
template <int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) single_kernel(const SingleArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[NW][kSlots];
  __shared__ __align__(8) uint64_t never_bar;
  __shared__ __align__(16) float P[NW][kWarpGroups][kSlotFloats];
  __shared__ __align__(16) SLink s_link[1];
  __shared__ int s_wa[NW], s_wb[NW];
  __shared__ int2 s_wg[NW];
  __shared__ float s_bv[NW];
  __shared__ int s_bi[NW];
  __shared__ int s_abort, s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = blockIdx.x, C = gridDim.x;
  Ctx x;
  x.c = c;
  x.C = C;
  x.s_abort = &s_abort;
  x.hdr = nullptr;  // no cross-CTA abort flag: nothing here waits on another CTA
  x.status = a.status;
  uint8_t* const ring_p = smem + warp * kSlots * kChunkBytes;
  const uint32_t ring = smem_u32(ring_p);
  uint8_t* const x16 = smem + NW * kSlots * kChunkBytes;
  float* const xinv = reinterpret_cast<float*>(x16 + rt::x16_bytes(a.k));
  const uint32_t bar0 = smem_u32(&full_bar[warp][0]);
  const uint64_t pol = l2_evict_first_policy();
  const int g0c = static_cast<int>(static_cast<int64_t>(a.groups) * c / C);
  const int g1c = static_cast<int>(static_cast<int64_t>(a.groups) * (c + 1) / C);
  const int ca = g0c * a.nsb, cb = g1c * a.nsb, gcount = g1c - g0c;
  if (tid == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&never_bar), 1);
    SLink& S = s_link[0];
    S.R = a.R;
    S.ext[0] = a.x;
    S.src_link[0] = -1;
    S.src_off[0] = 0;
    S.ca = ca;
    S.cb = cb;
    S.nsb = a.nsb;
    S.k = a.k;
  }
  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(bar0 + 8 * i, 1);
    int wa, wb;
    warp_range<NW>(ca, cb, warp, wa, wb);
    s_wa[warp] = wa;
    s_wb[warp] = wb;
    s_wg[warp] = wa < wb ? make_int2(wa / a.nsb, (wb - 1) / a.nsb) : make_int2(1, 0);
  }
  fence_mbarrier_init();
  __syncthreads();
  TileStream ts;
  ts.ps = 0;
  ts.issued = 0;
  ts.consumed = 0;
  pdl_allow_dependents();
  stream_enter<NW>(s_link, ts, warp);
  stream_settle<NW>(s_link, 1, ts, warp);
  for (int i = 0; i < kSlots; ++i) stream_issue<NW>(s_link, 1, ts, warp, lane, ring, bar0, pol);
  // under programmatic dependent launch, x (and the residual) may be the
  // previous kernel's output: read only after it has finished
  pdl_wait_prior_grid();
  volatile int* abort_flag = &s_abort;
  if ((a.flags & kFlagTestStallOneWait) != 0 && c == 0 && tid == 0)
    if (!mbar_wait(smem_u32(&never_bar), 0, &s_abort)) fail(x);

  // ---- stage x
  if (gcount > 0) {
    const SLink& S = s_link[0];
    Ent en[kStageQuads + 1];
    float4 v[kStageQuads + 1];
    en[kStageQuads].np = -1;
    for (int pass = 0; pass * NW * 256 < a.k; ++pass) {
      x_entries<NW>(s_link, nullptr, S, pass, tid, C, en);
      load_entries(en, x, v);  // plain loads: nothing to wait for
      convert_x<NW>(v, en, pass, tid, x16, xinv);
    }
  }
  bool stop = __syncthreads_or(*abort_flag) != 0;

  // ---- tiles, then the CTA's groups
  float bv = 0.f;
  int bi = -1;
  if (!stop) {
    run_tiles<NW>(s_link, 1, ts, x, warp, lane, ring_p, ring, bar0, x16, xinv, s_wa[warp],
                  s_wb[warp], s_wg[warp].x, a.nsb, P[warp]);
    stop = __syncthreads_or(*abort_flag) != 0;
  }
  if (!stop && (a.ops & kOpSwiglu)) {
    for (int idx = tid; idx < gcount * 8; idx += kThreads) {
      const int gl = idx >> 3, j = idx & 7, g = g0c + gl;
      float va = 0.f, vb = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int2 r = s_wg[w];
        if (g >= r.x && g <= r.y) {
          va += P[w][g - r.x][j];
          vb += P[w][g - r.x][j + 8];
        }
      }
      const float v = silu_gate(va, vb);
      if (a.y != nullptr) a.y[8 * g + j] = v;
      better(bv, bi, v, 8 * g + j);
    }
  } else if (!stop) {
    for (int idx = tid; idx < gcount * kSlotFloats; idx += kThreads) {
      const int gl = idx >> 4, row16 = idx & 15, g = g0c + gl, row = 16 * g + row16;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int2 r = s_wg[w];
        if (g >= r.x && g <= r.y) sum += P[w][g - r.x][row16];
      }
      if (row < a.n) {
        if (a.residual != nullptr) sum += __ldcg(a.residual + row);
        if (a.y != nullptr) a.y[row] = sum;
        better(bv, bi, sum, row);
      }
    }
  }
  if (a.ops & kOpArgmax) {
    // taken even after an abort, so that the tickets of every launch add up
    warp_best(bv, bi);
    if (lane == 0) {
      s_bv[warp] = bv;
      s_bi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float v = 0.f;
      int i = -1;
      for (int w = 0; w < NW; ++w)
        if (s_bi[w] >= 0) better(v, i, s_bv[w], s_bi[w]);
      uint32_t* rec = a.hdr + kHdrRecords + 2 * c;
      st_relaxed_u32(rec, __float_as_uint(i >= 0 ? v : 0.f));
      st_relaxed_u32(rec + 1, static_cast<uint32_t>(i));
      __threadfence();
      s_last = atomicAdd(a.hdr + kHdrTicket, 1u) == C - 1;
    }
    __syncthreads();
    if (s_last && warp == 0) {
      // every record was written before its CTA's ticket: read them after ours
      __threadfence();
      float v = 0.f;
      int i = -1;
      for (uint32_t cc = lane; cc < C; cc += 32) {
        const uint32_t* rec = a.hdr + kHdrRecords + 2 * cc;
        const int ri = static_cast<int>(ld_relaxed_u32(rec + 1));
        if (ri >= 0) better(v, i, __uint_as_float(ld_relaxed_u32(rec)), ri);
      }
      warp_best(v, i);
      if (lane == 0) {
        a.argmax[0] = i;
        a.argmax[1] = __float_as_int(i >= 0 ? v : __uint_as_float(0x7FC00000u));
        st_relaxed_u32(a.hdr + kHdrTicket, 0u);
      }
    }
  }
  for (int q = ts.consumed; q < ts.issued; ++q)
    mbar_wait(bar0 + 8 * static_cast<uint32_t>(q % kSlots),
              static_cast<uint32_t>((q / kSlots) & 1));
}

// ------------------------------------------------------------------ repack
// Thread per (tile, lane L = 4g + t, step quad j): the lane's 16 code bytes of
// steps 4j..4j+3 (rows 16G + g and 16G + g + 8, blocks 2j and 2j + 1 of the
// slice), and for t < 2 the scale word of block 2j + t of both rows.
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ W, int64_t n,
                                                     int64_t k, uint8_t* __restrict__ R) {
  const int64_t nb = k / 32, nsb = k / 256, tiles = (n + 15) / 16 * nsb;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= tiles * 128) return;
  const int64_t tile = idx >> 7;
  const int L = static_cast<int>(idx & 31), j = static_cast<int>((idx >> 5) & 3);
  const int g = L >> 2, tq = L & 3;
  const int64_t G = tile / nsb, t = tile - G * nsb;
  const int64_t r0 = 16 * G + g, r1 = r0 + 8;
  uint8_t* out = R + tile * rt::kTileBytes;
  // code of row r, block kb, element e (padding rows: 8)
  auto code = [&](int64_t r, int64_t kb, int e) -> uint32_t {
    if (r >= n) return 8u;
    const uint8_t* blk = W + (r * nb + kb) * kBlockBytes + 2;
    return e < 16 ? (blk[e] & 0xFu) : (blk[e - 16] >> 4);
  };
  uint32_t words[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int s = 4 * j + u;               // step
    const int64_t kb = 8 * t + s / 2;      // block of the step
    const int e0 = 16 * (s & 1) + 2 * tq;  // element of column 2t of the step
    uint32_t w = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int e = e0 + 8 * ((m >> 1) & 1) + (m >> 2);
      w |= code((m & 1) ? r1 : r0, kb, e) << (4 * m);
    }
    words[u] = w;
  }
  *reinterpret_cast<uint4*>(out + rt::kScaleBytes + rt::kStepBytes * j + 16 * L) =
      make_uint4(words[0], words[1], words[2], words[3]);
  if (tq < 2) {
    const int b = 2 * j + tq;
    const int64_t kb = 8 * t + b;
    auto dbits = [&](int64_t r) -> uint32_t {
      if (r >= n) return 0u;
      const uint8_t* blk = W + (r * nb + kb) * kBlockBytes;
      return blk[0] | (static_cast<uint32_t>(blk[1]) << 8);
    };
    *reinterpret_cast<uint32_t*>(out + 32 * g + 4 * b) = dbits(r0) | (dbits(r1) << 16);
  }
}

// ------------------------------------------------------------------ host side
Div make_div(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return {static_cast<uint32_t>(m), l, d};
}

inline bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

// Validates the links and fills the kernel arguments; returns the workspace
// bytes the chain needs in *ws.
q4_status chain_plan(const q4_chain_link* links, int32_t n, ChainArgs* A, size_t* ws) {
  if (links == nullptr || n < 1 || n > kMaxLinks) return Q4_ERR_INVALID_ARG;
  const uint32_t C = static_cast<uint32_t>(sm_count());
  int kmax = 256;
  uint32_t slot = 0, rec_floats = 0;
  // argmax records go after every link's slots; first count the slots
  uint32_t slots_total = 0;
  for (int32_t s = 0; s < n; ++s) {
    const q4_chain_link& l = links[s];
    if (l.n <= 0 || l.k <= 0 || l.n > (int64_t(1) << 28)) return Q4_ERR_INVALID_ARG;
    const int64_t groups = (l.n + 15) / 16;
    slots_total += static_cast<uint32_t>(groups + C);
  }
  for (int32_t s = 0; s < n; ++s) {
    const q4_chain_link& l = links[s];
    if (l.R == nullptr) return Q4_ERR_INVALID_ARG;
    if (l.k % 256 != 0 || l.k > kMaxK) return Q4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(l.R, 16)) return Q4_ERR_MISALIGNED;
    if (l.ops & ~uint32_t(Q4_OP_SWIGLU | Q4_OP_RESIDUAL | Q4_OP_ARGMAX)) return Q4_ERR_INVALID_ARG;
    if (l.y != nullptr && !aligned(l.y, 4)) return Q4_ERR_MISALIGNED;
    if ((l.ops & Q4_OP_ARGMAX) && (l.argmax == nullptr || !aligned(l.argmax, 4)))
      return Q4_ERR_INVALID_ARG;
    const bool gate = (l.ops & Q4_OP_SWIGLU) != 0;
    if (gate && (l.ops != Q4_OP_SWIGLU || l.n % 16 != 0)) return Q4_ERR_INVALID_ARG;
    const int64_t groups = (l.n + 15) / 16, nsb = l.k / 256, tiles = groups * nsb;
    if (tiles * C >= (int64_t(1) << 31)) return Q4_ERR_UNSUPPORTED_SHAPE;
    // Work is cut into whole 16-row groups when that costs the busiest CTA at
    // most 1/16 more tiles than cutting single tiles: a group then has one
    // owner, whose partial is its final value.
    const int64_t per_tile = (tiles + C - 1) / C, per_group = (groups + C - 1) / C * nsb;
    // A gated link is always cut at whole groups: the owner of a group applies
    // the gate to its 8 row pairs.
    const int64_t unit = (gate || per_group <= per_tile + per_tile / 16) ? nsb : 1;
    // bounded shared-memory bookkeeping per warp and per CTA
    const int64_t per_cta = unit == 1 ? per_tile : per_group;
    const int64_t per_warp = (per_cta + kWarps - 1) / kWarps;
    if (per_warp / nsb + 2 > kWarpGroups) return Q4_ERR_UNSUPPORTED_SHAPE;
    if ((l.ops & Q4_OP_RESIDUAL) && per_cta / nsb + 2 > kCtaGroups) return Q4_ERR_UNSUPPORTED_SHAPE;
    // sources: x (k elements) and the residual (n elements)
    const q4_chain_src* src[2] = {&l.x, &l.residual};
    const bool used[2] = {true, (l.ops & Q4_OP_RESIDUAL) != 0};
    const int64_t len[2] = {l.k, l.n};
    if (A != nullptr) {
      ChainLink& c = A->L[s];
      c.R = static_cast<const uint8_t*>(l.R);
      c.y = l.y;
      c.argmax = l.argmax;
      c.n = static_cast<int32_t>(l.n);
      c.k = static_cast<int32_t>(l.k);
      c.nsb = static_cast<int32_t>(nsb);
      c.groups = static_cast<int32_t>(groups);
      c.tiles = static_cast<int32_t>(tiles);
      c.ops = l.ops;
      c.slot0 = slot;
      c.unit = static_cast<int32_t>(unit);
      c.divU = make_div(static_cast<uint32_t>(tiles / unit));
      c.divNsb = make_div(static_cast<uint32_t>(nsb));
      c.rec0 = 0;
    }
    for (int j = 0; j < 2; ++j) {
      if (A != nullptr) {
        A->L[s].ext[j] = nullptr;
        A->L[s].src_link[j] = -1;
        A->L[s].src_off[j] = 0;
      }
      if (!used[j]) continue;
      const q4_chain_src& q = *src[j];
      if (q.offset < 0) return Q4_ERR_INVALID_ARG;
      if (q.offset % 4 != 0) return Q4_ERR_MISALIGNED;  // read in quads of elements
      if (j == 1 && l.n % 4 != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
      if (q.link >= 0) {
        if (q.link >= s) return Q4_ERR_INVALID_ARG;  // only earlier links
        const q4_chain_link& t = links[q.link];
        const int64_t out_len = (t.ops & Q4_OP_SWIGLU) ? t.n / 2 : t.n;
        if (q.offset + len[j] > out_len) return Q4_ERR_INVALID_ARG;
      } else {
        if (q.ptr == nullptr) return Q4_ERR_INVALID_ARG;
        if (!aligned(q.ptr, 16)) return Q4_ERR_MISALIGNED;
      }
      if (A != nullptr) {
        A->L[s].ext[j] = q.link >= 0 ? nullptr : q.ptr;
        A->L[s].src_link[j] = q.link;
        A->L[s].src_off[j] = q.offset;
      }
    }
    if (l.ops & Q4_OP_ARGMAX) {
      if (A != nullptr) A->L[s].rec0 = slots_total * kSlotFloats + rec_floats;
      rec_floats += 2 * C;
    }
    kmax = std::max<int>(kmax, static_cast<int>(l.k));
    slot += static_cast<uint32_t>(groups + C);
  }
  const uint64_t set_floats = (uint64_t(slots_total) * kSlotFloats + rec_floats + 63) / 64 * 64;
  *ws = kHeaderBytes + 2 * set_floats * 4;
  if (A != nullptr) {
    A->n_links = n;
    A->kmax = kmax;
    A->set_floats = static_cast<uint32_t>(set_floats);
    A->divC = make_div(C);
  }
  return Q4_OK;
}

size_t chain_smem_bytes(int kmax) {
  return static_cast<size_t>(kWarps) * kSlots * kChunkBytes +
         static_cast<size_t>(rt::x16_bytes(kmax)) + static_cast<size_t>(kmax / 256) * 4;
}

cudaError_t chain_launch(ChainArgs& A, void* workspace, cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(workspace);
  A.hdr = reinterpret_cast<uint32_t*>(w);
  A.set[0] = reinterpret_cast<float*>(w + kHeaderBytes);
  A.set[1] = A.set[0] + A.set_floats;
  const size_t smem = chain_smem_bytes(A.kmax);
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(chain_smem_bytes(kMaxK)));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chain_kernel, A);
}

// One link (its sources are in memory): the one-product kernel, unless the
// CTAs' whole-group shares do not fit its per-warp bookkeeping.
bool single_fits(const q4_chain_link& l, int nw) {
  const int64_t C = sm_count(), nsb = l.k / 256, groups = (l.n + 15) / 16;
  if (C > kMaxCtas) return false;
  const int64_t per_cta = (groups + C - 1) / C * nsb;
  const int64_t per_warp = (per_cta + nw - 1) / nw;
  return per_warp / nsb + 2 <= kWarpGroups;
}

size_t single_smem_bytes(int nw, int k) {
  return static_cast<size_t>(nw) * kSlots * kChunkBytes + static_cast<size_t>(rt::x16_bytes(k)) +
         static_cast<size_t>(k / 256) * 4;
}

template <int NW>
cudaError_t single_launch_nw(const SingleArgs& a, bool pdl, cudaStream_t s) {
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(single_kernel<NW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(single_smem_bytes(NW, kMaxK)));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = single_smem_bytes(NW, a.k);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, single_kernel<NW>, a);
}

// Alone: 16 warps, one CTA per SM.  With Q4_FLAG_PDL: the 8-warp shape when
// its per-warp bookkeeping fits (two CTAs per SM), else the 16-warp one.
bool single_usable(const q4_chain_link& l) { return single_fits(l, kWarps); }

cudaError_t single_launch(const q4_chain_link& l, void* workspace, int32_t* status, uint32_t flags,
                          cudaStream_t s) {
  SingleArgs a;
  a.R = static_cast<const uint8_t*>(l.R);
  a.x = l.x.ptr + l.x.offset;
  a.residual = (l.ops & Q4_OP_RESIDUAL) ? l.residual.ptr + l.residual.offset : nullptr;
  a.y = l.y;
  a.argmax = l.argmax;
  a.hdr = static_cast<uint32_t*>(workspace);
  a.status = status;
  a.n = static_cast<int32_t>(l.n);
  a.k = static_cast<int32_t>(l.k);
  a.nsb = static_cast<int32_t>(l.k / 256);
  a.groups = static_cast<int32_t>((l.n + 15) / 16);
  a.ops = l.ops;
  a.flags = flags;
  const bool pdl = (flags & Q4_FLAG_PDL) != 0;
  if (pdl && single_fits(l, 8)) return single_launch_nw<8>(a, true, s);
  return single_launch_nw<kWarps>(a, pdl, s);
}

cudaError_t repack_launch(const uint8_t* W, int64_t n, int64_t k, uint8_t* R, cudaStream_t s) {
  const int64_t work = (n + 15) / 16 * (k / 256) * 128;  // (tile, lane, step quad)
  const int64_t blocks = (work + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(W, n, k, R);
  return cudaGetLastError();
}

}  // namespace q4

// ------------------------------------------------------------------ C ABI
extern "C" {

size_t q4_repack_bytes(int64_t n, int64_t k) {
  if (n <= 0 || k <= 0 || k % 256 != 0 || n > (int64_t(1) << 40) || k > (int64_t(1) << 40))
    return 0;
  return static_cast<size_t>((n + 15) / 16 * (k / 256)) * q4::rt::kTileBytes;
}

q4_status q4_repack(const void* W, int64_t n, int64_t k, void* R, q4_stream_t s) {
  if (W == nullptr || R == nullptr || n <= 0 || k <= 0 || n > (int64_t(1) << 40) ||
      k > (int64_t(1) << 40))
    return Q4_ERR_INVALID_ARG;
  if (k % 256 != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (!q4::aligned(W, 16) || !q4::aligned(R, 16)) return Q4_ERR_MISALIGNED;
  return q4::repack_launch(static_cast<const uint8_t*>(W), n, k, static_cast<uint8_t*>(R),
                           reinterpret_cast<cudaStream_t>(s)) == cudaSuccess
             ? Q4_OK
             : Q4_ERR_CUDA;
}

size_t q4_chain_workspace_bytes(const q4_chain_link* links, int32_t n_links) {
  size_t ws = 0;
  return q4::chain_plan(links, n_links, nullptr, &ws) == Q4_OK ? ws : 0;
}

q4_status q4_chain(const q4_chain_link* links, int32_t n_links, void* workspace, size_t ws_bytes,
                   int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  static thread_local q4::ChainArgs A;  // ~14 KB: kept off the stack
  size_t need = 0;
  q4_status st = q4::chain_plan(links, n_links, &A, &need);
  if (st != Q4_OK) return st;
  if (workspace == nullptr || ws_bytes < need) return Q4_ERR_WORKSPACE;
  if (!q4::aligned(workspace, 256)) return Q4_ERR_MISALIGNED;
  A.status = status_dev;
  A.flags = flags;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  const cudaError_t e = (n_links == 1 && q4::single_usable(links[0]))
                            ? q4::single_launch(links[0], workspace, status_dev, flags, cs)
                            : q4::chain_launch(A, workspace, cs);
  return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

static q4_chain_link one_link(const void* R, int64_t n, int64_t k, const float* x, float* y) {
  q4_chain_link l = {};
  l.R = R;
  l.n = n;
  l.k = k;
  l.x.ptr = x;
  l.x.link = -1;
  l.residual.link = -1;
  l.y = y;
  return l;
}

size_t q4_gemv_r_workspace_bytes(int64_t n, int64_t k) {
  const q4_chain_link l = one_link(reinterpret_cast<const void*>(16), n, k,
                                   reinterpret_cast<const float*>(16), nullptr);
  return q4_chain_workspace_bytes(&l, 1);
}

q4_status q4_gemv_r(const void* R, int64_t n, int64_t k, const float* x, float* y, void* workspace,
                    size_t ws_bytes, int32_t* status_dev, uint32_t flags, q4_stream_t s) {
  if (x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
  const q4_chain_link l = one_link(R, n, k, x, y);
  return q4_chain(&l, 1, workspace, ws_bytes, status_dev, flags, s);
}

}  // extern "C"
