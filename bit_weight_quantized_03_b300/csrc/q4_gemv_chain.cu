// q4_gemv_chain.cu -- a chain of dependent batch-1 Q4_0 GEMVs in one persistent
// launch:  for s = 0, 1, ...:  y_s = W_s x_s,  where x_s may be (a slice of)
// y_{s-1} or any external vector.
//
// One decode step of the Voxtral Mini 4B Realtime port is such a chain: the
// per-token products of its 26 decoder layers (GeekNews,
// es.news.hada.io/topic?id=26595, "Arquitectura": hidden 3072, GQA 32Q/8KV),
// each reading the previous product's output.  Launched one GEMV at a time,
// every link pays a launch, a cold weight fetch and a split-K hand-off before
// the next can start.  Here the links run inside one cooperative grid of one
// 16-warp CTA per SM and the weight stream never stops: while an SM waits for
// the previous link to finish everywhere, its TMA rings already hold the
// next link's first tiles.
//
// Work split of a link with G row groups (32 rows) and nsb slices of 256 k:
//   * it is cut into items = (group, K-split p of P); P is chosen per link so
//     that the items fill the SMs evenly, and each CTA takes a contiguous run
//     of items (at most kMaxItems);
//   * inside the CTA the items' units (32 rows x 256 k, one 2-D TMA tile each)
//     are dealt to the 16 warps as contiguous ranges; warps that share an item
//     add their row sums in shared memory, in warp order;
//   * each item's sum is written once to a partial buffer part[s & 1][p][row]
//     in the workspace.  The link's output y_s is never reduced across SMs on
//     the critical path: after the grid-wide barrier each CTA sums the P
//     partials (in order, deterministic) while it stages x_{s+1} into shared
//     memory, and writes its share of the rows of y_s to the caller's buffer.
// The barrier is one counter in the workspace (release add per CTA, acquire
// poll by one thread, bounded); it is back at zero when the launch ends.
#include "q4_gemv_tile.cuh"

namespace q4 {
namespace {

using tile::unit_dot;
using tile::xpad_floats;
using tile::xpad_index;

constexpr int kWarps = 16;
constexpr int kStages = 2;                    // ring slots per warp
constexpr int kSlotBytes = 32 * kSuperBytes;  // 4608
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr int kPartBytes = kMaxChainItems * kWarps * 32 * 4;
constexpr int kSmemBudget = 219 * 1024;  // dynamic; the static tables take the rest

__device__ __forceinline__ void red_add_release_gpu(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ldcg_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// Bounded wait until *ctr >= target; false after kWaitLimitNs.
__device__ bool wait_counter(const int32_t* ctr, int target) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ld_acquire_gpu(ctr) >= target) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// The CTA's share of a link: items [i0, i1), holding `units` units in all.
struct Share {
  int i0, i1, units, pad;
};
__device__ __forceinline__ Share compute_share(const ChainStage& st, int c, int C) {
  Share sh;
  const int items = st.groups * st.P;
  sh.i0 = items * c / C;
  sh.i1 = items * (c + 1) / C;
  sh.units = 0;
  sh.pad = 0;
  for (int i = sh.i0; i < sh.i1; ++i) {
    const int p = i % st.P;
    sh.units += st.nsb * (p + 1) / st.P - st.nsb * p / st.P;
  }
  return sh;
}

// Walks one warp's units of link s in order: item, slice within the item.
struct Cursor {
  int s;          // link
  int item;       // current item
  int sb, sb_end; // current slice, end of the item's slices
  int left;       // units of this warp still to walk in link s
};

// Positions cur at the first unit of warp w in link s (left = 0 if it has none).
__device__ __forceinline__ void cursor_start(Cursor& cur, const ChainStage& st, const Share& sh,
                                             int s, int w) {
  const int u0 = sh.units * w / kWarps, u1 = sh.units * (w + 1) / kWarps;
  cur.s = s;
  cur.left = u1 - u0;
  int skip = u0, i = sh.i0;
  cur.item = i;
  cur.sb = 0;
  cur.sb_end = 0;
  if (cur.left == 0) return;
  for (; i < sh.i1; ++i) {
    const int p = i % st.P;
    const int a = st.nsb * p / st.P, b = st.nsb * (p + 1) / st.P;
    if (skip < b - a) {
      cur.item = i;
      cur.sb = a + skip;
      cur.sb_end = b;
      return;
    }
    skip -= b - a;
  }
}

__device__ __forceinline__ void cursor_next(Cursor& cur, const ChainStage& st) {
  --cur.left;
  if (cur.left == 0) return;
  if (++cur.sb == cur.sb_end) {
    ++cur.item;
    const int p = cur.item % st.P;
    cur.sb = st.nsb * p / st.P;
    cur.sb_end = st.nsb * (p + 1) / st.P;
  }
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    gemv_chain_kernel(const __grid_constant__ ChainParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ int abort_flag;
  // the links' parameters and this CTA's share of each, read from shared memory
  __shared__ ChainStage s_st[kMaxChain];
  __shared__ Share s_sh[kMaxChain];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = static_cast<int>(blockIdx.x), C = static_cast<int>(gridDim.x);
  const uint32_t ring = smem_u32(smem);
  const uint32_t slots = ring + warp * (kStages * kSlotBytes);
  float* part_smem = reinterpret_cast<float*>(smem + kRingBytes);  // [item][warp][32]
  const uint32_t xs = ring + kRingBytes + kPartBytes;
  float* xs_ptr = reinterpret_cast<float*>(smem + kRingBytes + kPartBytes);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);
  const uint64_t pol = l2_evict_first_policy();

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbarrier_init();
  }
  if (threadIdx.x == 0) abort_flag = 0;
  for (int t = threadIdx.x; t < P.n_stages; t += kWarps * 32) {
    s_st[t] = P.st[t];
    s_sh[t] = compute_share(P.st[t], c, C);
  }
  __syncthreads();

  // ---- producer: this warp's units across all links, issued ahead into the ring
  Cursor pc;
  int pseq = 0;  // units issued so far (sequence number of the next one)
  pc.s = 0;
  pc.left = 0;
  auto producer_settle = [&]() {  // move pc to the next link where this warp has units
    while (pc.left == 0 && pc.s < P.n_stages) {
      if (pc.s + 1 >= P.n_stages) {
        pc.s = P.n_stages;
        break;
      }
      cursor_start(pc, s_st[pc.s + 1], s_sh[pc.s + 1], pc.s + 1, warp);
    }
  };
  cursor_start(pc, s_st[0], s_sh[0], 0, warp);
  producer_settle();
  auto issue_next = [&]() {
    if (pc.s >= P.n_stages) return;
    if (lane == 0) {
      const ChainStage& st = s_st[pc.s];
      const int slot = pseq % kStages;
      const uint32_t bar = bar0 + 8 * slot;
      mbar_arrive_expect_tx(bar, kSlotBytes);
      tma_load_2d_hint(slots + slot * kSlotBytes, &P.tmap[pc.s],
                       static_cast<int32_t>(pc.sb * kSuperBytes),
                       static_cast<int32_t>((pc.item / st.P) * 32), bar, pol);
    }
    ++pseq;
    cursor_next(pc, s_st[pc.s]);
    producer_settle();
  };
  for (int i = 0; i < kStages; ++i) issue_next();

  pdl_allow_dependents();
  pdl_wait_prior_grid();

  const DecodeConsts dc = make_consts();
  const int j = lane & 3, rr = lane >> 2;
  int cseq = 0;  // units consumed so far
  bool ok = true;

  for (int s = 0; s <= P.n_stages; ++s) {
    // ---- wait until every CTA has finished link s - 1
    if (s > 0) {
      if (threadIdx.x == 0 && !abort_flag) {
        if (!wait_counter(P.done, C * s)) {
          abort_flag = 1;
          report(P.status, 6 /* Q4_ERR_TIMEOUT */);
        }
      }
      __syncthreads();
      if (abort_flag) break;
      // ---- write this CTA's share of y_{s-1} (sum of its P partials)
      const ChainStage& pv = s_st[s - 1];
      const float* part = P.part[(s - 1) & 1];
      const int r0 = pv.n * c / C;
      const int r1 = pv.n * (c + 1) / C;
      for (int r = r0 + static_cast<int>(threadIdx.x); r < r1; r += kWarps * 32) {
        float v = 0.f;
        for (int p = 0; p < pv.P; ++p) v += __ldcg(part + static_cast<int64_t>(p) * pv.n + r);
        pv.y[r] = v;
      }
    }
    if (s == P.n_stages) break;

    // ---- stage x_s into shared memory (padded layout)
    const ChainStage& st = s_st[s];
    const int k = st.nsb * kSuperElems;
    if (st.x_off >= 0) {
      const ChainStage& pv = s_st[s - 1];
      const float* part = P.part[(s - 1) & 1] + st.x_off;
      for (int e = 4 * static_cast<int>(threadIdx.x); e < k; e += 4 * kWarps * 32) {
        float4 v = ldcg_f4(part + e);
        for (int p = 1; p < pv.P; ++p) {
          const float4 u = ldcg_f4(part + static_cast<int64_t>(p) * pv.n + e);
          v.x += u.x;
          v.y += u.y;
          v.z += u.z;
          v.w += u.w;
        }
        *reinterpret_cast<float4*>(xs_ptr + xpad_index(e)) = v;
      }
    } else {
      for (int e = 4 * static_cast<int>(threadIdx.x); e < k; e += 4 * kWarps * 32)
        *reinterpret_cast<float4*>(xs_ptr + xpad_index(e)) = ldcg_f4(st.x + e);
    }
    __syncthreads();

    // ---- this warp's units of link s
    {
      Cursor cc;
      const Share& sh = s_sh[s];
      cursor_start(cc, st, sh, s, warp);
      float yv[4] = {0.f, 0.f, 0.f, 0.f};
      while (cc.left > 0 && ok) {
        const int slot = cseq % kStages;
        const uint32_t parity = static_cast<uint32_t>((cseq / kStages) & 1);
        const bool landed = mbar_wait(bar0 + 8 * slot, parity, &abort_flag);
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          if (lane == 0 && atomicExch(&abort_flag, 1) == 0) report(P.status, 6);
          break;
        }
        unit_dot(slots + slot * kSlotBytes, xs, cc.sb, j, rr, dc, yv);
        __syncwarp();
        fence_proxy_async_smem();
        ++cseq;
        issue_next();
        const bool item_end = (cc.sb + 1 == cc.sb_end) || (cc.left == 1);
        if (item_end) {
          // quad sum: the four lanes of a quad hold the same rows' block pairs
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float v = yv[i];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (j == 0) part_smem[((cc.item - sh.i0) * kWarps + warp) * 32 + rr + 8 * i] = v;
            yv[i] = 0.f;
          }
        }
        cursor_next(cc, st);
      }
    }
    __syncthreads();
    if (abort_flag) break;

    // ---- each item's row sums (warps in order) -> part[s & 1][p][row]
    {
      const Share& sh = s_sh[s];
      int u_lo = 0;
      for (int i = sh.i0; i < sh.i1; ++i) {
        const int p = i % st.P;
        const int len = st.nsb * (p + 1) / st.P - st.nsb * p / st.P;
        const int il = i - sh.i0;
        if ((il % kWarps) == warp) {
          const int w0 = ((u_lo + 1) * kWarps - 1) / sh.units;
          const int w1 = ((u_lo + len) * kWarps - 1) / sh.units;
          float v = 0.f;
          for (int w = w0; w <= w1; ++w)  // warps with no units hold no partial
            if (sh.units * w / kWarps < sh.units * (w + 1) / kWarps)
              v += part_smem[(il * kWarps + w) * 32 + lane];
          const int row = (i / st.P) * 32 + lane;
          if (row < st.n) P.part[s & 1][static_cast<int64_t>(p) * st.n + row] = v;
        }
        u_lo += len;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) red_add_release_gpu(P.done, 1);
  }

  // the last CTA to finish puts the counter back to zero for the next launch
  __syncthreads();
  if (threadIdx.x == 0 && !abort_flag) {
    const int old = atomicAdd(P.done, 1);
    if (old == C * (P.n_stages + 1) - 1) atomicExch(P.done, 0);
  }
  // let the copies this warp still has in flight land before the CTA exits
  for (int q = cseq; q < pseq; ++q)
    mbar_wait(bar0 + 8 * static_cast<uint32_t>(q % kStages),
              static_cast<uint32_t>((q / kStages) & 1));
}

}  // namespace

int64_t gemv_chain_max_k() {
  const int64_t avail = kSmemBudget - kRingBytes - kPartBytes;  // bytes for padded x
  int64_t k = avail / 4 * 64 / 68;
  return k / kSuperElems * kSuperElems;
}

int gemv_chain_split(int64_t groups, int64_t nsb, int ctas) {
  // Fewest units on the busiest CTA; ties go to fewer splits.
  int best = 1;
  int64_t best_cost = -1;
  for (int p = 1; p <= nsb && p <= 64; ++p) {
    const int64_t items = groups * p;
    const int64_t per_cta = (items + ctas - 1) / ctas;
    if (per_cta > kMaxChainItems) continue;
    const int64_t cost = per_cta * ((nsb + p - 1) / p);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = p;
    }
  }
  return best_cost < 0 ? 0 : best;
}

cudaError_t gemv_chain_launch(ChainParams& params, cudaStream_t s) {
  int64_t kmax = 0;
  for (int i = 0; i < params.n_stages; ++i)
    kmax = std::max<int64_t>(kmax, static_cast<int64_t>(params.st[i].nsb) * kSuperElems);
  const size_t smem = kRingBytes + kPartBytes + (xpad_floats(kmax) * 4 + 127) / 128 * 128;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemv_chain_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the barrier needs it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_chain_kernel, params);
}

}  // namespace q4
