// k_tc.cu -- decode projection y = x·Wᵀ on the tcgen05 tensor cores, for
// 17 <= M <= 64 tokens (16 when forced), where the projection is a real dense
// contraction (up to 64 flops per weight byte).
//
// Swap-AB: the weight tile is the MMA's A operand (128 rows x 64 k, K-major,
// 128B swizzle, straight from TMA) and the token tile its B operand (N = M
// rounded up to 16). The 128 x N fp32 accumulator lives in tensor memory,
// double-buffered so the epilogue of one output tile overlaps the MMAs of
// the next. Work is split stream-K exactly as in the CUDA-core/mma.sync
// kernel: one contiguous range of (tile, 128-wide k chunk) units per CTA,
// tiles shared by several CTAs finished by the last arriver in CTA order.
//
// Warp roles: warp 0 issues TMA, warp 1 allocates tensor memory and issues
// the MMAs (one thread), warps 2-9 drain the accumulator: each warp owns the
// 32 tensor-memory lanes of its quarter (warp % 4) and half of the token
// columns, so the split-K reduction of a tile's partials is spread over 256
// threads. For N with few 128-row tiles a second kernel splits each tile over
// the CTAs of a thread-block cluster instead (below), two CTAs per SM.
//
// "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 "针对工作负载调优形状"
// (split-K projections at larger batch).
#include <utility>

#include "launch.h"
#include "launch_util.cuh"
#include "tc_common.cuh"
#include "wstream.cuh"

namespace dg {

constexpr int kTcStages = 4;
constexpr int kTcXRows = 64;
constexpr int kTcXSub = kTcXRows * 128;                   // 8 KB per box column
constexpr int kTcThreads = 320;
constexpr int kTcEpi = 256;    // 8 epilogue warps: two per tensor-memory lane quarter
constexpr int kTcCols = kTcXRows / 2;  // token columns each epilogue warp drains

// PAIRED (SwiGLU gate/up): each stage holds the 128 gate rows of a tile and
// the 128 matching up rows (a.w_up_offset further down the weight); two MMAs
// per k step fill a gate and an up accumulator, and the epilogue writes
// bf16(silu(gate) * up). Two 80 KB stages; 256 tensor-memory columns.
template <bool PAIRED>
struct TcShape {
  static constexpr int kWB = (PAIRED ? 2 : 1) * kWBytes;       // weight bytes per stage
  static constexpr int kStage = kWB + kKSub * kTcXSub;         // stage bytes
  static constexpr int kStages = PAIRED ? 2 : kTcStages;
  static constexpr int kAcc = PAIRED ? 128 : 64;               // tensor-memory columns per tile
  static constexpr int kCols = 2 * kAcc;                       // double-buffered
  static constexpr int kStride = PAIRED ? 2 * kTileRows : kTileRows;  // floats per token in a slot
};

template <bool PAIRED = false>
constexpr int tc_smem() {
  return 1024 + TcShape<PAIRED>::kStages * TcShape<PAIRED>::kStage +
         8 * (2 * TcShape<PAIRED>::kStages + 5) + 64 + 4 * kMaxSlots;
}

template <int EPI, bool PAIRED = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_linear_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                     const StreamArgs a, const int NP, const uint32_t idesc) {
  using Sh = TcShape<PAIRED>;
  constexpr int kStages = Sh::kStages, kStage = Sh::kStage, kWB = Sh::kWB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStage);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;     // [2] accumulator ready
  uint64_t* tempty = tfull + 2;          // [2] accumulator drained
  uint64_t* mma_done = tempty + 2;       // [1]
  volatile int* s_flags = reinterpret_cast<volatile int*>(mma_done + 1);  // [0] abort [1] last
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(const_cast<int*>(s_flags) + 8);
  int* s_slot = reinterpret_cast<int*>(s_taddr + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kTcEpi / 32);
    }
    mbar_init(mma_done, 1);
    s_flags[0] = 0;
    s_flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_taddr, Sh::kCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&wmap);
    prefetch_tmap(&xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *s_taddr;
  griddep_launch_dependents();

  const int KB = a.KB, TILES = a.TILES;
  const long long T = (long long)TILES * KB;
  const long long c = blockIdx.x;
  const long long G = (long long)gridDim.x < T ? (long long)gridDim.x : T;
  const long long u0 = c < G ? cta_start(c, T, G) : 0;
  const long long u1 = c < G ? cta_start(c + 1, T, G) : 0;
  const int nunits = (int)(u1 - u0);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t bytes = kWB + kKSub * NP * 128;
      // unit positions advance one unit at a time (no division per stage)
      auto issue_w = [&](int s, const UnitPos& p) {
#pragma unroll
        for (int sb = 0; sb < kKSub; ++sb) {
          tma_load_2d(smem + s * kStage + sb * kWSub, &wmap, (p.kc * kKSub + sb) * kKBlk,
                      p.tile * kTileRows, &full[s], pol_w);
          if (PAIRED)  // the matching up rows
            tma_load_2d(smem + s * kStage + kWBytes + sb * kWSub, &wmap,
                        (p.kc * kKSub + sb) * kKBlk, a.w_up_offset + p.tile * kTileRows, &full[s],
                        pol_w);
        }
      };
      auto issue_x = [&](int s, const UnitPos& p) {
#pragma unroll
        for (int sb = 0; sb < kKSub; ++sb)
          tma_load_2d(smem + s * kStage + kWB + sb * kTcXSub, &xmap,
                      (p.kc * kKSub + sb) * kKBlk, 0, &full[s], pol_x);
      };
      // weights first (independent of the previous kernel), then tokens
      const int npre = nunits < kStages ? nunits : kStages;
      const UnitPos pos0 = unit_pos(u0, KB, TILES);
      UnitPos pos = pos0;
      int i = 0;
      for (; i < npre; ++i, pos.next(KB, TILES)) {
        mbar_arrive_expect_tx(&full[i], bytes);
        issue_w(i, pos);
      }
      griddep_wait();
      UnitPos px = pos0;
      for (int j = 0; j < npre; ++j, px.next(KB, TILES)) issue_x(j, px);
      for (; i < nunits; ++i, pos.next(KB, TILES)) {
        const int s = i % kStages;
        if (!mbar_wait(&empty[s], ((i / kStages) + 1) & 1, a.timeout_ns, a.status)) {
          s_flags[0] = 1;
          break;
        }
        if (s_flags[0]) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        issue_w(s, pos);
        issue_x(s, pos);
      }
      const int issued = i;
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int uses = (issued - s + kStages - 1) / kStages;
        mbar_wait(&full[s], (uses - 1) & 1, drain_ns(a.timeout_ns), nullptr);
      }
    } else {
      griddep_wait();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    griddep_wait();
    if (lane == 0) {
      long long cur = -1;
      int jt = -1;
      long long gt_next = u0 / KB;  // tile of unit u0 + i, advanced with its k chunk
      int kc_next = (int)(u0 - gt_next * KB);
      for (int i = 0; i < nunits; ++i) {
        const long long gt = gt_next;
        const bool tile_end = ++kc_next == KB;
        if (tile_end) {
          kc_next = 0;
          ++gt_next;
        }
        const bool first = gt != cur;
        if (first) {
          cur = gt;
          ++jt;
          if (jt >= 2 && !s_flags[0]) {
            if (!mbar_wait(&tempty[jt & 1], ((jt >> 1) - 1) & 1, a.timeout_ns, a.status))
              s_flags[0] = 1;
          }
          tc_fence_after();
        }
        const int s = i % kStages;
        if (!s_flags[0]) {
          if (!mbar_wait(&full[s], (i / kStages) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
        }
        tc_fence_after();
        const uint32_t d = taddr + (uint32_t)((jt & 1) * Sh::kAcc);
        if (!s_flags[0]) {
          const uint32_t wb = smem_u32(smem + s * kStage);
          const uint32_t xb = wb + kWB;
#pragma unroll
          for (int sb = 0; sb < kKSub; ++sb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (first && sb == 0 && kk == 0) ? 0u : 1u;
              const uint64_t bd = umma_desc_sw128(xb + sb * kTcXSub + kk * 32);
              umma_bf16(d, umma_desc_sw128(wb + sb * kWSub + kk * 32), bd, idesc, acc);
              if (PAIRED)  // up rows into the second accumulator of the tile
                umma_bf16(d + 64, umma_desc_sw128(wb + kWBytes + sb * kWSub + kk * 32), bd, idesc,
                          acc);
            }
        }
        umma_commit(&empty[s]);
        if (i == nunits - 1 || tile_end) umma_commit(&tfull[jt & 1]);
      }
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, drain_ns(a.timeout_ns), nullptr);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    griddep_wait();
    const int et = threadIdx.x - 64;         // 0..255
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;        // which half of the token columns it drains
    const int r = quarter * 32 + lane;       // tile row = TMEM lane
    const int t0 = half * kTcCols;           // first token column of this warp
    const GroupInfo gi{0, 0, a.M};
    if (nunits > 0) {
      const long long gfirst = u0 / KB, glast = (u1 - 1) / KB;
      int jt = -1;
      for (long long gt = gfirst; gt <= glast; ++gt) {
        ++jt;
        const int buf = jt & 1;
        if (!s_flags[0]) {
          if (!mbar_wait(&tfull[buf], (jt >> 1) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
        }
        tc_fence_after();
        float v[kTcCols];
        float vu[PAIRED ? kTcCols : 1];  // up sums (SwiGLU tiles)
#pragma unroll
        for (int cc = 0; cc < kTcCols / 16; ++cc)
          if (t0 + cc * 16 < NP) {
            const uint32_t ta = taddr + ((uint32_t)(quarter * 32) << 16) +
                                (uint32_t)(buf * Sh::kAcc + t0 + cc * 16);
            tmem_ld16_sync(ta, v + cc * 16);
            if constexpr (PAIRED) tmem_ld16_sync(ta + 64, vu + cc * 16);
          }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        const bool aborted = s_flags[0] != 0;
        const int tile = (int)gt;
        const int n = tile * kTileRows + r;
        const bool whole = (u0 <= gt * KB) && ((gt + 1) * KB <= u1);
        if (whole) {
          if (!aborted && n < a.nout) {
#pragma unroll
            for (int t = 0; t < kTcCols; ++t)
              if (t0 + t < gi.c) {
                if constexpr (PAIRED) store_swiglu(a, gi, t0 + t, n, v[t], vu[t]);
                else store_out<EPI, false>(a, gi, t0 + t, n, v[t]);
              }
          }
        } else {
          // slot [token][kStride]: the tile's rows, then (SwiGLU) its up rows
          constexpr long long kSlotFloats = (long long)Sh::kStride * kTcXRows;
          const int slot = (gt == u0 / KB) ? 0 : 1;
          const long long mine = (c * 2 + slot) * kSlotFloats;
#pragma unroll
          for (int t = 0; t < kTcCols; ++t)
            if (t0 + t < gi.c) {
              const long long o = mine + (t0 + t) * Sh::kStride + r;
              __stcg(DG_AT(a.status, a.ws, o, a.ws_len), v[t]);
              if constexpr (PAIRED) __stcg(DG_AT(a.status, a.ws, o + kTileRows, a.ws_len), vu[t]);
            }
          named_bar_sync(1, kTcEpi);
          const long long cf = cta_of(gt * KB, T, G);
          const long long cl = cta_of((gt + 1) * KB - 1, T, G);
          // barrier + release (and acquire + barrier on the last arriver)
          // order the partial slots; no separate fence needed
          if (et == 0) {
            int* cp = DG_AT(a.status, a.ctr, gt, a.ctr_len);
            const int old = atomic_add_acq_rel_gpu(cp, 1);
            const int is_last = (old == (int)(cl - cf)) ? 1 : 0;
            if (is_last) *cp = 0;
            s_flags[1] = is_last;
          }
          named_bar_sync(1, kTcEpi);
          if (s_flags[1]) {
            const int nc = (int)(cl - cf + 1);
            auto slot_of = [&](int j) -> long long {
              const long long cc = cf + j;
              return cc * 2 + ((gt == cta_start(cc, T, G) / KB) ? 0 : 1);
            };
            for (int j = et; j < nc && j < kMaxSlots; j += kTcEpi) s_slot[j] = (int)slot_of(j);
            named_bar_sync(1, kTcEpi);
            if (!aborted) {
              auto slot_at = [&](int j) -> long long {
                return j < kMaxSlots ? (long long)s_slot[j] : slot_of(j);
              };
              auto store = [&](int t, int rr, float v0, float v1) {
                const int nn = tile * kTileRows + rr;
                if (nn >= a.nout) return;
                if constexpr (PAIRED) store_swiglu(a, gi, t, nn, v0, v1);
                else store_out<EPI, false>(a, gi, t, nn, v0);
              };
              // 16 loads in flight per thread (4 items x 4 contributors), or
              // 8 for SwiGLU tiles (2 items x 2 contributors x (gate, up)),
              // whose 64 gate and up sums take most of the registers
              reduce_partials<kTcEpi, PAIRED, Sh::kStride, PAIRED ? 2 : 4, PAIRED ? 2 : 4>(
                  a.ws, kSlotFloats, nc, gi.c, et, slot_at, store, a.ws_len, a.status);
            }
          }
          named_bar_sync(1, kTcEpi);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(taddr, Sh::kCols);
  }
}

// ------------------------------------------------------------------ cluster split
// Small N: cluster i of S CTAs owns output tile i, rank r streams the r-th of
// S equal shares of its k chunks into one tensor-memory accumulator; after a
// cluster barrier every thread stores its row of the accumulator into the
// shared memory of the rank that owns the row, and after a second barrier
// each rank sums its rows over the S partials in rank order. No global
// partials, counters or atomics, deterministic. Two 48 KB stages (128 k) or
// four of 24 KB (64 k) keep a CTA near 100 KB of shared memory, so two fit on
// an SM: a call's CTAs load their first weight stages while the previous
// call's CTAs on those SMs finish.
constexpr int kTcClCols = 64;  // one accumulator of up to 64 token columns

// Stage shape of the cluster kernel: KSUB boxes of 64 k per stage (weights
// 128 rows x 64 k = 16 KB and 64 token rows x 64 k = 8 KB each), as many
// stages as fit in ~100 KB (two CTAs per SM).
template <int KSUB>
struct TcCl {
  static constexpr int kStage = KSUB * (kWSub + kTcXSub);
  static constexpr int kStages = (115712 - 1024 - 256) / kStage;
  static constexpr int kSmem = 1024 + kStages * kStage + 8 * (2 * kStages + 1) + 64;
  static_assert(kTileRows * kTcXRows * 4 <= kStages * kStage, "partial tile fits");
};

// ROUTE: the router's product (EPI_F32 logits); the last of the TILES clusters
// to write its logits then selects every token's top-k experts and gates.
template <int EPI, int KSUB, bool ROUTE = false>
__global__ void __launch_bounds__(kTcThreads, 2)
    tc_cluster_kernel(const __grid_constant__ CUtensorMap wmap,
                      const __grid_constant__ CUtensorMap xmap, const StreamArgs a, const int NP,
                      const uint32_t idesc) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int kTcClStages = TcCl<KSUB>::kStages, kStageB = TcCl<KSUB>::kStage;
  constexpr int kWB = KSUB * kWSub;  // weight bytes per stage
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcClStages * kStageB);
  uint64_t* empty = full + kTcClStages;
  uint64_t* tfull = empty + kTcClStages;  // [1] accumulator complete
  volatile int* s_flags = reinterpret_cast<volatile int*>(tfull + 1);  // [0] abort [2] route
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(const_cast<int*>(s_flags) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcClStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_taddr, kTcClCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&wmap);
    prefetch_tmap(&xmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *s_taddr;
  griddep_launch_dependents();

  const int KB = a.KB;
  const int cs = (int)cluster_size(), cr = (int)cluster_rank();
  // epilogue warps (2-9): the accumulator's row r, token columns t0..t0+31
  const int quarter = warp & 3;      // TMEM lanes this warp may access
  const int half = (warp - 2) >> 2;  // which half of the token columns it drains
  const int r = quarter * 32 + lane;
  const int t0 = half * kTcCols;
  float v[kTcCols];
  const int tile = (int)(blockIdx.x / cs);
  const int kc0 = cr * KB / cs;
  const int nunits = (cr + 1) * KB / cs - kc0;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t bytes = kWB + KSUB * NP * 128;
      auto issue_w = [&](int s, int kc) {
#pragma unroll
        for (int sb = 0; sb < KSUB; ++sb)
          tma_load_2d(smem + s * kStageB + sb * kWSub, &wmap, (kc * KSUB + sb) * kKBlk,
                      tile * kTileRows, &full[s], pol_w);
      };
      auto issue_x = [&](int s, int kc) {
#pragma unroll
        for (int sb = 0; sb < KSUB; ++sb)
          tma_load_2d(smem + s * kStageB + kWB + sb * kTcXSub, &xmap,
                      (kc * KSUB + sb) * kKBlk, 0, &full[s], pol_x);
      };
      // weights first (independent of the previous kernel), then tokens
      const int npre = nunits < kTcClStages ? nunits : kTcClStages;
      int i = 0;
      for (; i < npre; ++i) {
        mbar_arrive_expect_tx(&full[i], bytes);
        issue_w(i, kc0 + i);
      }
      griddep_wait();
      for (int j = 0; j < npre; ++j) issue_x(j, kc0 + j);
      for (; i < nunits; ++i) {
        const int s = i % kTcClStages;
        if (!mbar_wait(&empty[s], ((i / kTcClStages) + 1) & 1, a.timeout_ns, a.status)) {
          s_flags[0] = 1;
          break;
        }
        if (s_flags[0]) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        issue_w(s, kc0 + i);
        issue_x(s, kc0 + i);
      }
      const int issued = i;
      for (int s = 0; s < kTcClStages && s < issued; ++s) {
        const int uses = (issued - s + kTcClStages - 1) / kTcClStages;
        mbar_wait(&full[s], (uses - 1) & 1, drain_ns(a.timeout_ns), nullptr);
      }
    } else {
      griddep_wait();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    griddep_wait();
    if (lane == 0) {
      for (int i = 0; i < nunits; ++i) {
        const int s = i % kTcClStages;
        if (!s_flags[0]) {
          if (!mbar_wait(&full[s], (i / kTcClStages) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
        }
        tc_fence_after();
        if (!s_flags[0]) {
          const uint32_t wb = smem_u32(smem + s * kStageB);
          const uint32_t xb = wb + kWB;
#pragma unroll
          for (int sb = 0; sb < KSUB; ++sb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = umma_desc_sw128(wb + sb * kWSub + kk * 32);
              const uint64_t bd = umma_desc_sw128(xb + sb * kTcXSub + kk * 32);
              umma_bf16(taddr, ad, bd, idesc, (i == 0 && sb == 0 && kk == 0) ? 0u : 1u);
            }
        }
        umma_commit(&empty[s]);
      }
      // every MMA above is complete (and so every stage read) when this fires
      umma_commit(tfull);
      // The epilogue waits for it too, but gives up with the caller's bound:
      // the tensor memory is freed only once every MMA has completed.
      mbar_wait(tfull, 0, drain_ns(a.timeout_ns), nullptr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    griddep_wait();
    if (!s_flags[0]) {
      if (!mbar_wait(tfull, 0, a.timeout_ns, a.status)) s_flags[0] = 1;
    }
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < kTcCols / 16; ++cc)
      if (t0 + cc * 16 < NP)
        tmem_ld16_sync(taddr + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(t0 + cc * 16),
                       v + cc * 16);
    tc_fence_before();
  }
  // Rank q owns rows [q*R4, q*R4 + R4) of the tile (R4 = 128/cs rounded up to
  // a multiple of 4, the last run cut at 128). After a first barrier (every
  // rank's MMAs, and so its copies, are complete: its stage memory is free)
  // each thread stores its row of the drained accumulator straight into the
  // owner's shared memory, recv[source rank][token][row - owner's first row];
  // after a second barrier each rank sums its rows over the sources in rank
  // order from its own shared memory. Remote stores are posted: no remote
  // round trip (a version that loaded the partials from the other ranks took
  // ~2 us at 64 tokens).
  const int R4 = ((kTileRows + cs - 1) / cs + 3) / 4 * 4;
  float* recv = reinterpret_cast<float*>(smem);
  __syncwarp();
  cluster_sync_all();
  if (warp >= 2 && !s_flags[0]) {
    const int q = r / R4, rl = r - q * R4;
    float* dst = recv + (size_t)cr * kTcXRows * R4 + rl;  // this rank's slot in rank q
#pragma unroll
    for (int t = 0; t < kTcCols; ++t)
      if (t0 + t < a.M) st_dsmem_f32(dst + (t0 + t) * R4, (uint32_t)q, v[t]);
  }
  __syncwarp();
  cluster_sync_all();
  if (warp >= 2 && !s_flags[0]) {
    const int r0 = cr * R4 < kTileRows ? cr * R4 : kTileRows;
    const int r1 = r0 + R4 < kTileRows ? r0 + R4 : kTileRows;
    const int RR = r1 - r0;
    const GroupInfo gi{0, 0, a.M};
    for (int e = threadIdx.x - 64; e < RR * a.M; e += kTcEpi) {
      const int t = e / RR, rl = e - t * RR;
      float acc = 0.f;
      for (int src = 0; src < cs; ++src) acc += recv[((size_t)src * kTcXRows + t) * R4 + rl];
      const int n = tile * kTileRows + r0 + rl;
      if (n < a.nout) store_out<EPI, false>(a, gi, t, n, acc);
    }
  }
  if (ROUTE && a.route_k > 0) {
    // This cluster's logits are written (the barrier orders every thread's
    // stores before the release of the arrival below). The last of the TILES
    // clusters to arrive acquires them all and selects the experts: its
    // epilogue warps take the tokens in turn.
    __syncwarp();
    cluster_sync_all();
    if (cr == 0 && threadIdx.x == 0) {
      const int old = atomic_add_acq_rel_gpu(a.route_ctr, 1);
      const int last = old == a.TILES - 1 ? 1 : 0;
      if (last) *a.route_ctr = 0;
      for (int q = 0; q < cs; ++q) st_dsmem_s32(const_cast<int*>(&s_flags[2]), (uint32_t)q, last);
    }
    __syncwarp();
    cluster_sync_all();
    if (s_flags[2] && warp >= 2) {
      const int K = a.route_k, nwc = kTcEpi / 32;
      for (int m = cr * nwc + (warp - 2); m < a.M; m += cs * nwc)
        if (DG_OK(a.status, (long long)(m + 1) * K <= a.pairs &&
                                (long long)m * a.ldo + a.route_E <= a.out_len, m))
          warp_topk_gates(reinterpret_cast<const float*>(a.out) + (long long)m * a.ldo, a.route_E,
                          K, lane, a.route_idx + m * K, a.route_gate + m * K,
                          a.route_idx_user ? a.route_idx_user + m * K : nullptr,
                          a.route_w_user ? a.route_w_user + m * K : nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(taddr, kTcClCols);
  }
}

template <int EPI, int KSUB>
static cudaError_t run_tc_cluster(const Ctx& cx, const void* x, const void* W, const void* res,
                                  void* y, int M, int N, int K, int cl) {
  constexpr int SMEM = TcCl<KSUB>::kSmem;
  static_assert(2 * (SMEM + 1024) <= kSmemPerSm, "two CTAs per SM");
  auto kern = tc_cluster_kernel<EPI, KSUB>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM, true); e != cudaSuccess) return e;
  const int NP = (M + 15) / 16 * 16;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W, (uint64_t)N, (uint64_t)K, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)K, (uint32_t)NP, false, (uint64_t)cx.ldx))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = K;
  a.KB = (K + KSUB * kKBlk - 1) / (KSUB * kKBlk);  // work units of KSUB boxes
  a.TILES = (N + kTileRows - 1) / kTileRows;
  a.nout = N;
  a.M = M;
  a.out = y;
  a.ldo = N;
  a.res = reinterpret_cast<const uint16_t*>(res);
  a.status = cx.status;
  a.out_len = (long long)M * N;
  a.res_len = res ? (long long)M * N : 0;
  a.timeout_ns = cx.timeout_ns;
  return launch_kc(kern, dim3(a.TILES * cl), dim3(kTcThreads), SMEM, cx.stream, cx.pdl, cl, wmap,
                   xmap, a, NP, umma_idesc_bf16(128, NP));
}

cudaError_t launch_dense_tc_cluster(const Ctx& cx, bool residual, const void* x, const void* W,
                                    const void* res, void* y, int M, int N, int K, int cl) {
  if (M < 16 || M > kTcXRows || cl < 2 || cl > 8 || cl > (K + kKChunk - 1) / kKChunk)
    return cudaErrorInvalidValue;
  // Stages of 64 k (four of 24 KB) when each rank streams 768 k or more,
  // else of 128 k (two of 48 KB). Same-GPU A/B, us, 128-k -> 64-k stages:
  // 2048 x 7168 at M = 17 / 32 / 64: 9.55 / 9.88 / 11.46 -> 9.40 / 9.77 /
  // 10.94; 2048 x 16384 at M = 32 / 64: 17.1 / 18.9 -> 16.2 / 17.5; but
  // 2048 x 4096 at M = 24 (512 k per rank): 7.15 -> 7.37.
  if (K / cl >= 768)
    return residual ? run_tc_cluster<EPI_BF16_RES, 1>(cx, x, W, res, y, M, N, K, cl)
                    : run_tc_cluster<EPI_BF16, 1>(cx, x, W, res, y, M, N, K, cl);
  return residual ? run_tc_cluster<EPI_BF16_RES, 2>(cx, x, W, res, y, M, N, K, cl)
                  : run_tc_cluster<EPI_BF16, 2>(cx, x, W, res, y, M, N, K, cl);
}

// Router scores and top-k on the tensor cores (17-64 tokens): logits =
// x·Wrᵀ in fp32 over E + L rows (router rows, then the latent input rows),
// cl CTAs per 128-row tile in one cluster, the top-k of the first E columns
// in the last cluster.
template <int KSUB>
static cudaError_t run_router_tc(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E,
                                 int L, int k, int cl, const RouteOut& ro) {
  constexpr int SMEM = TcCl<KSUB>::kSmem;
  auto kern = tc_cluster_kernel<EPI_F32, KSUB, true>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM, true); e != cudaSuccess) return e;
  const int N = E + L, NP = (M + 15) / 16 * 16;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Wr, (uint64_t)N, (uint64_t)H, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)H, (uint32_t)NP, false))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = H;
  a.KB = (H + KSUB * kKBlk - 1) / (KSUB * kKBlk);
  a.TILES = (N + kTileRows - 1) / kTileRows;
  a.nout = N;
  a.M = M;
  a.out = ro.logits;
  a.ldo = N;
  a.status = cx.status;
  a.out_len = (long long)M * N;
  a.timeout_ns = cx.timeout_ns;
  a.route_k = k;
  a.route_E = E;
  a.route_ctr = ro.ctr;
  a.route_idx = ro.idx;
  a.route_gate = ro.gate;
  a.route_idx_user = ro.idx_user;
  a.route_w_user = ro.w_user;
  a.pairs = M * k;
  return launch_kc(kern, dim3(a.TILES * cl), dim3(kTcThreads), SMEM, cx.stream, cx.pdl, cl, wmap,
                   xmap, a, NP, umma_idesc_bf16(128, NP));
}

cudaError_t launch_router_tc(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E,
                             int L, int k, int cl, const RouteOut& ro) {
  if (M < 16 || M > kTcXRows || cl < 1 || cl > 8 || cl > (H + kKChunk - 1) / kKChunk)
    return cudaErrorInvalidValue;
  if (H / cl >= 768) return run_router_tc<1>(cx, x, Wr, M, H, E, L, k, cl, ro);
  return run_router_tc<2>(cx, x, Wr, M, H, E, L, k, cl, ro);
}

// PAIRED: W is [2I, K] (gate rows, then up rows) and N = I; y = bf16(silu(x·W1ᵀ)
// * (x·W3ᵀ)) is [M, I].
template <int EPI, bool PAIRED = false>
static cudaError_t run_tc(const Ctx& cx, const void* x, const void* W, const void* res, void* y,
                          int M, int N, int K, int grid, float* ws, int* ctr) {
  constexpr int SMEM = tc_smem<PAIRED>();
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = tc_linear_kernel<EPI, PAIRED>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  const int NP = (M + 15) / 16 * 16;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W, (uint64_t)(PAIRED ? 2 * N : N), (uint64_t)K, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)K, (uint32_t)NP, false, (uint64_t)cx.ldx))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = K;
  a.KB = (K + kKChunk - 1) / kKChunk;
  a.TILES = (N + kTileRows - 1) / kTileRows;
  a.nout = N;
  a.M = M;
  a.out = y;
  a.ldo = N;
  a.res = reinterpret_cast<const uint16_t*>(res);
  a.ws = ws;
  a.ctr = ctr;
  a.status = cx.status;
  a.out_len = (long long)M * N;
  a.res_len = res ? (long long)M * N : 0;
  a.ws_len = cx.ws_len;
  a.ctr_len = cx.ctr_len;
  a.timeout_ns = cx.timeout_ns;
  a.w_up_offset = PAIRED ? N : 0;
  const long long T = (long long)a.TILES * a.KB;
  if (grid > T) grid = (int)T;
  return launch_k(kern, dim3(grid), dim3(kTcThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a, NP,
                  umma_idesc_bf16(128, NP));
}

cudaError_t launch_dense_tc_f32(const Ctx& cx, const void* x, const void* W, float* y, int M, int N,
                                int K, int grid, float* ws, int* ctr) {
  if (M < 16 || M > kTcXRows) return cudaErrorInvalidValue;
  return run_tc<EPI_F32>(cx, x, W, nullptr, y, M, N, K, grid, ws, ctr);
}

cudaError_t launch_swiglu_tc(const Ctx& cx, const void* x, const void* W13, void* h, int M, int I,
                             int K, int grid, float* ws, int* ctr) {
  if (M < 16 || M > kTcXRows) return cudaErrorInvalidValue;
  return run_tc<EPI_SWIGLU, true>(cx, x, W13, nullptr, h, M, I, K, grid, ws, ctr);
}

cudaError_t launch_dense_tc(const Ctx& cx, bool residual, const void* x, const void* W,
                            const void* res, void* y, int M, int N, int K, int grid, float* ws,
                            int* ctr) {
  if (M < 16 || M > kTcXRows) return cudaErrorInvalidValue;
  return residual ? run_tc<EPI_BF16_RES>(cx, x, W, res, y, M, N, K, grid, ws, ctr)
                  : run_tc<EPI_BF16>(cx, x, W, res, y, M, N, K, grid, ws, ctr);
}

}  // namespace dg
