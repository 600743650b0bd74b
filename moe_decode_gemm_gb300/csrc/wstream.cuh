// wstream.cuh -- persistent weight-streaming GEMM for decode shapes (swap-AB:
// weight rows are the long side, the 1..64 tokens the short side).
//
// One producer warp streams weight stages -- 128 weight rows x 128 k (two
// 128-row x 64-column bf16 TMA boxes with 128B swizzle, 32 KB), or twice that
// for SwiGLU gate/up pairs and 256-row tiles -- and the matching token tile
// into a ring of shared-memory stages; eight consumer warps reduce them. The
// work is the list of (group, output tile, 128-wide k chunk) units, cut into
// one contiguous range per CTA ("stream-K"), so every CTA streams the same
// number of weight bytes whatever the shape. An output tile whose k range
// spans several CTAs is finished by the last CTA to arrive on the tile's
// counter, which sums the partials in CTA order: the result does not depend on
// arrival order. Small projections instead split each tile over the CTAs of
// one thread-block cluster, which sum their partials through distributed
// shared memory.
//
// Consumers: a CUDA-core path for groups of fewer than mma_min_tokens tokens
// (the projections of 1-2 tokens: a GEMV has no dense contraction to give the
// tensor cores) and an mma.sync m16n8k16 path for the rest (every group of
// the MoE kernels, where it measured faster even at 1 token). Groups are the
// routed experts of an MoE block (the token list of each comes from the
// router's scheduler) or one dense matrix.
//
// Sources: "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 (small-matrix
// kernel at batch 1-2, split-K beyond) and Part 1 §3 (routed experts).
#pragma once

#include "dg_common.cuh"
#include "routing.cuh"

namespace dg {

constexpr int kNCW = 8;                    // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;  // + one producer warp
constexpr int kTileRows = 128;             // weight rows per stage
constexpr int kKBlk = 64;                  // k elements per TMA box (128 bytes, one swizzle span)
constexpr int kKSub = 2;                   // boxes along k per stage
constexpr int kKChunk = kKBlk * kKSub;     // k elements per stage (one work unit)
constexpr int kWSub = kTileRows * 128;     // 16 KB of weights per box column
constexpr int kWBytes = kWSub * kKSub;     // 32 KB of weights per stage

enum Epi : int { EPI_BF16 = 0, EPI_BF16_RES = 1, EPI_F32 = 2, EPI_SWIGLU = 3 };

// An expert chosen by more tokens than this is split into several groups of
// at most this many (its weights are then streamed once per group). It sizes
// the token rows of an expert kernel's pipeline stage beyond 16 tokens.
constexpr int kGroupTokens = 32;
// Groups of at most this many tokens load a token box of this height when
// the stage holds more rows (the smaller box fills the first rows of the
// same shared-memory slot): the token rows a stage moves follow the group.
constexpr int kNarrowRows = 16;

constexpr int kMaxSlots = 512;  // contributor slot table entries in shared memory
// Weight bytes per CTA a plain projection prefetches into L2 before waiting
// for its predecessor, beyond the ones its ring loads (152 CTAs: 39 MB, under
// a third of L2).
constexpr int kPrefetchBytes = 256 * 1024;

// Dynamic shared memory of one wstream_kernel instantiation: 1 KB alignment
// slack, the stage ring, full/empty barriers, flags, slot table, and `extra`.
constexpr int wstream_smem(int xr, int stages, int extra, bool paired = false) {
  return 1024 + stages * ((paired ? 2 : 1) * kWBytes + kKSub * xr * 128) + 2 * 8 * stages + 32 +
         4 * kMaxSlots + extra;
}

struct StreamArgs {
  int K, KB, TILES;
  int nout;                  // valid output features per group
  int M;                     // dense token count
  int mma_min_tokens;        // groups with at least this many tokens use mma.sync
  // grouped (MoE) mode; all null in dense mode
  const int* nact;
  const int* grp_exp;
  const int* grp_off;
  int w_group_rows;          // weight rows per expert
  int w_up_offset;           // paired (SwiGLU) tiles: row offset of the up block
  // grouped mode: the group tables were complete before the previous kernel
  // let this one launch (it does so only after its own wait), so they may be
  // read, and the weights streamed, before waiting for it
  int tables_ready;
  // output
  void* out;
  long long ldo;             // elements between output rows
  const uint16_t* res;       // residual for EPI_BF16_RES ([M, ldo] bf16)
  const float* addf;         // optional fp32 [M, ldo] added to the product before
                             // the residual (EPI_BF16 / EPI_BF16_RES); null: none
  // split-K workspace
  float* ws;                 // [grid][2][128][XR] fp32 partial tiles
  int* ctr;                  // per output tile arrival counters (zero at rest)
  int* status;
  long long timeout_ns;
  // router role: with route_k > 0 the last cluster to finish its logits
  // selects every token's top route_k experts and their gates
  int route_k;
  int route_E;               // scores the top-k ranks: columns 0..route_E-1 of each row
  int* route_ctr;            // arrival counter (zero at rest)
  int* route_idx;            // [M][route_k]
  float* route_gate;         // [M][route_k]
  int32_t* route_idx_user;   // optional copies for the caller
  float* route_w_user;
  // extents (elements) of the buffers above, checked by the index checks of
  // a DEC_DEBUG build: out, res, ws (floats), ctr; pairs = rows of the pair
  // tables (grouped: M*k; router: M*k of route_idx); groups_len = entries of
  // grp_exp (grp_off has one more)
  long long out_len, res_len, ws_len, ctr_len, addf_len;
  int pairs, groups_len;
};

struct GroupInfo {
  int e;       // expert id (0 in dense mode)
  int p0;      // first output row (pair) of the group
  int c;       // tokens in the group
};

// Group g; gsz is the most tokens a group of this instantiation may hold.
template <bool GROUPED>
__device__ __forceinline__ GroupInfo load_group(const StreamArgs& a, int g, int gsz = 0) {
  GroupInfo gi;
  if (GROUPED) {
    gi.e = *DG_AT(a.status, a.grp_exp, g, a.groups_len);
    gi.p0 = *DG_AT(a.status, a.grp_off, g, a.groups_len + 1);
    gi.c = *DG_AT(a.status, a.grp_off, g + 1, a.groups_len + 1) - gi.p0;
    if (!DG_OK(a.status, gi.p0 >= 0 && gi.c >= 0 && gi.p0 + gi.c <= a.pairs && gi.c <= gsz,
               (long long)gi.c * 1000000 + gi.p0)) {
      gi.p0 = 0;
      gi.c = 0;
    }
  } else {
    gi.e = 0;
    gi.p0 = 0;
    gi.c = a.M;
  }
  return gi;
}

// Position of work unit u in (group, tile, k chunk) order: u = (g * TILES +
// tile) * KB + kc. Walked one unit at a time with next().
struct UnitPos {
  int kc, tile, g;
  __device__ __forceinline__ void next(int KB, int TILES) {
    if (++kc == KB) {
      kc = 0;
      if (++tile == TILES) {
        tile = 0;
        ++g;
      }
    }
  }
};

__device__ __forceinline__ UnitPos unit_pos(long long u, int KB, int TILES) {
  const long long gt = u / KB;
  return UnitPos{(int)(u - gt * KB), (int)(gt % TILES), (int)(gt / TILES)};
}

__device__ __forceinline__ long long cta_start(long long c, long long T, long long G) {
  return (c * T) / G;
}

// CTA whose unit range contains unit v: largest c with start(c) <= v.
__device__ __forceinline__ long long cta_of(long long v, long long T, long long G) {
  return ((v + 1) * G + T - 1) / T - 1;
}

// ------------------------------------------------------------------ epilogue
template <int EPI, bool GROUPED>
__device__ __forceinline__ void store_out(const StreamArgs& a, const GroupInfo& gi, int t, int n,
                                          float v) {
  const long long row = (long long)gi.p0 + t;
  const long long i = row * a.ldo + n;
  if (EPI == EPI_F32) {
    *DG_AT(a.status, reinterpret_cast<float*>(a.out), i, a.out_len) = v;
    return;
  }
  if (a.addf) v += *DG_AT(a.status, a.addf, i, a.addf_len);
  if (EPI == EPI_BF16_RES) {
    const float r = bf_bits2f(*DG_AT(a.status, a.res, i, a.res_len));
    *DG_AT(a.status, reinterpret_cast<uint16_t*>(a.out), i, a.out_len) = f2bf_bits(r + v);
  } else {
    *DG_AT(a.status, reinterpret_cast<uint16_t*>(a.out), i, a.out_len) = f2bf_bits(v);
  }
}

__device__ __forceinline__ void store_swiglu(const StreamArgs& a, const GroupInfo& gi, int t, int i,
                                             float gate, float up) {
  const long long row = (long long)gi.p0 + t;
  const float h = silu_f(gate) * up;
  *DG_AT(a.status, reinterpret_cast<uint16_t*>(a.out), row * a.ldo + i, a.out_len) = f2bf_bits(h);
}

// ------------------------------------------------------------------ routing tail
// ------------------------------------------------------------------ split-K fixup
// Sum the partial tiles of all nc contributors of one output tile, in
// contributor order, and hand each total to `store(t, r, v, v_up)`. A partial
// slot is [token][STRIDE] fp32 at ws + slot * slot_floats: 128 rows of output
// features, followed for SwiGLU tiles (PAIRED) by the 128 matching up rows.
// Work item e is one float4 (4 rows of one token); thread tid takes items
// tid, tid + NT, ... so that every warp-wide load reads 512 contiguous bytes.
// A round loads EB items from JB contributors at once, so each thread keeps
// EB x JB loads in flight (twice that for SwiGLU tiles); each item's
// contributions are still added in contributor order.
// ws_len and st: the workspace's extent in floats and the status word, for
// the index checks of a DEC_DEBUG build.
template <int NT, bool PAIRED, int STRIDE, int EB, int JB, typename Slot, typename Store>
__device__ __forceinline__ void reduce_partials(const float* ws, long long slot_floats, int nc,
                                                int c, int tid, Slot slot_of, Store store,
                                                long long ws_len, int* st) {
  constexpr int R4 = (PAIRED ? kTileRows : STRIDE) / 4;  // output rows per token, in fours
  const int nel4 = R4 * c;
  for (int base = 0; base < nel4; base += NT * EB) {
    float4 g[EB], u[EB];
    int off[EB];
    bool ok[EB];
#pragma unroll
    for (int q = 0; q < EB; ++q) {
      g[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      u[q] = g[q];
      const int e = base + q * NT + tid;
      ok[q] = e < nel4;
      const int t = e / R4;
      off[q] = t * STRIDE + (e - t * R4) * 4;
    }
    auto add = [](float4& acc, const float4& v) {
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    };
    // JB contributors per round, the last round predicated: every round keeps
    // all of its loads in flight, however few contributors are left.
    for (int j = 0; j < nc; j += JB) {
      float4 pg[JB][EB], pu[JB][EB];
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        if (j + jj < nc) {
          const long long b = slot_of(j + jj) * slot_floats;
#pragma unroll
          for (int q = 0; q < EB; ++q) {
            if (ok[q]) {
              pg[jj][q] = __ldcg(reinterpret_cast<const float4*>(DG_AT(st, ws, b + off[q], ws_len - 3)));
              if (PAIRED)
                pu[jj][q] = __ldcg(reinterpret_cast<const float4*>(
                    DG_AT(st, ws, b + off[q] + kTileRows, ws_len - 3)));
            }
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        if (j + jj < nc) {
#pragma unroll
          for (int q = 0; q < EB; ++q) {
            if (ok[q]) {
              add(g[q], pg[jj][q]);
              if (PAIRED) add(u[q], pu[jj][q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < EB; ++q) {
      if (!ok[q]) continue;
      const int e = base + q * NT + tid;
      const int t = e / R4, r = (e - t * R4) * 4;
      store(t, r + 0, g[q].x, u[q].x);
      store(t, r + 1, g[q].y, u[q].y);
      store(t, r + 2, g[q].z, u[q].z);
      store(t, r + 3, g[q].w, u[q].w);
    }
  }
}

// Items per thread and round for reduce_partials, for at most `loads` float4
// loads in flight per thread (SwiGLU tiles load two halves per item): as many
// items as one round needs at XR token rows, the rest of the budget spent on
// contributors.
constexpr int reduce_eb(int nt, bool paired, int stride, int xr, int loads) {
  const int per = ((paired ? kTileRows : stride) / 4) * xr / nt;
  const int cap = paired ? loads / 2 : loads;
  return per < 1 ? 1 : per > cap ? cap : per;
}
constexpr int reduce_jb(bool paired, int eb, int loads) {
  const int jb = loads / (eb * (paired ? 2 : 1));
  return jb < 1 ? 1 : jb;
}

// ------------------------------------------------------------------ the kernel
// XR: token rows per stage (8, 16 or 64). STAGES: ring depth.
// PAIRED: SwiGLU tiles (128 gate rows and the 128 matching up rows per stage
// column). WIDE: 256-row output tiles (two 128-row halves per stage column).
// GROUPED: MoE groups. ROLE: which step of the decode layer launches the
// instantiation; it changes no code, only the kernel's name, so that launch
// lists and profiles tell the router and shared expert from the projections.
// MINB: CTAs per SM the build must fit (registers and shared memory). With 2,
// a call's CTA can start on an SM while the previous call's CTA there is
// still finishing, and stream its weights before waiting for that call.
// CLUSTER (dense 128-row tiles only): the kernel is launched in clusters of S
// CTAs, cluster i owning output tile i and CTA r of it the r-th of S equal
// shares of its k chunks; the S partial tiles are summed through distributed
// shared memory, in rank order, behind two cluster barriers -- no global
// partials, counters or atomics.
enum Role : int { ROLE_PROJECTION = 0, ROLE_ROUTER = 1, ROLE_EXPERT = 2, ROLE_SHARED = 3 };
// PATH: which consumers the instantiation carries. PATH_ANY chooses per group
// (CUDA cores below mma_min_tokens tokens, mma.sync from there): expert groups
// hold 1..XR tokens each. PATH_CORE carries the CUDA-core consumer only, for
// projections of 1-2 tokens.
enum Path : int { PATH_ANY = 0, PATH_CORE = 1 };
template <int XR, int STAGES, int EPI, bool PAIRED, bool GROUPED, bool WIDE = false,
          int ROLE = ROLE_PROJECTION, int MINB = 1, bool CLUSTER = false, int PATH = PATH_ANY>
__global__ void __launch_bounds__(kThreads, MINB)
    wstream_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const __grid_constant__ CUtensorMap xmap_narrow, const StreamArgs a) {
  constexpr int H2 = (PAIRED || WIDE) ? 2 : 1;  // 128-row weight halves per box column
  // CUDA-core dot form. Both give the same bits. The bf16-operand form
  // (fma.rn.f32.bf16) issues half the instructions; the widened form is kept
  // in the two-CTA-per-SM instantiations that carry the mma.sync path too,
  // where at 112 registers the compiler's allocation of the mma loop spilled
  // more with the other form and that path lost 6-8 % (M = 4 / 16 tokens,
  // N = 2048, K = 7168, same-GPU A/B).
  constexpr bool kMixedDot = PATH == PATH_CORE || MINB == 1;
  constexpr int kTileOut = PAIRED ? kTileRows : H2 * kTileRows;  // output features per tile
  constexpr int kXSub = XR * 128;              // token rows of one box column
  constexpr int kXBytes = kXSub * kKSub;
  constexpr int kWStage = H2 * kWBytes;
  constexpr int kStageBytes = kWStage + kXBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStageBytes);
  uint64_t* empty = full + STAGES;
  // [0] abort [1] last arriver of a split tile [2] last cluster of the router
  volatile int* s_flags = reinterpret_cast<volatile int*>(empty + STAGES);
  int* s_slot = const_cast<int*>(s_flags) + 8;                                 // [kMaxSlots]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
    s_flags[2] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&wmap);
    prefetch_tmap(&xmap);
    if (GROUPED && XR > kNarrowRows) prefetch_tmap(&xmap_narrow);
  }
  __syncthreads();
  // Kernels that can stream weights before their predecessor finishes let
  // their own dependents launch at once. A grouped kernel that must wait for
  // the group tables does so only after that wait: its dependents' CTAs would
  // otherwise take SMs early and sit idle there, and they may then read the
  // tables before waiting.
  const bool early = !GROUPED || a.tables_ready;
  if (early) griddep_launch_dependents();

  const long long c = blockIdx.x;
  const int KB = a.KB, TILES = a.TILES;

  long long T;
  if (GROUPED) {
    if (!early) {
      griddep_wait();
      griddep_launch_dependents();
    }
    T = (long long)(*a.nact) * TILES * KB;
  } else {
    T = (long long)TILES * KB;
  }
  // Only the first min(grid, T) CTAs take units, so every working CTA has at
  // least one and the contributors of a tile are exactly the CTAs between
  // the owners of its first and last unit.
  const long long G = (long long)gridDim.x < T ? (long long)gridDim.x : T;
  long long u0, u1;
  if (CLUSTER) {
    static_assert(!CLUSTER || (!GROUPED && !PAIRED && !WIDE), "cluster split: dense 128-row tiles");
    const long long cs = cluster_size(), cr = cluster_rank();
    const long long tile = c / cs;
    u0 = tile * KB + cr * KB / cs;
    u1 = tile * KB + (cr + 1) * KB / cs;
    if (tile >= TILES) u0 = u1 = 0;
  } else {
    u0 = c < G ? cta_start(c, T, G) : 0;
    u1 = c < G ? cta_start(c + 1, T, G) : 0;
  }
  const int nunits = (int)(u1 - u0);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int gcur = -1;
      GroupInfo gi{0, 0, 0};
      // Unit positions advance one unit at a time: no 64-bit division per
      // stage on the path that refills the ring.
      auto issue_w = [&](int s, const UnitPos& p) {
        uint8_t* wdst = smem + s * kStageBytes;
        const CUtensorMap* wm = &wmap;
        const int rbase = gi.e * a.w_group_rows;
#pragma unroll
        for (int sb = 0; sb < kKSub; ++sb) {
          const int k0 = (p.kc * kKSub + sb) * kKBlk;
          uint8_t* d = wdst + sb * H2 * kWSub;
          tma_load_2d(d, wm, k0, rbase + p.tile * kTileOut, &full[s], pol_w);
          if (H2 == 2)
            tma_load_2d(d + kWSub, wm, k0,
                        rbase + (PAIRED ? a.w_up_offset + p.tile * kTileRows
                                        : p.tile * kTileOut + kTileRows),
                        &full[s], pol_w);
        }
      };
      auto narrow_group = [&](const GroupInfo& g_) {
        return GROUPED && XR > kNarrowRows && g_.c <= kNarrowRows;
      };
      auto issue_x = [&](int s, int kc, const GroupInfo& g_) {
        uint8_t* xdst = smem + s * kStageBytes + kWStage;
#pragma unroll
        for (int sb = 0; sb < kKSub; ++sb) {
          const int k0 = (kc * kKSub + sb) * kKBlk;
          uint8_t* d = xdst + sb * kXSub;
          // Grouped: the token rows of a group are contiguous in the token
          // tensor (pairs are stored in expert order), so one box of XR rows
          // at the group's first pair covers them; rows past the group are
          // never read.
          tma_load_2d(d, narrow_group(g_) ? &xmap_narrow : &xmap, k0, GROUPED ? g_.p0 : 0,
                      &full[s], pol_x);
        }
      };
      // The same weight boxes as issue_w for group g_, into L2 only.
      auto prefetch_w = [&](const UnitPos& p, const GroupInfo& g_) {
        const CUtensorMap* wm = &wmap;
        const int rbase = g_.e * a.w_group_rows;
#pragma unroll
        for (int sb = 0; sb < kKSub; ++sb) {
          const int k0 = (p.kc * kKSub + sb) * kKBlk;
          tma_prefetch_2d(wm, k0, rbase + p.tile * kTileOut);
          if (H2 == 2)
            tma_prefetch_2d(wm, k0,
                            rbase + (PAIRED ? a.w_up_offset + p.tile * kTileRows
                                            : p.tile * kTileOut + kTileRows));
        }
      };
      auto tx_bytes = [&](const GroupInfo& g_) -> uint32_t {
        return kWStage + (narrow_group(g_) ? (uint32_t)(kKSub * kNarrowRows * 128) : (uint32_t)kXBytes);
      };
      UnitPos pos = unit_pos(u0, KB, TILES);
      int i = 0;
      if (early) {
        // Weights do not depend on the previous kernel: start streaming them
        // before waiting for it, then fetch the token tiles.
        const int npre = nunits < STAGES ? nunits : STAGES;
        GroupInfo pg[STAGES];
        const UnitPos pos0 = pos;
        for (; i < npre; ++i, pos.next(KB, TILES)) {
          if (pos.g != gcur) {
            gcur = pos.g;
            gi = load_group<GROUPED>(a, pos.g, XR);
          }
          pg[i] = gi;
          mbar_arrive_expect_tx(&full[i], tx_bytes(gi));
          issue_w(i, pos);
        }
        // The units beyond the ring: pull up to kPrefetchBytes of them into
        // L2 while the previous kernel finishes, so that after the wait they
        // arrive at L2 rather than HBM latency and bandwidth.
        // (not in cluster mode: there the shares are small and it did not pay)
        constexpr int kPfUnits = CLUSTER ? 0 : kPrefetchBytes / kWStage;
        const int npf = nunits - npre < kPfUnits ? nunits - npre : kPfUnits;
        int pgrp = -1;
        GroupInfo pgi{0, 0, 0};
        UnitPos pp = pos;
        for (int j = 0; j < npf; ++j, pp.next(KB, TILES)) {
          if (pp.g != pgrp) {
            pgrp = pp.g;
            pgi = load_group<GROUPED>(a, pp.g, XR);
          }
          prefetch_w(pp, pgi);
        }
        griddep_wait();
        UnitPos px = pos0;
        for (int j = 0; j < npre; ++j, px.next(KB, TILES)) issue_x(j, px.kc, pg[j]);
      }
      for (; i < nunits; ++i, pos.next(KB, TILES)) {
        const int s = i % STAGES;
        if (i >= STAGES) {
          if (!mbar_wait(&empty[s], ((i / STAGES) + 1) & 1, a.timeout_ns, a.status)) {
            s_flags[0] = 1;
            break;
          }
        }
        if (s_flags[0]) break;
        if (GROUPED && pos.g != gcur) {
          // new expert group: read its id and pair range once
          gcur = pos.g;
          gi = load_group<GROUPED>(a, pos.g, XR);
        }
        mbar_arrive_expect_tx(&full[s], tx_bytes(gi));
        issue_w(s, pos);
        issue_x(s, pos.kc, gi);
      }
      // Drain: wait until every issued copy has landed before the CTA may exit.
      const int issued = i;
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const int uses = (issued - s + STAGES - 1) / STAGES;
        mbar_wait(&full[s], (uses - 1) & 1, drain_ns(a.timeout_ns), nullptr);
      }
    }
    if (early && lane != 0) griddep_wait();
    if (CLUSTER) {
      // the producer warp takes part in the consumers' cluster barriers
      __syncwarp();
      cluster_sync_all();
      cluster_sync_all();
      if (ROLE == ROLE_ROUTER && a.route_k > 0) cluster_sync_all();
    }
  } else {
    // ---------------------------------------------------------------- consumers
    if (early) griddep_wait();
    const int w = warp - 1;
    const int ct = threadIdx.x - 32;
    const int q = lane & 7, rho = lane >> 3;  // CUDA-core path: chunk and row group
    const int gq = lane >> 2, tq = lane & 3;  // mma path: fragment row and column pair

    // Thread-held rows (within each 128-row half of a stage):
    //   CUDA-core path: rows 16w + rho + 4r, r = 0..3, 16-byte chunk q of each;
    //   mma path: rows 16w + gq and 16w + gq + 8 of the m16 fragment.
    // Half 0 is the plain weight tile (or the gate rows), half 1 the up rows.
    constexpr int kSlotStride = H2 * kTileRows;  // floats per token in a partial slot
    float dacc[H2][4][2];
    float macc[H2][XR / 8][4];
    long long cur = -1;
    GroupInfo gi{0, 0, 0};
    bool use_mma = false;

    auto zero_acc = [&]() {
#pragma unroll
      for (int h = 0; h < H2; ++h) {
#pragma unroll
        for (int r = 0; r < 4; ++r) dacc[h][r][0] = dacc[h][r][1] = 0.f;
#pragma unroll
        for (int tg = 0; tg < XR / 8; ++tg)
#pragma unroll
          for (int j = 0; j < 4; ++j) macc[h][tg][j] = 0.f;
      }
    };

    // The CUDA-core path's sums are complete only in lanes with q == 0 after
    // this shuffle reduction over the 8 chunks of a row.
    auto reduce_dots = [&]() {
#pragma unroll
      for (int h = 0; h < H2; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            float v = dacc[h][r][t];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            dacc[h][r][t] = v;
          }
    };

    // One output of tile row r (0 .. kTileOut-1): SwiGLU of the gate sum v0
    // and the up sum v1, or the plain sum v0.
    auto emit = [&](int tile, int r, int t, float v0, float v1) {
      const int n = tile * kTileOut + r;
      if (n >= a.nout) return;
      if (PAIRED) store_swiglu(a, gi, t, n, v0, v1);
      else store_out<EPI, GROUPED>(a, gi, t, n, v0);
    };

    // Final values held in registers (the CTA covered the tile's whole k range).
    auto reg_epilogue = [&](int tile) {
      if (!use_mma) {
        if (q != 0) return;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= gi.c) continue;
            const int row = 16 * w + rho + 4 * r;
            if (PAIRED) {
              emit(tile, row, t, dacc[0][r][t], dacc[1][r][t]);
            } else {
#pragma unroll
              for (int h = 0; h < H2; ++h) emit(tile, h * kTileRows + row, t, dacc[h][r][t], 0.f);
            }
          }
        return;
      }
#pragma unroll
      for (int tg = 0; tg < XR / 8; ++tg)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int t = tg * 8 + 2 * tq + hh;
          if (t >= gi.c) continue;
          if (PAIRED) {
            emit(tile, 16 * w + gq, t, macc[0][tg][hh], macc[1][tg][hh]);
            emit(tile, 16 * w + gq + 8, t, macc[0][tg][2 + hh], macc[1][tg][2 + hh]);
          } else {
#pragma unroll
            for (int h = 0; h < H2; ++h) {
              emit(tile, h * kTileRows + 16 * w + gq, t, macc[h][tg][hh], 0.f);
              emit(tile, h * kTileRows + 16 * w + gq + 8, t, macc[h][tg][2 + hh], 0.f);
            }
          }
        }
    };

    // This CTA's share of a tile that other CTAs also contribute to, written
    // to its workspace slot as [token][kSlotStride] fp32.
    // Partial tiles go to global memory (L2) for the split-K fixup, or to
    // this CTA's shared memory in cluster mode.
    auto put = [&](float* p, float v) {
      if (CLUSTER) *p = v;
      else __stcg(DG_AT(a.status, a.ws, p - a.ws, a.ws_len), v);
    };
    auto write_partial = [&](float* mine) {
      if (!use_mma) {
        if (q != 0) return;
#pragma unroll
        for (int h = 0; h < H2; ++h)
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < 2; ++t)
              if (t < gi.c)
                put(mine + t * kSlotStride + h * kTileRows + 16 * w + rho + 4 * r, dacc[h][r][t]);
        return;
      }
#pragma unroll
      for (int h = 0; h < H2; ++h)
#pragma unroll
        for (int tg = 0; tg < XR / 8; ++tg)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int t = tg * 8 + 2 * tq + hh;
            if (t < gi.c) {
              float* p = mine + t * kSlotStride + h * kTileRows + 16 * w + gq;
              put(p, macc[h][tg][hh]);
              put(p + 8, macc[h][tg][2 + hh]);
            }
          }
    };

    constexpr long long kSlotFloats = (long long)kSlotStride * XR;
    // Contributors of split tile gt: CTAs cf..cl.
    auto first_cta = [&](long long gt) { return cta_of(gt * KB, T, G); };
    auto last_cta = [&](long long gt) { return cta_of((gt + 1) * KB - 1, T, G); };

    // The last contributor of tile gt sums every contributor's slot in CTA
    // order (so the result does not depend on who arrived last). Called by all
    // consumer threads after the arrival atomic's result is in s_flags[1].
    auto reduce_tile = [&](long long gt, bool aborted) {
      const int tile = (int)(gt % TILES);
      const long long cf = first_cta(gt);
      const int nc = (int)(last_cta(gt) - cf + 1);
      auto slot_of = [&](int j) -> long long {
        const long long cc = cf + j;
        return cc * 2 + ((gt == cta_start(cc, T, G) / KB) ? 0 : 1);
      };
      for (int j = ct; j < nc && j < kMaxSlots; j += kNCW * 32) s_slot[j] = (int)slot_of(j);
      named_bar_sync(1, kNCW * 32);
      if (!aborted) {
        auto slot_at = [&](int j) -> long long {
          return j < kMaxSlots ? (long long)s_slot[j] : slot_of(j);
        };
        auto store = [&](int t, int r, float vg, float vu) { emit(tile, r, t, vg, vu); };
        // fewer registers for two CTAs per SM, and for SwiGLU tiles at 64
        // token rows, whose accumulators take most of them
        constexpr int kLoads = (MINB == 2 || (PAIRED && XR == 64)) ? 4 : 8;
        constexpr int kEB = reduce_eb(kNCW * 32, PAIRED, kSlotStride, XR, kLoads);
        constexpr int kJB = reduce_jb(PAIRED, kEB, kLoads);
        reduce_partials<kNCW * 32, PAIRED, kSlotStride, kEB, kJB>(a.ws, kSlotFloats, nc, gi.c, ct,
                                                                  slot_at, store, a.ws_len,
                                                                  a.status);
      }
    };

    // Thread 0's share of the arrival on tile gt's counter, given the counter's
    // value before its own increment: flags the last contributor and resets
    // the counter for the next call.
    auto settle = [&](long long gt, int old) {
      const int is_last = (old == (int)(last_cta(gt) - first_cta(gt))) ? 1 : 0;
      if (is_last) *DG_AT(a.status, a.ctr, gt, a.ctr_len) = 0;
      s_flags[1] = is_last;
    };

    // A split tile met in the middle of the range (the CTA's first tile, whose
    // other contributors precede it) has its arrival deferred: the atomic is
    // issued and the consumers move on to the next tile at once; its result is
    // read, and the tile reduced if this CTA arrived last, after the range.
    long long dgt = -1;  // deferred tile
    int dold = 0;        // its counter's value before this CTA's increment (thread 0)
    GroupInfo dgi{0, 0, 0};

    auto finish_tile = [&](long long gt, bool defer) {
      const int tile = (int)(gt % TILES);
      const bool aborted = s_flags[0] != 0;
      if (!use_mma) reduce_dots();
      const bool whole = (u0 <= gt * KB) && ((gt + 1) * KB <= u1);
      if (whole) {
        if (!aborted) reg_epilogue(tile);
      } else {
        const int slot = (gt == u0 / KB) ? 0 : 1;
        write_partial(a.ws + (c * 2 + slot) * kSlotFloats);
        // The barrier orders every consumer thread's partial stores before
        // thread 0's release; the acquire side of the same atomic, followed by
        // a barrier, orders the last arriver's reads of the other slots after
        // every contributor's release. No separate fence needed.
        named_bar_sync(1, kNCW * 32);
        if (defer) {
          if (ct == 0) dold = atomic_add_acq_rel_gpu(DG_AT(a.status, a.ctr, gt, a.ctr_len), 1);
          dgt = gt;
          dgi = gi;
          return;
        }
        if (ct == 0) settle(gt, atomic_add_acq_rel_gpu(DG_AT(a.status, a.ctr, gt, a.ctr_len), 1));
        named_bar_sync(1, kNCW * 32);
        if (s_flags[1]) reduce_tile(gt, aborted);
      }
      named_bar_sync(1, kNCW * 32);  // partial slots and flags may be reused next tile
    };

    // tile of the current unit, advanced with its k chunk (no division per stage)
    long long gt_next = u0 / KB;
    int kc_next = (int)(u0 - gt_next * KB);
    for (int i = 0; i < nunits; ++i) {
      const long long gt = gt_next;
      if (++kc_next == KB) {
        kc_next = 0;
        ++gt_next;
      }
      if (gt != cur) {
        if (cur >= 0) finish_tile(cur, cur == u0 / KB);
        cur = gt;
        zero_acc();
        gi = load_group<GROUPED>(a, (int)(gt / TILES), XR);
        use_mma = PATH == PATH_ANY && gi.c >= a.mma_min_tokens;
      }
      const int s = i % STAGES;
      if (!s_flags[0]) {
        if (!mbar_wait(&full[s], (i / STAGES) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
      }
#pragma unroll
      for (int sb = 0; sb < kKSub; ++sb) {
        const uint8_t* wbase = smem + s * kStageBytes + sb * H2 * kWSub;
        const uint8_t* xs_base = smem + s * kStageBytes + kWStage + sb * kXSub;
        if (!use_mma) {
          // CUDA-core path: lane reads 16-byte chunk q of rows 16w + rho + 4r
          // and multiplies it with the same chunk of each token.
          if constexpr (kMixedDot) {
            // bf16 operands, fp32 sums: no widening instructions
            uint4 xq[2];
#pragma unroll
            for (int t = 0; t < 2; ++t)
              xq[t] = t < gi.c ? *reinterpret_cast<const uint4*>(xs_base + t * 128 +
                                                                  ((q ^ (t & 7)) << 4))
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int row = 16 * w + rho + 4 * r;
#pragma unroll
              for (int h = 0; h < H2; ++h) {
                const uint4 wv = *reinterpret_cast<const uint4*>(wbase + h * kWSub + row * 128 +
                                                                 ((q ^ (row & 7)) << 4));
                dacc[h][r][0] = dot8_bf16(wv, xq[0], dacc[h][r][0]);
                if (gi.c > 1) dacc[h][r][1] = dot8_bf16(wv, xq[1], dacc[h][r][1]);
              }
            }
          } else {
            float xv[2][8];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t < gi.c) {
                const uint4 v =
                    *reinterpret_cast<const uint4*>(xs_base + t * 128 + ((q ^ (t & 7)) << 4));
                unpack8(v, xv[t]);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) xv[t][j] = 0.f;
              }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int row = 16 * w + rho + 4 * r;
#pragma unroll
              for (int h = 0; h < H2; ++h) {
                const uint4 wv = *reinterpret_cast<const uint4*>(wbase + h * kWSub + row * 128 +
                                                                 ((q ^ (row & 7)) << 4));
                dacc[h][r][0] = dot8(wv, xv[0], dacc[h][r][0]);
                if (gi.c > 1) dacc[h][r][1] = dot8(wv, xv[1], dacc[h][r][1]);
              }
            }
          }
        } else {
          const int ntg = (gi.c + 7) >> 3;
          const uint32_t wb = smem_u32(wbase), xb = smem_u32(xs_base);
          const int mi = lane >> 3, r8 = lane & 7;
          const int a_row = 16 * w + (mi & 1) * 8 + r8;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint32_t af[H2][4];
            const int ach = kk * 2 + (mi >> 1);
#pragma unroll
            for (int h = 0; h < H2; ++h)
              ldmatrix_x4(af[h][0], af[h][1], af[h][2], af[h][3],
                          wb + h * kWSub + a_row * 128 + ((ach ^ r8) << 4));
#pragma unroll
            for (int tg = 0; tg < XR / 8; ++tg) {
              if (tg < ntg) {
                const int t = tg * 8 + r8;
                const int bch = kk * 2 + (mi & 1);
                uint32_t b0, b1;
                ldmatrix_x2(b0, b1, xb + t * 128 + ((bch ^ r8) << 4));
#pragma unroll
                for (int h = 0; h < H2; ++h) mma_bf16_16816(macc[h][tg], af[h], b0, b1);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (CLUSTER) {
      // Partial tile [token][128] at the start of this CTA's shared memory
      // (every stage has been consumed and no copy is in flight once all
      // consumer warps are past their last stage).
      float* part = reinterpret_cast<float*>(smem);
      const bool aborted = s_flags[0] != 0;
      if (cur >= 0 && !use_mma) reduce_dots();
      named_bar_sync(1, kNCW * 32);
      if (cur >= 0) {
        write_partial(part);
      } else {
        // no k chunks (more ranks than chunks): this rank's share is zero
        for (int e = ct; e < a.M * kTileRows; e += kNCW * 32) part[e] = 0.f;
      }
      cluster_sync_all();
      // Rank r sums its run of R4 rows of every token over the S partials,
      // in rank order, and writes them: R4 = 128/S rounded up to a multiple
      // of 4, the last rank's run cut at 128 (S need not divide 128: the
      // router's clusters have up to 8 CTAs, one per 128 k of the hidden
      // size; with 128/S rounded down, rows 125-127 of a tile were lost).
      const int cs = (int)cluster_size(), cr = (int)cluster_rank();
      const int R4 = ((kTileRows + cs - 1) / cs + 3) / 4 * 4;
      const int r0 = cr * R4 < kTileRows ? cr * R4 : kTileRows;
      const int r1 = r0 + R4 < kTileRows ? r0 + R4 : kTileRows;
      const int tile = (int)(blockIdx.x / cs);
      if (!aborted && tile < TILES && nunits > 0) {
        const int RR = r1 - r0;
        for (int e = ct; e < RR * gi.c; e += kNCW * 32) {
          const int t = e / RR, r = r0 + (e - t * RR);
          float v = 0.f;
          for (int qr = 0; qr < cs; ++qr) v += ld_dsmem_f32(part + t * kTileRows + r, (uint32_t)qr);
          emit(tile, r, t, v, 0.f);
        }
      }
      cluster_sync_all();  // no CTA leaves while another still reads its partial
      if (ROLE == ROLE_ROUTER && a.route_k > 0) {
        // This cluster's logits are written (the barrier orders every
        // thread's stores before the release of the arrival below). The last
        // of the TILES clusters to arrive acquires them all and selects the
        // experts: its consumer warps take the tokens in turn.
        if (cr == 0 && ct == 0) {
          const int old = atomic_add_acq_rel_gpu(a.route_ctr, 1);
          const int last = old == TILES - 1 ? 1 : 0;
          if (last) *a.route_ctr = 0;
          for (int qr = 0; qr < cs; ++qr)
            st_dsmem_s32(const_cast<int*>(&s_flags[2]), (uint32_t)qr, last);
        }
        cluster_sync_all();
        if (s_flags[2]) {
          const int K = a.route_k;
          for (int m = cr * kNCW + w; m < a.M; m += cs * kNCW)
            if (DG_OK(a.status, (long long)(m + 1) * K <= a.pairs &&
                                    (long long)m * a.ldo + a.route_E <= a.out_len, m))
              warp_topk_gates(reinterpret_cast<const float*>(a.out) + (long long)m * a.ldo, a.route_E,
                            K, lane, a.route_idx + m * K, a.route_gate + m * K,
                            a.route_idx_user ? a.route_idx_user + m * K : nullptr,
                            a.route_w_user ? a.route_w_user + m * K : nullptr);
        }
      }
    } else if (cur >= 0) {
      finish_tile(cur, false);
    }
    if (dgt >= 0) {
      if (ct == 0) settle(dgt, dold);
      named_bar_sync(1, kNCW * 32);
      if (s_flags[1]) {
        gi = dgi;
        reduce_tile(dgt, s_flags[0] != 0);
      }
    }
  }
  __syncthreads();
}

}  // namespace dg
