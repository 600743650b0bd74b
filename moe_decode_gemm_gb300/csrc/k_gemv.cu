// k_gemv.cu -- decode projection y = x·Wᵀ for 1-16 tokens without splitting K
// across CTAs: each CTA owns R consecutive weight rows (R = 8 to 64) over
// the whole K, so no partial sums leave the CTA -- no workspace, counters,
// atomics or cluster barriers. What split-K spends after the last weight
// byte (the wait for the slowest rank of a tile, the reduction of the
// partial tiles and the barrier that keeps partials alive) is gone; the sum
// over K ends with a reduction inside the CTA.
//
// Two kernels share that plan. In both, one producer thread streams stages
// of weights with one 3-D TMA box (R rows x k blocks of 64, 128-byte swizzle)
// and the tokens' matching k range (issued once the previous kernel has
// finished; the weights of the first stages are in flight before that), and
// eight consumer warps split each stage by k block.
//
// gemv_slab_kernel (1-2 tokens, CUDA cores): 32 KB stages of R rows x 16384/R
// k, the token slices by one bulk copy per token; lane l of warp w takes row
// l % R of k block w*(32/R) + l/R and its 8
// chunks of 16 bytes, multiplying them with the tokens' matching chunks
// (fma.rn.f32.bf16, fp32 sums). The 32/R lanes of a row and then the 8 warps
// are summed in a fixed order, so results do not vary from run to run.
//
// gemv_mma_kernel (1-16 tokens, mma.sync): see its own comment below.
//
// "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 "针对工作负载调优形状"
// (a small-matrix kernel for batch 1-2).
#include <utility>

#include "launch.h"
#include "launch_util.cuh"
#include "wstream.cuh"

namespace dg {

constexpr int kGvStage = 32768;         // weight bytes per stage
constexpr int kGvThreads = 9 * 32;      // producer warp + 8 consumer warps
constexpr int kGvMaxTokens = 2;        // CUDA-core slabs
constexpr int kMmaMaxTokens = 16;      // tensor-core slabs

// Bytes of one stage: the weights, then each token's k range (16384/R k).
constexpr int gemv_stage_bytes(int R) { return kGvStage + kGvMaxTokens * (kGvStage / R); }

// Stages: three, or two at R = 8, whose stages carry 8 KB of token slices
// (two CTAs per SM either way).
constexpr int gemv_stages(int R) { return R == 8 ? 2 : 3; }

// Shared memory: stages, barriers, the cross-warp partials.
constexpr int gemv_smem(int R) {
  return 1024 + gemv_stages(R) * gemv_stage_bytes(R) + 8 * 2 * gemv_stages(R) + 32 +
         8 * R * kGvMaxTokens * 4;
}

template <int R, int EPI>
__global__ void __launch_bounds__(kGvThreads, 2)
    gemv_slab_kernel(const __grid_constant__ CUtensorMap wmap, const uint16_t* x, long long ldx,
                     const StreamArgs a) {
  static_assert(R == 8 || R == 16 || R == 32, "rows per CTA");
  constexpr int STAGES = gemv_stages(R);
  constexpr int KS = kGvStage / (2 * R);   // k elements per stage
  constexpr int KBS = KS / 64;             // 64-wide k blocks per stage
  constexpr int LPR = 32 / R;              // lanes per row in a warp
  constexpr int SB = gemv_stage_bytes(R);
  static_assert(KBS == 8 * LPR, "one k block per lane");
  static_assert(SB % 1024 == 0, "stages stay 1024-byte aligned");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int M = a.M, K = a.K;
  // stage s: [weights 32 KB][token t's k range: KS bf16, t < 2]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * SB);
  uint64_t* empty = full + STAGES;
  volatile int* s_flags = reinterpret_cast<volatile int*>(empty + STAGES);  // [0] abort
  float* red = reinterpret_cast<float*>(const_cast<int*>(s_flags) + 8);      // [8][R][2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) prefetch_tmap(&wmap);
  __syncthreads();
  // The weights do not depend on the previous kernel: this one may launch at
  // once and stream its first stages while that kernel finishes.
  griddep_launch_dependents();

  const int row0 = blockIdx.x * R;
  const int nst = (K + KS - 1) / KS;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      // the tokens' k range of stage i: from k = i*KS, up to K
      auto xbytes = [&](int i) -> uint32_t {
        const int n = K - i * KS;
        return (uint32_t)((n < KS ? n : KS) * 2);
      };
      auto issue_x = [&](int s, int i) {
        uint16_t* xs = reinterpret_cast<uint16_t*>(smem + s * SB + kGvStage);
        for (int m = 0; m < M; ++m)
          bulk_copy_g2s(xs + m * KS, x + m * ldx + (long long)i * KS, xbytes(i), &full[s]);
      };
      const int npre = nst < STAGES ? nst : STAGES;
      int i = 0;
      for (; i < npre; ++i) {
        mbar_arrive_expect_tx(&full[i], kGvStage + M * xbytes(i));
        tma_load_3d(smem + i * SB, &wmap, 0, row0, i * KBS, &full[i], pol_w);
      }
      griddep_wait();
      for (int j = 0; j < npre; ++j) issue_x(j, j);
      for (; i < nst; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], ((i / STAGES) + 1) & 1, a.timeout_ns, a.status)) {
          s_flags[0] = 1;
          break;
        }
        if (s_flags[0]) break;
        mbar_arrive_expect_tx(&full[s], kGvStage + M * xbytes(i));
        tma_load_3d(smem + s * SB, &wmap, 0, row0, i * KBS, &full[s], pol_w);
        issue_x(s, i);
      }
      // Drain: every issued copy has landed before the CTA may exit.
      const int issued = i;
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const int uses = (issued - s + STAGES - 1) / STAGES;
        mbar_wait(&full[s], (uses - 1) & 1, drain_ns(a.timeout_ns), nullptr);
      }
    } else {
      griddep_wait();
    }
  } else {
    // ---------------------------------------------------------------- consumers
    griddep_wait();
    const int w = warp - 1;
    const int r = lane % R;                // this lane's row within the slab
    const int kb = w * LPR + lane / R;     // this lane's k block within a stage
    float acc[kGvMaxTokens] = {0.f, 0.f};
    for (int i = 0; i < nst; ++i) {
      const int s = i % STAGES;
      if (!s_flags[0]) {
        if (!mbar_wait(&full[s], (i / STAGES) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
      }
      const int k0 = (i * KBS + kb) * 64;  // first k of this lane's block
      if (k0 < K && !s_flags[0]) {
        const uint8_t* wrow = smem + s * SB + (kb * R + r) * 128;
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + s * SB + kGvStage) + kb * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 wv = *reinterpret_cast<const uint4*>(wrow + ((c ^ (r & 7)) << 4));
#pragma unroll
          for (int t = 0; t < kGvMaxTokens; ++t)
            if (t < M) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * KS + c * 8);
              acc[t] = dot8_bf16(wv, xv, acc[t]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // lanes of a row (lane, lane + R, ...), then warps, in a fixed order
#pragma unroll
    for (int t = 0; t < kGvMaxTokens; ++t)
#pragma unroll
      for (int off = R; off < 32; off <<= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    if (lane < R)
#pragma unroll
      for (int t = 0; t < kGvMaxTokens; ++t) red[(w * R + lane) * kGvMaxTokens + t] = acc[t];
    named_bar_sync(1, kNCW * 32);
    const int ct = threadIdx.x - 32;
    if (ct < R * M && !s_flags[0]) {
      const int rr = ct % R, t = ct / R;
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < kNCW; ++q) v += red[(q * R + rr) * kGvMaxTokens + t];
      const int n = row0 + rr;
      if (n < a.nout) store_out<EPI, false>(a, GroupInfo{0, 0, M}, t, n, v);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- mma slabs
// The same whole-row slabs with the dot products on the tensor cores
// (mma.sync.m16n8k16: the weights are the 16-row operand, the tokens the
// 8-column one, columns past M zero). On the CUDA cores the multiply-adds of
// a stage cost more than its copies once the dependency has resolved (~0.5 us
// per 32 KB stage of one token; a copy of the kernel with them left out was
// 1-2 us faster per call), while a stage here is 32-64 MMAs. A stage is KBS k
// blocks of 64 of the slab's R rows (16 KB of weights, 24 KB at R = 48: one
// 3-D TMA box, 128-byte swizzle) and the same k range of XR = 4, 8 or 16 token rows (one
// 3-D TMA box, rows past M zero-filled, same swizzle). Warp w works on row
// group w % (R/16) and takes every (warps of that group)-th k block of a
// stage; it keeps one accumulator tile over all its tasks, and the warps of a
// row group are summed in order at the end, so results do not vary from run
// to run.
//
// Every CTA reads the tokens' rows over all of K, XR/R of its weight bytes.
// Measured alternatives (us per call, CUDA graph, N x K = 2048 x 7168): a bulk
// copy per token row instead of the token box cost more with every token
// (13.8 at 16 tokens, the box 8.9); slabs of 32 or 64 rows shared by a cluster
// of 2 or 4 CTAs that split K (fewer token bytes per CTA, partials summed
// through distributed shared memory) lost to one CTA per slab at every size
// (8 tokens: 9.0 / 9.7 against 6.9).
template <int R, int XR, int KBS, int MINB>
struct MmaSlab {
  static constexpr int RG = R / 16;                     // 16-row groups
  static constexpr int XN = (XR + 7) / 8;               // 8-token column tiles
  static constexpr int KS = KBS * 64;                   // k per stage
  static constexpr int WB = R * KS * 2;                 // weight bytes per stage
  static constexpr int XB = KBS * XR * 128;             // token bytes per stage (full box)
  static constexpr int SB = (WB + XB + 1023) / 1024 * 1024;
  static constexpr int RED = kNCW * 16 * XR * 4;        // per-warp tiles (token rows only)
  static constexpr int FIXED = 1024 + RED + 256;        // alignment, tiles, barriers, flags
  // two CTAs per SM (MINB = 2), or one with a ring twice as deep (MINB = 1)
  static constexpr int STAGES = ((MINB == 2 ? 115712 : 225000) - FIXED) / SB;
  static constexpr int SMEM = FIXED + STAGES * SB;
  static_assert(RG >= 1 && RG <= kNCW, "row groups");
  static_assert(STAGES >= 2, "ring depth");
};

template <int R, int XR, int KBS, int MINB, int EPI>
__global__ void __launch_bounds__(kGvThreads, MINB)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    const StreamArgs a) {
  using P = MmaSlab<R, XR, KBS, MINB>;
  constexpr int STAGES = P::STAGES, KS = P::KS, SB = P::SB, RG = P::RG;
  constexpr int XN = P::XN;                            // 8-token column tiles
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int M = a.M, K = a.K;
  float* red = reinterpret_cast<float*>(smem + STAGES * SB);     // [warp][16][XR]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * SB + P::RED);
  uint64_t* empty = full + STAGES;
  volatile int* s_flags = reinterpret_cast<volatile int*>(empty + STAGES);  // [0] abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&wmap);
    prefetch_tmap(&xmap);
  }
  __syncthreads();
  griddep_launch_dependents();

  const int row0 = blockIdx.x * R;
  const int nst = (K + KS - 1) / KS;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      auto issue_x = [&](int s, int i) {
        tma_load_3d(smem + s * SB + P::WB, &xmap, 0, 0, i * KBS, &full[s], pol_x);
      };
      const int npre = nst < STAGES ? nst : STAGES;
      int i = 0;
      for (; i < npre; ++i) {
        mbar_arrive_expect_tx(&full[i], P::WB + P::XB);
        tma_load_3d(smem + i * SB, &wmap, 0, row0, i * KBS, &full[i], pol_w);
      }
      griddep_wait();
      for (int j = 0; j < npre; ++j) issue_x(j, j);
      for (; i < nst; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], ((i / STAGES) + 1) & 1, a.timeout_ns, a.status)) {
          s_flags[0] = 1;
          break;
        }
        if (s_flags[0]) break;
        mbar_arrive_expect_tx(&full[s], P::WB + P::XB);
        tma_load_3d(smem + s * SB, &wmap, 0, row0, i * KBS, &full[s], pol_w);
        issue_x(s, i);
      }
      // Drain: every issued copy has landed before the CTA may exit.
      const int issued = i;
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const int uses = (issued - s + STAGES - 1) / STAGES;
        mbar_wait(&full[s], (uses - 1) & 1, drain_ns(a.timeout_ns), nullptr);
      }
    } else {
      griddep_wait();
    }
  } else {
    // ---------------------------------------------------------------- consumers
    griddep_wait();
    const int w = warp - 1;
    const int rg = w % RG;                   // this warp's row group (every task of it)
    const int nw = (kNCW - rg + RG - 1) / RG;  // warps of that row group
    const int mi = lane >> 3, r8 = lane & 7;
    const int a_row = rg * 16 + (mi & 1) * 8 + r8;
    const int bn = lane >> 2, bk = (lane & 3) * 2;  // B fragment: token, k pair
    float d[XN][4];
#pragma unroll
    for (int nt = 0; nt < XN; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[nt][e] = 0.f;
    for (int i = 0; i < nst; ++i) {
      const int s = i % STAGES;
      if (!s_flags[0]) {
        if (!mbar_wait(&full[s], (i / STAGES) & 1, a.timeout_ns, a.status)) s_flags[0] = 1;
      }
      if (!s_flags[0]) {
        const uint32_t wst = smem_u32(smem + s * SB);
        const uint8_t* xs = smem + s * SB + P::WB;   // [k block][XR tokens][128 B], swizzled
#pragma unroll
        // the nw warps of row group rg take the stage's k blocks in turn
        for (int kb = w / RG; kb < KBS; kb += nw) {
          if ((i * KBS + kb) * 64 < K) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint32_t af[4];
              const int ach = kk * 2 + (mi >> 1);
              ldmatrix_x4(af[0], af[1], af[2], af[3],
                          wst + (kb * R + a_row) * 128 + ((ach ^ r8) << 4));
#pragma unroll
              for (int nt = 0; nt < XN; ++nt) {
                // token t's 16-byte chunks kk*2 and kk*2+1 of k block kb, the
                // lane's k pair at byte bk*2 within each
                const int t = nt * 8 + bn;
                const int xrow = kb * XR + t;
                uint32_t b0 = 0u, b1 = 0u;
                if (t < M) {
                  const uint8_t* xr = xs + xrow * 128 + bk * 2;
                  b0 = *reinterpret_cast<const uint32_t*>(xr + (((kk * 2) ^ (xrow & 7)) << 4));
                  b1 = *reinterpret_cast<const uint32_t*>(xr + (((kk * 2 + 1) ^ (xrow & 7)) << 4));
                }
                if (nt * 8 < M) mma_bf16_16816(d[nt], af, b0, b1);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // this warp's tile of its row group: rows g, g + 8; tokens 2(l%4), +1
    const int g = lane >> 2, tc = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < XN; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = g + (e >> 1) * 8, t = nt * 8 + tc + (e & 1);
        if (t < XR) red[(w * 16 + rr) * XR + t] = d[nt][e];
      }
    named_bar_sync(1, kNCW * 32);
    const int ct = threadIdx.x - 32;
    for (int e = ct; e < R * M; e += kNCW * 32) {
      const int r = e % R, t = e / R;
      const int grp = r / 16, rr = r % 16;
      float v = 0.f;
#pragma unroll
      for (int q = grp; q < kNCW; q += RG) v += red[(q * 16 + rr) * XR + t];
      const int n = row0 + r;
      if (!s_flags[0] && n < a.nout) store_out<EPI, false>(a, GroupInfo{0, 0, M}, t, n, v);
    }
  }
  __syncthreads();
}

template <int R, int XR, int KBS, int MINB, int EPI>
static cudaError_t run_gemv_mma(const Ctx& cx, const void* x, long long ldx, const void* W,
                                const void* res, const float* addf, void* y, int M, int N, int K) {
  if (M > XR) return cudaErrorInvalidValue;
  auto kern = gemv_mma_kernel<R, XR, KBS, MINB, EPI>;
  constexpr int SMEM = MmaSlab<R, XR, KBS, MINB>::SMEM;
  static_assert(MINB * (SMEM + 1024) <= kSmemPerSm, "CTAs per SM");
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM, true); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap_slab(&wmap, W, (uint64_t)N, (uint64_t)K, R, KBS) ||
      !make_tmap_slab(&xmap, x, (uint64_t)M, (uint64_t)K, XR, KBS, (uint64_t)ldx))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = K;
  a.nout = N;
  a.M = M;
  a.out = y;
  a.ldo = N;
  a.res = reinterpret_cast<const uint16_t*>(res);
  a.status = cx.status;
  a.timeout_ns = cx.timeout_ns;
  a.out_len = (long long)M * N;
  a.res_len = res ? (long long)M * N : 0;
  a.addf = addf;
  a.addf_len = addf ? (long long)M * N : 0;
  const int grid = (N + R - 1) / R;
  return launch_k(kern, dim3(grid), dim3(kGvThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

template <int R, int EPI>
static cudaError_t run_gemv(const Ctx& cx, const void* x, long long ldx, const void* W,
                            const void* res, void* y, int M, int N, int K) {
  auto kern = gemv_slab_kernel<R, EPI>;
  constexpr int SMEM = gemv_smem(R);
  static_assert(2 * (SMEM + 1024) <= kSmemPerSm, "two CTAs per SM");
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM, true); e != cudaSuccess) return e;
  CUtensorMap wmap;
  if (!make_tmap_slab(&wmap, W, (uint64_t)N, (uint64_t)K, R, kGvStage / (2 * R) / 64))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = K;
  a.nout = N;
  a.M = M;
  a.out = y;
  a.ldo = N;
  a.res = reinterpret_cast<const uint16_t*>(res);
  a.status = cx.status;
  a.timeout_ns = cx.timeout_ns;
  a.out_len = (long long)M * N;
  a.res_len = res ? (long long)M * N : 0;
  const int grid = (N + R - 1) / R;
  return launch_k(kern, dim3(grid), dim3(kGvThreads), SMEM, cx.stream, cx.pdl, wmap,
                  reinterpret_cast<const uint16_t*>(x), ldx, a);
}

// Rows per CTA for N rows on `sms` SMs: the smallest R in {8, 16, 32} whose
// grid fits on the SMs, if that grid keeps at least three quarters of them
// busy; 0 when the slab kernel does not apply (then split-K does).
int gemv_slab_rows(int M, int N, int K, int sms) {
  if (M < 1 || M > kGvMaxTokens || (K % 64) != 0) return 0;
  for (int R = 8; R <= 32; R <<= 1) {
    const long long grid = ((long long)N + R - 1) / R;
    if (grid <= sms) return grid * 4 < 3LL * sms ? 0 : R;
  }
  return 0;
}

// Rows per CTA of the mma slabs: 16, 32, 48 or 64 (1-4 row groups), the
// smallest whose grid fits on the SMs, if that grid keeps at least three
// quarters of them busy; 0 when none does (or more than 16 tokens, or
// K % 64 != 0).
int gemv_mma_rows(int M, int N, int K, int sms) {
  if (M < 1 || M > kMmaMaxTokens || (K % 64) != 0) return 0;
  for (int R = 16; R <= 64; R += 16) {
    const long long grid = ((long long)N + R - 1) / R;
    if (grid <= sms) return grid * 4 < 3LL * sms ? 0 : R;
  }
  return 0;
}

// One CTA per SM with a ring twice as deep when a CTA streams more than
// 320 KB (its weight rows and token rows over all of K): same-GPU A/B, us,
// two CTAs per SM -> one: 2048 x 7168 at M = 5 / 8 / 16: 6.89 / 6.90 / 8.87
// -> 6.35 / 6.33 / 7.09 (344-459 KB); 2048 x 16384 at M = 1 / 8: 13.45 /
// 13.93 -> 12.45 / 11.80; 4096 x 7168 at M = 4: 11.09 -> 10.70. Below, the
// next call's CTAs loading their first stages while this one finishes
// count for more: 4096 x 4096 at M = 1: 7.07 -> 7.37 (295 KB); 2048 x 7168
// at M = 4: 6.40 -> 6.60 (287 KB).
constexpr long long kDeepRingBytes = 320 * 1024;

template <int R, int XR, int KBS>
static cudaError_t mma_epi(const Ctx& cx, bool residual, const void* x, long long ldx,
                           const void* W, const void* res, const float* addf, void* y, int M,
                           int N, int K) {
  if ((long long)(R + XR) * K * 2 > kDeepRingBytes)
    return residual
               ? run_gemv_mma<R, XR, KBS, 1, EPI_BF16_RES>(cx, x, ldx, W, res, addf, y, M, N, K)
               : run_gemv_mma<R, XR, KBS, 1, EPI_BF16>(cx, x, ldx, W, res, addf, y, M, N, K);
  return residual
             ? run_gemv_mma<R, XR, KBS, 2, EPI_BF16_RES>(cx, x, ldx, W, res, addf, y, M, N, K)
             : run_gemv_mma<R, XR, KBS, 2, EPI_BF16>(cx, x, ldx, W, res, addf, y, M, N, K);
}

// Token rows per stage XR = 4, 8 or 16 (the least that holds M); k blocks
// per stage so that a stage holds 16 KB of weights (8 at R = 16, 4 at 32, 2
// at 64), 24 KB at R = 48 (4 k blocks, two per warp of a row group).
template <int R>
static cudaError_t mma_rows(const Ctx& cx, bool residual, const void* x, long long ldx,
                            const void* W, const void* res, const float* addf, void* y, int M,
                            int N, int K) {
  constexpr int KBS = R == 48 ? 4 : 128 / R;
  if (M <= 4) return mma_epi<R, 4, KBS>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  if (M <= 8) return mma_epi<R, 8, KBS>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  return mma_epi<R, 16, KBS>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
}

cudaError_t launch_gemv_mma(const Ctx& cx, bool residual, const void* x, const void* W,
                            const void* res, void* y, int M, int N, int K, int R,
                            const float* addf) {
  const long long ldx = cx.ldx ? cx.ldx : K;
  if (R == 16) return mma_rows<16>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  if (R == 32) return mma_rows<32>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  if (R == 48) return mma_rows<48>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  if (R == 64) return mma_rows<64>(cx, residual, x, ldx, W, res, addf, y, M, N, K);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_slab(const Ctx& cx, bool residual, const void* x, const void* W,
                             const void* res, void* y, int M, int N, int K, int R) {
  const long long ldx = cx.ldx ? cx.ldx : K;
  if (R == 8)
    return residual ? run_gemv<8, EPI_BF16_RES>(cx, x, ldx, W, res, y, M, N, K)
                    : run_gemv<8, EPI_BF16>(cx, x, ldx, W, res, y, M, N, K);
  if (R == 16)
    return residual ? run_gemv<16, EPI_BF16_RES>(cx, x, ldx, W, res, y, M, N, K)
                    : run_gemv<16, EPI_BF16>(cx, x, ldx, W, res, y, M, N, K);
  if (R == 32)
    return residual ? run_gemv<32, EPI_BF16_RES>(cx, x, ldx, W, res, y, M, N, K)
                    : run_gemv<32, EPI_BF16>(cx, x, ldx, W, res, y, M, N, K);
  return cudaErrorInvalidValue;
}

}  // namespace dg
