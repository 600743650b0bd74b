// k_gemv.cu -- decode projection y = x·Wᵀ for 1-2 tokens without splitting K
// across CTAs: each CTA owns R consecutive weight rows (R = 8, 16 or 32) over
// the whole K, so no partial sums leave the CTA -- no workspace, counters,
// atomics or cluster barriers. What split-K spends after the last weight
// byte (the wait for the slowest rank of a tile, the reduction of the
// partial tiles and the barrier that keeps partials alive) is gone; the sum
// over K ends with a reduction inside the CTA.
//
// One producer thread streams stages of 32 KB of weights, each R rows x
// 16384/R k, with one 3-D TMA box (rows x k blocks of 64, 128-byte swizzle),
// and the tokens' matching k range (a bulk copy per token, issued once the
// previous kernel has finished; the weights of the first stages are in
// flight before that). Eight consumer warps split each stage by k block:
// lane l of warp w takes row l % R of k block w*(32/R) + l/R and its 8 chunks
// of 16 bytes, multiplying them with the tokens' matching chunks
// (fma.rn.f32.bf16, fp32 sums). The 32/R lanes of a row and then the 8 warps
// are summed in a fixed order, so results do not vary from run to run.
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
constexpr int kGvMaxTokens = 2;

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
