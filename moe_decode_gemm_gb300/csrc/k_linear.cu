// k_linear.cu -- dense decode projections y = x·Wᵀ on the weight-streaming
// kernel: the CUDA-core small-matrix path (M <= 2) and the mma.sync split-K
// path (3 <= M <= 16, and up to 64 when forced), each with stream-K, 256-row
// (wide) or cluster-split instances. "vLLM 如何用智能体辅助优化 Kimi K3 解码性能",
// Part 1 §1.
#include <utility>

#include "launch.h"
#include "launch_util.cuh"
#include "wstream.cuh"

namespace dg {

// Narrow tiles at 8 or 16 token rows: 3 stages (about 105 KB of shared memory)
// so that two CTAs fit on an SM -- the next call's CTA starts and streams its
// weights while the previous call's CTA on that SM finishes its split-K
// reduction. Wide tiles and 64 token rows: one CTA per SM, deeper rings.
template <int XR, bool WIDE>
constexpr int dense_minb() {
  return (!WIDE && XR <= 16) ? 2 : 1;
}

template <int XR, bool WIDE>
constexpr int dense_stages() {
  return WIDE ? 3 : dense_minb<XR, WIDE>() == 2 ? 3 : 4;
}

template <int XR, bool WIDE>
constexpr int dense_smem() {
  return wstream_smem(XR, dense_stages<XR, WIDE>(), 0, WIDE);
}

// WIDE: 256-row output tiles, 64 KB weight stages (two 128-row halves).
// CL > 0: cluster split, CL CTAs per output tile (grid = tiles * CL).
// PATH: PATH_CORE (1-2 tokens, CUDA cores only) or PATH_ANY with every group
// on mma.sync (mma_min_tokens = 1). The mma.sync instances keep the CUDA-core
// branch: without it the compiler scheduled their loop into more spills at
// 112 registers (M = 4 / 16, N = 2048: 8.3 / 9.1 us against 10.1 / 11.0 us).
template <int XR, int EPI, bool WIDE, bool CLUSTER, int PATH>
static cudaError_t run_dense_path(const Ctx& cx, const void* x, const void* W, const void* res,
                                  void* y, int M, int N, int K, int grid, float* ws, int* ctr,
                                  int cl) {
  constexpr int S = dense_stages<XR, WIDE>();
  constexpr int MINB = dense_minb<XR, WIDE>();
  constexpr int SMEM = dense_smem<XR, WIDE>();
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  static_assert(MINB == 1 || 2 * (SMEM + 1024) <= kSmemPerSm, "two CTAs per SM");
  static_assert(!CLUSTER || kTileRows * XR * 4 <= S * (kWBytes + kKSub * XR * 128),
                "the partial tile fits in the stage ring");
  auto kern = wstream_kernel<XR, S, EPI, false, false, WIDE, ROLE_PROJECTION, MINB, CLUSTER, PATH>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM, MINB > 1); e != cudaSuccess) return e;
  constexpr int kTile = WIDE ? 2 * kTileRows : kTileRows;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W, (uint64_t)N, (uint64_t)K, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)K, XR, false, (uint64_t)cx.ldx))
    return cudaErrorInvalidValue;
  StreamArgs a = {};
  a.K = K;
  a.KB = (K + kKChunk - 1) / kKChunk;
  a.TILES = (N + kTile - 1) / kTile;
  a.nout = N;
  a.M = M;
  a.mma_min_tokens = PATH == PATH_CORE ? 1 << 30 : 1;
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
  if (CLUSTER)
    return launch_kc(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, cl, wmap, xmap, xmap,
                     a);
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, xmap, a);
}

// The CUDA-core consumer takes at most two tokens and only runs at 8 token
// rows per stage (the small-matrix regime); every other instance is mma.sync.
template <int XR, int EPI, bool WIDE = false, bool CLUSTER = false>
static cudaError_t run_dense(const Ctx& cx, bool mma, const void* x, const void* W, const void* res,
                             void* y, int M, int N, int K, int grid, float* ws, int* ctr,
                             int cl = 0) {
  if (mma)
    return run_dense_path<XR, EPI, WIDE, CLUSTER, PATH_ANY>(cx, x, W, res, y, M, N, K, grid, ws,
                                                            ctr, cl);
  if constexpr (XR == 8) {
    if (M <= 2)
      return run_dense_path<8, EPI, WIDE, CLUSTER, PATH_CORE>(cx, x, W, res, y, M, N, K, grid, ws,
                                                              ctr, cl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dense_cluster(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                                 const void* W, const void* res, void* y, int M, int N, int K,
                                 int cl) {
  const int grid = (N + kTileRows - 1) / kTileRows * cl;
  if (xr == 8)
    return residual ? run_dense<8, EPI_BF16_RES, false, true>(cx, mma, x, W, res, y, M, N, K, grid,
                                                              nullptr, nullptr, cl)
                    : run_dense<8, EPI_BF16, false, true>(cx, mma, x, W, res, y, M, N, K, grid,
                                                          nullptr, nullptr, cl);
  if (xr == 16)
    return residual ? run_dense<16, EPI_BF16_RES, false, true>(cx, mma, x, W, res, y, M, N, K,
                                                               grid, nullptr, nullptr, cl)
                    : run_dense<16, EPI_BF16, false, true>(cx, mma, x, W, res, y, M, N, K, grid,
                                                           nullptr, nullptr, cl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_dense_wide(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                              const void* W, const void* res, void* y, int M, int N, int K,
                              int grid, float* ws, int* ctr) {
  if (xr == 8)
    return residual
               ? run_dense<8, EPI_BF16_RES, true>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr)
               : run_dense<8, EPI_BF16, true>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr);
  if (xr == 16)
    return residual
               ? run_dense<16, EPI_BF16_RES, true>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr)
               : run_dense<16, EPI_BF16, true>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr);
  return cudaErrorInvalidValue;
}

cudaError_t launch_dense_f32(const Ctx& cx, int xr, bool mma, const void* x, const void* W,
                             float* y, int M, int N, int K, int grid, float* ws, int* ctr) {
  if (xr == 8) return run_dense<8, EPI_F32>(cx, mma, x, W, nullptr, y, M, N, K, grid, ws, ctr);
  if (xr == 16) return run_dense<16, EPI_F32>(cx, mma, x, W, nullptr, y, M, N, K, grid, ws, ctr);
  return run_dense<64, EPI_F32>(cx, mma, x, W, nullptr, y, M, N, K, grid, ws, ctr);
}

cudaError_t launch_dense(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                         const void* W, const void* res, void* y, int M, int N, int K, int grid,
                         float* ws, int* ctr) {
  if (xr == 8)
    return residual ? run_dense<8, EPI_BF16_RES>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr)
                    : run_dense<8, EPI_BF16>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr);
  if (xr == 16)
    return residual ? run_dense<16, EPI_BF16_RES>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr)
                    : run_dense<16, EPI_BF16>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr);
  return residual ? run_dense<64, EPI_BF16_RES>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr)
                  : run_dense<64, EPI_BF16>(cx, mma, x, W, res, y, M, N, K, grid, ws, ctr);
}

}  // namespace dg
