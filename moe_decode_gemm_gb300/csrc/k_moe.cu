// k_moe.cu -- the MoE decode block's kernels: router scoring with the
// top-k / gate / expert-gather tail, the routed experts' gate-up (SwiGLU) and
// down projections over the selected experts only, the shared expert, and the
// gate-weighted combine. Plus the residual add, the L2 prefetch kernel and the
// failure-detection self test.
// "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §3 "改进 MoE 调度与重叠" and
// Part 1 §4 "将即将使用的权重预取到缓存".
#include <utility>

#include "launch.h"
#include "launch_util.cuh"
#include "wstream.cuh"

namespace dg {

constexpr int kMoeXR = 64;                  // router and shared expert: every token (M <= 64)
constexpr int kMoeStages = 4;
constexpr int kRouterStages = 3;
constexpr int kExpertXR = kGroupTokens;     // routed experts: one group's tokens
constexpr int kExpertPairStages = 3;        // gate/up: 64 KB stages (gate and up halves)
constexpr int kSharedPairStages = 2;        // shared gate/up: 64 KB + 16 KB of tokens
constexpr int kRouteScratch = 36 * 1024;

constexpr int moe_smem(int stages, int extra) { return wstream_smem(kMoeXR, stages, extra); }
constexpr int expert_pair_smem() { return wstream_smem(kExpertXR, kExpertPairStages, 0, true); }

template <typename K>
static cudaError_t smem_once(K kern, int bytes, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = allow_smem(kern, bytes);
  if (e == cudaSuccess) done = true;
  return e;
}

static StreamArgs base_args(const Ctx& cx, float* ws, int* ctr) {
  StreamArgs a = {};
  a.mma_min_tokens = 3;  // 1-2 tokens: CUDA-core dot products
  a.ws = ws;
  a.ctr = ctr;
  a.status = cx.status;
  a.timeout_ns = cx.timeout_ns;
  return a;
}

cudaError_t launch_router(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E, int k,
                          int32_t* idx_user, float* w_user, const MoeBufs& b, float* ws, int* ctr) {
  constexpr int SMEM = moe_smem(kRouterStages, kRouteScratch);
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<kMoeXR, kRouterStages, EPI_F32, false, false, true>;
  static bool done = false;
  cudaError_t e = smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Wr, (uint64_t)E, (uint64_t)H, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)H, kMoeXR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = H;
  a.KB = (H + kKChunk - 1) / kKChunk;
  a.TILES = (E + kTileRows - 1) / kTileRows;
  a.nout = E;
  a.M = M;
  a.out = b.logits;
  a.ldo = E;
  a.done = b.done;
  a.total_tiles_dense = a.TILES;
  a.route.M = M;
  a.route.E = E;
  a.route.k = k;
  a.route.logits = b.logits;
  a.route.idx_user = idx_user;
  a.route.w_user = w_user;
  a.route.nact = b.nact;
  a.route.grp_exp = b.grp_exp;
  a.route.grp_off = b.grp_off;
  a.route.pair_tok = b.pair_tok;
  a.route.pair_of = b.pair_of;
  a.route.gate = b.gate;
  a.route.done = b.done;
  a.route.total_tiles = a.TILES;
  // The router streams only E*H bf16 (5.5 MB for 384 x 7168) and is latency
  // bound: a sixth of the SMs keeps the number of CTAs per output tile, and so
  // the split-K fixup, small.
  const long long T = (long long)a.TILES * a.KB;
  const int cap = router_grid(cx.sms);  // the shared expert uses the other SMs
  const int grid = (int)(T < cap ? T : cap);
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

cudaError_t launch_experts_w13(const Ctx& cx, const void* x, const void* W13, int M, int H, int E,
                               int k, int I, const MoeBufs& b, float* ws, int* ctr) {
  constexpr int SMEM = expert_pair_smem();
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<kExpertXR, kExpertPairStages, EPI_SWIGLU, true, true, false>;
  static bool done = false;
  cudaError_t e = smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W13, (uint64_t)E * 2 * I, (uint64_t)H, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.xs, (uint64_t)M * k, (uint64_t)H, kExpertXR, false))
    return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = H;
  a.KB = (H + kKChunk - 1) / kKChunk;
  a.TILES = (I + kTileRows - 1) / kTileRows;
  a.nout = I;
  a.M = M;
  a.nact = b.nact;
  a.grp_exp = b.grp_exp;
  a.grp_off = b.grp_off;
  a.w_group_rows = 2 * I;
  a.w_up_offset = I;
  a.out = b.h;
  a.ldo = I;
  return launch_k(kern, dim3(cx.sms), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

cudaError_t launch_experts_w2(const Ctx& cx, const void* W2, int M, int H, int E, int k, int I,
                              const MoeBufs& b, float* ws, int* ctr) {
  // 256-row output tiles: two 128-row halves, 64 KB weight stages
  constexpr int SMEM = expert_pair_smem();
  auto kern = wstream_kernel<kExpertXR, kExpertPairStages, EPI_F32, false, true, false, true>;
  static bool done = false;
  cudaError_t e = smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W2, (uint64_t)E * H, (uint64_t)I, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.h, (uint64_t)M * k, (uint64_t)I, kExpertXR, false))
    return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = I;
  a.KB = (I + kKChunk - 1) / kKChunk;
  a.TILES = (H + 2 * kTileRows - 1) / (2 * kTileRows);
  a.nout = H;
  a.M = M;
  a.nact = b.nact;
  a.grp_exp = b.grp_exp;
  a.grp_off = b.grp_off;
  a.w_group_rows = H;
  a.out = b.o;
  a.ldo = H;
  return launch_k(kern, dim3(cx.sms), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

cudaError_t launch_shared_w13(const Ctx& cx, const void* x, const void* Ws13, int M, int H, int I,
                              const MoeBufs& b, int grid, float* ws, int* ctr) {
  constexpr int SMEM = wstream_smem(kMoeXR, kSharedPairStages, 0, true);
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<kMoeXR, kSharedPairStages, EPI_SWIGLU, true, false, false>;
  static bool done = false;
  cudaError_t e = smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Ws13, (uint64_t)2 * I, (uint64_t)H, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)H, kMoeXR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = H;
  a.KB = (H + kKChunk - 1) / kKChunk;
  a.TILES = (I + kTileRows - 1) / kTileRows;
  a.nout = I;
  a.M = M;
  a.w_up_offset = I;
  a.out = b.hs;
  a.ldo = I;
  const long long T = (long long)a.TILES * a.KB;
  if (grid > T) grid = (int)T;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

cudaError_t launch_shared_w2(const Ctx& cx, const void* Ws2, int M, int H, int I, const MoeBufs& b,
                             int grid, float* ws, int* ctr) {
  constexpr int SMEM = moe_smem(kMoeStages, 0);
  auto kern = wstream_kernel<kMoeXR, kMoeStages, EPI_F32, false, false, false>;
  static bool done = false;
  cudaError_t e = smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Ws2, (uint64_t)H, (uint64_t)I, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.hs, (uint64_t)M, (uint64_t)I, kMoeXR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = I;
  a.KB = (I + kKChunk - 1) / kKChunk;
  a.TILES = (H + kTileRows - 1) / kTileRows;
  a.nout = H;
  a.M = M;
  a.out = b.s;
  a.ldo = H;
  const long long T = (long long)a.TILES * a.KB;
  if (grid > T) grid = (int)T;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, a);
}

// ------------------------------------------------------------------ token gather
// xs[p] = x[pair_tok[p]] for every (token, slot) pair p: the routed experts'
// token rows in expert order, so that each expert group's rows are contiguous
// and reach shared memory as one TMA box. 16-byte vectors, grid-stride.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x,
                                                     const int* __restrict__ pair_tok,
                                                     uint4* __restrict__ xs, int npairs,
                                                     int row_vecs) {
  griddep_launch_dependents();
  griddep_wait();
  const long long total = (long long)npairs * row_vecs;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < total;
       v += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(v / row_vecs);
    const int c = (int)(v - (long long)p * row_vecs);
    xs[v] = x[(long long)pair_tok[p] * row_vecs + c];
  }
}

cudaError_t launch_gather(const Ctx& cx, const void* x, int M, int H, int k, const MoeBufs& b) {
  const int row_vecs = H / 8;
  const long long total = (long long)M * k * row_vecs;
  long long grid = (total + 255) / 256;
  if (grid > 2 * cx.sms) grid = 2 * cx.sms;
  if (grid < 1) grid = 1;
  return launch_k(gather_kernel, dim3((unsigned)grid), dim3(256), 0, cx.stream, cx.pdl,
                  reinterpret_cast<const uint4*>(x), (const int*)b.pair_tok,
                  reinterpret_cast<uint4*>(b.xs), M * k, row_vecs);
}

// ------------------------------------------------------------------ combine
// out[m,n] = bf16( res[m,n] + (sum_{j<k} g[m,j] * o[pair(m,j), n] + s[m,n]) ),
// j summed in order 0..k-1, then the shared term, then the residual.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o,
                                                      const float* __restrict__ s,
                                                      const float* __restrict__ gate,
                                                      const int* __restrict__ pair_of,
                                                      const uint16_t* res,  // may alias out
                                                      uint16_t* out, int M, int H,
                                                      int k) {
  griddep_launch_dependents();
  griddep_wait();
  const int per_row = H / 4;
  const long long total = (long long)M * per_row;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < total;
       v += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(v / per_row);
    const int n = (int)(v - (long long)m * per_row) * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const float g = gate[m * k + j];
      const int p = pair_of[m * k + j];
      const float4 ov = *reinterpret_cast<const float4*>(o + (long long)p * H + n);
      acc[0] = fmaf(g, ov.x, acc[0]);
      acc[1] = fmaf(g, ov.y, acc[1]);
      acc[2] = fmaf(g, ov.z, acc[2]);
      acc[3] = fmaf(g, ov.w, acc[3]);
    }
    if (s) {
      const float4 sv = *reinterpret_cast<const float4*>(s + (long long)m * H + n);
      acc[0] += sv.x;
      acc[1] += sv.y;
      acc[2] += sv.z;
      acc[3] += sv.w;
    }
    if (res) {
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = bf_bits2f(res[(long long)m * H + n + q]) + acc[q];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) out[(long long)m * H + n + q] = f2bf_bits(acc[q]);
  }
}

cudaError_t launch_combine(const Ctx& cx, const MoeBufs& b, bool with_shared, const void* res,
                           void* out, int M, int H, int k) {
  const long long total = (long long)M * (H / 4);
  int grid = (int)((total + 255) / 256);
  if (grid > 4 * cx.sms) grid = 4 * cx.sms;
  if (grid < 1) grid = 1;
  return launch_k(combine_kernel, dim3(grid), dim3(256), 0, cx.stream, cx.pdl, (const float*)b.o,
                  (const float*)(with_shared ? b.s : nullptr), (const float*)b.gate,
                  (const int*)b.pair_of, reinterpret_cast<const uint16_t*>(res),
                  reinterpret_cast<uint16_t*>(out), M, H, k);
}

// ------------------------------------------------------------------ residual add
// out may alias a or b: each element is read and written by one thread.
__global__ void __launch_bounds__(256) add_kernel(const uint16_t* a, const uint16_t* b,
                                                  uint16_t* out, long long n) {
  griddep_launch_dependents();
  griddep_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = f2bf_bits(bf_bits2f(a[i]) + bf_bits2f(b[i]));
}

cudaError_t launch_add(const Ctx& cx, const void* a, const void* b, void* out, size_t n) {
  long long grid = ((long long)n + 255) / 256;
  if (grid > 4 * cx.sms) grid = 4 * cx.sms;
  if (grid < 1) grid = 1;
  return launch_k(add_kernel, dim3((unsigned)grid), dim3(256), 0, cx.stream, cx.pdl,
                  reinterpret_cast<const uint16_t*>(a), reinterpret_cast<const uint16_t*>(b),
                  reinterpret_cast<uint16_t*>(out), (long long)n);
}

// ------------------------------------------------------------------ L2 prefetch
// Each thread issues bulk L2 prefetches of 32 KB chunks of the range.
__global__ void __launch_bounds__(128) prefetch_kernel(const uint8_t* __restrict__ p,
                                                       long long bytes) {
  constexpr long long kChunk = 32 * 1024;
  const long long nchunks = (bytes + kChunk - 1) / kChunk;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < nchunks;
       c += (long long)gridDim.x * blockDim.x) {
    const long long off = c * kChunk;
    const long long len = (bytes - off) < kChunk ? (bytes - off) : kChunk;
    bulk_prefetch_l2(p + off, (uint32_t)len);
  }
}

cudaError_t launch_prefetch(const Ctx& cx, const void* ptr, size_t bytes) {
  const long long nchunks = ((long long)bytes + 32767) / 32768;
  long long grid = (nchunks + 127) / 128;
  if (grid > cx.sms) grid = cx.sms;
  if (grid < 1) grid = 1;
  // No PDL: the prefetch has no data dependency and must not delay dependents.
  return launch_k(prefetch_kernel, dim3((unsigned)grid), dim3(128), 0, cx.stream, false,
                  reinterpret_cast<const uint8_t*>(ptr), (long long)bytes);
}

// ------------------------------------------------------------------ self test
// Waits, with the same bounded wait every kernel uses, on a barrier that no
// one arrives at. The wait must give up and set the status word.
__global__ void selftest_timeout_kernel(int* status, long long ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, ns, status);
  }
}

cudaError_t launch_selftest_timeout(const Ctx& cx, long long ns) {
  return launch_k(selftest_timeout_kernel, dim3(1), dim3(32), 0, cx.stream, false, cx.status, ns);
}

}  // namespace dg
