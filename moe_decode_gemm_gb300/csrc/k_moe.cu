// k_moe.cu -- the MoE decode block's kernels: router scoring with the top-k
// and renormalised gates in the same kernel (routing.cuh), the expert-gather
// schedule and token gather, the routed
// experts' gate-up (SwiGLU) and down projections over the selected experts
// only, the shared expert, and the gate-weighted combine. Plus the residual
// add, the L2 prefetch kernel and the failure-detection self test.
// "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §3 "改进 MoE 调度与重叠" and
// Part 1 §4 "将即将使用的权重预取到缓存".
#include <utility>

#include "launch.h"
#include "launch_util.cuh"
#include "wstream.cuh"

namespace dg {

constexpr int kExpertPairStages = 3;  // gate/up: 64 KB stages (gate and up halves)

// Token rows per stage of the routed-expert kernels: a group's tokens. Up to
// 16 tokens no expert can have more than 16, and the 16-row instances are
// used; beyond, the 32-row instances, so that an expert chosen by 17-32 tokens
// streams its weights once. Groups of at most 16 tokens load a 16-row token
// box there (kNarrowRows).
template <int XR>
constexpr int expert_pair_smem() {
  return wstream_smem(XR, kExpertPairStages, 0, true);
}


static StreamArgs base_args(const Ctx& cx, float* ws, int* ctr) {
  StreamArgs a = {};
  // mma.sync dot products for groups of any size: same-GPU A/B of the MoE
  // block, us at M = 1 / 4 / 16 / 64, CUDA cores for groups of 1-2 tokens ->
  // mma.sync: 142.0 / 428.4 / 1453.2 / 3745.9 -> 140.6 / 425.4 / 1446.0 /
  // 3712.8 (most groups hold 1-2 tokens under uniform routing)
  a.mma_min_tokens = 1;
  a.ws = ws;
  a.ctr = ctr;
  a.status = cx.status;
  a.timeout_ns = cx.timeout_ns;
  a.ws_len = cx.ws_len;
  a.ctr_len = cx.ctr_len;
  return a;
}

// ------------------------------------------------------------------ router
// logits[m, e] = x[m]·Wr[e] in fp32 (not rounded): the weight-streaming kernel
// with fp32 output, token rows per stage sized to M. The router streams only
// E*H bf16 (5.5 MB for 384 x 7168) and is latency bound: it runs in the
// cluster split, router_clusters(H) CTAs per 128-row tile of experts summing
// their partial tiles through distributed shared memory, so no split-K fixup
// through L2 sits on the routing path; the shared expert streams on the
// other SMs meanwhile. The last cluster to write its logits then selects
// every token's top-k experts and gates (one warp per token), so no separate
// top-k kernel and launch sits between the scores and the schedule.
template <int XR>
static cudaError_t run_router(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E,
                              int k, int32_t* idx_user, float* w_user, const MoeBufs& b, int L) {
  constexpr int STAGES = XR == 64 ? 4 : 6;
  constexpr int SMEM = wstream_smem(XR, STAGES, 0);
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<XR, STAGES, EPI_F32, false, false, false, ROLE_ROUTER, 1, true>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Wr, (uint64_t)(E + L), (uint64_t)H, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)H, XR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, nullptr, nullptr);
  a.K = H;
  a.KB = (H + kKChunk - 1) / kKChunk;
  a.TILES = (E + L + kTileRows - 1) / kTileRows;
  a.nout = E + L;
  a.M = M;
  a.out = b.logits;
  a.ldo = E + L;
  a.route_k = k;
  a.route_E = E;
  a.route_ctr = b.route_ctr;
  a.route_idx = b.topk;
  a.route_gate = b.gate;
  a.route_idx_user = idx_user;
  a.route_w_user = w_user;
  a.out_len = (long long)M * (E + L);
  a.pairs = M * k;
  const int cl = router_clusters(H);
  return launch_kc(kern, dim3(a.TILES * cl), dim3(kThreads), SMEM, cx.stream, cx.pdl, cl, wmap,
                   xmap, xmap, a);
}

// From 17 tokens the router's product is a dense contraction (352 MFLOP at
// 64 tokens over 384 x 7168): tcgen05 with the accumulator in tensor memory,
// in the same cluster split and with the same top-k in the last cluster.
// Same-GPU A/B, us per block, mma.sync -> tcgen05 router: MoE block at
// M = 64: 3709 -> 3702 (the shared expert hides most of the router there);
// latent block (L = 512) at M = 32 / 64: 238.9 / 343.3 -> 234.6 / 333.5.
cudaError_t launch_router(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E, int k,
                          int32_t* idx_user, float* w_user, const MoeBufs& b, int L) {
  if (k < 1 || k > 32 || k > E || E > 1024 || L < 0) return cudaErrorInvalidValue;
  if (M <= 8) return run_router<8>(cx, x, Wr, M, H, E, k, idx_user, w_user, b, L);
  if (M <= 16) return run_router<16>(cx, x, Wr, M, H, E, k, idx_user, w_user, b, L);
  const RouteOut ro{b.logits, b.route_ctr, b.topk, b.gate, idx_user, w_user};
  return launch_router_tc(cx, x, Wr, M, H, E, L, k, router_clusters(H), ro);
}

// ------------------------------------------------------------------ schedule + gather
// Every CTA builds the expert-gather schedule from the M x k chosen indices
// (cheap: at most 2048 pairs over at most 1024 experts); CTA 0 publishes it:
//   groups  : experts with at least one token, in expert order, split into
//             groups of at most kGroupTokens tokens (grp_exp, grp_off, nact);
//   pairs   : (token, slot) pairs in expert order, by token within an expert
//             (pair_tok = token of pair p, pair_of[m*k + j] = pair of (m, j)).
// Then all CTAs copy xs[p] = x[pair_tok[p]] (16-byte vectors), so each expert
// group's token rows are contiguous for the expert kernels' TMA boxes.
constexpr int kSchedThreads = 256;
constexpr int kMaxE = 1024;
constexpr int kMaxPairs = 64 * 32;

// LATENT: the rows copied are the latent inputs, fp32 scores at columns
// E..E+row_vecs*8-1 of rows of src_ld floats, rounded to bf16 on the way;
// otherwise bf16 token rows of x.
// status / src_len / groups_cap: for the index checks of a DEC_DEBUG build
// (src_len in floats for LATENT, else in 16-byte vectors).
template <bool LATENT>
__global__ void __launch_bounds__(kSchedThreads) schedule_gather_kernel(
    const void* __restrict__ src, long long src_ld, const int* __restrict__ topk, int M, int E,
    int K, int row_vecs, uint4* __restrict__ xs, int* nact, int* grp_exp, int* grp_off,
    int* pair_tok, int* pair_of, int* status, long long src_len, int groups_cap) {
  // Dynamic shared memory sized to E and M*k (about 9 KB at E = 384, M = 64,
  // k = 8), so a CTA fits on an SM beside a weight-streaming CTA:
  // [E] token masks, [E] pair offsets, [M*k] chosen experts, [M*k] pair tokens.
  extern __shared__ __align__(16) uint8_t s_dyn[];
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(s_dyn);
  int* s_off = reinterpret_cast<int*>(s_mask + E);
  int* s_idx = s_off + E;
  int* s_tok = s_idx + M * K;
  __shared__ int s_warp[64];
  // The expert kernel that follows can do nothing before this schedule is
  // complete: it is let launch only at the end (see below), so that its CTAs
  // do not take SMs early and sit idle while routing runs.
  griddep_wait();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int P = M * K;
  const bool publish = blockIdx.x == 0;
  for (int p = t; p < P; p += kSchedThreads) {
    const int e = topk[p];
    s_idx[p] = DG_OK(status, e >= 0 && e < E, e) ? e : 0;
  }
  for (int e = t; e < E; e += kSchedThreads) s_mask[e] = 0ull;
  __syncthreads();
  for (int p = t; p < P; p += kSchedThreads) atomicOr(&s_mask[s_idx[p]], 1ull << (p / K));
  __syncthreads();
  // exclusive scans over experts of token counts and of group counts
  constexpr int PER = kMaxE / kSchedThreads;  // 4 experts per thread
  int cnt[PER], grp[PER], csum = 0, gsum = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = t * PER + q;
    cnt[q] = (e < E) ? __popcll(s_mask[e]) : 0;
    grp[q] = (cnt[q] + kGroupTokens - 1) / kGroupTokens;
    csum += cnt[q];
    gsum += grp[q];
  }
  int cinc = csum, ginc = gsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int c2 = __shfl_up_sync(0xffffffffu, cinc, off);
    const int g2 = __shfl_up_sync(0xffffffffu, ginc, off);
    if (lane >= off) {
      cinc += c2;
      ginc += g2;
    }
  }
  if (lane == 31) {
    s_warp[warp] = cinc;
    s_warp[32 + warp] = ginc;
  }
  __syncthreads();
  int cpre = 0, gpre = 0;
  for (int w2 = 0; w2 < warp; ++w2) {
    cpre += s_warp[w2];
    gpre += s_warp[32 + w2];
  }
  cpre += cinc - csum;
  gpre += ginc - gsum;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = t * PER + q;
    if (e < E) {
      s_off[e] = cpre;
      if (publish)
        for (int j = 0; j < grp[q]; ++j) {
          *DG_AT(status, grp_exp, gpre + j, groups_cap) = e;
          *DG_AT(status, grp_off, gpre + j, groups_cap + 1) = cpre + j * kGroupTokens;
        }
    }
    cpre += cnt[q];
    gpre += grp[q];
  }
  if (publish && t == kSchedThreads - 1) {
    int total = 0;
    for (int w2 = 0; w2 < kSchedThreads / 32; ++w2) total += s_warp[32 + w2];
    *DG_AT(status, grp_off, total, groups_cap + 1) = P;
    *nact = total;
  }
  __syncthreads();
  // pairs: position of (m, j) among expert e's pairs = tokens below m that chose e
  for (int p = t; p < P; p += kSchedThreads) {
    const int m = p / K;
    const int e = s_idx[p];
    const unsigned long long below = (m == 0) ? 0ull : (s_mask[e] & ((1ull << m) - 1ull));
    const int pos = s_off[e] + __popcll(below);
    *DG_AT(status, s_tok, pos, P) = m;
    if (publish) {
      *DG_AT(status, pair_tok, pos, P) = m;
      pair_of[p] = pos;
    }
  }
  __syncthreads();
  // gather this CTA's share of the token rows
  const long long total = (long long)P * row_vecs;
  for (long long v = blockIdx.x * (long long)kSchedThreads + t; v < total;
       v += (long long)gridDim.x * kSchedThreads) {
    const int p = (int)(v / row_vecs);
    const int c = (int)(v - (long long)p * row_vecs);
    const int m = s_tok[p];
    if constexpr (LATENT) {
      const long long f0 = (long long)m * src_ld + E + (long long)c * 8;
      const float* f = DG_AT(status, reinterpret_cast<const float*>(src), f0, src_len - 7);
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = (uint32_t)f2bf_bits(__ldcg(f + 2 * q)) |
               ((uint32_t)f2bf_bits(__ldcg(f + 2 * q + 1)) << 16);
      xs[v] = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      xs[v] = *DG_AT(status, reinterpret_cast<const uint4*>(src), (long long)m * row_vecs + c,
                     src_len);
    }
  }
  griddep_launch_dependents();
}

cudaError_t launch_gather(const Ctx& cx, const void* x, int M, int H, int E, int k,
                          const MoeBufs& b, int L) {
  if (E > kMaxE || M * k > kMaxPairs) return cudaErrorInvalidValue;
  const int row_vecs = (L > 0 ? L : H) / 8;
  const long long total = (long long)M * k * row_vecs;
  long long grid = (total + kSchedThreads - 1) / kSchedThreads;
  if (grid > cx.sms) grid = cx.sms;
  if (grid < 1) grid = 1;
  const int smem = E * 8 + E * 4 + 2 * M * k * 4;
  if (L > 0)
    return launch_k(schedule_gather_kernel<true>, dim3((unsigned)grid), dim3(kSchedThreads), smem,
                    cx.stream, cx.pdl, (const void*)b.logits, (long long)(E + L),
                    (const int*)b.topk, M, E, k, row_vecs, reinterpret_cast<uint4*>(b.xs), b.nact,
                    b.grp_exp, b.grp_off, b.pair_tok, b.pair_of, cx.status,
                    (long long)M * (E + L), b.groups_cap);
  return launch_k(schedule_gather_kernel<false>, dim3((unsigned)grid), dim3(kSchedThreads), smem,
                  cx.stream, cx.pdl, x, (long long)0, (const int*)b.topk, M, E, k, row_vecs,
                  reinterpret_cast<uint4*>(b.xs), b.nact, b.grp_exp, b.grp_off, b.pair_tok,
                  b.pair_of, cx.status, (long long)M * row_vecs, b.groups_cap);
}

template <int XR>
static cudaError_t run_experts_w13(const Ctx& cx, const void* W13, int M, int H, int E, int k,
                                   int I, const MoeBufs& b, int grid, float* ws, int* ctr) {
  constexpr int SMEM = expert_pair_smem<XR>();
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<XR, kExpertPairStages, EPI_SWIGLU, true, true, false, ROLE_EXPERT>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W13, (uint64_t)E * 2 * I, (uint64_t)H, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.xs, (uint64_t)M * k, (uint64_t)H, XR, false))
    return cudaErrorInvalidValue;
  CUtensorMap xnarrow = xmap;
  if (XR > kNarrowRows &&
      !make_tmap(&xnarrow, b.xs, (uint64_t)M * k, (uint64_t)H, kNarrowRows, false))
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
  a.out_len = (long long)M * k * I;
  a.pairs = M * k;
  a.groups_len = b.groups_cap;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, xnarrow,
                  a);
}

template <int XR>
static cudaError_t run_experts_w2(const Ctx& cx, const void* W2, int M, int H, int E, int k, int I,
                                  const MoeBufs& b, int grid, float* ws, int* ctr) {
  // 256-row output tiles: two 128-row halves, 64 KB weight stages
  constexpr int SMEM = expert_pair_smem<XR>();
  auto kern = wstream_kernel<XR, kExpertPairStages, EPI_F32, false, true, true, ROLE_EXPERT>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, W2, (uint64_t)E * H, (uint64_t)I, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.h, (uint64_t)M * k, (uint64_t)I, XR, false))
    return cudaErrorInvalidValue;
  CUtensorMap xnarrow = xmap;
  if (XR > kNarrowRows &&
      !make_tmap(&xnarrow, b.h, (uint64_t)M * k, (uint64_t)I, kNarrowRows, false))
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
  a.tables_ready = 1;  // the gate/up kernel lets this one launch only after its own wait
  a.out = b.o;
  a.ldo = H;
  a.out_len = (long long)M * k * H;
  a.pairs = M * k;
  a.groups_len = b.groups_cap;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, xnarrow,
                  a);
}

cudaError_t launch_experts_w13(const Ctx& cx, const void* x, const void* W13, int M, int H, int E,
                               int k, int I, const MoeBufs& b, int grid, float* ws, int* ctr) {
  (void)x;
  if (M <= kNarrowRows) return run_experts_w13<kNarrowRows>(cx, W13, M, H, E, k, I, b, grid, ws, ctr);
  return run_experts_w13<kGroupTokens>(cx, W13, M, H, E, k, I, b, grid, ws, ctr);
}

cudaError_t launch_experts_w2(const Ctx& cx, const void* W2, int M, int H, int E, int k, int I,
                              const MoeBufs& b, int grid, float* ws, int* ctr) {
  if (M <= kNarrowRows) return run_experts_w2<kNarrowRows>(cx, W2, M, H, E, k, I, b, grid, ws, ctr);
  return run_experts_w2<kGroupTokens>(cx, W2, M, H, E, k, I, b, grid, ws, ctr);
}

// Shared expert: a dense (ungrouped) pass over every token. Up to 16 tokens
// the weight-streaming kernel, token rows per stage sized to M like the dense
// projections (8 rows for 1-2 tokens, 16 up to 16; mma.sync, as every MoE kernel); from 17
// tokens the gate/up and down projections are dense contractions for the
// tcgen05 tensor cores (the SwiGLU gate/up kernel with both accumulators in
// tensor memory, and the fp32-output projection).
template <int XR>
static cudaError_t run_shared_w13(const Ctx& cx, const void* x, const void* Ws13, int M, int H,
                                  int I, const MoeBufs& b, int grid, float* ws, int* ctr) {
  constexpr int STAGES = 3;  // 64 KB of gate + up weights per stage
  constexpr int SMEM = wstream_smem(XR, STAGES, 0, true);
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<XR, STAGES, EPI_SWIGLU, true, false, false, ROLE_SHARED>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Ws13, (uint64_t)2 * I, (uint64_t)H, kTileRows, true))
    return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, x, (uint64_t)M, (uint64_t)H, XR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = H;
  a.KB = (H + kKChunk - 1) / kKChunk;
  a.TILES = (I + kTileRows - 1) / kTileRows;
  a.nout = I;
  a.M = M;
  a.w_up_offset = I;
  a.out = b.hs;
  a.ldo = I;
  a.out_len = (long long)M * I;
  const long long T = (long long)a.TILES * a.KB;
  if (grid > T) grid = (int)T;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, xmap, a);
}

template <int XR>
static cudaError_t run_shared_w2(const Ctx& cx, const void* Ws2, int M, int H, int I,
                                 const MoeBufs& b, int grid, float* ws, int* ctr) {
  constexpr int STAGES = 6;
  constexpr int SMEM = wstream_smem(XR, STAGES, 0);
  static_assert(SMEM <= kMaxDynSmem, "shared memory");
  auto kern = wstream_kernel<XR, STAGES, EPI_F32, false, false, false, ROLE_SHARED>;
  static DevOnce once;
  if (cudaError_t e = setup_smem(once, kern, SMEM); e != cudaSuccess) return e;
  CUtensorMap wmap, xmap;
  if (!make_tmap(&wmap, Ws2, (uint64_t)H, (uint64_t)I, kTileRows, true)) return cudaErrorInvalidValue;
  if (!make_tmap(&xmap, b.hs, (uint64_t)M, (uint64_t)I, XR, false)) return cudaErrorInvalidValue;
  StreamArgs a = base_args(cx, ws, ctr);
  a.K = I;
  a.KB = (I + kKChunk - 1) / kKChunk;
  a.TILES = (H + kTileRows - 1) / kTileRows;
  a.nout = H;
  a.M = M;
  a.out = b.s;
  a.ldo = H;
  a.out_len = (long long)M * H;
  const long long T = (long long)a.TILES * a.KB;
  if (grid > T) grid = (int)T;
  return launch_k(kern, dim3(grid), dim3(kThreads), SMEM, cx.stream, cx.pdl, wmap, xmap, xmap, a);
}

cudaError_t launch_shared_w13(const Ctx& cx, const void* x, const void* Ws13, int M, int H, int I,
                              const MoeBufs& b, int grid, float* ws, int* ctr) {
  if (M <= 2) return run_shared_w13<8>(cx, x, Ws13, M, H, I, b, grid, ws, ctr);
  if (M <= 16) return run_shared_w13<16>(cx, x, Ws13, M, H, I, b, grid, ws, ctr);
  return launch_swiglu_tc(cx, x, Ws13, b.hs, M, I, H, grid, ws, ctr);
}

cudaError_t launch_shared_w2(const Ctx& cx, const void* Ws2, int M, int H, int I, const MoeBufs& b,
                             int grid, float* ws, int* ctr) {
  if (M <= 2) return run_shared_w2<8>(cx, Ws2, M, H, I, b, grid, ws, ctr);
  if (M <= 16) return run_shared_w2<16>(cx, Ws2, M, H, I, b, grid, ws, ctr);
  return launch_dense_tc_f32(cx, b.hs, Ws2, b.s, M, H, I, grid, ws, ctr);
}

// ------------------------------------------------------------------ combine
// out[m,n] = bf16( res[m,n] + (sum_{j<k} g[m,j] * o[pair(m,j), n] + s[m,n]) ),
// j summed in order 0..k-1, then the shared term, then the residual. Without
// gates (gate == nullptr, k = 1) the sum is o[m, n] itself: the latent
// block's up-projection plus the shared expert and the residual.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o,
                                                      const float* __restrict__ s,
                                                      const float* __restrict__ gate,
                                                      const int* __restrict__ pair_of,
                                                      const uint16_t* res,  // may alias out
                                                      uint16_t* out, int M, int H,
                                                      int k, int* status, long long o_len) {
  griddep_launch_dependents();
  griddep_wait();
  const int per_row = H / 4;
  const long long total = (long long)M * per_row;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < total;
       v += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(v / per_row);
    const int n = (int)(v - (long long)m * per_row) * 4;
    // Eight slots at a time: their gates and pair positions are loaded, then
    // their expert outputs (independent loads, one round trip per batch of
    // eight instead of two per slot), then added in slot order.
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      float g[8];
      int p[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        g[jj] = j < k ? (gate ? gate[m * k + j] : 1.0f) : 0.f;
        p[jj] = j < k ? (gate ? pair_of[m * k + j] : m) : -1;
      }
      float4 ov[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (p[jj] >= 0)
          ov[jj] = *reinterpret_cast<const float4*>(
              DG_AT(status, o, (long long)p[jj] * H + n, o_len - 3));
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (p[jj] >= 0) {
          acc[0] = fmaf(g[jj], ov[jj].x, acc[0]);
          acc[1] = fmaf(g[jj], ov[jj].y, acc[1]);
          acc[2] = fmaf(g[jj], ov[jj].z, acc[2]);
          acc[3] = fmaf(g[jj], ov[jj].w, acc[3]);
        }
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
                  reinterpret_cast<uint16_t*>(out), M, H, k, cx.status, (long long)M * k * H);
}

cudaError_t launch_combine_up(const Ctx& cx, const MoeBufs& b, bool with_shared, const void* res,
                              void* out, int M, int H) {
  const long long total = (long long)M * (H / 4);
  int grid = (int)((total + 255) / 256);
  if (grid > 4 * cx.sms) grid = 4 * cx.sms;
  if (grid < 1) grid = 1;
  return launch_k(combine_kernel, dim3(grid), dim3(256), 0, cx.stream, cx.pdl, (const float*)b.u,
                  (const float*)(with_shared ? b.s : nullptr), (const float*)nullptr,
                  (const int*)nullptr, reinterpret_cast<const uint16_t*>(res),
                  reinterpret_cast<uint16_t*>(out), M, H, 1, cx.status, (long long)M * H);
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
