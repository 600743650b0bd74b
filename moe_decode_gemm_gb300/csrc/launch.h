// launch.h -- host-side launchers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dg {

// Tensor map of a row-major bf16 matrix [rows, cols] read in boxes of
// 64 columns x box_rows rows with 128-byte swizzle. Returns false on failure.
bool make_tmap(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
               bool l2_promote_256, uint64_t ld = 0);

// Rows [N, K] (K % 64 == 0; rows ld elements apart, ld = 0 meaning K, else
// ld % 8 == 0) read in boxes of `rows` rows x `kboxes` 64-wide k blocks (a
// 3-D view), 128-byte swizzle; rows past N read as zeros. Returns false on
// failure.
bool make_tmap_slab(CUtensorMap* map, const void* W, uint64_t N, uint64_t K, uint32_t rows,
                    uint32_t kboxes, uint64_t ld = 0);

struct Ctx {
  int sms;
  long long timeout_ns;
  int* status;
  cudaStream_t stream;
  bool pdl;
  long long ldx = 0;  // dense projections: elements between rows of x (0: K)
  // extents of the split-K workspace given to a launch (floats, ints): the
  // index checks of a DEC_DEBUG build test against them
  long long ws_len = 0, ctr_len = 0;
};

// Dense projection: y = x·Wᵀ (+ res), XR in {8, 16, 64} token rows per stage.
// grid: CTAs to launch (stream-K ranges). ws/ctr: split-K workspace.
// mma: reduce with mma.sync (otherwise CUDA-core dot products, M <= 2 only).
cudaError_t launch_dense(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                         const void* W, const void* res, void* y, int M, int N, int K, int grid,
                         float* ws, int* ctr);

// Same with 256-row output tiles and 64 KB weight stages (xr 8 or 16): for
// matrices large enough that every CTA gets ten or more stages of work.
// Cluster split for narrow projections (xr 8 or 16): cl CTAs per 128-row tile,
// 2 <= cl <= 8 and cl <= ceil(K/128); needs no workspace.
cudaError_t launch_dense_cluster(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                                 const void* W, const void* res, void* y, int M, int N, int K,
                                 int cl);
cudaError_t launch_dense_wide(const Ctx& cx, int xr, bool mma, bool residual, const void* x,
                              const void* W, const void* res, void* y, int M, int N, int K,
                              int grid, float* ws, int* ctr);

// Projection for 1-2 tokens without a split over K: R rows per CTA (R from
// gemv_slab_rows; 0 there means the shape does not suit it).
int gemv_slab_rows(int M, int N, int K, int sms);
cudaError_t launch_gemv_slab(const Ctx& cx, bool residual, const void* x, const void* W,
                             const void* res, void* y, int M, int N, int K, int R);

// The same slabs for up to 16 tokens with mma.sync dot products: R = 16, 32,
// 48 or 64 rows per CTA (R from gemv_mma_rows; 0 means the shape does not
// suit it). addf: optional fp32 [M, N] added to the product before the
// residual, y = bf16(res + (x·Wᵀ + addf)).
int gemv_mma_rows(int M, int N, int K, int sms);
cudaError_t launch_gemv_mma(const Ctx& cx, bool residual, const void* x, const void* W,
                            const void* res, void* y, int M, int N, int K, int R,
                            const float* addf = nullptr);

// tcgen05 projection for 16 <= M <= 64.
cudaError_t launch_dense_tc(const Ctx& cx, bool residual, const void* x, const void* W,
                            const void* res, void* y, int M, int N, int K, int grid, float* ws,
                            int* ctr);
// tcgen05 projection with an fp32 output (no residual), 16 <= M <= 64.
cudaError_t launch_dense_tc_f32(const Ctx& cx, const void* x, const void* W, float* y, int M, int N,
                                int K, int grid, float* ws, int* ctr);
// tcgen05 SwiGLU gate/up: W13 [2I, K] (gate rows, then up rows), h = bf16(silu(x·W1ᵀ) *
// (x·W3ᵀ)) [M, I], 16 <= M <= 64; stream-K over `grid` CTAs.
cudaError_t launch_swiglu_tc(const Ctx& cx, const void* x, const void* W13, void* h, int M, int I,
                             int K, int grid, float* ws, int* ctr);
// Router outputs: fp32 logits [M, E + L], the arrival counter (zero at rest),
// the chosen experts and gates [M, k], optional copies for the caller.
struct RouteOut {
  float* logits;
  int* ctr;
  int* idx;
  float* gate;
  int32_t* idx_user;
  float* w_user;
};
// Router scores and top-k on tcgen05, 16 <= M <= 64: cl CTAs (a cluster) per
// 128-row tile of the E + L rows.
cudaError_t launch_router_tc(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E,
                             int L, int k, int cl, const RouteOut& ro);
// tcgen05 cluster split: cl CTAs per 128-row tile (grid = tiles * cl).
cudaError_t launch_dense_tc_cluster(const Ctx& cx, bool residual, const void* x, const void* W,
                                    const void* res, void* y, int M, int N, int K, int cl);

struct MoeBufs {
  float* logits;   // [M,E]
  int* nact;
  int* grp_exp;    // [E]
  int* grp_off;    // [E+1]
  int* pair_tok;   // [M*k]
  int* pair_of;    // [M*k]
  float* gate;     // [M*k]
  int* topk;       // [M*k] chosen experts
  uint16_t* xs;    // [M*k, H] token rows in expert-sorted pair order
  uint16_t* h;     // [M*k, I]
  float* o;        // [M*k, H]
  uint16_t* hs;    // [M, I]
  float* s;        // [M, H]
  int* route_ctr;  // router clusters arrived (zero at rest)
  uint16_t* z;     // latent block: [M, L] gate-weighted sum of the experts, bf16
  float* u;        // latent block: [M, H] its up-projection, fp32
  int groups_cap;  // entries of grp_exp (grp_off has one more)
};

// Router: CTAs per 128-row tile of experts (one thread-block cluster each),
// at most 8 and at most the number of 128-wide k chunks; and its CTA count.
inline int router_clusters(int H) {
  const int kb = (H + 127) / 128;
  return kb < 8 ? kb : 8;
}
inline int router_ctas(int E, int H) { return (E + 127) / 128 * router_clusters(H); }

// Router scores and, in the same kernel, the top-k experts and gates. With
// L > 0 the weight stacks the E router rows on the latent input projection's
// L rows (one product, [M, E + L] fp32 into b.logits); the top-k ranks the
// first E columns.
cudaError_t launch_router(const Ctx& cx, const void* x, const void* Wr, int M, int H, int E, int k,
                          int32_t* idx_user, float* w_user, const MoeBufs& b, int L = 0);
// Schedule + gather of the token rows (width H, bf16 from x); with L > 0 the
// rows are the latent inputs instead: columns E..E+L-1 of b.logits rounded to
// bf16 (width L).
cudaError_t launch_gather(const Ctx& cx, const void* x, int M, int H, int E, int k,
                          const MoeBufs& b, int L = 0);
// grid: CTAs (the expert kernels split their work statically over them).
cudaError_t launch_experts_w13(const Ctx& cx, const void* x, const void* W13, int M, int H, int E,
                               int k, int I, const MoeBufs& b, int grid, float* ws, int* ctr);
cudaError_t launch_experts_w2(const Ctx& cx, const void* W2, int M, int H, int E, int k, int I,
                              const MoeBufs& b, int grid, float* ws, int* ctr);
// out = bf16(res + (sum_{j<k} g_j o_j + s)) over [M, H] (s when with_shared,
// res nullable); o in expert-sorted pair order.
cudaError_t launch_combine(const Ctx& cx, const MoeBufs& b, bool with_shared, const void* res,
                           void* out, int M, int H, int k);
cudaError_t launch_shared_w13(const Ctx& cx, const void* x, const void* Ws13, int M, int H, int I,
                              const MoeBufs& b, int grid, float* ws, int* ctr);
cudaError_t launch_shared_w2(const Ctx& cx, const void* Ws2, int M, int H, int I,
                             const MoeBufs& b, int grid, float* ws, int* ctr);
// out = bf16(res + (u + s)) over [M, H]: the latent block's last step (s the
// shared expert's output when with_shared, res nullable).
cudaError_t launch_combine_up(const Ctx& cx, const MoeBufs& b, bool with_shared, const void* res,
                              void* out, int M, int H);
// Dense projection with an fp32 output (no residual): stream-K over `grid` CTAs.
cudaError_t launch_dense_f32(const Ctx& cx, int xr, bool mma, const void* x, const void* W,
                             float* y, int M, int N, int K, int grid, float* ws, int* ctr);
cudaError_t launch_add(const Ctx& cx, const void* a, const void* b, void* out, size_t n);
cudaError_t launch_prefetch(const Ctx& cx, const void* ptr, size_t bytes);
cudaError_t launch_selftest_timeout(const Ctx& cx, long long ns);

// Status bits of the allocation-free projection's fixed array on the current
// device, read and cleared (0 if none or never used; -1 if the read failed).
int noalloc_take_status();

// Shared memory each dense/MoE kernel needs (bytes), for cudaFuncSetAttribute.
constexpr int kMaxDynSmem = 232448;
constexpr int kSmemPerSm = 233472;  // per SM; each resident CTA also reserves 1 KB

}  // namespace dg
