/*
 * decgemm.h -- C ABI of a GB300 (sm_103a) library for the weight-bandwidth-
 * bound decode step of a large MoE transformer at batch 1-64.
 *
 * Conventions for every call below
 * --------------------------------
 *  - Pointers named x, W, y, out, ... are DEVICE pointers owned by the caller.
 *    The library never frees or retains them after the call's kernels end.
 *  - bf16 means IEEE bfloat16 (the upper half of a binary32 word). Matrices
 *    are dense row-major: a [R,C] matrix has element (r,c) at r*C + c.
 *  - Activations, weights and outputs must be 16-byte aligned, and every
 *    reduction length (K, H, I) a multiple of 8, because weights and
 *    activations move as 16-byte vectors and TMA tiles.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream. Every call only enqueues work: no host synchronisation, no
 *    device-to-host copy. Results are ready once the stream reaches them.
 *  - Return value: DEC_OK (0) or a negative DEC_E* code. Nothing throws
 *    across this boundary. Argument errors are detected on the host before
 *    any launch. A device-side wait that gives up (see dec_sync_check) is
 *    reported as DEC_ETIMEOUT by dec_sync_check or by the next call.
 *  - The library owns a per-device workspace (split-K partials, arrival
 *    counters, routing tables, MoE intermediates), one side stream for the
 *    shared expert, and events. They are created on first use, grown when a
 *    larger shape arrives, and released by dec_shutdown. Calls that may
 *    allocate must not be the first ones issued inside a CUDA graph capture:
 *    make one call of each shape outside capture first. Calls that share the
 *    workspace must be ordered on one stream (the library orders its own
 *    side stream).
 *
 * Sources. The method is described, in prose only, by web pages on the Kimi
 * K3 specialised decode path for GB300. The ones cited below:
 *   [tune-shapes]  "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1
 *                  "针对工作负载调优形状" (small-matrix kernel at batch 1-2,
 *                  split-K kernel at larger batch).
 *   [moe-overlap]  same page, Part 1 §3 "改进 MoE 调度与重叠" (router,
 *                  routed experts, shared expert on its own stream).
 *   [prefetch]     same page, Part 1 §4 "将即将使用的权重预取到缓存"
 *                  (side-stream kernel that warms the cache with upcoming
 *                  weights).
 *   [trace-path]   same page, Part 2 §1 "隔离变更" (the optimised path must be
 *                  traceable at run time: when it is chosen and how execution
 *                  returns to the standard path).
 */
#ifndef DECGEMM_H
#define DECGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error codes. */
#define DEC_OK            0
#define DEC_EINVAL       -1  /* NULL required pointer, bad size, misaligned pointer, K % 8 != 0 */
#define DEC_EUNSUPPORTED -2  /* outside the decode envelope: M > 64, topk > 32 or > E, E > 1024 */
#define DEC_ECUDA        -3  /* a CUDA runtime call or a launch failed */
#define DEC_ETIMEOUT     -4  /* a bounded device-side wait gave up */
#define DEC_ENOMEM       -5  /* the workspace could not be allocated */
#define DEC_ENODEV       -6  /* no sm_103 device is current */
#define DEC_EBOUNDS      -7  /* a device-side index check failed (DEC_DEBUG builds only) */

/* Kernel regimes reported by dec_last_choice (low 8 bits). */
#define DEC_REGIME_NONE   0
#define DEC_REGIME_SMALLM 1  /* CUDA-core small-matrix kernels, M <= 2 */
#define DEC_REGIME_MMA    2  /* mma.sync: split-K at 3 <= M <= 16, whole-row slabs at M <= 16 */
#define DEC_REGIME_TC     3  /* split-K with tcgen05 tensor cores and TMEM, M >= 17 */

/*
 * dec_linear -- decode projection y = x·Wᵀ. [tune-shapes]
 *
 *   x : [M,K] bf16 activations          W : [N,K] bf16 weights (row n = output n)
 *   y : [M,N] bf16 output               1 <= M <= 64, N >= 1, K >= 8, K % 8 == 0
 *
 * Accumulates in fp32 and rounds once to bf16 (nearest even). The kernel is
 * chosen from M: M <= 2 the small-matrix kernels; 3 <= M <= 16 split-K on
 * mma.sync; M >= 17 split-K on tcgen05 (at exactly 16 tokens mma.sync streams
 * faster). For 1-16 tokens, when K % 64 == 0 and slabs of 16, 32, 48 or 64 whole
 * weight rows per CTA fill between three quarters of the SMs and all of them,
 * no CTA splits K (the sum over K stays inside the CTA; dot products on
 * mma.sync, reported as DEC_REGIME_MMA); for 1-2 tokens where only slabs of 8
 * rows fill the SMs, the same on the CUDA cores; otherwise split-K.
 * Split-K partial sums are reduced in a fixed order (by the last-arriving CTA
 * of each output tile, or -- when N has few 128-row tiles, on every kernel --
 * by the CTAs of one thread-block cluster per tile, in rank order), so the
 * result is identical from run to run. The environment variable
 * DEC_FORCE=smallm|mma|tc overrides the choice (smallm only for M <= 2: the
 * CUDA-core kernels, slabs of 8, 16 or 32 rows included); DEC_FORCE=splitk
 * keeps 1-16 tokens on the split-K kernels.
 * Errors: DEC_EINVAL, DEC_EUNSUPPORTED, DEC_ECUDA, DEC_ENOMEM.
 */
int dec_linear(const void* x, const void* W, void* y, int M, int N, int K, void* stream);

/*
 * dec_linear_residual -- y = bf16(res + x·Wᵀ), the projection with the residual
 * add fused into its epilogue (accumulate in fp32, add res in fp32, round
 * once). res is [M,N] bf16 and may alias y. Same rules as dec_linear.
 */
int dec_linear_residual(const void* x, const void* W, const void* res, void* y,
                        int M, int N, int K, void* stream);

/*
 * dec_linear_ex -- dec_linear with a row stride for x and an optional residual:
 * y = bf16(x·Wᵀ), or bf16(res + x·Wᵀ) when res is not NULL, where row m of x
 * starts ldx elements after row m-1 (ldx >= K, ldx % 8 == 0). A column slice
 * of a wider activation -- the q part of a fused q|kv projection's output,
 * say -- is then read in place. res ([M,N] bf16) may alias y. x must be
 * 16-byte aligned. Errors as dec_linear; DEC_EINVAL also for a bad ldx.
 */
int dec_linear_ex(const void* x, int ldx, const void* W, const void* res, void* y,
                  int M, int N, int K, void* stream);

/*
 * dec_linear_splitk -- dec_linear with the split factor forced to S
 * (1 <= S <= min(256, ceil(K/128))): the grid has S CTAs per 128-row output
 * tile and each takes an equal share of the tile's 128-wide K chunks (shares
 * differ by at most one chunk when S does not divide the chunk count). A test
 * and tuning hook for the split-K regime. [tune-shapes]
 */
int dec_linear_splitk(const void* x, const void* W, void* y, int M, int N, int K,
                      int S, void* stream);

/*
 * moe_decode -- one MoE decode block. [moe-overlap]
 *
 *   x    : [M,H] bf16 token activations, 1 <= M <= 64
 *   Wr   : [E,H] bf16 router weights
 *   W13  : [E,2I,H] bf16; for expert e, rows 0..I-1 are the gate projection W1
 *          and rows I..2I-1 the up projection W3
 *   W2   : [E,H,I] bf16 down projections
 *   Ws13 : [2I,H] bf16 shared-expert gate/up, Ws2 : [H,I] bf16 shared down;
 *          both NULL for a block without a shared expert
 *   out  : [M,H] bf16 output
 *   topk_idx : optional [M,topk] int32 output, topk_w : optional [M,topk] fp32
 *
 * Computes, per token m:
 *   logits = x·Wrᵀ (fp32, not rounded);
 *   idx    = the topk largest logits, ordered by (value desc, index asc);
 *   g_j    = exp(l_j - l_max) / sum_{j' < topk} exp(l_j' - l_max);
 *   h      = silu(x·W1ᵀ) * (x·W3ᵀ) per chosen expert (rounded to bf16);
 *   out    = bf16( sum_{j=0..topk-1} g_j · h_j·W2ᵀ  +  shared(x) ).
 * Only the chosen experts' weights are read: each once per call, or once per
 * group of 32 tokens if more than 32 tokens chose it. Kernels on `stream`:
 * router projection with the top-k (one warp per token, in the router's last
 * cluster), schedule + token gather, expert gate/up with SwiGLU, expert down,
 * combine. The shared expert runs on a library-owned side stream of the
 * lowest priority that waits on `stream` at entry: its kernels take the SMs
 * the router leaves free and stream their weights while routing runs;
 * `stream` joins it before the combine.
 * The number of active experts never returns to the host.
 * Limits: H % 8 == 0, I % 8 == 0, 1 <= topk <= min(E, 32), E <= 1024.
 * Errors: DEC_EINVAL, DEC_EUNSUPPORTED, DEC_ECUDA, DEC_ENOMEM.
 */
int moe_decode(const void* x, const void* Wr, const void* W13, const void* W2,
               const void* Ws13, const void* Ws2, void* out,
               int M, int H, int E, int topk, int I,
               int32_t* topk_idx, float* topk_w, void* stream);

/*
 * moe_decode_residual -- moe_decode whose combine adds a residual:
 * out = bf16(res + sum_j g_j·o_j + shared). res is [M,H] bf16 and may alias x
 * or out (the residual stream of a decode layer is usually the block's own
 * input). out may alias x: x is last read before the combine starts.
 */
int moe_decode_residual(const void* x, const void* Wr, const void* W13, const void* W2,
                        const void* Ws13, const void* Ws2, const void* res, void* out,
                        int M, int H, int E, int topk, int I,
                        int32_t* topk_idx, float* topk_w, void* stream);

/*
 * moe_decode_latent -- an MoE decode block whose routed experts work on a
 * latent width L. [moe-overlap] The router scores and the latent input
 * projection are computed as one product over a stacked weight (the pages
 * merge the two into one matrix multiplication); the steps after it are the
 * library's reading of the block, the pages naming only that product:
 *
 *   x    : [M,H] bf16               Wrl : [E+L,H] bf16, rows 0..E-1 the router,
 *                                         rows E..E+L-1 the latent input projection
 *   W13  : [E,2I,L] bf16 (gate rows 0..I-1, up rows I..2I-1)   W2 : [E,L,I] bf16
 *   Wup  : [H,L] bf16 up-projection     Ws13 [2I,H] / Ws2 [H,I]: shared expert on x
 *   res  : optional [M,H] bf16 residual (may alias x or out)   out : [M,H] bf16
 *
 *   sc     = x·Wrlᵀ (fp32);  logits = sc[:, :E];  lat = bf16(sc[:, E:])
 *   idx, g = top-k of logits, renormalised softmax gates (as moe_decode)
 *   z      = bf16( sum_{j=0..topk-1} g_j · expert_{idx_j}(lat) )   (width L)
 *   out    = bf16( res + (z·Wupᵀ + shared(x)) )   (fp32 sum, one rounding)
 *
 * Kernels on `stream`: the router over E+L rows with the top-k, schedule +
 * gather of the latent rows (rounded to bf16 as they are copied), expert
 * gate/up, expert down, the gate-weighted sum z, the up-projection, and the
 * final sum; the shared expert on the library's side stream as in
 * moe_decode. Limits as moe_decode; L >= 8, L % 8 == 0.
 * Errors: DEC_EINVAL, DEC_EUNSUPPORTED, DEC_ECUDA, DEC_ENOMEM.
 */
int moe_decode_latent(const void* x, const void* Wrl, const void* W13, const void* W2,
                      const void* Wup, const void* Ws13, const void* Ws2, const void* res,
                      void* out, int M, int H, int L, int E, int topk, int I,
                      int32_t* topk_idx, float* topk_w, void* stream);

/*
 * l2_prefetch -- enqueue a light kernel on `stream` that pulls
 * [ptr, ptr + bytes) into L2, so that a later kernel reading the range hits
 * in cache. [prefetch] It has no data dependency and changes no memory;
 * ordering against other streams is the caller's. bytes is rounded down to a
 * multiple of 16 and capped at half the L2 size. ptr must be 16-byte aligned.
 */
int l2_prefetch(const void* ptr, size_t bytes, void* stream);

/*
 * dec_add -- out = bf16(a + b) elementwise over n bf16 values (the residual
 * add of a decode layer when it is not fused). out may alias a or b.
 */
int dec_add(const void* a, const void* b, void* out, size_t n, void* stream);

/*
 * dec_last_choice -- regime and split of this thread's last dec_linear* call.
 * [trace-path] Returns regime | (S << 8) | (C << 16) | (Wd << 17) | (Sl << 18)
 * where regime
 * is a DEC_REGIME_* value, S the number of CTAs that share each output tile's
 * K range (1 = none), rounded up, C is 1 when those S CTAs form one
 * thread-block cluster and sum their partial tiles through distributed shared
 * memory (small projections: few 128-row tiles, M <= 16), 0 when the split is
 * the stream-K one with a last-arriver fixup, and Wd is 1 when the output
 * tiles are 256 rows high (large projections at M <= 16), and Sl is 1 when
 * each CTA owned whole weight rows (1-16 tokens, S = 1). DEC_REGIME_NONE before
 * any call.
 */
int dec_last_choice(void);

/* dec_last_grid -- CTAs launched by this thread's last dec_linear* call. */
int dec_last_grid(void);

/* dec_strerror -- static text for a DEC_* code. */
const char* dec_strerror(int code);

/*
 * dec_sync_check -- synchronise `stream` (and the library's side stream),
 * then read and clear the device status words that kernels set when a bounded
 * wait gives up: the library's own and the one in dec_linear_noalloc's fixed
 * array. Returns DEC_OK, DEC_ETIMEOUT, or DEC_ECUDA if the synchronisation
 * itself failed. Allocates nothing: in a process that has only called
 * dec_linear_noalloc it sets up no workspace, stream or event.
 */
int dec_sync_check(void* stream);

/*
 * dec_set_wait_timeout_ns -- upper bound, in nanoseconds of %globaltimer, on
 * every device-side wait of later launches (default 2e9). A wait that runs
 * out sets the status word, drains its own copies in flight and returns.
 * Returns the previous value.
 */
long long dec_set_wait_timeout_ns(long long ns);

/*
 * dec_selftest_timeout -- launch one CTA that waits, with the bounded wait
 * used by every kernel, on a barrier that nothing will complete, with limit
 * `ns`. The wait must give up; dec_sync_check then returns DEC_ETIMEOUT.
 * Exercises failure detection without faulting or hanging the GPU.
 */
int dec_selftest_timeout(long long ns, void* stream);

/*
 * dec_debug_build -- 1 for the index-checking build of this library
 * (libdecgemm_debug.so, compiled with DEC_DEBUG), 0 otherwise. In that build
 * every index a kernel computes into a global buffer (output rows and
 * columns, split-K slots and counters, expert group tables, pair positions,
 * gathered token rows) is checked against the buffer's extent; an access out
 * of range is skipped, and dec_sync_check returns DEC_EBOUNDS.
 * dec_debug_check_site -- the source line of the first failed check and the
 * offending index, as read by the dec_sync_check that returned DEC_EBOUNDS;
 * returns 1 if there was one, 0 if not.
 */
int dec_debug_build(void);
int dec_debug_check_site(int* line, long long* index);

/* dec_launch_count -- kernels launched by this library since load (all threads). */
long long dec_launch_count(void);

/*
 * dec_probe_begin / dec_probe_end -- time every launch of one kernel kind with
 * CUDA events recorded on the stream the kernel is launched on.
 * kind: 0 = routed-expert gate/up kernel, 1 = routed-expert down kernel,
 *       2 = projection kernels, 3 = router projection kernel, 4 = combine kernel.
 * dec_probe_begin arms the probe for up to `capacity` launches (0 disarms).
 * dec_probe_end synchronises those events and returns, through the
 * pointers, the summed duration in ms and the number of launches timed.
 */
int dec_probe_begin(int kind, int capacity);
int dec_probe_end(double* total_ms, int* launches);

/*
 * dec_linear_noalloc -- dec_linear for callers that must not allocate device
 * memory. The pages describe no counterpart: this entry point exists for
 * integration, not for the method.
 *
 * Who needs it: code whose device memory is owned by someone else (a
 * framework's caching allocator that has reserved the GPU, an engine with a
 * memory budget fixed before the first request) and latency-critical loops
 * in which cudaMalloc/cudaFree, which may synchronise the device, must never
 * run. dec_linear allocates its split-K workspace on first use and grows it
 * for larger shapes; this variant allocates nothing and calls no allocating
 * routine.
 *
 * Same arguments, layouts and result as dec_linear (fp32 accumulation, one
 * bf16 rounding), computed by the same weight-streaming kernel: CUDA-core for
 * M <= 2, mma.sync for 3 <= M <= 16. Its split-K partial sums and arrival
 * counters live in one 4 MiB array compiled into the library; every GPU that
 * loads the library holds that array until the process exits.
 *
 * Limits (DEC_EUNSUPPORTED beyond them): M <= 16; ceil(N/128) <= 16384 output
 * tiles; the partial tiles of the launch, min(SMs, ceil(N/128)*ceil(K/128))
 * CTAs x 2 x 128 x (8 if M <= 2 else 16) floats, within 4 MiB - 64 KiB - 256 B
 * (a 152-SM GB300 needs at most 2.4 MiB, so every N and K fit there).
 * Argument errors as for dec_linear (DEC_EINVAL); DEC_ENODEV without an sm_103
 * device; DEC_ECUDA if a runtime call fails.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. Every call shares the one array, which keeps the
 * last call's contents (each call clears the counters it uses): calls that can
 * overlap on the GPU -- on unordered streams or from several host threads --
 * race and corrupt each other's results. A bounded device-side wait that
 * gives up ends the kernel as in dec_linear (y is then incomplete) and sets a
 * status word in the fixed array; the word is not cleared by later calls, and
 * dec_sync_check reports it as DEC_ETIMEOUT (and clears it) -- call it before
 * trusting y where a give-up must not pass unseen. A first call made while
 * `stream` is being captured returns DEC_EINVAL (the set-up above cannot run
 * inside a capture). Does not update dec_last_choice or dec_launch_count.
 */
int dec_linear_noalloc(const void* x, const void* W, void* y, int M, int N, int K, void* stream);

/* dec_shutdown -- free the workspace, side stream and events of the current device. */
void dec_shutdown(void);

/* dec_version -- ABI version of this header (major*100 + minor). */
int dec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DECGEMM_H */
