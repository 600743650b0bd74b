// api.cu -- the C ABI: argument validation, kernel-regime selection, the
// per-device workspace, the shared-expert side stream, launch accounting and
// the timing probe. Everything here runs on the host; every step of the
// decode path runs in the kernels of k_linear.cu, k_tc.cu and k_moe.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/decgemm.h"
#include "launch.h"

namespace dg {

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

bool make_tmap(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
               bool l2_promote_256, uint64_t ld) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(ld ? ld : cols) * 2};  // bytes between rows
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        l2_promote_256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Weight rows [N, K] (K % 64 == 0) as a 3-D tensor: element (x, n, j) is
// W[n][64 j + x]. A box of `rows` rows and `kboxes` 64-wide k blocks lands in
// shared memory as kboxes x rows lines of 128 bytes (128-byte swizzle), one
// TMA instruction for what would take `kboxes` 2-D boxes.
bool make_tmap_slab(CUtensorMap* map, const void* W, uint64_t N, uint64_t K, uint32_t rows,
                    uint32_t kboxes, uint64_t ld) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode || N == 0 || K == 0 || (K % 64) != 0) return false;
  if (ld == 0) ld = K;
  if (ld < K || (ld % 8) != 0) return false;
  cuuint64_t dims[3] = {64, N, K / 64};
  cuuint64_t strides[2] = {ld * 2, 128};  // bytes: next row, next 64-wide k block
  cuuint32_t box[3] = {64, rows, kboxes};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ device state
struct Buf {
  void* p = nullptr;
  size_t bytes = 0;
};

struct DevState {
  bool init = false;
  int sms = 0;
  int l2 = 0;
  int cc_major = 0, cc_minor = 0;
  cudaStream_t side = nullptr;            // shared expert
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  int* status = nullptr;                  // device status word
  Buf ws_main, ctr_main, ws_side, ctr_side;
  Buf moe;                                // routing tables + intermediates
  int moe_M = 0, moe_E = 0, moe_k = 0, moe_I = 0, moe_H = 0, moe_L = 0;
  MoeBufs mb = {};
};

static std::mutex g_mu;
static std::vector<DevState> g_dev;
static std::atomic<long long> g_launches{0};
static long long g_timeout_ns = 2000000000LL;
static thread_local int t_last_choice = DEC_REGIME_NONE;
static thread_local int t_last_grid = 0;

// timing probe
static std::mutex g_probe_mu;
static int g_probe_kind = -1;
static int g_probe_cap = 0;
static std::vector<cudaEvent_t> g_probe_ev;  // start/end pairs
static int g_probe_n = 0;

static int to_err(cudaError_t e) { return e == cudaSuccess ? DEC_OK : DEC_ECUDA; }

// The status word's bit for a failed index check (the device-side
// kStatusBounds of the kernels).
constexpr int kStatusBoundsBit = 2;

static int get_dev(DevState** out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return DEC_ENODEV;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_dev.size() <= d) g_dev.resize(d + 1);
  DevState& s = g_dev[d];
  if (!s.init) {
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, d) != cudaSuccess) return DEC_ENODEV;
    if (p.major != 10 || p.minor != 3) return DEC_ENODEV;  // the library is built for sm_103a
    s.sms = p.multiProcessorCount;
    s.l2 = p.l2CacheSize;
    s.cc_major = p.major;
    s.cc_minor = p.minor;
    // The shared expert's stream has the lowest priority: a CTA of the
    // routed path (router -> top-k -> gather -> experts) never waits behind
    // one of its CTAs for an SM. (A pending CTA of a higher-priority stream
    // also holds back the dispatch of every lower-priority launch.)
    int lo = 0, hi = 0;
    cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (cudaStreamCreateWithPriority(&s.side, cudaStreamNonBlocking, lo) != cudaSuccess)
      return DEC_ECUDA;
    if (cudaEventCreateWithFlags(&s.ev_fork, cudaEventDisableTiming) != cudaSuccess) return DEC_ECUDA;
    if (cudaEventCreateWithFlags(&s.ev_join, cudaEventDisableTiming) != cudaSuccess) return DEC_ECUDA;
    if (cudaMalloc(&s.status, 256) != cudaSuccess) return DEC_ENOMEM;
    if (cudaMemset(s.status, 0, 256) != cudaSuccess) return DEC_ECUDA;
    s.init = true;
  }
  *out = &s;
  return DEC_OK;
}

// Grow a zero-initialised device buffer. Growing synchronises the device.
static int ensure(Buf& b, size_t bytes, cudaStream_t st) {
  if (b.bytes >= bytes) return DEC_OK;
  if (b.p) {
    cudaDeviceSynchronize();
    cudaFree(b.p);
    b.p = nullptr;
    b.bytes = 0;
  }
  size_t want = bytes + bytes / 4;
  if (cudaMalloc(&b.p, want) != cudaSuccess) return DEC_ENOMEM;
  if (cudaMemsetAsync(b.p, 0, want, st) != cudaSuccess) return DEC_ECUDA;
  b.bytes = want;
  return DEC_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static Ctx make_ctx(DevState* s, cudaStream_t st) {
  Ctx c;
  c.sms = s->sms;
  c.timeout_ns = g_timeout_ns;
  c.status = s->status;
  c.stream = st;
  c.pdl = true;
  return c;
}

// Probe: time launches of one kind with events on their stream.
struct ProbeScope {
  bool on = false;
  cudaStream_t st;
  int slot = -1;
  ProbeScope(int kind, cudaStream_t s) : st(s) {
    std::lock_guard<std::mutex> lk(g_probe_mu);
    if (kind == g_probe_kind && g_probe_n < g_probe_cap) {
      slot = g_probe_n++;
      on = true;
      cudaEventRecord(g_probe_ev[2 * slot], st);
    }
  }
  ~ProbeScope() {
    if (on) cudaEventRecord(g_probe_ev[2 * slot + 1], st);
  }
};

static int counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return to_err(e);
}

// ------------------------------------------------------------------ projections
static bool forced(const char* what) {
  const char* f = std::getenv("DEC_FORCE");
  return f && !std::strcmp(f, what);
}

static bool force_splitk() { return forced("splitk"); }


static int regime_for(int M) {
  const char* f = std::getenv("DEC_FORCE");
  if (f) {
    if (!std::strcmp(f, "smallm") && M <= 2) return DEC_REGIME_SMALLM;
    if (!std::strcmp(f, "mma")) return DEC_REGIME_MMA;
    if (!std::strcmp(f, "tc") && M >= 16) return DEC_REGIME_TC;
  }
  // tcgen05 from 17 tokens: at exactly 16 the mma.sync kernel with 16 token
  // rows per stage streams faster on GB300 (N = 2048 / 8192 / 16384, K = 7168:
  // 9.7 / 22.9 / 37.2 us against 12.7 / 24.2 / 42.4 us); from 24 tokens the
  // tensor-memory kernel wins (13.0 against 20.5 us at N = 2048).
  if (M <= 2) return DEC_REGIME_SMALLM;
  if (M <= 16) return DEC_REGIME_MMA;
  return DEC_REGIME_TC;
}

// Weight bytes one CTA of the CUDA-core / mma.sync cluster split may stream.
// Measured (us, stream-K over every SM -> cluster split): 2048 x 16384 at
// M = 1 / 4 / 8 / 16: 16.0 / 17.4 / 17.5 / 18.4 -> 14.4 / 15.7 / 15.9 / 17.2
// (512 KB per CTA); 4096 x 7168 at M = 1 / 8: 13.2 / 15.0 -> 12.8 / 14.0
// (448 KB).
constexpr long long kClusterMaxBytes = 1024LL * 1024;

// Weight bytes one CTA of the tcgen05 cluster split may stream. Measured (us,
// tile-aligned stream-K split -> cluster split, 8 CTAs per tile): 2048 x 7168
// at M = 64 / 32 / 17: 14.1 / 11.2 / 10.6 -> 11.4 / 9.6 / 9.2 (224 KB per
// CTA); 2048 x 16384 at M = 64 / 32: 19.9 / 16.9 -> 18.7 / 16.9 (512 KB).
constexpr long long kTcClusterMaxBytes = 1024LL * 1024;

static int linear_impl(const void* x, const void* W, const void* res, void* y, int M, int N, int K,
                       int S, void* stream, long long ldx = 0) {
  if (!x || !W || !y) return DEC_EINVAL;
  if (M < 1 || N < 1 || K < 8 || (K % 8) != 0) return DEC_EINVAL;
  if (ldx != 0 && (ldx < K || (ldx % 8) != 0)) return DEC_EINVAL;
  if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (res && !aligned16(res))) return DEC_EINVAL;
  if (M > 64) return DEC_EUNSUPPORTED;
  const int KB = (K + 127) / 128;  // 128-wide k chunks (one pipeline stage each)
  if (S != 0 && (S < 1 || S > KB || S > 256)) return DEC_EINVAL;
  DevState* s = nullptr;
  int rc = get_dev(&s);
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int regime = regime_for(M);
  // Whole-row slabs (R weight rows per CTA, no split over K) when such slabs
  // fill between three quarters of the SMs and all of them: up to 16 tokens
  // on the tensor cores (16, 32, 48 or 64 rows per CTA), 1-2 tokens on the CUDA cores
  // where only 8 rows per CTA fill the SMs (or under DEC_FORCE=smallm).
  // Same-GPU A/B, us per call in a CUDA graph, split-K -> slab: N x K =
  // 2048 x 7168 at M = 1 / 2 / 4 / 5 / 8 / 12 / 16: 8.0 / 8.3 / 8.7 / 8.7 /
  // 8.9 / 9.3 / 9.5 -> 6.4 / 6.4 / 6.4 / 7.0 / 6.9 / 8.8 / 8.9; 2048 x 16384
  // at M = 8: 16.6 -> 14.0; 4096 x 4096 at M = 1 / 8: 8.6 / 9.6 -> 7.2 / 7.4;
  // 4096 x 7168 at M = 8 / 16: 14.6 / 15.9 -> 11.6 / 14.4 (the CUDA-core
  // slabs: 6.8 / 7.8 at M = 1 / 2 of 2048 x 7168); 48-row slabs: 7168 x 7168
  // at M = 1 / 16: 18.6 / 20.8 -> 17.1 / 18.2; 64-row slabs: 8192 x 7168 at
  // M = 1 / 8 / 16: 20.4 / 21.5 / 22.4 -> 18.9 / 19.4 / 21.3, 8192 x 4096 at
  // M = 4: 16.7 -> 12.2. DEC_FORCE=splitk keeps the split-K kernels.
  if (S == 0 && !force_splitk()) {
    const bool core_only = forced("smallm");
    const int Rm = (regime != DEC_REGIME_TC && !core_only) ? gemv_mma_rows(M, N, K, s->sms) : 0;
    const int Rc = (!Rm && regime == DEC_REGIME_SMALLM) ? gemv_slab_rows(M, N, K, s->sms) : 0;
    if (Rm || Rc) {
      Ctx cx = make_ctx(s, st);
      cx.ldx = ldx;
      const int R = Rm ? Rm : Rc;
      t_last_choice = (Rm ? DEC_REGIME_MMA : DEC_REGIME_SMALLM) | (1 << 8) | (1 << 18);
      t_last_grid = (N + R - 1) / R;
      ProbeScope probe(2, st);
      return counted(Rm ? launch_gemv_mma(cx, res != nullptr, x, W, res, y, M, N, K, Rm)
                        : launch_gemv_slab(cx, res != nullptr, x, W, res, y, M, N, K, Rc));
    }
  }
  // token rows per stage of the CUDA-core / mma.sync kernel; the tcgen05
  // kernel's partial tiles always hold 64 token columns
  const int xr = regime == DEC_REGIME_TC ? 64 : regime == DEC_REGIME_SMALLM ? 8 : (M <= 16 ? 16 : 64);
  // 256-row tiles with 64 KB stages stream faster; they are used when every
  // CTA still gets ten or more stages of work (so the split stays balanced).
  const long long wide_units = ((N + 255) / 256) * (long long)KB;
  const bool wide = S == 0 && regime != DEC_REGIME_TC && xr <= 16 && wide_units >= 10LL * s->sms;
  const long long tiles = wide ? (N + 255) / 256 : (N + 127) / 128;
  const long long T = tiles * KB;
  // Cluster split for narrow projections: cl CTAs per 128-row tile (a
  // thread-block cluster), the largest portable size (<= 8) with
  // tiles * cl <= SMs and cl <= KB. Used when it keeps at least three quarters
  // of the SMs busy and each CTA streams at most kClusterMaxBytes of weights.
  // No split-K workspace, counters or atomics.
  int cl = 0;
  if (S == 0 && regime != DEC_REGIME_TC && !wide && xr <= 16) {
    for (int c = 8; c >= 2; c >>= 1)
      if (tiles * c <= s->sms && c <= KB) {
        cl = c;
        break;
      }
    if (cl && (tiles * cl * 4 < 3LL * s->sms || 256LL * K / cl > kClusterMaxBytes)) cl = 0;
  }
  // The same split for the tcgen05 kernel (17-64 tokens), whose stream-K
  // fixups sum partial tiles of 32 KB per contributor at 64 tokens, but only
  // with 8 ranks per tile: with 2-4 partials per tile the tile-aligned split
  // below sums them cheaply and its 4-stage ring streams a large share faster
  // than the cluster kernel's 2-stage one (M = 64, us, cluster -> aligned:
  // 4096 x 7168 17.8 -> 16.2 at 4 ranks, 8192 x 7168 31.9 -> 24.9 at 2; with
  // the cluster kernel's current stages and reduction, M = 32 / 64: 4096 x
  // 7168 at 4 ranks 15.2 / 17.0 against 14.9 / 17.4, at 2 ranks 7168 x 7168
  // 25.8 / 28.9 against 21.6 / 24.4, 8192 x 7168 29.9 against 26.1).
  if (S == 0 && regime == DEC_REGIME_TC && tiles * 8 <= s->sms && KB >= 8 &&
      tiles * 8 * 4 >= 3LL * s->sms && 256LL * K / 8 <= kTcClusterMaxBytes)
    cl = 8;
  if (cl) {
    Ctx cx = make_ctx(s, st);
    cx.ldx = ldx;
    t_last_choice = regime | (cl << 8) | (1 << 16);
    t_last_grid = (int)(tiles * cl);
    ProbeScope probe(2, st);
    if (regime == DEC_REGIME_TC)
      return counted(launch_dense_tc_cluster(cx, res != nullptr, x, W, res, y, M, N, K, cl));
    return counted(launch_dense_cluster(cx, xr, regime != DEC_REGIME_SMALLM, res != nullptr, x, W,
                                        res, y, M, N, K, cl));
  }
  long long grid = S ? tiles * S : (T < s->sms ? T : s->sms);
  // tcgen05: a tile-aligned split -- tiles * sa CTAs, sa dividing the k chunks,
  // so that every CTA covers whole k ranges of one tile -- when it keeps at
  // least three quarters of the SMs busy. Its fixups sum sa equal partials
  // (none at sa = 1) instead of the uneven ones of a split over every SM,
  // each partial 32 KB at 64 token columns. Measured, us (stream-K over 152
  // SMs -> aligned): M = 64, N x K = 2048 x 7168: 15.9 -> 14.0 (sa = 8);
  // 2048 x 16384: 21.0 -> 20.0 (8); 16384 x 7168: 42.4 -> 38.6 (1). At
  // 7168 x 7168 the only aligned split (2) leaves a quarter of the SMs idle
  // and is slower (23.1 against 22.2).
  if (S == 0 && regime == DEC_REGIME_TC) {
    for (long long sa = KB < 16 ? KB : 16; sa >= 1; --sa)
      if (tiles * sa <= s->sms && KB % sa == 0) {
        if (tiles * sa * 4 >= 3LL * s->sms) grid = tiles * sa;
        break;
      }
  }
  if (grid > T) grid = T;
  const size_t slot_rows = wide ? 256 : 128;
  if ((rc = ensure(s->ws_main, (size_t)grid * 2 * slot_rows * xr * sizeof(float), st))) return rc;
  if ((rc = ensure(s->ctr_main, (size_t)tiles * sizeof(int), st))) return rc;
  Ctx cx = make_ctx(s, st);
  cx.ldx = ldx;
  cx.ws_len = (long long)(s->ws_main.bytes / sizeof(float));
  cx.ctr_len = (long long)(s->ctr_main.bytes / sizeof(int));
  long long seff = (KB * grid + T - 1) / T;
  if (seff < 1) seff = 1;
  t_last_choice = regime | ((int)seff << 8) | ((wide ? 1 : 0) << 17);
  t_last_grid = (int)grid;
  ProbeScope probe(2, st);
  if (regime == DEC_REGIME_TC)
    return counted(launch_dense_tc(cx, res != nullptr, x, W, res, y, M, N, K, (int)grid,
                                   (float*)s->ws_main.p, (int*)s->ctr_main.p));
  if (wide)
    return counted(launch_dense_wide(cx, xr, regime != DEC_REGIME_SMALLM, res != nullptr, x, W,
                                     res, y, M, N, K, (int)grid, (float*)s->ws_main.p,
                                     (int*)s->ctr_main.p));
  return counted(launch_dense(cx, xr, regime != DEC_REGIME_SMALLM, res != nullptr, x, W, res, y,
                              M, N, K, (int)grid,
                              (float*)s->ws_main.p, (int*)s->ctr_main.p));
}

// ------------------------------------------------------------------ MoE
// L: the latent width of a latent block (0 for the plain block).
static int moe_bufs(DevState* s, int M, int H, int E, int k, int I, int L, cudaStream_t st) {
  if (M <= s->moe_M && H <= s->moe_H && E <= s->moe_E && k <= s->moe_k && I <= s->moe_I &&
      L <= s->moe_L)
    return DEC_OK;
  const int Mx = 64;  // sized for the whole decode envelope at once
  const int Ex = E > s->moe_E ? E : s->moe_E;
  const int kx = k > s->moe_k ? k : s->moe_k;
  const int Ix = I > s->moe_I ? I : s->moe_I;
  const int Hx = H > s->moe_H ? H : s->moe_H;
  const int Lx = L > s->moe_L ? L : s->moe_L;
  const int Wx = Hx > Lx ? Hx : Lx;  // expert model width: H, or L in a latent block
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  size_t off = 0;
  size_t o_logits = off; off += al((size_t)Mx * (Ex + Lx) * 4);
  size_t o_nact = off; off += al(4);
  // expert groups: at most one per expert plus one per 16 (token, slot) pairs
  // (a bound for groups of 16 or more tokens)
  const size_t Gx = (size_t)Ex + ((size_t)Mx * kx + 15) / 16;
  size_t o_gexp = off; off += al(Gx * 4);
  size_t o_goff = off; off += al((Gx + 1) * 4);
  size_t o_ptok = off; off += al((size_t)Mx * kx * 4);
  size_t o_pof = off; off += al((size_t)Mx * kx * 4);
  size_t o_gate = off; off += al((size_t)Mx * kx * 4);
  size_t o_topk = off; off += al((size_t)Mx * kx * 4);
  size_t o_xs = off; off += al((size_t)Mx * kx * Wx * 2);
  size_t o_h = off; off += al((size_t)Mx * kx * Ix * 2);
  size_t o_o = off; off += al((size_t)Mx * kx * Wx * 4);
  size_t o_hs = off; off += al((size_t)Mx * Ix * 2);
  size_t o_s = off; off += al((size_t)Mx * Hx * 4);
  size_t o_rctr = off; off += al(4);
  size_t o_z = off; off += al((size_t)Mx * (Lx > 0 ? Lx : 1) * 2);
  size_t o_u = off; off += al((size_t)Mx * Hx * 4);
  int rc = ensure(s->moe, off, st);
  if (rc) return rc;
  // The layout has changed even when the buffer did not have to grow (its
  // slack held the larger shapes): the arrival counters that must be zero at
  // rest now sit on bytes of the old layout. Clear it, on the stream that
  // orders every earlier use of the buffer.
  if (cudaMemsetAsync(s->moe.p, 0, off, st) != cudaSuccess) return DEC_ECUDA;
  uint8_t* b = (uint8_t*)s->moe.p;
  s->mb.logits = (float*)(b + o_logits);
  s->mb.nact = (int*)(b + o_nact);
  s->mb.grp_exp = (int*)(b + o_gexp);
  s->mb.grp_off = (int*)(b + o_goff);
  s->mb.pair_tok = (int*)(b + o_ptok);
  s->mb.pair_of = (int*)(b + o_pof);
  s->mb.gate = (float*)(b + o_gate);
  s->mb.topk = (int*)(b + o_topk);
  s->mb.xs = (uint16_t*)(b + o_xs);
  s->mb.h = (uint16_t*)(b + o_h);
  s->mb.o = (float*)(b + o_o);
  s->mb.hs = (uint16_t*)(b + o_hs);
  s->mb.s = (float*)(b + o_s);
  s->mb.route_ctr = (int*)(b + o_rctr);
  s->mb.z = (uint16_t*)(b + o_z);
  s->mb.u = (float*)(b + o_u);
  s->mb.groups_cap = (int)Gx;
  s->moe_M = Mx;
  s->moe_L = Lx;
  s->moe_E = Ex;
  s->moe_k = kx;
  s->moe_I = Ix;
  s->moe_H = Hx;
  return DEC_OK;
}

// The MoE block; with L > 0 the latent block: Wr stacks the E router rows on
// the latent input projection's L rows, the experts work on width L, and Wup
// [H, L] projects their gate-weighted sum back to the hidden width.
static int moe_impl(const void* x, const void* Wr, const void* W13, const void* W2, const void* Ws13,
                    const void* Ws2, const void* res, void* out, int M, int H, int E, int topk,
                    int I, int32_t* topk_idx, float* topk_w, void* stream, int L = 0,
                    const void* Wup = nullptr) {
  if (!x || !Wr || !W13 || !W2 || !out) return DEC_EINVAL;
  if ((Ws13 == nullptr) != (Ws2 == nullptr)) return DEC_EINVAL;
  if (M < 1 || H < 8 || E < 1 || topk < 1 || I < 8 || (H % 8) || (I % 8)) return DEC_EINVAL;
  if (L < 0 || (L > 0 && (L < 8 || (L % 8) || !Wup))) return DEC_EINVAL;
  const void* ptrs[] = {x, Wr, W13, W2, Ws13, Ws2, res, out, topk_idx, topk_w, Wup};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DEC_EINVAL;
  if (M > 64 || E > 1024 || topk > 32 || topk > E) return DEC_EUNSUPPORTED;
  DevState* s = nullptr;
  int rc = get_dev(&s);
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = moe_bufs(s, M, H, E, topk, I, L, st))) return rc;
  const int Wd = L > 0 ? L : H;  // the experts' model width
  // partial slots: 2 per CTA, up to 256 rows (gate + up halves) x 64 tokens
  const size_t ws_bytes = (size_t)s->sms * 2 * 256 * 64 * sizeof(float);
  const int tiles13 = (I + 127) / 128, tiles2 = ((Wd > H ? Wd : H) + 127) / 128;
  int maxt = tiles13 > tiles2 ? tiles13 : tiles2;
  // an expert chosen by more tokens than a group holds forms several groups:
  // at most E + M*topk/16 groups, each with its own tile counters
  const int max_groups = E + (M * topk + 15) / 16;
  const size_t ctr_bytes = (size_t)(max_groups * (size_t)maxt + 64) * sizeof(int);
  if ((rc = ensure(s->ws_main, ws_bytes, st))) return rc;
  if ((rc = ensure(s->ctr_main, ctr_bytes, st))) return rc;
  const bool shared = Ws13 != nullptr;
  if (shared) {
    if ((rc = ensure(s->ws_side, ws_bytes, st))) return rc;
    if ((rc = ensure(s->ctr_side, (size_t)(maxt + 64) * sizeof(int), st))) return rc;
  }
  Ctx cx = make_ctx(s, st);
  cx.ws_len = (long long)(s->ws_main.bytes / sizeof(float));
  cx.ctr_len = (long long)(s->ctr_main.bytes / sizeof(int));
  float* ws = (float*)s->ws_main.p;
  int* ctr = (int*)s->ctr_main.p;
  // Shared expert, forked first to the side stream (lowest priority), one CTA
  // on each SM the router leaves free, so its weights stream while the
  // latency-bound router, top-k and gather run on the other SMs. Its down
  // projection is launched without the early-start dependency, so its CTAs do
  // not take SMs early and sit waiting for the gate/up kernel. The routed
  // experts take the SMs as the shared expert's CTAs leave them; the streams
  // join before the combine.
  //
  // Small batches: the routed experts read few bytes, and the shared expert,
  // packed into the routing window, then delays the routed gate/up kernel's
  // start on most SMs and leaves its down projection as a tail. There it gets
  // gd dedicated SMs for the whole block instead -- its share of the block's
  // bytes, from the expected number of distinct experts under uniform routing
  // and a routed expert's bytes per shared-expert byte (Wd / H: the latent
  // block's experts are narrower) -- and the routed experts the others. Used
  // when few experts are expected (eu <= 32: M <= 4 at E = 384, k = 8) and
  // 4 <= gd < SMs / 2. Same-GPU A/B of the latent block (L = 512), us at
  // M = 1 / 2 / 4 / 8 / 16 / 64, the share without the Wd / H weight ->
  // with it: 81.5 / 150.6 / 247.6 / 103.7 / 152.7 / 344.4 -> 56.4 / 66.7 /
  // 78.5 / 106.9 / 157.3 / 382.8 (dedicated SMs from 8 tokens on lose: hence
  // the bound on eu).
  const double eu = E * (1.0 - std::pow(1.0 - (double)topk / E, (double)M));
  const int gd = (int)(s->sms / (1.0 + eu * Wd / H) + 0.5);
  const bool dedicated = shared && eu <= 32.0 && gd >= 4 && gd < s->sms / 2;
  const int egrid = dedicated ? s->sms - gd : s->sms;
  if (shared) {
    const int rc_ctas = router_ctas(E + L, H);
    const int sgrid = dedicated ? gd : (s->sms - rc_ctas > 0 ? s->sms - rc_ctas : 1);
    if (cudaEventRecord(s->ev_fork, st) != cudaSuccess) return DEC_ECUDA;
    if (cudaStreamWaitEvent(s->side, s->ev_fork, 0) != cudaSuccess) return DEC_ECUDA;
    Ctx sx = make_ctx(s, s->side);
    sx.pdl = false;
    sx.ws_len = (long long)(s->ws_side.bytes / sizeof(float));
    sx.ctr_len = (long long)(s->ctr_side.bytes / sizeof(int));
    if ((rc = counted(launch_shared_w13(sx, x, Ws13, M, H, I, s->mb, sgrid, (float*)s->ws_side.p,
                                        (int*)s->ctr_side.p))))
      return rc;
    if ((rc = counted(launch_shared_w2(sx, Ws2, M, H, I, s->mb, sgrid, (float*)s->ws_side.p,
                                       (int*)s->ctr_side.p))))
      return rc;
    if (cudaEventRecord(s->ev_join, s->side) != cudaSuccess) return DEC_ECUDA;
  }
  {
    ProbeScope p(3, st);
    if ((rc = counted(launch_router(cx, x, Wr, M, H, E, topk, topk_idx, topk_w, s->mb, L))))
      return rc;
  }
  if ((rc = counted(launch_gather(cx, x, M, H, E, topk, s->mb, L)))) return rc;
  {
    ProbeScope p(0, st);
    if ((rc = counted(launch_experts_w13(cx, x, W13, M, Wd, E, topk, I, s->mb, egrid, ws, ctr))))
      return rc;
  }
  {
    ProbeScope p(1, st);
    if ((rc = counted(launch_experts_w2(cx, W2, M, Wd, E, topk, I, s->mb, egrid, ws, ctr))))
      return rc;
  }
  // Latent block, 1-16 tokens, where whole-row slabs of Wup fill the SMs: the
  // up-projection after the join, on the slab kernel, with the shared
  // expert's output and the residual added in its epilogue (one launch and
  // one pass over u fewer than the split-K projection and the final sum).
  // Same-GPU A/B (L = 512, hidden 7168), us per block at M = 1 / 2 / 4 / 8 /
  // 16, split-K projection and final sum -> slab tail: 55.8 / 62.7 / 74.8 /
  // 101.9 / 149.9 -> 52.8 / 58.4 / 69.6 / 101.8 / 149.0.
  const int Ru = (L > 0 && !forced("splitk")) ? gemv_mma_rows(M, H, L, s->sms) : 0;
  if (L > 0) {
    // z = bf16(sum_j g_j o_j) on width L
    if ((rc = counted(launch_combine(cx, s->mb, false, nullptr, s->mb.z, M, L, topk)))) return rc;
  }
  if (L > 0 && !Ru) {
    // u = z·Wupᵀ in fp32 (stream-K over every SM); out = bf16(res + (u + s)) below
    const int xr = M <= 2 ? 8 : (M <= 16 ? 16 : 64);
    const long long T = (long long)((H + 127) / 128) * ((L + 127) / 128);
    const int ugrid = (int)(T < s->sms ? T : s->sms);
    if ((rc = counted(launch_dense_f32(cx, xr, M > 2, s->mb.z, Wup, s->mb.u, M, H, L, ugrid, ws,
                                       ctr))))
      return rc;
  }
  if (shared) {
    if (cudaStreamWaitEvent(st, s->ev_join, 0) != cudaSuccess) return DEC_ECUDA;
  }
  // After the join the final sum depends on two streams: launch it without
  // the programmatic (early-start) dependency so both are complete ones.
  cx.pdl = !shared;
  ProbeScope p(4, st);
  if (Ru) {
    cx.ldx = 0;
    return counted(launch_gemv_mma(cx, res != nullptr, s->mb.z, Wup, res, out, M, H, L, Ru,
                                   shared ? s->mb.s : nullptr));
  }
  if (L > 0) return counted(launch_combine_up(cx, s->mb, shared, res, out, M, H));
  return counted(launch_combine(cx, s->mb, shared, res, out, M, H, topk));
}

}  // namespace dg

using namespace dg;

extern "C" {

int dec_version(void) { return 100; }

int dec_linear(const void* x, const void* W, void* y, int M, int N, int K, void* stream) {
  return linear_impl(x, W, nullptr, y, M, N, K, 0, stream);
}

int dec_linear_residual(const void* x, const void* W, const void* res, void* y, int M, int N, int K,
                        void* stream) {
  if (!res) return DEC_EINVAL;
  return linear_impl(x, W, res, y, M, N, K, 0, stream);
}

int dec_linear_ex(const void* x, int ldx, const void* W, const void* res, void* y, int M, int N,
                  int K, void* stream) {
  if (ldx < 1) return DEC_EINVAL;
  return linear_impl(x, W, res, y, M, N, K, 0, stream, ldx);
}

int dec_linear_splitk(const void* x, const void* W, void* y, int M, int N, int K, int S,
                      void* stream) {
  if (S < 1) return DEC_EINVAL;
  return linear_impl(x, W, nullptr, y, M, N, K, S, stream);
}

int moe_decode(const void* x, const void* Wr, const void* W13, const void* W2, const void* Ws13,
               const void* Ws2, void* out, int M, int H, int E, int topk, int I, int32_t* topk_idx,
               float* topk_w, void* stream) {
  return moe_impl(x, Wr, W13, W2, Ws13, Ws2, nullptr, out, M, H, E, topk, I, topk_idx, topk_w,
                  stream);
}

int moe_decode_residual(const void* x, const void* Wr, const void* W13, const void* W2,
                        const void* Ws13, const void* Ws2, const void* res, void* out, int M, int H,
                        int E, int topk, int I, int32_t* topk_idx, float* topk_w, void* stream) {
  if (!res) return DEC_EINVAL;
  return moe_impl(x, Wr, W13, W2, Ws13, Ws2, res, out, M, H, E, topk, I, topk_idx, topk_w, stream);
}

int moe_decode_latent(const void* x, const void* Wrl, const void* W13, const void* W2,
                      const void* Wup, const void* Ws13, const void* Ws2, const void* res,
                      void* out, int M, int H, int L, int E, int topk, int I, int32_t* topk_idx,
                      float* topk_w, void* stream) {
  if (L < 1) return DEC_EINVAL;
  return moe_impl(x, Wrl, W13, W2, Ws13, Ws2, res, out, M, H, E, topk, I, topk_idx, topk_w, stream,
                  L, Wup);
}

int l2_prefetch(const void* ptr, size_t bytes, void* stream) {
  if (!ptr || !aligned16(ptr)) return DEC_EINVAL;
  bytes &= ~size_t(15);
  if (bytes == 0) return DEC_OK;
  DevState* s = nullptr;
  int rc = get_dev(&s);
  if (rc) return rc;
  const size_t cap = (size_t)s->l2 / 2;
  if (bytes > cap) bytes = cap;
  Ctx cx = make_ctx(s, reinterpret_cast<cudaStream_t>(stream));
  return counted(launch_prefetch(cx, ptr, bytes));
}

int dec_add(const void* a, const void* b, void* out, size_t n, void* stream) {
  if (!a || !b || !out) return DEC_EINVAL;
  if (n == 0) return DEC_OK;
  DevState* s = nullptr;
  int rc = get_dev(&s);
  if (rc) return rc;
  Ctx cx = make_ctx(s, reinterpret_cast<cudaStream_t>(stream));
  return counted(launch_add(cx, a, b, out, n));
}

int dec_last_choice(void) { return t_last_choice; }
int dec_last_grid(void) { return t_last_grid; }

const char* dec_strerror(int code) {
  switch (code) {
    case DEC_OK: return "ok";
    case DEC_EINVAL: return "invalid argument (null pointer, size, alignment or K % 8)";
    case DEC_EUNSUPPORTED: return "outside the decode envelope (M > 64, topk > 32 or > E, E > 1024)";
    case DEC_ECUDA: return "CUDA runtime or launch error";
    case DEC_ETIMEOUT: return "a bounded device-side wait gave up";
    case DEC_ENOMEM: return "workspace allocation failed";
    case DEC_ENODEV: return "no sm_103 (GB300) device is current";
    case DEC_EBOUNDS: return "a device-side index check failed (DEC_DEBUG build)";
    default: return "unknown error code";
  }
}

// The device state of the current device if it has been set up, else null
// (sets up nothing).
static DevState* peek_dev() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_dev.size() <= d || !g_dev[d].init) return nullptr;
  return &g_dev[d];
}

// Where the first failed index check of a DEC_DEBUG build was, as read by the
// last dec_sync_check that reported DEC_EBOUNDS.
static int g_check_line = 0;
static long long g_check_index = 0;

int dec_sync_check(void* stream) {
  // Allocates nothing: a device whose state was never set up (a process that
  // only calls dec_linear_noalloc) is not set up here.
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DEC_ECUDA;
  const int nst = noalloc_take_status();
  if (nst < 0) return DEC_ECUDA;
  DevState* s = peek_dev();
  if (!s) return nst ? DEC_ETIMEOUT : DEC_OK;
  if (cudaStreamSynchronize(s->side) != cudaSuccess) return DEC_ECUDA;
  int words[4] = {0, 0, 0, 0};
  if (cudaMemcpy(words, s->status, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DEC_ECUDA;
  const int st = words[0];
  if (st == 0 && nst != 0) return DEC_ETIMEOUT;
  if (st != 0) {
    if (st & kStatusBoundsBit) {
      g_check_line = words[1];
      g_check_index = (long long)(unsigned)words[2] | ((long long)words[3] << 32);
    }
    // Reset the status word and every arrival counter a timed-out kernel may
    // have left behind.
    cudaMemset(s->status, 0, sizeof(int));
    if (s->ctr_main.p) cudaMemset(s->ctr_main.p, 0, s->ctr_main.bytes);
    if (s->ctr_side.p) cudaMemset(s->ctr_side.p, 0, s->ctr_side.bytes);
    if (s->mb.route_ctr) cudaMemset(s->mb.route_ctr, 0, sizeof(int));
    cudaMemset(s->status, 0, sizeof(words));
    cudaDeviceSynchronize();
    return (st & kStatusBoundsBit) ? DEC_EBOUNDS : DEC_ETIMEOUT;
  }
  return DEC_OK;
}

int dec_debug_check_site(int* line, long long* index) {
  if (line) *line = g_check_line;
  if (index) *index = g_check_index;
  return g_check_line != 0 ? 1 : 0;
}

int dec_debug_build(void) {
#ifdef DEC_DEBUG
  return 1;
#else
  return 0;
#endif
}

long long dec_set_wait_timeout_ns(long long ns) {
  long long old = g_timeout_ns;
  if (ns >= 0) g_timeout_ns = ns;
  return old;
}

int dec_selftest_timeout(long long ns, void* stream) {
  DevState* s = nullptr;
  int rc = get_dev(&s);
  if (rc) return rc;
  Ctx cx = make_ctx(s, reinterpret_cast<cudaStream_t>(stream));
  return counted(launch_selftest_timeout(cx, ns));
}

long long dec_launch_count(void) { return g_launches.load(); }

int dec_probe_begin(int kind, int capacity) {
  std::lock_guard<std::mutex> lk(g_probe_mu);
  for (cudaEvent_t e : g_probe_ev) cudaEventDestroy(e);
  g_probe_ev.clear();
  g_probe_n = 0;
  g_probe_cap = 0;
  g_probe_kind = -1;
  if (capacity <= 0) return DEC_OK;
  g_probe_ev.resize(2 * (size_t)capacity);
  for (auto& e : g_probe_ev)
    if (cudaEventCreate(&e) != cudaSuccess) return DEC_ECUDA;
  g_probe_cap = capacity;
  g_probe_kind = kind;
  return DEC_OK;
}

int dec_probe_end(double* total_ms, int* launches) {
  std::lock_guard<std::mutex> lk(g_probe_mu);
  double tot = 0.0;
  for (int i = 0; i < g_probe_n; ++i) {
    if (cudaEventSynchronize(g_probe_ev[2 * i + 1]) != cudaSuccess) return DEC_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_probe_ev[2 * i], g_probe_ev[2 * i + 1]) != cudaSuccess)
      return DEC_ECUDA;
    tot += ms;
  }
  if (total_ms) *total_ms = tot;
  if (launches) *launches = g_probe_n;
  g_probe_kind = -1;
  return DEC_OK;
}

void dec_shutdown(void) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_dev.size() <= d || !g_dev[d].init) return;
  DevState& s = g_dev[d];
  cudaDeviceSynchronize();
  Buf* bufs[] = {&s.ws_main, &s.ctr_main, &s.ws_side, &s.ctr_side, &s.moe};
  for (Buf* b : bufs) {
    if (b->p) cudaFree(b->p);
    b->p = nullptr;
    b->bytes = 0;
  }
  if (s.status) cudaFree(s.status);
  if (s.side) cudaStreamDestroy(s.side);
  if (s.ev_fork) cudaEventDestroy(s.ev_fork);
  if (s.ev_join) cudaEventDestroy(s.ev_join);
  s = DevState();
}

}  // extern "C"
