// dg_common.cuh -- inline-PTX building blocks for sm_103a: mbarriers with
// bounded waits, TMA tile loads with L2 cache hints, programmatic dependent
// launch, ldmatrix / mma.sync, and a few bf16 helpers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dg {

// Status word bits set by device code (read and cleared by dec_sync_check).
// kStatusBounds: an index check of a DEC_DEBUG build failed; the status words
// after the first then hold the source line of the first failed check and
// the offending index (low and high 32 bits).
enum : int { kStatusTimeout = 1, kStatusBounds = 2 };

// ------------------------------------------------------------------ index checks
// DG_AT(status, base, idx, len) is base + idx. In a DEC_DEBUG build an index
// outside [0, len) is not accessed: the first failure records its line and
// index in the status words (status[1..3]), sets kStatusBounds, and the
// access goes to a scratch word of this translation unit instead, so the
// kernel runs on (with wrong results, reported) rather than faulting.
#ifdef DEC_DEBUG
static __device__ __align__(16) unsigned char g_dbg_sink[64];

static __device__ __noinline__ void dbg_check_failed(int* status, int line, long long idx) {
  if (!status) return;
  if (atomicCAS(status + 1, 0, line) == 0) {
    status[2] = (int)(idx & 0xFFFFFFFFLL);
    status[3] = (int)(idx >> 32);
  }
  atomicOr(status, kStatusBounds);
}

template <typename T>
__device__ __forceinline__ T* dbg_at(T* base, long long idx, long long len, int* status,
                                     int line) {
  if (idx >= 0 && idx < len) return base + idx;
  dbg_check_failed(status, line, idx);
  return reinterpret_cast<T*>(const_cast<unsigned char*>(g_dbg_sink));
}
#define DG_AT(status, base, idx, len) \
  ::dg::dbg_at((base), (long long)(idx), (long long)(len), (status), __LINE__)
#define DG_OK(status, cond, v) \
  ((cond) ? true : (::dg::dbg_check_failed((status), __LINE__, (long long)(v)), false))
#else
#define DG_AT(status, base, idx, len) ((base) + (idx))
#define DG_OK(status, cond, v) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up after
// about timeout_ns (counted in SM clock cycles at 2 GHz, so a slower clock
// only lengthens the bound): sets the status word and returns false. The
// clock is read only every 64 polls, so a wait that succeeds costs nothing
// extra.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long timeout_ns,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = timeout_ns * 2;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0 && clock64() - t0 > limit) {
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// Bound of a drain: the wait, after a kernel has given up, for its own copies
// and MMAs still in flight, so that no copy lands in (and no MMA writes to) a
// CTA's shared or tensor memory after the CTA has released it. Issued copies
// always complete, so this bound is never reached in practice; it is at least
// one second whatever the caller's wait bound, which may be far shorter.
__device__ __forceinline__ long long drain_ns(long long timeout_ns) {
  return timeout_ns > 1000000000LL ? timeout_ns : 1000000000LL;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load: box at (c0 = inner coordinate, c1 = row) into smem,
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load: box at (c0, c1, c2) into smem, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global memory into this CTA's shared memory, completing on
// `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk prefetch of [src, src+bytes) into L2 (bytes % 16 == 0).
// Prefetch one tensor-map box into L2 (no shared-memory destination, no
// barrier): the box a later tma_load_2d at the same coordinates will read.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire): shared-memory writes before it are visible to the whole cluster
// after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 load from the shared memory of CTA `rank` of this cluster, at the
// address `local` has in this CTA's shared memory.
__device__ __forceinline__ float ld_dsmem_f32(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// fp32 store into the shared memory of CTA `rank` of this cluster, at the
// address `local` has in this CTA's shared memory.
__device__ __forceinline__ void st_dsmem_f32(void* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// int store into the shared memory of CTA `rank` of this cluster, at the
// address `local` has in this CTA's shared memory.
__device__ __forceinline__ void st_dsmem_s32(void* local, uint32_t rank, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// ------------------------------------------------------------------ PDL
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ sync
// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ mma.sync
__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// D[16x8] += A[16x16] (row) * B[16x8] (col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ bf16
// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f2bf_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float bf_bits2f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// acc + w0*x0 + w1*x1 for the two bf16 halves of w and x (low half first),
// each step one fma.rn.f32.bf16: the bf16 operands enter at full precision
// (a bf16 x bf16 product is exact in fp32) and the sum rounds once per step,
// as fmaf on the widened values would -- without widening them first.
__device__ __forceinline__ float dot2_bf16(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// The same dot with the activations widened to fp32 beforehand (unpack8) and
// each weight widened in the loop: bit-identical to dot8_bf16.
__device__ __forceinline__ float dot8(const uint4& w, const float* xv, float acc) {
  acc = fmaf(bf16lo(w.x), xv[0], acc);
  acc = fmaf(bf16hi(w.x), xv[1], acc);
  acc = fmaf(bf16lo(w.y), xv[2], acc);
  acc = fmaf(bf16hi(w.y), xv[3], acc);
  acc = fmaf(bf16lo(w.z), xv[4], acc);
  acc = fmaf(bf16hi(w.z), xv[5], acc);
  acc = fmaf(bf16lo(w.w), xv[6], acc);
  acc = fmaf(bf16hi(w.w), xv[7], acc);
  return acc;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* o) {
  o[0] = bf16lo(v.x); o[1] = bf16hi(v.x);
  o[2] = bf16lo(v.y); o[3] = bf16hi(v.y);
  o[4] = bf16lo(v.z); o[5] = bf16hi(v.z);
  o[6] = bf16lo(v.w); o[7] = bf16hi(v.w);
}

// Dot of 8 bf16 weights with 8 bf16 activations (one uint4 each), in order.
__device__ __forceinline__ float dot8_bf16(const uint4& w, const uint4& x, float acc) {
  acc = dot2_bf16(w.x, x.x, acc);
  acc = dot2_bf16(w.y, x.y, acc);
  acc = dot2_bf16(w.z, x.z, acc);
  acc = dot2_bf16(w.w, x.w, acc);
  return acc;
}

// silu(z) = z / (1 + e^-z), with CUDA's expf.
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ atomics
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace dg
