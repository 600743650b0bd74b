// k_noalloc.cu -- dec_linear_noalloc: the decode projection for callers that
// must not allocate device memory.
//
// dec_linear keeps its split-K partial sums and arrival counters in a
// workspace that the library allocates with cudaMalloc on first use and
// grows when a larger shape arrives. Some callers cannot allow that: a
// framework whose caching allocator has already reserved the device's memory,
// an engine whose memory budget is fixed before the first request, or a
// latency-critical loop where cudaMalloc / cudaFree (which can synchronise the
// device) must never run. This entry point runs the same weight-streaming
// kernel (CUDA-core for M <= 2, mma.sync for 3 <= M <= 16) with its scratch in
// a fixed array compiled into the library instead.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/decgemm.h"
#include "launch.h"

namespace dg {
namespace {

// Scratch layout: [status word, 256 B][arrival counters][split-K partial tiles].
constexpr size_t kNoAllocBytes = size_t(4) << 20;     // 4 MiB per device
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocCtrBytes = size_t(64) << 10;  // counters for up to 16384 output tiles
constexpr size_t kNoAllocPartBytes = kNoAllocBytes - kNoAllocStatusBytes - kNoAllocCtrBytes;
constexpr int kNoAllocMaxM = 16;
constexpr int kNoAllocMaxDevices = 64;

// Every GPU that loads the library holds this array until the process exits.
// In host code its name is only a host-side stand-in: the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Once per device, with that device current: look up the array's device
// address and the SM count. Allocates nothing.
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DEC_ENODEV;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DEC_ENODEV;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DEC_ENODEV;
    if (major != 10 || minor != 3) return DEC_ENODEV;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DEC_ECUDA;
    d.base = static_cast<unsigned char*>(p);
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return DEC_OK;
}

// As noalloc_setup, but a device that is not set up yet is not set up inside a
// stream capture: the set-up's runtime calls have to run outside it.
int noalloc_setup_checked(void* stream, NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DEC_ENODEV;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DEC_ENODEV;
  bool ready = false;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    ready = g_noalloc_dev[dev].ready;
  }
  if (!ready) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess ||
        cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();  // a query refused during capture leaves no sticky error
      return DEC_EINVAL;
    }
  }
  return noalloc_setup(out);
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Read and clear the status word of the array on the current device: the
// bits a bounded wait of an earlier call set when it gave up. Synchronous
// (callers synchronise the streams first); allocates nothing; 0 when the
// entry point has not run on this device.
int noalloc_take_status() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return 0;
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_dev[dev].ready) return 0;
    base = g_noalloc_dev[dev].base;
  }
  int st = 0;
  if (cudaMemcpy(&st, base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (st != 0 && cudaMemset(base, 0, sizeof(int)) != cudaSuccess) return -1;
  return st;
}

}  // namespace dg

extern "C" int dec_linear_noalloc(const void* x, const void* W, void* y, int M, int N, int K,
                                  void* stream) {
  using namespace dg;
  if (!x || !W || !y) return DEC_EINVAL;
  if (M < 1 || N < 1 || K < 8 || (K % 8) != 0) return DEC_EINVAL;
  if (!is_aligned16(x) || !is_aligned16(W) || !is_aligned16(y)) return DEC_EINVAL;
  if (M > kNoAllocMaxM) return DEC_EUNSUPPORTED;
  NoAllocDevice* d = nullptr;
  int rc = noalloc_setup_checked(stream, &d);
  if (rc) return rc;
  const int xr = M <= 2 ? 8 : 16;  // token rows per pipeline stage
  const long long tiles = (N + 127) / 128;
  const long long KB = (K + 127) / 128;
  const long long T = tiles * KB;
  const long long grid = T < d->sms ? T : d->sms;
  const size_t ctr_bytes = (size_t)tiles * sizeof(int);
  const size_t part_bytes = (size_t)grid * 2 * 128 * xr * sizeof(float);
  if (ctr_bytes > kNoAllocCtrBytes || part_bytes > kNoAllocPartBytes) return DEC_EUNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = reinterpret_cast<int*>(d->base);
  int* ctr = reinterpret_cast<int*>(d->base + kNoAllocStatusBytes);
  float* ws = reinterpret_cast<float*>(d->base + kNoAllocStatusBytes + kNoAllocCtrBytes);
  // The array keeps whatever the last call left: the counters this launch
  // uses must start at zero (a launch that gave up may have left some set).
  // The status word is not cleared here: it keeps a give-up until
  // dec_sync_check reads it.
  if (cudaMemsetAsync(d->base + kNoAllocStatusBytes, 0, ctr_bytes, st) != cudaSuccess)
    return DEC_ECUDA;
  Ctx cx;
  cx.sms = d->sms;
  cx.timeout_ns = dec_set_wait_timeout_ns(-1);  // current bound, unchanged
  cx.status = status;
  cx.stream = st;
  cx.pdl = true;
  cx.ws_len = (long long)(kNoAllocPartBytes / sizeof(float));
  cx.ctr_len = (long long)(kNoAllocCtrBytes / sizeof(int));
  const cudaError_t e = launch_dense(cx, xr, M > 2, false, x, W, nullptr, y, M, N, K, (int)grid,
                                     ws, ctr);
  return e == cudaSuccess ? DEC_OK : DEC_ECUDA;
}
