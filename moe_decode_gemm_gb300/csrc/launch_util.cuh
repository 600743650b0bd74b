// launch_util.cuh -- kernel launch with programmatic dependent launch (PDL).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace dg {

// Launch `kern` on `stream`. With pdl, the launch carries the programmatic
// stream serialisation attribute: the kernel may start while the previous
// kernel in the stream is finishing, and must call griddepcontrol.wait before
// it touches anything that kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// As launch_k, in thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared memory limit.
template <typename K>
cudaError_t allow_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Once per device: a kernel's function attributes are set for the current
// device only, so a flag per device (bit d for device d < 64; devices beyond
// set them on every call). Two threads may both run the set-up the first
// time; setting an attribute twice is harmless.
struct DevOnce {
  std::atomic<unsigned long long> bits{0};
  template <typename F>
  cudaError_t run(F&& setup) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    const unsigned long long b = d < 64 ? 1ull << d : 0ull;
    if (b && (bits.load(std::memory_order_acquire) & b)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess && b) bits.fetch_or(b, std::memory_order_release);
    return e;
  }
};

// A kernel's dynamic shared memory limit (and, with max_carveout, the largest
// shared-memory carveout), once per device.
template <typename K>
cudaError_t setup_smem(DevOnce& once, K kern, int bytes, bool max_carveout = false) {
  return once.run([&]() -> cudaError_t {
    cudaError_t e = allow_smem(kern, bytes);
    if (e == cudaSuccess && max_carveout)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    return e;
  });
}

}  // namespace dg
