// Host helpers for launching the kernels: `launch` (every kernel, as a
// programmatic dependent of the work before it in the stream), and for the
// shared-memory-staged kernels `resident_ctas`, which raises a kernel's dynamic
// shared-memory limit to the device's opt-in maximum once per (kernel, device)
// and asks the occupancy calculator how many CTAs fit on an SM, with the
// answers cached.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "tuning.h"

namespace ep {

// Launches `kernel` on `stream`, with EP_PDL as a programmatic dependent of the
// work before it in the stream: its CTAs may be scheduled while that work
// drains, and they wait for it (pdl_wait) before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args... args) {
  static_assert(sizeof...(KArgs) == sizeof...(Args), "one argument per kernel parameter");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = EP_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Resident CTAs per SM of `fn` with `threads` threads and `smem` bytes of
// dynamic shared memory on the current device (>= 1).
inline cudaError_t resident_ctas(const void* fn, int threads, size_t smem, int* per_sm) {
  struct Limit {
    const void* fn;
    int dev;
  };
  struct Occ {
    const void* fn;
    int dev;
    int threads;
    size_t smem;
    int per_sm;
  };
  constexpr int kCache = 512;
  static std::mutex mu;
  static Limit limits[kCache];
  static Occ occs[kCache];
  static int n_limits = 0, n_occs = 0;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n_occs; ++i)
    if (occs[i].fn == fn && occs[i].dev == dev && occs[i].threads == threads && occs[i].smem == smem) {
      *per_sm = occs[i].per_sm;
      return cudaSuccess;
    }
  bool raised = false;
  for (int i = 0; i < n_limits && !raised; ++i) raised = limits[i].fn == fn && limits[i].dev == dev;
  if (!raised) {
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
    if (n_limits < kCache) limits[n_limits++] = Limit{fn, dev};
  }
  int r = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, fn, threads, smem);
  if (e != cudaSuccess) return e;
  r = std::max(r, 1);
  if (n_occs < kCache) occs[n_occs++] = Occ{fn, dev, threads, smem, r};
  *per_sm = r;
  return cudaSuccess;
}

}  // namespace ep
