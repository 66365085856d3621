// Kernel launches with programmatic dependent launch (PDL).
//
// Every kernel of the step is launched with the programmatic-serialization
// attribute, so the next kernel in the stream may be scheduled as soon as all
// CTAs of the current one have exited (no kernel triggers earlier), before the
// grid's completion is processed.  Each kernel does its private set-up first
// (barriers, TMEM, tensor-map and weight prefetches) and calls dev::pdl_wait()
// before it touches memory that an earlier kernel writes or reads
// (activations, workspaces, the KV pool); the wait returns when every earlier
// kernel of the stream has completed and its writes are visible, so the chain
// keeps stream order for all data.  Measured on GB300 (Llama-3-8B-shaped step,
// T = 576): 0.383 ms without the attribute, 0.365 ms with it; triggering the
// dependents at kernel start instead made it 0.435 ms, since the waiting CTAs
// of the next kernel then sit beside the running one.  Build with -DMB_PDL=0 to
// launch without the attribute (the waits are then no-ops).
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#ifndef MB_PDL
#define MB_PDL 1
#endif

namespace mb {

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per (kernel, device): the attribute belongs to the device's context, so a
// process that launches on several GPUs sets it on each.
inline cudaError_t ensure_max_smem(const void *kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void *, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto &d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (MB_PDL) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mb
