// Host-side launch of one forward-kernel configuration: opt in to its shared
// memory size, size the grid to the resident CTAs of the device (one wave, so
// the grid barrier can complete), and launch cooperatively on the caller's stream.
#pragma once
#include <cuda_runtime.h>

#include <atomic>

#include "fwd_kernel.cuh"

namespace dsf {

constexpr int kMaxDevices = 64;

// The grid size is computed on the first launch per device and cached; host
// threads may race on that first computation (each gets the same value), so
// the cache words are atomics.
template <class C>
int grid_for_device(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  const int known = cache[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  constexpr int smem = smem_bytes<C>();
  static_assert(smem <= 227 * 1024, "shared memory per block above the sm_100-family limit");
  int optin = 0, nsm = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  if (optin < smem) return 0;
  if (cudaFuncSetAttribute(dsf_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dsf_fwd_kernel<C>, kThreads, smem) != cudaSuccess)
    return 0;
  if (occ < 1) return 0;
  int g = nsm * occ;
  if (g > kMaxG) g = kMaxG;
  cache[dev].store(g, std::memory_order_release);
  return g;
}

// Returns 0 on success, 2 if this device cannot run the configuration, 3 on a
// launch error.
template <class C>
int launch_fwd(const FwdParams& p, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 3;
  const int G = grid_for_device<C>(dev);
  if (G <= 0) return 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<C>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dsf_fwd_kernel<C>, p);
  return e == cudaSuccess ? 0 : 3;
}

// Dispatch entry points, one per translation unit group.
int launch_pool(int D, bool bf16, const FwdParams& p, cudaStream_t s);
int launch_attn_tc(int D, bool bf16, const FwdParams& p, cudaStream_t s);
int launch_attn_f32(int D, bool bf16, const FwdParams& p, cudaStream_t s);
int grid_pool(int D, bool bf16, int dev);
int grid_attn_tc(int D, bool bf16, int dev);
int grid_attn_f32(int D, bool bf16, int dev);

}  // namespace dsf
