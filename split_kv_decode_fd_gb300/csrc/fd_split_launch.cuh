// fd_split_launch.cuh -- host-side launch of one fd_split_kernel instantiation.
#pragma once

#include <atomic>

#include "fd_internal.h"
#include "fd_split.cuh"

namespace fdk {

template <int D, class KV, int G>
cudaError_t launch_split_t(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p, dim3 grid,
                           cudaStream_t stream) {
  using C = SplitCfg<D, KV, G>;
  static std::atomic<int> configured_device{-1};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device.load(std::memory_order_acquire) != dev) {
    e = cudaFuncSetAttribute(fd_split_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured_device.store(dev, std::memory_order_release);
  }
  // Programmatic dependent launch: the kernel may be scheduled while the
  // kernel before it on the stream is still finishing; it touches no memory
  // before griddepcontrol.wait, so only its set-up overlaps the earlier kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fd_split_kernel<C>, tk, tv, p);
}

template <class KV>
cudaError_t launch_split_dispatch(int D, int gpad, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const SplitParams& p, dim3 grid, cudaStream_t stream) {
#define FD_CASE(DD, GG) \
  if (D == DD && gpad == GG) return launch_split_t<DD, KV, GG>(tk, tv, p, grid, stream);
  FD_CASE(128, 1) FD_CASE(128, 2) FD_CASE(128, 4) FD_CASE(128, 8)
  FD_CASE(64, 1) FD_CASE(64, 2) FD_CASE(64, 4) FD_CASE(64, 8)
  if constexpr (sizeof(KV) == 2) {
    FD_CASE(128, 16) FD_CASE(64, 16)
  }
#undef FD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fdk
