// fd_split_bf16.cu -- split kernels for bf16 K/V caches (D = 64, 128; 1..8 heads per CTA).
#include "fd_split_launch.cuh"

namespace fdk {
cudaError_t launch_split_bf16(int D, int gpad, const CUtensorMap& tk, const CUtensorMap& tv,
                              const SplitParams& p, dim3 grid, cudaStream_t stream) {
  return launch_split_dispatch<__nv_bfloat16>(D, gpad, tk, tv, p, grid, stream);
}
}  // namespace fdk
