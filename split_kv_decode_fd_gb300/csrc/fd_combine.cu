// fd_combine.cu -- stand-alone log-sum-exp merge of split partials, one warp
// per (batch, head) (the combine walkthrough of "Kernel visualization: Flash
// Decoding", one thread block per (batch, head) there).  It runs the same
// merge_head as the merge fused into fd_decode, so both give identical bits.
#include "fd_internal.h"
#include "fd_split.cuh"

namespace fdk {

template <int D>
__global__ void __launch_bounds__(128) fd_combine_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ m_part,
                                                         const float* __restrict__ l_part, float* out,
                                                         float* lse, int BH, int n_splits) {
  __shared__ __align__(16) float wsm[4][128];
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= BH) return;
  const GlobalPartials<D> src{o_part, m_part, l_part, (size_t)row * n_splits, 1};
  merge_head<D>(src, n_splits, out + (size_t)row * D, lse ? lse + row : nullptr, threadIdx.x & 31,
                wsm[threadIdx.x >> 5]);
}

cudaError_t launch_combine(int D, const float* o_part, const float* m_part, const float* l_part, float* out,
                           float* lse, int BH, int n_splits, cudaStream_t stream) {
  const dim3 grid((BH + 3) / 4);
  if (D == 128)
    fd_combine_kernel<128><<<grid, 128, 0, stream>>>(o_part, m_part, l_part, out, lse, BH, n_splits);
  else if (D == 64)
    fd_combine_kernel<64><<<grid, 128, 0, stream>>>(o_part, m_part, l_part, out, lse, BH, n_splits);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fdk
