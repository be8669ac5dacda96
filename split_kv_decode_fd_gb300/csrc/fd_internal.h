// fd_internal.h -- launch entry points shared between the library's
// translation units (kernels are compiled in several units so that the build
// runs in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fd_plan.h"

namespace fdk {

struct SplitParams;

// Launch the split kernel for (head_dim, kv element bytes, heads per CTA).
// Returns cudaErrorInvalidValue for a combination that is not compiled.
cudaError_t launch_split_bf16(int D, int gpad, const CUtensorMap& tk, const CUtensorMap& tv,
                              const SplitParams& p, dim3 grid, cudaStream_t stream);
cudaError_t launch_split_f32(int D, int gpad, const CUtensorMap& tk, const CUtensorMap& tv,
                             const SplitParams& p, dim3 grid, cudaStream_t stream);

cudaError_t launch_combine(int D, const float* o_part, const float* m_part, const float* l_part, float* out,
                           float* lse, int BH, int n_splits, cudaStream_t stream);

}  // namespace fdk
