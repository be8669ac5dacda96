// fd_prefill.h -- parameters of the many-row (prefill) attention kernel,
// shared by the host entry points and the kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fdk {

struct PrefillParams {
  const float* q;              // [B, Hq, n_q, D] fp32
  float* out;                  // [B, Hq, n_q, D] fp32
  float* lse;                  // [B, Hq, n_q] natural log, or null
  const int32_t* seq_lens;     // [B] keys per sequence (the n_q rows are its last n_q tokens), or null
  const int32_t* block_table;  // paged: [B, max_pages]
  unsigned* err;               // error word (timeouts, bad pages)
  unsigned* work;              // [2] item queue: next item, CTAs done (zero between launches)
  int32_t B, Hq, Hkv, g, n_q, max_len, causal;
  int32_t paged, page_size, max_pages, num_pages;
  float qk_scale;              // scale * log2(e)
  uint64_t wait_ns;            // limit of every mbarrier wait (0: the default, 2 s)
  int32_t stall_u;             // testing hook: the K/V copy (slot use) every CTA skips, or -1
};

// Query rows per CTA and keys per tile of the prefill kernel.
constexpr int kPrefillRows = 128;
constexpr int kPrefillKeys = 128;

// D = 64 or 128; cudaErrorInvalidValue otherwise.
// `tq`, `to`: q and the output as [B*Hq, n_q, D] fp32, 32-column x 128-row
// boxes with the 128-byte swizzle (the kernel loads q tiles and stores output
// tiles through them).
cudaError_t launch_prefill(int D, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);

}  // namespace fdk
