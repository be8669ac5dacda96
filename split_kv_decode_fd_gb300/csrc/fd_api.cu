// fd_api.cu -- the C ABI of libfdecode: argument checks, workspace layout,
// TMA descriptors, the host-side plan inspector and kernel dispatch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/fdecode.h"
#include "fd_internal.h"
#include "fd_prefill.h"
#include "fd_split.cuh"

using namespace fdk;

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;  // error word + reserved
constexpr size_t kPrefillWorkOff = 128;  // the prefill's item-queue counters, inside the header
// Arrival counters of the fused merge live in a region of fixed size right
// after the header, whatever the problem shape, so that no call ever writes
// partials where another shape keeps its counters; every call leaves the
// counters it used at zero.
constexpr int64_t kMaxFusedPairs = 65536;
constexpr size_t kCounterBytes = (size_t)kMaxFusedPairs * 4;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Balanced plan CTA count for the current device (one CTA per SM).
int sm_count(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64) {
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return 1;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return 1;
}

struct WsLayout {
  size_t err, counters, o, m, l, q_stage, out_stage, lse_stage, len_stage, total;
};

// Workspace: [header | counters | o | m | l | host staging (q, out, lse, lens)].
int group_cap(int dtype) { return dtype == FD_BF16 ? kMaxGroupBf16 : kMaxGroupF32; }

WsLayout ws_layout(int B, int Hq, int Hkv, int D, int n_splits, int grid, int cap) {
  const Groups gr = make_groups(Hq, Hkv, cap);
  const size_t pairs = (size_t)B * gr.hv;
  size_t states;  // number of (slot, head) partial states
  if (n_splits == 0)
    states = ((size_t)grid + pairs) * gr.gpad;  // slots <= grid + pairs - 1
  else
    states = (size_t)B * Hq * n_splits;
  WsLayout w;
  w.err = 0;
  w.counters = kHeaderBytes;
  w.o = w.counters + kCounterBytes;
  w.m = w.o + align_up(states * D * 4);
  w.l = w.m + align_up(states * 4);
  w.q_stage = w.l + align_up(states * 4);
  w.out_stage = w.q_stage + align_up((size_t)B * Hq * D * 4);
  w.lse_stage = w.out_stage + align_up((size_t)B * Hq * D * 4);
  w.len_stage = w.lse_stage + align_up((size_t)B * Hq * 4);
  w.total = w.len_stage + align_up((size_t)B * 4);
  return w;
}

fd_status check_shape(int B, int Hq, int Hkv, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return FD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FD_ERR_UNSUPPORTED;
  const Groups gr = make_groups(Hq, Hkv, kMaxGroupF32);  // the larger hv of the two caps
  if ((int64_t)B * gr.hv > (int64_t)1 << 30) return FD_ERR_UNSUPPORTED;
  return FD_OK;
}

fd_status check_kv(const fd_kv_desc* kv, int B, int Hkv, int max_seq_len) {
  if (!kv || !kv->k || !kv->v) return FD_ERR_INVALID_ARG;
  if (!aligned16(kv->k) || !aligned16(kv->v)) return FD_ERR_INVALID_ARG;
  if (kv->dtype != FD_F32 && kv->dtype != FD_BF16) return FD_ERR_UNSUPPORTED;
  if (max_seq_len < 0) return FD_ERR_INVALID_ARG;
  const int64_t tiles = (int64_t)B * Hkv * ((max_seq_len + kPlanTile - 1) / kPlanTile);
  if (tiles >= ((int64_t)1 << 31) / kMaxGroupBf16) return FD_ERR_UNSUPPORTED;
  if (kv->layout == FD_KV_CONTIGUOUS) {
    if (kv->capacity < 1 || kv->capacity < max_seq_len) return FD_ERR_INVALID_ARG;
    if (kv->capacity > ((int64_t)1 << 31) - 1) return FD_ERR_UNSUPPORTED;
  } else if (kv->layout == FD_KV_PAGED) {
    if (!kv->block_table || kv->page_size < 16 || kv->page_size % 16 != 0 || kv->num_pages < 1 ||
        kv->max_pages_per_seq < 1)
      return FD_ERR_INVALID_ARG;
    if ((int64_t)kv->max_pages_per_seq * kv->page_size < max_seq_len) return FD_ERR_INVALID_ARG;
    if ((int64_t)kv->num_pages * Hkv > INT32_MAX) return FD_ERR_UNSUPPORTED;  // TMA row-block coordinate
  } else {
    return FD_ERR_INVALID_ARG;
  }
  return FD_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 16-row x 128-byte boxes with the 128-byte swizzle, over the contiguous
// cache [B*Hkv, T_cap, D] or the page pool [num_pages, Hkv, page_size, D].
fd_status make_maps(const fd_kv_desc* kv, int B, int Hkv, int D, CUtensorMap* tk, CUtensorMap* tv) {
  auto encode = encode_fn();
  if (!encode) return FD_ERR_CUDA;
  const CUtensorMapDataType dt =
      kv->dtype == FD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t es = kv->dtype == FD_BF16 ? 2 : 4;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  cuuint32_t rank;
  if (kv->layout == FD_KV_CONTIGUOUS) {
    rank = 3;
    dims[0] = (cuuint64_t)D;
    dims[1] = (cuuint64_t)kv->capacity;
    dims[2] = (cuuint64_t)B * Hkv;
    strides[0] = (cuuint64_t)D * es;
    strides[1] = (cuuint64_t)kv->capacity * D * es;
    box[0] = (cuuint32_t)(128 / es);
    box[1] = 16;
    box[2] = 1;
  } else {
    // the pool [num_pages, Hkv, page_size, D] as [num_pages * Hkv, page_size, D]
    // (measured faster than the 4-D view of the same boxes)
    rank = 3;
    dims[0] = (cuuint64_t)D;
    dims[1] = (cuuint64_t)kv->page_size;
    dims[2] = (cuuint64_t)kv->num_pages * Hkv;
    strides[0] = (cuuint64_t)D * es;
    strides[1] = (cuuint64_t)kv->page_size * D * es;
    box[0] = (cuuint32_t)(128 / es);
    box[1] = 16;
    box[2] = 1;
  }
  // Encoding costs a driver call per map; decode steps usually repeat the same
  // cache, so the last few (K, V) pairs are kept per host thread, keyed by
  // every input of the encoding (a map holds nothing else).
  struct MapEntry {
    const void *k, *v;
    CUtensorMapDataType dt;
    cuuint64_t dims[3], strides[2];
    CUtensorMap tk, tv;
    bool valid;
  };
  thread_local MapEntry cache[4];
  thread_local int next_slot = 0;
  for (const MapEntry& e : cache) {
    if (e.valid && e.k == kv->k && e.v == kv->v && e.dt == dt && e.dims[0] == dims[0] && e.dims[1] == dims[1] &&
        e.dims[2] == dims[2] && e.strides[0] == strides[0] && e.strides[1] == strides[1]) {
      *tk = e.tk;
      *tv = e.tv;
      return FD_OK;
    }
  }
  const void* ptrs[2] = {kv->k, kv->v};
  CUtensorMap* maps[2] = {tk, tv};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(maps[i], dt, rank, const_cast<void*>(ptrs[i]), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FD_ERR_INVALID_ARG;
  }
  MapEntry& e = cache[next_slot];
  next_slot = (next_slot + 1) % 4;
  e.k = kv->k;
  e.v = kv->v;
  e.dt = dt;
  for (int i = 0; i < 3; ++i) e.dims[i] = dims[i];
  for (int i = 0; i < 2; ++i) e.strides[i] = strides[i];
  e.tk = *tk;
  e.tv = *tv;
  e.valid = true;
  return FD_OK;
}

// The prefill's q or output [B*Hq][n_q][D] fp32 as a tensor map: boxes of 32
// columns (128 bytes, the 128-byte swizzle) x 128 query rows of one head, so
// that a tile's rows past n_q fall outside the map: loads read zeros there,
// stores leave them alone.
fd_status make_rows_map(const float* base, int64_t heads, int32_t n_q, int32_t D, CUtensorMap* to) {
  auto encode = encode_fn();
  if (!encode) return FD_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n_q, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)n_q * D * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)kPrefillRows, 1}, estr[3] = {1, 1, 1};
  CUresult r = encode(to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FD_OK : FD_ERR_INVALID_ARG;
}

// Testing hook of the bounded waits (fd_debug_stall): off by default.
std::atomic<int32_t> g_stall_it{-1};
std::atomic<int64_t> g_wait_ns{0};

SplitParams base_params(const float* q, const fd_kv_desc* kv, int B, int Hq, int Hkv,
                        const int32_t* seq_lens, int max_seq_len, float scale) {
  SplitParams p;
  std::memset(&p, 0, sizeof(p));
  const Groups gr = make_groups(Hq, Hkv, group_cap(kv->dtype));
  p.q = q;
  p.seq_lens = seq_lens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = gr.g;
  p.gpad = gr.gpad;
  p.nsub = gr.nsub;
  p.hv = gr.hv;
  p.max_len = max_seq_len;
  p.paged = kv->layout == FD_KV_PAGED;
  p.block_table = kv->block_table;
  p.page_size = kv->page_size;
  p.max_pages = kv->max_pages_per_seq;
  p.num_pages = kv->num_pages;
  p.qk_scale = (float)((double)scale * 1.4426950408889634);
  p.n_q = 1;
  p.causal = 0;
  p.stall_it = g_stall_it.load(std::memory_order_relaxed);
  p.wait_ns = (uint64_t)g_wait_ns.load(std::memory_order_relaxed);
  return p;
}

// Split count used when the balanced plan does not apply (batch above
// FD_AUTO_MAX_BATCH): about two CTAs per SM over all (b, virtual kv head).
int fallback_splits(int B, int hv, int max_seq_len, int sms) {
  const int64_t pairs = (int64_t)B * hv;
  int64_t n = (2 * (int64_t)sms + pairs - 1) / pairs;
  const int64_t cap = (max_seq_len + kPlanTile - 1) / kPlanTile;
  if (n > cap) n = cap;
  return (int)(n < 1 ? 1 : (n > 65535 ? 65535 : n));
}

fd_status launch(const fd_kv_desc* kv, int D, const SplitParams& p, dim3 grid, cudaStream_t stream) {
  CUtensorMap tk, tv;
  fd_status st = make_maps(kv, p.B, p.Hkv, D, &tk, &tv);
  if (st != FD_OK) return st;
  cudaError_t e = kv->dtype == FD_BF16 ? launch_split_bf16(D, p.gpad, tk, tv, p, grid, stream)
                                       : launch_split_f32(D, p.gpad, tk, tv, p, grid, stream);
  return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

// Host copy of the per-sequence cost-unit table, for the plan inspector.
struct HostTiles {
  const int64_t* pre;
  const int32_t* ln;
  int32_t piece_units;
  FD_HD int32_t piece() const { return piece_units; }
  FD_HD int64_t prefix(int32_t b) const { return pre[b]; }
  FD_HD int32_t tiles(int32_t b) const { return ceil_div(ln[b], kPlanTile); }
  FD_HD int32_t len(int32_t b) const { return ln[b]; }
};

// Device address of host memory that is pinned and mapped into the device's
// address space (cudaHostAlloc / cudaHostRegister under unified addressing);
// false for pageable memory.  Asked on every call: a buffer freed and another
// allocated at the same address must not inherit the old answer.
template <class T>
bool host_mapped(T* host, T** dev) {
  cudaPointerAttributes a;
  void* d = nullptr;
  if (cudaPointerGetAttributes(&a, host) == cudaSuccess && a.type == cudaMemoryTypeHost && a.devicePointer)
    d = a.devicePointer;
  cudaGetLastError();  // a pageable pointer may leave an error behind on older runtimes
  *dev = static_cast<T*>(d);
  return d != nullptr;
}

}  // namespace

extern "C" {

const char* fd_status_string(fd_status s) {
  switch (s) {
    case FD_OK: return "ok";
    case FD_ERR_INVALID_ARG: return "invalid argument";
    case FD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case FD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FD_ERR_BAD_INDEX: return "block-table entry out of range";
    case FD_ERR_CUDA: return "CUDA error";
    case FD_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

int32_t fd_version(void) { return 100; }

void fd_debug_stall(int32_t stage, int64_t wait_limit_ns) {
  g_wait_ns.store(stage >= 0 && wait_limit_ns > 0 ? wait_limit_ns : 0, std::memory_order_relaxed);
  g_stall_it.store(stage >= 0 ? stage : -1, std::memory_order_relaxed);
}

int32_t fd_split_size(int32_t max_seq_len, int32_t n_splits) {
  return explicit_split_size(max_seq_len, n_splits);
}

size_t fd_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_splits, int32_t num_sms) {
  if (check_shape(B, Hq, Hkv, D) != FD_OK || n_splits < 0 || n_splits > 65535) return 0;
  int grid = num_sms;
  if (grid <= 0 && !sm_count(&grid)) return 0;
  // The size must hold for either cache dtype (their group caps differ).
  size_t most = 0;
  for (const int cap : {kMaxGroupF32, kMaxGroupBf16}) {
    const Groups gr = make_groups(Hq, Hkv, cap);
    size_t a;
    if (n_splits == 0 && (B > FD_AUTO_MAX_BATCH || (int64_t)B * gr.hv > kMaxFusedPairs))
      // the fallback split count depends on max_seq_len; size for the largest it can be
      a = ws_layout(B, Hq, Hkv, D, fallback_splits(B, gr.hv, 1 << 30, grid), grid, cap).total;
    else
      a = ws_layout(B, Hq, Hkv, D, n_splits, grid, cap).total;
    most = a > most ? a : most;
  }
  return most;
}

fd_status fd_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kHeaderBytes) return FD_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) == cudaSuccess ? FD_OK
                                                                                                : FD_ERR_CUDA;
}

fd_status fd_workspace_status(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kHeaderBytes) return FD_ERR_INVALID_ARG;
  unsigned word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FD_ERR_CUDA;
  if (word == 0) return FD_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return FD_ERR_CUDA;
  if (word & kErrTimeout) return FD_ERR_TIMEOUT;
  return FD_ERR_BAD_INDEX;
}

}  // extern "C"

namespace {

// fd_decode over Hq "virtual heads" = query heads x rows (n_q rows per head).
// Variants of the decode: several query rows per head; the fused append.
struct DecodeExtras {
  int32_t n_q = 1, causal = 0;
  const void* k_new = nullptr;  // non-null: append the new token before attending
  const void* v_new = nullptr;
};

fd_status decode_impl(const float* q, const fd_kv_desc* kv, float* out, float* lse, int32_t B, int32_t Hq,
                      int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len, int32_t D, float scale,
                      int32_t n_splits, void* workspace, size_t workspace_bytes, void* stream,
                      const DecodeExtras& x) {
  fd_status st = check_shape(B, Hq, Hkv, D);
  if (st != FD_OK) return st;
  if (!q || !out || !workspace || !aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return FD_ERR_INVALID_ARG;
  if (n_splits < 0 || n_splits > 65535) return FD_ERR_INVALID_ARG;
  const int32_t append = x.k_new ? 1 : 0;
  if (append && (!x.v_new || !aligned16(x.k_new) || !aligned16(x.v_new) || max_seq_len < 0)) return FD_ERR_INVALID_ARG;
  if (max_seq_len > INT32_MAX - append) return FD_ERR_UNSUPPORTED;
  max_seq_len += append;  // from here on: lengths as the kernel sees them (the new token included)
  if ((st = check_kv(kv, B, Hkv, max_seq_len)) != FD_OK) return st;
  const Groups gr = make_groups(Hq, Hkv, group_cap(kv->dtype));
  const int64_t pairs = (int64_t)B * gr.hv;
  int sms = 0;
  if (n_splits == 0) {
    if (!sm_count(&sms)) return FD_ERR_CUDA;
    if (B > FD_AUTO_MAX_BATCH || pairs > kMaxFusedPairs) n_splits = fallback_splits(B, gr.hv, max_seq_len, sms);
  }
  const WsLayout w = ws_layout(B, Hq, Hkv, D, n_splits, sms, group_cap(kv->dtype));
  if (workspace_bytes < w.total) return FD_ERR_WORKSPACE_TOO_SMALL;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SplitParams p = base_params(q, kv, B, Hq, Hkv, seq_lens, max_seq_len, scale);
  p.n_q = x.n_q;
  p.causal = x.causal;
  p.append = append;
  p.k_new = x.k_new;
  p.v_new = x.v_new;
  p.k_cache = const_cast<void*>(kv->k);
  p.v_cache = const_cast<void*>(kv->v);
  p.capacity = kv->capacity;
  p.out = out;
  p.lse = lse;
  p.o_part = reinterpret_cast<float*>(ws + w.o);
  p.m_part = reinterpret_cast<float*>(ws + w.m);
  p.l_part = reinterpret_cast<float*>(ws + w.l);
  p.err = reinterpret_cast<unsigned*>(ws + w.err);
  cudaStream_t s = (cudaStream_t)stream;
  if (n_splits == 0) {
    p.n_splits = 0;
    p.counters = reinterpret_cast<int*>(ws + w.counters);
    return launch(kv, D, p, dim3((unsigned)sms, 1, 1), s);
  }
  p.n_splits = n_splits;
  p.split_tokens = max_seq_len > 0 ? explicit_split_size(max_seq_len, n_splits) : kSplitAlign;
  const dim3 grid((unsigned)pairs, (unsigned)n_splits, 1);
  if (pairs <= kMaxFusedPairs) {
    p.counters = reinterpret_cast<int*>(ws + w.counters);
    return launch(kv, D, p, grid, s);
  }
  // Too many sequences for the counter region: split, then a separate merge.
  p.counters = nullptr;
  if ((st = launch(kv, D, p, grid, s)) != FD_OK) return st;
  const cudaError_t e = launch_combine(D, p.o_part, p.m_part, p.l_part, out, lse, B * Hq, n_splits, s);
  return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace

extern "C" {

fd_status fd_decode(const float* q, const fd_kv_desc* kv, float* out, float* lse, int32_t B, int32_t Hq,
                    int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len, int32_t D, float scale,
                    int32_t n_splits, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, kv, out, lse, B, Hq, Hkv, seq_lens, max_seq_len, D, scale, n_splits, workspace,
                     workspace_bytes, stream, DecodeExtras{});
}

fd_status fd_append_decode(const float* q, const void* k_new, const void* v_new, const fd_kv_desc* kv, float* out,
                           float* lse, int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t D, float scale, int32_t n_splits, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!k_new || !v_new) return FD_ERR_INVALID_ARG;
  DecodeExtras x;
  x.k_new = k_new;
  x.v_new = v_new;
  return decode_impl(q, kv, out, lse, B, Hq, Hkv, seq_lens, max_seq_len, D, scale, n_splits, workspace,
                     workspace_bytes, stream, x);
}

fd_status fd_decode_rows(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out,
                         float* lse, int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens,
                         int32_t max_seq_len, int32_t D, float scale, int32_t n_splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (n_q < 1 || n_q > 64 || (causal != 0 && causal != 1)) return FD_ERR_INVALID_ARG;
  if (Hq < 1 || (int64_t)Hq * n_q > ((int64_t)1 << 24)) return FD_ERR_INVALID_ARG;
  DecodeExtras x;
  x.n_q = n_q;
  x.causal = causal;
  return decode_impl(q, kv, out, lse, B, Hq * n_q, Hkv, seq_lens, max_seq_len, D, scale, n_splits, workspace,
                     workspace_bytes, stream, x);
}

fd_status fd_prefill(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out, float* lse,
                     int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len, int32_t D,
                     float scale, void* workspace, size_t workspace_bytes, void* stream) {
  fd_status st = check_shape(B, Hq, Hkv, D);
  if (st != FD_OK) return st;
  if (!q || !out || !workspace || !aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return FD_ERR_INVALID_ARG;
  if (n_q < 1 || (causal != 0 && causal != 1)) return FD_ERR_INVALID_ARG;
  if (workspace_bytes < kHeaderBytes) return FD_ERR_WORKSPACE_TOO_SMALL;
  if ((st = check_kv(kv, B, Hkv, max_seq_len)) != FD_OK) return st;
  if (kv->dtype != FD_BF16) return FD_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535 || (int64_t)B * Hq * n_q * D > ((int64_t)1 << 40)) return FD_ERR_UNSUPPORTED;
  if ((int64_t)B * Hq > INT32_MAX) return FD_ERR_UNSUPPORTED;  // a tensor-map coordinate
  CUtensorMap tk, tv, tq, to;
  if ((st = make_maps(kv, B, Hkv, D, &tk, &tv)) != FD_OK) return st;
  if ((st = make_rows_map(q, (int64_t)B * Hq, n_q, D, &tq)) != FD_OK) return st;
  if ((st = make_rows_map(out, (int64_t)B * Hq, n_q, D, &to)) != FD_OK) return st;
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.seq_lens = seq_lens;
  p.block_table = kv->block_table;
  p.err = reinterpret_cast<unsigned*>(workspace);
  p.work = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + kPrefillWorkOff);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.n_q = n_q;
  p.max_len = max_seq_len;
  p.causal = causal;
  p.paged = kv->layout == FD_KV_PAGED;
  p.page_size = kv->page_size;
  p.max_pages = kv->max_pages_per_seq;
  p.num_pages = kv->num_pages;
  p.qk_scale = (float)((double)scale * 1.4426950408889634);
  p.stall_u = g_stall_it.load(std::memory_order_relaxed);
  p.wait_ns = (uint64_t)g_wait_ns.load(std::memory_order_relaxed);
  return launch_prefill(D, tk, tv, tq, to, p, (cudaStream_t)stream) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

int32_t fd_attend_backend(int32_t n_q, int32_t Hq, int32_t Hkv, int32_t D, int32_t kv_dtype) {
  if (n_q < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return -1;
  if (n_q == 1) return FD_BACKEND_DECODE;
  const bool prefill_ok = (D == 64 || D == 128) && kv_dtype == FD_BF16;
  if ((int64_t)n_q * (Hq / Hkv) <= kMaxGroupBf16 || (!prefill_ok && n_q <= 64)) return FD_BACKEND_DECODE_ROWS;
  return prefill_ok ? FD_BACKEND_PREFILL : -1;
}

const char* fd_backend_name(int32_t backend) {
  switch (backend) {
    case FD_BACKEND_DECODE: return "decode (fd_split_kernel, one query row)";
    case FD_BACKEND_DECODE_ROWS: return "decode_rows (fd_split_kernel, rows as virtual heads)";
    case FD_BACKEND_PREFILL: return "prefill (fd_prefill_kernel, tcgen05 query tiles)";
    default: return "none";
  }
}

fd_status fd_attend(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out, float* lse,
                    int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len, int32_t D,
                    float scale, int32_t n_splits, void* workspace, size_t workspace_bytes, void* stream,
                    int32_t* backend) {
  const int32_t be = fd_attend_backend(n_q, Hq, Hkv, D, kv ? kv->dtype : -1);
  if (backend) *backend = be;
  switch (be) {
    case FD_BACKEND_DECODE:
      return fd_decode(q, kv, out, lse, B, Hq, Hkv, seq_lens, max_seq_len, D, scale, n_splits, workspace,
                       workspace_bytes, stream);
    case FD_BACKEND_DECODE_ROWS:
      return fd_decode_rows(q, n_q, causal, kv, out, lse, B, Hq, Hkv, seq_lens, max_seq_len, D, scale, n_splits,
                            workspace, workspace_bytes, stream);
    case FD_BACKEND_PREFILL:
      return fd_prefill(q, n_q, causal, kv, out, lse, B, Hq, Hkv, seq_lens, max_seq_len, D, scale, workspace,
                        workspace_bytes, stream);
    default:
      return n_q < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ? FD_ERR_INVALID_ARG : FD_ERR_UNSUPPORTED;
  }
}

fd_status fd_split_partial(const float* q, const fd_kv_desc* kv, int32_t B, int32_t Hq, int32_t Hkv,
                           const int32_t* seq_lens, int32_t max_seq_len, int32_t D, float scale,
                           int32_t n_splits, float* o_part, float* m_part, float* l_part, void* stream) {
  fd_status st = check_shape(B, Hq, Hkv, D);
  if (st != FD_OK) return st;
  if (!q || !o_part || !m_part || !l_part || !aligned16(q) || !aligned16(o_part)) return FD_ERR_INVALID_ARG;
  if (n_splits < 1 || n_splits > 65535) return FD_ERR_INVALID_ARG;
  if ((st = check_kv(kv, B, Hkv, max_seq_len)) != FD_OK) return st;
  SplitParams p = base_params(q, kv, B, Hq, Hkv, seq_lens, max_seq_len, scale);
  p.o_part = o_part;
  p.m_part = m_part;
  p.l_part = l_part;
  p.n_splits = n_splits;
  p.split_tokens = max_seq_len > 0 ? explicit_split_size(max_seq_len, n_splits) : kSplitAlign;
  const dim3 grid((unsigned)(B * p.hv), (unsigned)n_splits, 1);
  return launch(kv, D, p, grid, (cudaStream_t)stream);
}

fd_status fd_combine(const float* o_part, const float* m_part, const float* l_part, float* out, float* lse,
                     int32_t B, int32_t Hq, int32_t D, int32_t n_splits, void* stream) {
  if (!o_part || !m_part || !l_part || !out || B < 1 || Hq < 1 || n_splits < 1) return FD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FD_ERR_UNSUPPORTED;
  if (!aligned16(o_part) || !aligned16(out)) return FD_ERR_INVALID_ARG;
  if ((int64_t)B * Hq > ((int64_t)1 << 31) - 4) return FD_ERR_UNSUPPORTED;
  cudaError_t e = launch_combine(D, o_part, m_part, l_part, out, lse, B * Hq, n_splits, (cudaStream_t)stream);
  return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

fd_status fd_decode_host(const float* q_host, const fd_kv_desc* kv, float* out_host, float* lse_host, int32_t B,
                         int32_t Hq, int32_t Hkv, const int32_t* seq_lens_host, int32_t max_seq_len, int32_t D,
                         float scale, int32_t n_splits, void* workspace, size_t workspace_bytes,
                         void* stream) {
  fd_status st = check_shape(B, Hq, Hkv, D);
  if (st != FD_OK) return st;
  if (!q_host || !out_host || !workspace) return FD_ERR_INVALID_ARG;
  if (n_splits < 0 || n_splits > 65535) return FD_ERR_INVALID_ARG;
  int grid_ctas = 0;
  if (n_splits == 0 && !sm_count(&grid_ctas)) return FD_ERR_CUDA;
  if (!kv) return FD_ERR_INVALID_ARG;
  if (kv->dtype != FD_F32 && kv->dtype != FD_BF16) return FD_ERR_UNSUPPORTED;
  int n_eff = n_splits;
  const Groups gr = make_groups(Hq, Hkv, group_cap(kv->dtype));
  if (n_splits == 0 && (B > FD_AUTO_MAX_BATCH || (int64_t)B * gr.hv > kMaxFusedPairs))
    n_eff = fallback_splits(B, gr.hv, max_seq_len, grid_ctas);
  const WsLayout w = ws_layout(B, Hq, Hkv, D, n_eff, grid_ctas, group_cap(kv->dtype));
  if (workspace_bytes < w.total) return FD_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  float* q_dev = reinterpret_cast<float*>(ws + w.q_stage);
  float* out_dev = reinterpret_cast<float*>(ws + w.out_stage);
  float* lse_dev = reinterpret_cast<float*>(ws + w.lse_stage);
  int32_t* len_dev = reinterpret_cast<int32_t*>(ws + w.len_stage);
  const size_t qbytes = (size_t)B * Hq * D * 4;
  // Buffers in pinned host memory that the device can address are read and
  // written by the kernels in place, over the host link (no staging copy, no
  // copy back: on a coherent host link that is what a copy would move, with
  // one operation less on the stream); others go through the workspace.
  float* out_k = out_host;
  float* lse_k = lse_host;
  const float* q_k = nullptr;
  const int32_t* len_k = nullptr;
  if (!host_mapped(out_host, &out_k) || !aligned16(out_k)) out_k = nullptr;
  if (lse_host && !host_mapped(lse_host, &lse_k)) lse_k = nullptr;
  if (!host_mapped(q_host, &q_k) || !aligned16(q_k)) q_k = nullptr;
  if (seq_lens_host && !host_mapped(seq_lens_host, &len_k)) len_k = nullptr;
  if (!q_k && cudaMemcpyAsync(q_dev, q_host, qbytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return FD_ERR_CUDA;
  if (seq_lens_host && !len_k &&
      cudaMemcpyAsync(len_dev, seq_lens_host, (size_t)B * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FD_ERR_CUDA;
  st = fd_decode(q_k ? q_k : q_dev, kv, out_k ? out_k : out_dev, lse_host ? (lse_k ? lse_k : lse_dev) : nullptr, B,
                 Hq, Hkv, seq_lens_host ? (len_k ? len_k : len_dev) : nullptr,
                 max_seq_len, D, scale, n_splits, workspace, workspace_bytes, stream);
  if (st != FD_OK) return st;
  if (!out_k && cudaMemcpyAsync(out_host, out_dev, qbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FD_ERR_CUDA;
  if (lse_host && !lse_k &&
      cudaMemcpyAsync(lse_host, lse_dev, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FD_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

int64_t fd_plan_pieces(int32_t B, int32_t Hq, int32_t Hkv, int32_t kv_dtype, const int32_t* seq_lens_host,
                       int32_t max_seq_len, int32_t n_splits, int32_t grid, int32_t* pieces, int64_t capacity) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_seq_len < 0 || n_splits < 0) return -1;
  if (kv_dtype != FD_F32 && kv_dtype != FD_BF16) return -1;
  const Groups gr = make_groups(Hq, Hkv, group_cap(kv_dtype));
  std::vector<int32_t> ln(B);
  std::vector<int64_t> pre(B + 1, 0);
  for (int b = 0; b < B; ++b) ln[b] = clamp_len(seq_lens_host ? seq_lens_host[b] : max_seq_len, max_seq_len);
  // the kernels charge a piece per pair only when given per-sequence lengths
  const int32_t piece = seq_lens_host ? kPieceUnits : 0;
  for (int b = 0; b < B; ++b) pre[b + 1] = pre[b] + pair_units(ceil_div(ln[b], kPlanTile), piece);
  int64_t count = 0;
  auto emit = [&](int32_t cta, const Piece& pc, int32_t npieces) {
    if (pieces && count < capacity) {
      int32_t* r = pieces + count * 7;
      r[0] = cta;
      r[1] = pc.b;
      r[2] = pc.vkv;
      r[3] = pc.tok_begin;
      r[4] = pc.tok_end;
      r[5] = pc.slot;
      r[6] = npieces;
    }
    ++count;
  };
  if (n_splits == 0) {
    if (grid < 1) return -1;
    HostTiles tl{pre.data(), ln.data(), piece};
    const int64_t total = (int64_t)gr.hv * pre[B];
    if (total == 0) return 0;
    const int32_t used = balanced_ctas(total, grid);
    for (int32_t cta = 0; cta < used; ++cta) {
      BalancedWalk<HostTiles> w(tl, B, gr.hv, total, used, cta);
      Piece pc;
      while (w.next(pc)) {
        int32_t first, last;
        balanced_pair_ctas(tl, gr.hv, total, used, pc.b, pc.vkv, &first, &last);
        emit(cta, pc, last - first + 1);
      }
    }
  } else {
    const int32_t S = max_seq_len > 0 ? explicit_split_size(max_seq_len, n_splits) : kSplitAlign;
    for (int32_t pair = 0; pair < B * gr.hv; ++pair) {
      for (int32_t s = 0; s < n_splits; ++s) {
        Piece pc;
        pc.b = pair / gr.hv;
        pc.vkv = pair % gr.hv;
        const int64_t L = ln[pc.b];
        const int64_t lo = (int64_t)s * S;
        const int64_t hi = std::min<int64_t>(lo + S, L);
        pc.tok_begin = (int32_t)std::min<int64_t>(lo, L);
        pc.tok_end = (int32_t)std::max<int64_t>(hi, pc.tok_begin);
        pc.slot = s;
        pc.len = (int32_t)L;
        emit(pair * n_splits + s, pc, n_splits);
      }
    }
  }
  return count;
}

}  // extern "C"

// --------------------------------------------------------------------------
// fd_decode_static: fd_decode for callers that cannot allocate device memory.
//
// The scratch that fd_decode takes from the caller's workspace (error word,
// arrival counters, split partials) lives here in one file-scope device array
// instead.  It is loaded with the library, so every GPU that loads the library
// holds these bytes until the process exits.
namespace {

constexpr size_t kStaticScratchBytes = (size_t)FD_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  The host-side
// symbol is only a stand-in and must never reach a kernel; the address is
// looked up on every call (cheap once the library's module is loaded on the
// device), so a context that was torn down and created again is never handed
// a stale address.
fd_status static_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FD_ERR_CUDA;
  *out = p;
  return FD_OK;
}

}  // namespace

extern "C" fd_status fd_decode_static(const float* q, const fd_kv_desc* kv, float* out, float* lse, int32_t B,
                                      int32_t Hq, int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len,
                                      int32_t D, float scale, int32_t n_splits, void* stream) {
  fd_status st = check_shape(B, Hq, Hkv, D);
  if (st != FD_OK) return st;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FD_ERR_INVALID_ARG;
  if (n_splits < 0 || n_splits > 65535) return FD_ERR_INVALID_ARG;
  if ((st = check_kv(kv, B, Hkv, max_seq_len)) != FD_OK) return st;
  const Groups gr = make_groups(Hq, Hkv, group_cap(kv->dtype));
  const int64_t pairs = (int64_t)B * gr.hv;
  int sms = 0;
  if (n_splits == 0) {
    if (!sm_count(&sms)) return FD_ERR_CUDA;
    if (B > FD_AUTO_MAX_BATCH || pairs > kMaxFusedPairs) n_splits = fallback_splits(B, gr.hv, max_seq_len, sms);
  }
  const WsLayout w = ws_layout(B, Hq, Hkv, D, n_splits, sms, group_cap(kv->dtype));
  // Only the scratch part of the layout is used here (no host staging area).
  if (w.q_stage > kStaticScratchBytes) return FD_ERR_WORKSPACE_TOO_SMALL;
  void* base = nullptr;
  if ((st = static_scratch(&base)) != FD_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(base);
  cudaStream_t s = (cudaStream_t)stream;
  // The array keeps the previous call's contents; the error word and the
  // arrival counters must start at zero.
  if (cudaMemsetAsync(ws, 0, w.o, s) != cudaSuccess) return FD_ERR_CUDA;

  SplitParams p = base_params(q, kv, B, Hq, Hkv, seq_lens, max_seq_len, scale);
  p.out = out;
  p.lse = lse;
  p.o_part = reinterpret_cast<float*>(ws + w.o);
  p.m_part = reinterpret_cast<float*>(ws + w.m);
  p.l_part = reinterpret_cast<float*>(ws + w.l);
  p.err = reinterpret_cast<unsigned*>(ws + w.err);
  if (n_splits == 0) {
    p.n_splits = 0;
    p.counters = reinterpret_cast<int*>(ws + w.counters);
    return launch(kv, D, p, dim3((unsigned)sms, 1, 1), s);
  }
  p.n_splits = n_splits;
  p.split_tokens = max_seq_len > 0 ? explicit_split_size(max_seq_len, n_splits) : kSplitAlign;
  const dim3 grid((unsigned)pairs, (unsigned)n_splits, 1);
  if (pairs <= kMaxFusedPairs) {
    p.counters = reinterpret_cast<int*>(ws + w.counters);
    return launch(kv, D, p, grid, s);
  }
  p.counters = nullptr;
  if ((st = launch(kv, D, p, grid, s)) != FD_OK) return st;
  const cudaError_t e = launch_combine(D, p.o_part, p.m_part, p.l_part, out, lse, B * Hq, n_splits, s);
  return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

extern "C" fd_status fd_static_status(void* stream) {
  void* base = nullptr;
  fd_status st = static_scratch(&base);
  if (st != FD_OK) return st;
  // the error word sits at the start of the array, where fd_decode_static puts
  // the workspace header
  return fd_workspace_status(base, kHeaderBytes, stream);
}
