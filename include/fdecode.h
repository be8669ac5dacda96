/*
 * fdecode.h -- C ABI of libfdecode: split-KV decode attention (Flash-Decoding)
 * for NVIDIA GB300 (sm_103a).
 *
 * What is computed (per batch b and query head h, one query row each):
 *
 *     out[b,h,:] = softmax(scale * q[b,h,:] . K_b^T) . V_b     over keys t < L_b
 *     lse[b,h]   = ln sum_t exp(scale * q[b,h,:] . k_t)
 *
 * The KV sequence is cut into splits; each split runs an online softmax and
 * leaves an unnormalised partial output O_s with its running max m_s and sum
 * l_s; a log-sum-exp merge rescales each partial by exp(m_s - M), sums, and
 * divides once by the global sum.  Sources, by page and section:
 *   - "Kernel visualization: Flash Decoding" (tinyvolt.com): the fd_split
 *     walkthrough (per-split online softmax, partials written unnormalised)
 *     and "Combine kernel -- one thread block per (batch, head)" (the merge);
 *   - "attn-flash-decoding" (zenaique.com): "What decode looks like" (shapes
 *     Q (batch, n_heads, 1, d_head), K/V (batch, n_kv_heads, T, d_head)) and
 *     the answer on why the log-sum-exp combine is exact;
 *   - "FlashDecoding and split-KV" (guide.dupenodi.dev), "Walking through it":
 *     paged or ragged KV layouts and GQA head grouping.
 *
 * Conventions fixed by this library where the pages are silent:
 *   - GQA: g = Hq / Hkv; query head h reads KV head h / g (integer division).
 *   - lse is a natural log; m_part is in the natural units of scale*q.k.
 *   - L_b == 0 gives out = 0 and lse = -inf.  Keys at t >= L_b (padding, and
 *     block-table entries at index >= ceil(L_b / page_size)) are never read.
 *   - Paged pool layout [num_pages, Hkv, page_size, D]: token t of sequence b
 *     is row t % page_size of page block_table[b * max_pages_per_seq + t / page_size].
 *
 * General rules for every call:
 *   - Pointers are DEVICE pointers unless the name ends in _host.
 *   - All memory is owned by the caller; the library allocates nothing.  The
 *     one exception is the fixed FD_STATIC_SCRATCH_BYTES device array that
 *     fd_decode_static uses in place of a workspace (see there).
 *   - Calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return without waiting, except fd_decode_host and
 *     fd_workspace_status, which synchronise the stream.
 *   - Arguments are checked on the host before anything is enqueued; on an
 *     error no kernel is launched and no memory is touched.
 *   - Supported: D in {64, 128}; K/V in FD_BF16 or FD_F32; q, out, lse, partials
 *     in fp32; Hq % Hkv == 0; page_size a multiple of 16.  q, out, o_part, k, v
 *     must be 16-byte aligned; q/out/partials are dense row-major.
 *   - Results are deterministic: no floating-point atomics; repeated calls
 *     give bit-identical outputs.
 */
#ifndef FDECODE_H_
#define FDECODE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FD_API __attribute__((visibility("default")))
#else
#define FD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fd_status {
  FD_OK = 0,
  FD_ERR_INVALID_ARG = 1,         /* null pointer, bad size, misalignment, Hq % Hkv != 0 ... */
  FD_ERR_UNSUPPORTED = 2,         /* head_dim, dtype or size outside what this build handles */
  FD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < fd_workspace_bytes(...) */
  FD_ERR_BAD_INDEX = 4,           /* a kernel met a block-table entry outside [0, num_pages) */
  FD_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed (launch, copy, ...) */
  FD_ERR_TIMEOUT = 6              /* a kernel's internal wait gave up (never expected) */
} fd_status;

typedef enum fd_dtype { FD_F32 = 0, FD_BF16 = 1 } fd_dtype;

typedef enum fd_kv_layout { FD_KV_CONTIGUOUS = 0, FD_KV_PAGED = 1 } fd_kv_layout;

/* n_splits value asking the library to plan the split itself (balanced over the SMs). */
#define FD_SPLITS_AUTO 0

/*
 * Largest batch the balanced (FD_SPLITS_AUTO) plan handles in one fused
 * launch; larger batches, or more than 65536 (batch, KV head) pairs, are run
 * with a fixed split count chosen by the library instead.
 */
#define FD_AUTO_MAX_BATCH 1024

/*
 * The KV cache.  All pointers are device pointers.
 *   contiguous: k, v are [B, Hkv, capacity, D]; block_table etc. are ignored.
 *   paged:      k, v are [num_pages, Hkv, page_size, D]; block_table is
 *               [B, max_pages_per_seq] int32, row-major; capacity is ignored.
 */
typedef struct fd_kv_desc {
  fd_kv_layout layout;
  fd_dtype dtype;               /* element type of k and v */
  const void* k;
  const void* v;
  int64_t capacity;             /* contiguous: padded length T_cap of every sequence */
  const int32_t* block_table;   /* paged only */
  int32_t max_pages_per_seq;    /* paged only: row length of block_table */
  int32_t page_size;            /* paged only: tokens per page, multiple of 16 */
  int32_t num_pages;            /* paged only: pages in the pool */
} fd_kv_desc;

/*
 * Bytes of device workspace needed by fd_decode and fd_decode_host.
 * n_splits: FD_SPLITS_AUTO or the explicit split count that will be passed.
 * num_sms:  SM count of the device that will run the call; 0 = query the
 *           current device.  Returns 0 for invalid arguments.
 * The workspace must be zero-filled once after allocation (fd_workspace_init);
 * every successful call, of any shape, leaves it valid for the next call (the
 * merge's arrival counters sit in a fixed-size region and end each call at
 * zero).  One workspace serves one call at a time: calls that share a
 * workspace must be ordered (same stream, or synchronised).
 */
FD_API size_t fd_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_splits,
                          int32_t num_sms);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
FD_API fd_status fd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronise `stream`, then report (and clear) the error word that kernels
 * of earlier calls on this workspace may have raised: FD_OK, FD_ERR_BAD_INDEX
 * or FD_ERR_TIMEOUT.  Kernels never trap; they record and skip instead.
 */
FD_API fd_status fd_workspace_status(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Tokens per split when the caller fixes n_splits > 0:
 *   S = 16 * ceil(ceil(max_seq_len / n_splits) / 16);
 * split s of sequence b covers tokens [s*S, min((s+1)*S, L_b)).
 * (The fd_split sketch takes the split size S as a parameter with
 * n_start = s*S, n_end = min(n_start + S, N).)  Returns 0 on bad arguments.
 */
FD_API int32_t fd_split_size(int32_t max_seq_len, int32_t n_splits);

/*
 * Full decode attention: split + merge, enqueued on `stream`.
 *   q        [B, Hq, D] fp32.
 *   out      [B, Hq, D] fp32 (written).
 *   lse      [B, Hq] fp32 natural-log softmax denominator, or NULL.
 *   seq_lens [B] int32 valid lengths L_b, or NULL (= every L_b is max_seq_len).
 *            Values are clamped to [0, max_seq_len] on the device.
 *   max_seq_len  upper bound of every L_b; contiguous: <= capacity;
 *            paged: <= max_pages_per_seq * page_size.
 *   scale    multiplies q.k (callers usually pass 1/sqrt(D)).
 *   n_splits FD_SPLITS_AUTO (the library balances the keys of all
 *            sequences over one CTA per SM) or the number of splits per sequence.
 *   workspace/workspace_bytes  zero-initialised device scratch of at least
 *            fd_workspace_bytes(B, Hq, Hkv, D, n_splits, 0) bytes.
 * One kernel launch (split with the merge fused in: the last CTA to finish a
 * sequence merges it); two launches only when more than 65536 (batch, KV head)
 * pairs need merging.  Errors in arguments return before any launch.
 */
FD_API fd_status fd_decode(const float* q, const fd_kv_desc* kv, float* out, float* lse, int32_t B,
                    int32_t Hq, int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len, int32_t D,
                    float scale, int32_t n_splits, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Decode with n_q query rows per (batch, head) sharing one read of K/V, for a
 * few new tokens per sequence (e.g. verifying speculative tokens): the page
 * "FlashDecoding and split-KV", section "Walking through it", lets decode carry
 * n_q slightly above one and leaves the masking of those rows open.
 *   q    [B, Hq, n_q, D] fp32; out [B, Hq, n_q, D]; lse [B, Hq, n_q] or NULL.
 *   causal = 1: the n_q rows are the last n_q tokens, already in the cache, and
 *            row i attends keys t < L_b - (n_q - 1 - i); causal = 0: every row
 *            attends all L_b keys.  A row with no key gives out = 0, lse = -inf.
 *   1 <= n_q <= 64.  Other arguments as in fd_decode; the workspace is
 *   fd_workspace_bytes(B, Hq * n_q, Hkv, D, n_splits, 0).  The rows of a GQA
 *   group are served together (up to 16 rows x heads per bf16 K/V read, 8 per
 *   fp32 read).
 */
FD_API fd_status fd_decode_rows(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out,
                                float* lse, int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens,
                                int32_t max_seq_len, int32_t D, float scale, int32_t n_splits, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Fused append-KV + decode (the "fused append-KV" path named in "FlashDecoding
 * and split-KV", section "Walking through it"; the operation is this
 * library's reading of it): for every sequence b the new token's key and
 * value are written into the cache at position L_b and the decode then
 * attends the L_b + 1 keys, in one launch.  The result equals writing the row
 * first and calling fd_decode with lengths L_b + 1 (bit for bit).
 *   k_new, v_new  [B, Hkv, D] device, in the cache dtype (kv->dtype), 16-byte
 *                 aligned; their bits are stored unchanged.
 *   seq_lens / max_seq_len  the lengths BEFORE the append (seq_lens is read,
 *                 not updated: the caller advances its lengths).
 *   kv            kv->k and kv->v are written (one row per (b, KV head)).
 *                 Contiguous: capacity >= max_seq_len + 1.  Paged: the page
 *                 holding position L_b must already be in the block table;
 *                 an entry outside [0, num_pages) skips the cache write and
 *                 is reported as FD_ERR_BAD_INDEX by fd_workspace_status (the
 *                 output still includes the new token).
 *   Other arguments as in fd_decode; the workspace is the same size.
 */
FD_API fd_status fd_append_decode(const float* q, const void* k_new, const void* v_new, const fd_kv_desc* kv,
                                  float* out, float* lse, int32_t B, int32_t Hq, int32_t Hkv,
                                  const int32_t* seq_lens, int32_t max_seq_len, int32_t D, float scale,
                                  int32_t n_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention for many query rows per sequence (prefill, or a long window of new
 * tokens): the same operation as fd_decode_rows -- q [B, Hq, n_q, D], the rows
 * are the last n_q tokens of each sequence, causal or not -- computed with
 * query tiles of 128 rows on the tensor cores (tcgen05.mma, TMEM
 * accumulators) instead of rows-as-heads.  "FlashDecoding and split-KV",
 * section "Walking through it": prefill has many query rows and wants
 * FlashAttention's tiling along them; decode has one.
 *   Supports D = 64 and 128 with a bf16 cache (contiguous or paged); any n_q >= 1.
 *   workspace: at least 256 bytes, zero-filled once (its first word is the
 *   kernels' error word, read by fd_workspace_status; bytes 128-135 hold the
 *   kernel's work-queue counters, which every call leaves at zero, so calls
 *   that share a workspace must not overlap in time).  out, lse as in
 *   fd_decode_rows.  One launch, asynchronous on `stream`.
 *   FD_ERR_CUDA, with nothing launched, also when the kernel variant for an odd
 *   group size (one query head per CTA, which redistributes registers between
 *   its warps) was not compiled with the register count it assumes.
 */
FD_API fd_status fd_prefill(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out,
                            float* lse, int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens,
                            int32_t max_seq_len, int32_t D, float scale, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Phase dispatch ("FlashDecoding and split-KV", "Walking through it": serving
 * engines pick a kernel per phase and should log which one ran).  fd_attend
 * picks the backend for n_q query rows per sequence and reports it:
 *   FD_BACKEND_DECODE       n_q == 1                      -> fd_decode
 *   FD_BACKEND_DECODE_ROWS  n_q * (Hq / Hkv) <= 16, or no prefill kernel for
 *                           this D / dtype and n_q <= 64  -> fd_decode_rows
 *   FD_BACKEND_PREFILL      otherwise (D = 64 or 128, bf16) -> fd_prefill
 * fd_attend_backend returns the choice without running anything (-1: no
 * backend); fd_backend_name names it.  The workspace must fit the chosen
 * backend: fd_workspace_bytes(B, Hq * n_q, Hkv, D, n_splits, 0) for the decode
 * backends, 256 bytes for prefill.  *backend (may be NULL) receives the choice.
 */
#define FD_BACKEND_DECODE 0
#define FD_BACKEND_DECODE_ROWS 1
#define FD_BACKEND_PREFILL 2
FD_API int32_t fd_attend_backend(int32_t n_q, int32_t Hq, int32_t Hkv, int32_t D, int32_t kv_dtype);
FD_API const char* fd_backend_name(int32_t backend);
FD_API fd_status fd_attend(const float* q, int32_t n_q, int32_t causal, const fd_kv_desc* kv, float* out,
                           float* lse, int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t D, float scale, int32_t n_splits, void* workspace,
                           size_t workspace_bytes, void* stream, int32_t* backend);

/*
 * Split step only ("fd_split" of the walkthrough), with n_splits > 0 splits
 * per sequence of fd_split_size(max_seq_len, n_splits) tokens each.  Writes:
 *   o_part [B, Hq, n_splits, D]  unnormalised sum_t exp(s_t - m_s) v_t
 *   m_part [B, Hq, n_splits]     running max m_s of scale*q.k (natural units)
 *   l_part [B, Hq, n_splits]     sum_t exp(s_t - m_s)
 * A split with no keys holds O = 0, m = -inf, l = 0.  Other arguments as in
 * fd_decode.  Needs no workspace.
 */
FD_API fd_status fd_split_partial(const float* q, const fd_kv_desc* kv, int32_t B, int32_t Hq, int32_t Hkv,
                           const int32_t* seq_lens, int32_t max_seq_len, int32_t D, float scale,
                           int32_t n_splits, float* o_part, float* m_part, float* l_part,
                           void* stream);

/*
 * Merge step only (the combine walkthrough): per (b, h), over splits with
 * l > 0:  M = max m_s,  L = sum exp(m_s - M) l_s,
 *         out = sum exp(m_s - M) O_s / L,  lse = M + ln L  (lse may be NULL).
 * If no split has keys: out = 0, lse = -inf.  Layouts as in fd_split_partial.
 */
FD_API fd_status fd_combine(const float* o_part, const float* m_part, const float* l_part, float* out,
                     float* lse, int32_t B, int32_t Hq, int32_t D, int32_t n_splits, void* stream);

/*
 * fd_decode with the per-step inputs and outputs in HOST memory: q_host
 * [B,Hq,D], seq_lens_host [B] (or NULL), out_host [B,Hq,D] and lse_host
 * [B,Hq] (or NULL).  Pinned (page-locked, device-mapped) buffers are used in
 * place: the kernels read q and the lengths and write out and lse over the
 * host link, with no staging copy (q_host and out_host must then start on a
 * 16-byte boundary, else they are staged).  Pageable buffers are copied
 * through the staging area inside `workspace` (q and lengths in, out and lse
 * back).  Synchronises `stream` before returning, so the host may rewrite
 * q_host and seq_lens_host as soon as the call returns.  The KV cache (kv)
 * stays device-resident.  Workspace as for fd_decode.
 */
FD_API fd_status fd_decode_host(const float* q_host, const fd_kv_desc* kv, float* out_host, float* lse_host,
                         int32_t B, int32_t Hq, int32_t Hkv, const int32_t* seq_lens_host,
                         int32_t max_seq_len, int32_t D, float scale, int32_t n_splits,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * fd_decode without a workspace, for callers that cannot allocate device
 * memory: code handed only its input and output buffers by a host framework
 * (plugin or custom-operator interfaces that own every allocation), and code
 * that must not call cudaMalloc on its path because cudaMalloc can synchronise
 * the device and stall work running on other streams.  The pages have no
 * counterpart to this call; it is a deployment variant of fd_decode.
 *   Arguments as in fd_decode, minus the workspace.  The scratch (error word,
 *   merge counters, split partials) is one file-scope device array of
 *   FD_STATIC_SCRATCH_BYTES inside the library; every GPU that loads the
 *   library holds it until the process exits.
 *   Every call looks the array's device address up on the current device
 *   (cudaGetSymbolAddress); the first call on a device also loads the
 *   library's module there, so make that first call before any stream capture.
 *   Returns FD_ERR_WORKSPACE_TOO_SMALL, before any launch, when the problem
 *   needs more scratch than the array holds (fd_workspace_bytes of the same
 *   problem, minus its host-staging part, is the amount needed).
 *   Allocates nothing: no cudaMalloc or cudaFree.  Each call clears the error
 *   word and the counters (cudaMemsetAsync) and then launches as fd_decode.
 *   All calls share the one array, and it keeps the last call's contents:
 *   calls that overlap on the GPU (different streams, other host threads)
 *   race on it and must be ordered by the caller.
 *   Kernel-side errors (a block-table entry outside the pool, a wait that
 *   gave up) are recorded in the array's error word: read them with
 *   fd_static_status after the call and before the next fd_decode_static
 *   call on that device, which clears the word.
 */
#define FD_STATIC_SCRATCH_BYTES (16u << 20)

FD_API fd_status fd_decode_static(const float* q, const fd_kv_desc* kv, float* out, float* lse, int32_t B,
                                  int32_t Hq, int32_t Hkv, const int32_t* seq_lens, int32_t max_seq_len,
                                  int32_t D, float scale, int32_t n_splits, void* stream);

/*
 * fd_workspace_status for fd_decode_static: synchronise `stream`, then report
 * (and clear) the error word in the library's static scratch array on the
 * current device -- FD_OK, FD_ERR_BAD_INDEX or FD_ERR_TIMEOUT, raised by the
 * kernels of the most recent fd_decode_static call there.  Like that call it
 * has no counterpart on the pages and allocates nothing.
 */
FD_API fd_status fd_static_status(void* stream);

/*
 * Host-side description of the work decomposition, for inspection and tests
 * (touches no GPU).  Enumerates every split piece that fd_decode would run
 * for these lengths on `grid` CTAs (FD_SPLITS_AUTO) or for n_splits > 0, for
 * a cache of dtype kv_dtype (an fd_dtype).
 * Each piece is 7 int32: {cta, b, virtual_kv_head, tok_begin, tok_end, slot,
 * pieces_of_its_sequence} (the last is the arrival count that triggers the
 * fused merge).  A virtual KV head is a KV head with up to 16 (bf16 cache) or
 * 8 (fp32 cache) of its query heads; when Hq / Hkv is at most that, it is the
 * KV head itself.
 * Writes at most `capacity` pieces and returns the total count (negative on
 * bad arguments).  seq_lens_host may be NULL (every L_b = max_seq_len).
 */
FD_API int64_t fd_plan_pieces(int32_t B, int32_t Hq, int32_t Hkv, int32_t kv_dtype, const int32_t* seq_lens_host,
                              int32_t max_seq_len, int32_t n_splits, int32_t grid, int32_t* pieces,
                              int64_t capacity);

/*
 * Testing hook for the kernels' bounded waits; off by default.  Every
 * mbarrier wait of the split and prefill kernels gives up after a time limit
 * (2 s by default), records FD_ERR_TIMEOUT in the error word, lets the copies
 * it issued land and exits, so the context stays usable.  With stage >= 0, the
 * kernels launched afterwards skip, in every CTA that reaches it, the copies of
 * stage number `stage` (split kernels: fd_decode and every call built on it,
 * fd_split_partial) or K/V tile copy number `stage` (fd_prefill, K and V
 * counted separately), so the waits for it run out; wait_limit_ns > 0 shortens
 * every wait of those kernels to that many nanoseconds (0 keeps the default).  The
 * call's output is then undefined and fd_workspace_status (or
 * fd_static_status) reports FD_ERR_TIMEOUT; the workspace stays valid for the
 * next call.  stage < 0 switches the hook off and restores the default limit.
 * A process-wide setting, read when a call is made.
 */
FD_API void fd_debug_stall(int32_t stage, int64_t wait_limit_ns);

/* Static description of a status code. */
FD_API const char* fd_status_string(fd_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
FD_API int32_t fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FDECODE_H_ */
