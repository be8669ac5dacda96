// fd_split.cuh -- the split-KV decode kernel for sm_103a (GB300).
//
// One CTA streams K/V for one (batch, KV head) run of keys -- or, in the
// balanced plan, a fixed share of all runs -- and serves every query head of
// the GQA group from that single read.  Per CTA:
//
//   warp W (producer): walks the CTA's pieces and, per stage of kBT keys,
//     issues 16-row x 128-byte TMA boxes of K and V into a ring of kStages
//     shared-memory stages (128-byte swizzle), plus one bulk copy of the
//     piece's q rows.  mbarriers carry the byte counts.
//   warps 0..W-1 (consumers): warp w owns rows [32w, 32w+32) of every stage.
//     q.k:  lane = key row; the lane walks its row in 16-byte chunks (the
//           swizzle makes the 8 rows of each quarter-warp hit distinct banks)
//           while q is read from shared memory as a broadcast;
//     softmax: per warp and head, max over the 32 rows, one exp2 per row;
//           each warp keeps its own running (m, l, O) -- the online softmax
//           of the fd_split walkthrough, one level per warp;
//     p.V:  lane = a D/32-wide slice of the output; the warp walks the valid
//           rows with p broadcast from shared memory.
//   At the end of a piece the W warp states are merged in shared memory with
//   the log-sum-exp rule, giving the piece's (O, m, l).  A piece that covers
//   its whole sequence is normalised and written as the output directly;
//   otherwise its partial is written and, when the merge is fused, the last
//   CTA to finish a sequence merges all of its partials (arrival counter,
//   no waiting on other CTAs).
//
// Scores are kept in base 2 (q.k times scale*log2 e); m written to memory is
// converted back to natural units.  Masking is by index only: rows past the
// valid length get score -inf and are skipped in p.V, so nothing stored there
// (even NaN) reaches a sum.
#pragma once

#include <cuda_bf16.h>

#include "fd_device.cuh"
#include "fd_plan.h"

#ifndef FD_USE_FFMA2
#define FD_USE_FFMA2 1
#endif

namespace fdk {

constexpr int kAutoMaxBatch = 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct SplitParams {
  const float* q;          // [B, Hq, D]
  float* out;              // [B, Hq, D]      (fused merge only)
  float* lse;              // [B, Hq] or null (fused merge only)
  float* o_part;           // balanced: [slots, gpad, D]; explicit: [B, Hq, n_splits, D]
  float* m_part;           // balanced: [slots, gpad];    explicit: [B, Hq, n_splits]
  float* l_part;
  int* counters;           // [B * hv] arrival counters; null = write partials only
  unsigned* err;           // error word or null
  const int32_t* seq_lens; // [B] or null
  const int32_t* block_table;
  int32_t B, Hq, Hkv;
  int32_t g, gpad, nsub, hv;
  int32_t max_len;
  int32_t n_splits;        // 0 = balanced plan
  int32_t split_tokens;    // explicit plan: S
  int32_t paged;
  int32_t page_size, max_pages, num_pages;
  float qk_scale;          // scale * log2(e)
  int32_t n_q;             // query rows per (b, head): virtual head h' = head * n_q + row
  int32_t causal;          // rows see keys t < L_b - (n_q - 1 - row) (else all L_b keys)
  // Fused append: the new token's k/v ([B, Hkv, D], cache dtype) join every
  // sequence at position L_b (seq_lens are the lengths before the append; the
  // plan sees L_b + 1) and are written into the cache at that position.
  int32_t append;
  const void* k_new;
  const void* v_new;
  void* k_cache;           // the cache's K and V base pointers (pool when paged)
  void* v_cache;
  int64_t capacity;        // contiguous: rows per (b, KV head)
  // Bounded waits: every mbarrier wait gives up after wait_ns (0 = kWaitLimitNs).
  // Testing hook: stall_it >= 0 makes the producer of every CTA skip the copies
  // of its stage number stall_it, so that the consumers' wait on it runs out.
  uint64_t wait_ns;
  int32_t stall_it;
};

__device__ __forceinline__ unsigned long long wait_limit(const SplitParams& p) {
  return p.wait_ns ? (unsigned long long)p.wait_ns : kWaitLimitNs;
}

// Keys seen by the heads of one piece: head0 + j for j < nh; virtual head
// h' = head * n_q + row sees keys t < len - (n_q - 1 - row) when causal.
struct RowLimits {
  int32_t head0, nh, len, n_q, causal;
  __device__ __forceinline__ int32_t operator()(int32_t j) const {
    if (j >= nh) return 0;
    if (!causal || n_q <= 1) return len;
    const int32_t lim = len - (n_q - 1 - (head0 + j) % n_q);
    return lim < 0 ? 0 : lim;
  }
};

template <int D_, class KV, int G_>
struct SplitCfg {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int kEs = (int)sizeof(KV);
  static constexpr bool kBf16 = kEs == 2;
  static constexpr int kRowBytes = D * kEs;
  static constexpr int kNB = kRowBytes / 128;  // 128-byte column blocks per row
  static constexpr int kWarps = kRowBytes <= 256 ? 4 : 2;
  static constexpr int kThreads = 32 * (kWarps + 1);
  static constexpr int kBT = 32 * kWarps;      // keys per stage
  static constexpr int kTileBytes = kBT * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStagesFit = 196608 / kStageBytes;
  static constexpr int kStages = kStagesFit > 4 ? 4 : kStagesFit;
  static constexpr int kEPL = D / 32;          // output elements per lane in p.V
  static constexpr int kChunkElems = 16 / kEs; // elements per 16-byte chunk
  static constexpr int kChunks = kRowBytes / 16; // 16-byte chunks per row
  // Independent q.k accumulator chains per head: eight chains in all keep the
  // packed FMAs of one lane from waiting on each other.
  static constexpr int kAcc = G >= 8 ? 1 : 8 / G;
  static constexpr int kBoxBytes = 16 * 128;

  // bf16 caches with four or more query heads per CTA run q.k and p.V on
  // mma.sync; there the CUDA-core FMAs (and bf16 widening) bound the kernel
  // well above its streaming time, while one or two heads per CTA stay cheap.
  static constexpr bool kMma = kBf16 && G >= 4;
  // Sixteen heads per CTA (bf16 only): each lane's MMA fragments carry two
  // heads.  q lives in registers after the first read, so one q buffer is
  // enough (released as soon as every warp has its fragments), and the warp
  // states are merged eight heads at a time to keep the merge buffer small.
  static constexpr bool kWide = G > 8;
  static constexpr int kQBufs = kWide ? 1 : 2;
  static constexpr int kPubHeads = kWide ? 8 : G;  // heads per merge round
  static_assert(!kWide || (kBf16 && G == 16), "sixteen heads per CTA need a bf16 cache");
  static_assert(kNB >= 1 && kStages >= 2, "unsupported row size");

  // shared-memory layout (byte offsets from a 1024-aligned base)
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kQBytes = G * D * 4;
  static constexpr int kUOff = kQOff + kQBufs * kQBytes;
  static constexpr int kPBytes = kMma ? 0 : kWarps * 32 * G * 8;  // CUDA-core engine's p rows
  // Warp states are published in rows of kObStride floats: the padding keeps
  // the MMA engines' float2 stores (eight heads of one warp at a time) off
  // each other's banks.
  static constexpr int kObStride = D + 8;
  static constexpr int kObBytes = kWarps * kPubHeads * kObStride * 4;
  static constexpr int kWsBytes = kWarps * 128 * 4;  // merge_head weight scratch (fused merge)
  static constexpr int kUBytes0 = kPBytes > kObBytes ? kPBytes : kObBytes;
  static constexpr int kUBytes = kUBytes0 > kWsBytes ? kUBytes0 : kWsBytes;
  static constexpr int kMlOff = kUOff + kUBytes;
  static constexpr int kFinOff = kMlOff + kWarps * kPubHeads * 8;
  static constexpr int kLenOff = kFinOff + kPubHeads * 8;
  static constexpr int kPreOff = kLenOff + (kAutoMaxBatch + 4) * 4;
  static constexpr int kBarOff = kPreOff + (kAutoMaxBatch + 4) * 4;
  static constexpr int kFlagOff = kBarOff + (2 * kStages + 6) * 8;
  static constexpr int kDescOff = (kFlagOff + 16 + 15) / 16 * 16;  // PieceDesc per q slot
  static constexpr int kBytes = kDescOff + 2 * 48;
  static constexpr int kSmemAlloc = kBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory over the sm_100 limit");
};

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
#if FD_USE_FFMA2
  return __ffma2_rn(a, b, c);
#else
  return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
#endif
}

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// Lengths and per-sequence tile counts seen by every thread of a CTA.
struct CtaTiles {
  const int32_t* pre;  // shared: cost-unit prefix per sequence, per pair (balanced with lengths)
  const int32_t* ln;   // shared: clamped lengths
  int32_t ut, ul;      // uniform tile count / length when no lengths are given
  int uniform;
  FD_HD int32_t piece() const { return uniform ? 0 : kPieceUnits; }
  FD_HD int64_t prefix(int32_t b) const { return uniform ? (int64_t)b * pair_units(ut, 0) : pre[b]; }
  FD_HD int32_t tiles(int32_t b) const { return uniform ? ut : ceil_div(ln[b], kPlanTile); }
  FD_HD int32_t len(int32_t b) const { return uniform ? ul : ln[b]; }
};

// Log-sum-exp merge of `count` split states of one head (the combine
// walkthrough), by one warp.  The states come from a partials source P:
// P::m(k), P::l(k) and P::slice(k, lane, v) (this lane's D/32 elements of
// O_k); GlobalPartials reads them from the workspace (L2).  `wsm` is the
// warp's scratch of 128 floats in shared memory (16-byte aligned).  The loads are issued in
// batches so that the merge costs a few round trips rather than one per
// split.  Summation order is fixed: per output element, four partial sums
// over k = 0, 1, 2, 3 (mod 4) in increasing k, then ((s0 + s1) + s2) + s3 --
// bit-reproducible, and the same in the fused merge and in fd_combine, which
// therefore give identical bits.
template <int D>
__device__ __forceinline__ void load_slice(const float* row, float (&v)[D / 32]) {
  if constexpr (D / 32 == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(row));
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(row));
    v[0] = x.x;
    v[1] = x.y;
  }
}

// Split k of one head at o + (base + k*stride)*D, m/l + base + k*stride.
template <int D>
struct GlobalPartials {
  const float *o, *m_, *l_;
  size_t base, stride;
  __device__ __forceinline__ float m(int k) const { return __ldcg(m_ + base + (size_t)k * stride); }
  __device__ __forceinline__ float l(int k) const { return __ldcg(l_ + base + (size_t)k * stride); }
  __device__ __forceinline__ void slice(int k, int lane, float (&v)[D / 32]) const {
    load_slice<D>(o + (base + (size_t)k * stride) * D + lane * (D / 32), v);
  }
};

// The merge's weights, computed by one warp for one head: lane holds the split
// states k = r*32 + lane (r < kMergeKR) as (mk[r], lk[r]), with l = 0 for k at
// or past the count.  `mx` is the largest m over splits with l > 0 (already
// reduced over the warp); wk[r] = exp2((m_k - mx) log2 e) (0 for an empty
// split) and lsum is this lane's part of L = sum_k w_k l_k.  Shared by every
// merge path so that they give identical bits.
constexpr int kMergeKR = 4;

__device__ __forceinline__ float merge_max(const float (&mk)[kMergeKR], const float (&lk)[kMergeKR]) {
  float mx = -INFINITY;
#pragma unroll
  for (int r = 0; r < kMergeKR; ++r)
    if (lk[r] > 0.f) mx = fmaxf(mx, mk[r]);
  return mx;
}

__device__ __forceinline__ float merge_weights(const float (&mk)[kMergeKR], const float (&lk)[kMergeKR], float mx,
                                               float (&wk)[kMergeKR]) {
  float lsum = 0.f;
#pragma unroll
  for (int r = 0; r < kMergeKR; ++r) {
    wk[r] = lk[r] > 0.f ? exp2f((mk[r] - mx) * kLog2e) : 0.f;
    lsum = fmaf(wk[r], lk[r], lsum);
  }
  return lsum;
}

template <int D, class P>
__device__ __forceinline__ void merge_head(const P& src, int count, float* out_row, float* lse_slot, int lane,
                                           float* wsm) {
  constexpr int EPL = D / 32;
  constexpr int KR = kMergeKR;          // splits per lane whose (m, l) stay in registers: count <= 128
  constexpr int NB = 128 / EPL;         // splits per batch of O loads (128 registers)
  // Round trip 1: every (m, l) and the first batch of O slices, all in flight together.
  float mk[KR], lk[KR];
#pragma unroll
  for (int r = 0; r < KR; ++r) {
    const int k = r * 32 + lane;
    mk[r] = -INFINITY;
    lk[r] = 0.f;
    if (k < count) {
      lk[r] = src.l(k);
      mk[r] = src.m(k);
    }
  }
  float v[NB][EPL];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[j][e] = 0.f;
    if (j < count) src.slice(j, lane, v[j]);
  }
  float mx = merge_max(mk, lk);
  for (int k = KR * 32 + lane; k < count; k += 32)
    if (src.l(k) > 0.f) mx = fmaxf(mx, src.m(k));
  mx = warp_max(mx);
  if (mx == -INFINITY) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out_row[lane * EPL + e] = 0.f;
    if (lse_slot && lane == 0) *lse_slot = -INFINITY;
    return;
  }
  float wk[KR];
  float lsum = merge_weights(mk, lk, mx, wk);
  for (int k = KR * 32 + lane; k < count; k += 32) {
    const float lv = src.l(k);
    if (lv > 0.f) lsum = fmaf(exp2f((src.m(k) - mx) * kLog2e), lv, lsum);
  }
  const float L = warp_sum(lsum);
  // weight of split k (< 128) at wsm[k]; 0 past `count` (there l = 0)
  __syncwarp();  // the warp's reads of an earlier merge are done
#pragma unroll
  for (int r = 0; r < KR; ++r) wsm[r * 32 + lane] = wk[r];
  __syncwarp();
  float acc[4][EPL];
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[s4][e] = 0.f;
  for (int k0 = 0; k0 < count; k0 += NB) {
    if (k0 > 0) {  // later batches
#pragma unroll
      for (int j = 0; j < NB; ++j) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[j][e] = 0.f;
        if (k0 + j < count) src.slice(k0 + j, lane, v[j]);
      }
    }
    // Weights four splits per shared-memory load (the warp's scratch), the
    // rest (count > 128) from the source.  Splits past `count` have w = 0 and
    // v = 0, and fmaf(0, 0, a) == a: the padding leaves the sums' bits as they are.
#pragma unroll
    for (int j4 = 0; j4 < NB; j4 += 4) {
      float w[4] = {0.f, 0.f, 0.f, 0.f};
      if (k0 + j4 < KR * 32) {
        const float4 x = *reinterpret_cast<const float4*>(wsm + k0 + j4);
        w[0] = x.x;
        w[1] = x.y;
        w[2] = x.z;
        w[3] = x.w;
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int k = k0 + j4 + jj;
          if (k < count) {
            const float lv = src.l(k);
            w[jj] = lv > 0.f ? exp2f((src.m(k) - mx) * kLog2e) : 0.f;
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          acc[(j4 + jj) & 3][e] = fmaf(w[jj], v[j4 + jj][e], acc[(j4 + jj) & 3][e]);
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) out_row[lane * EPL + e] = (((acc[0][e] + acc[1][e]) + acc[2][e]) + acc[3][e]) / L;
  if (lse_slot && lane == 0) *lse_slot = mx + logf(L);
}

// A piece as the producer announces it to the consumers: written to the
// shared-memory slot of the piece's q rows before the arrival on that slot's
// "q full" barrier, read by the consumers after their wait on it.  b < 0 ends
// the CTA's work.
struct PieceDesc {
  int32_t b, vkv, tok_begin, tok_end, slot, len;
  int32_t npieces;  // pieces of the sequence (b, vkv) over all CTAs: the arrival count
  int32_t first;    // balanced plan: first CTA holding the sequence
  int32_t more;     // this CTA has a piece after this one
  int32_t has_q;    // the piece's q rows were loaded (not after an abort)
  int32_t pad[2];
};
static_assert(sizeof(PieceDesc) == 48, "PieceDesc layout");

// The pieces of this CTA, walked by the producer, which announces each one.
struct PieceIter {
  BalancedWalk<CtaTiles> walk;
  const SplitParams& p;
  bool balanced, pending;

  __device__ __forceinline__ static int32_t walk_grid(const SplitParams& p, int64_t total) {
    const int32_t g = p.n_splits == 0 ? balanced_ctas(total, (int32_t)gridDim.x) : 0;
    return g > 0 ? g : 1;
  }
  __device__ __forceinline__ static bool walk_active(const SplitParams& p, int64_t total) {
    return p.n_splits == 0 && total > 0 && (int32_t)blockIdx.x < balanced_ctas(total, (int32_t)gridDim.x);
  }

  __device__ __forceinline__ PieceIter(const SplitParams& p_, const CtaTiles& tl, int64_t total)
      : walk(tl, p_.B, p_.hv, walk_active(p_, total) ? total : 0, walk_grid(p_, total),
             walk_active(p_, total) ? (int32_t)blockIdx.x : 0),
        p(p_), balanced(p_.n_splits == 0), pending(p_.n_splits != 0) {}

  // Does this CTA have a piece after the one last returned?
  __device__ __forceinline__ bool more() const { return balanced ? !walk.done() : pending; }

  __device__ __forceinline__ bool next(Piece& pc) {
    if (balanced) return walk.next(pc);
    if (!pending) return false;
    pending = false;
    const int32_t pair = blockIdx.x, s = blockIdx.y;
    pc.b = pair / p.hv;
    pc.vkv = pair % p.hv;
    const int32_t L = p.seq_lens ? clamp_len(__ldg(p.seq_lens + pc.b) + p.append, p.max_len) : p.max_len;
    const int64_t lo = (int64_t)s * p.split_tokens;
    const int64_t hi = lo + p.split_tokens < L ? lo + p.split_tokens : L;
    pc.tok_begin = (int32_t)(lo < L ? lo : L);
    pc.tok_end = (int32_t)(hi > pc.tok_begin ? hi : pc.tok_begin);
    pc.slot = s;
    pc.len = L;
    return true;
  }
};

// ----------------------------------------------------------------- producer
template <class C>
__device__ __forceinline__ void producer_warp(const CUtensorMap* tk, const CUtensorMap* tv,
                                              const SplitParams& p, const CtaTiles& tl, int64_t total,
                                              uint8_t* smem, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + 2;
  uint32_t it = 0, qi = 0;
  uint32_t stalled = 0xffffffffu;  // stage skipped by the testing hook
  bool ok = true;
  Groups gr;
  gr.g = p.g;
  gr.gpad = p.gpad;
  gr.nsub = p.nsub;
  gr.hv = p.hv;

  constexpr int kPageAhead = 4;
  // Contiguous caches: K/V are read once, so their L2 lines go first (measured
  // faster).  The paged pool keeps the default policy (evict-first measured ~1 %
  // slower there).
  const uint64_t stream_policy = policy_evict_first();
  // one tile advances a lane's position by step_q pages and step_r rows
  const int32_t step_q = p.paged ? C::kBT / p.page_size : 0;
  const int32_t step_r = p.paged ? C::kBT % p.page_size : 0;

  PieceDesc* desc = reinterpret_cast<PieceDesc*>(smem + C::kDescOff);
  const int32_t grid_used = p.n_splits == 0 ? balanced_ctas(total, (int32_t)gridDim.x) : 0;
  PieceIter pieces(p, tl, total);
  Piece pc;
  bool waited = false, live = true;  // live: the consumers still take announcements
  while (pieces.next(pc)) {
    const bool nonempty = pc.tok_end > pc.tok_begin;
    if (!waited) {  // first memory access of this warp: q, the block table, K/V
      pdl_wait();
      waited = true;
    }
    int32_t head0, nh;
    vkv_heads(gr, pc.vkv, &head0, &nh);
    const int32_t kvh = kv_head_of_vkv(gr, pc.vkv);
    // The piece's arrival count (the consumers' registers are scarcer than the producer's).
    int32_t npieces = p.n_splits, first = 0;
    if (p.n_splits == 0) {
      int32_t last;
      balanced_pair_ctas(tl, p.hv, total, grid_used, pc.b, pc.vkv, &first, &last);
      npieces = last - first + 1;
    }
    // Announce it with its q rows.  After an abort (!ok) the pieces are still
    // announced, without q and without tiles, so that every arrival count
    // completes and the counters end at zero.
    if (lane == 0) {
      const uint32_t slot = qi % C::kQBufs;
      if (!mbar_wait_for(qempty + slot, ((qi / C::kQBufs) & 1) ^ 1, wait_limit(p))) {
        live = false;  // the consumers stopped taking pieces
      } else {
        const bool load_q = ok && nonempty;
        PieceDesc* d = desc + slot;
        d->b = pc.b;
        d->vkv = pc.vkv;
        d->tok_begin = pc.tok_begin;
        d->tok_end = pc.tok_end;
        d->slot = pc.slot;
        d->len = pc.len;
        d->npieces = npieces;
        d->first = first;
        d->more = pieces.more() ? 1 : 0;
        d->has_q = load_q ? 1 : 0;
        if (load_q) {
          const uint32_t bytes = (uint32_t)nh * C::D * 4;
          mbar_arrive_expect_tx(qfull + slot, bytes);
          bulk_load(smem + C::kQOff + slot * C::kQBytes, p.q + ((size_t)pc.b * p.Hq + head0) * C::D, bytes,
                    qfull + slot);
        } else {
          mbar_arrive(qfull + slot);
        }
      }
    }
    ++qi;
    live = __shfl_sync(0xffffffffu, live, 0);
    if (!live) {
      ok = false;
      break;
    }
    if (!ok || !nonempty) continue;
    // Paged: lane j looks up the page of row block j of a tile kPageAhead tiles
    // ahead, so the table loads -- which miss L2 once the K/V stream has
    // evicted the table -- overlap several stages.  The tile loop is unrolled
    // by kPageAhead so that each queue slot stays in its own register (moving
    // a register would wait for its load).  Positions advance by a fixed
    // (pages, rows) step per tile: no division in the loop.  Only entries of
    // keys below tok_end (<= L_b) are ever read.
    const int32_t* trow = p.paged ? p.block_table + (size_t)pc.b * p.max_pages : nullptr;
    int32_t pq[kPageAhead];
    int32_t cur_row = 0, a_tn = 0, a_idx = 0, a_row = 0;
    if (p.paged) {
      const int32_t tn0 = pc.tok_begin + 16 * lane;
#pragma unroll
      for (int a = 0; a < kPageAhead; ++a) {
        const int32_t tn = tn0 + a * C::kBT;
        pq[a] = tn < pc.tok_end ? __ldg(trow + tn / p.page_size) : 0;
      }
      cur_row = tn0 % p.page_size;
      a_tn = tn0 + kPageAhead * C::kBT;
      a_idx = a_tn / p.page_size;
      a_row = a_tn - a_idx * p.page_size;
    }
    for (int32_t t0 = pc.tok_begin; ok && t0 < pc.tok_end;) {
#pragma unroll
      for (int slot = 0; slot < kPageAhead; ++slot) {
        if (!ok || t0 >= pc.tok_end) break;
        const int32_t nvalid = pc.tok_end - t0 < C::kBT ? pc.tok_end - t0 : C::kBT;
        const int32_t nbox = ceil_div(nvalid, 16);
        bool mine = lane < nbox;
        int32_t page = 0, row = t0 + 16 * lane;
        if (p.paged) {
          page = pq[slot];
          row = cur_row;
          cur_row += step_r;
          if (cur_row >= p.page_size) cur_row -= p.page_size;
          pq[slot] = a_tn < pc.tok_end ? __ldg(trow + a_idx) : 0;
          a_tn += C::kBT;
          a_idx += step_q;
          a_row += step_r;
          if (a_row >= p.page_size) {
            a_row -= p.page_size;
            ++a_idx;
          }
          if (mine && (page < 0 || page >= p.num_pages)) {
            raise_error(p.err, kErrBadIndex);
            mine = false;
          }
        }
        const unsigned issue = __ballot_sync(0xffffffffu, mine);
        const uint32_t stage = it % C::kStages;
        const uint32_t phase = (it / C::kStages) & 1;
        const bool stall = p.stall_it >= 0 && it == (uint32_t)p.stall_it;
        if (lane == 0) {
          if (*abort_flag || !mbar_wait_for(empty + stage, phase ^ 1, wait_limit(p))) {
            ok = false;
          } else if (!stall) {
            mbar_arrive_expect_tx(full + stage, (uint32_t)__popc(issue) * C::kNB * 2 * C::kBoxBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (stall) stalled = it;  // nothing issued: this stage never completes
        if (mine && !stall) {
          uint8_t* kdst = smem + stage * C::kStageBytes + lane * C::kBoxBytes;
          uint8_t* vdst = kdst + C::kTileBytes;
          // paged pool viewed as [num_pages * Hkv, page_size, D]; contiguous [B * Hkv, T_cap, D]
          const int32_t z = p.paged ? page * p.Hkv + kvh : pc.b * p.Hkv + kvh;
#pragma unroll
          for (int nb = 0; nb < C::kNB; ++nb) {
            const int32_t x = nb * (128 / C::kEs);
            const int32_t off = nb * C::kBT * 128;
            if (p.paged) {
              tma_load_3d(kdst + off, tk, full + stage, x, row, z);
              tma_load_3d(vdst + off, tv, full + stage, x, row, z);
            } else {
              tma_load_3d_hint(kdst + off, tk, full + stage, x, row, z, stream_policy);
              tma_load_3d_hint(vdst + off, tv, full + stage, x, row, z, stream_policy);
            }
          }
        }
        t0 += C::kBT;
        ++it;
      }
    }
  }
  // No more pieces: tell the consumers.
  if (live && lane == 0) {
    const uint32_t slot = qi % C::kQBufs;
    if (mbar_wait_for(qempty + slot, ((qi / C::kQBufs) & 1) ^ 1, wait_limit(p))) {
      desc[slot].b = -1;
      mbar_arrive(qfull + slot);
    } else {
      ok = false;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) {
    raise_error(p.err, kErrTimeout);
    *abort_flag = 1;
  }
  // Do not leave while copies this warp issued may still be landing.
  if (lane == 0) {
    const uint32_t n = it < (uint32_t)C::kStages ? it : (uint32_t)C::kStages;
    for (uint32_t j = it - n; j < it; ++j) {
      if (j == stalled) continue;
      if (!mbar_wait_for(full + (j % C::kStages), (j / C::kStages) & 1, wait_limit(p))) raise_error(p.err, kErrTimeout);
    }
  }
}

// The last arriver's merge of a whole (b, virtual KV head), for a CTA with no
// piece after this one: its K/V ring is idle, so the pair's partial outputs
// come into it with bulk copies (one round trip to L2 for all heads and
// splits), and the (m, l) of every state with a small copy of their own on a
// second barrier, so that the weights are ready while the outputs still land;
// the weighted sums then run out of shared memory, every thread's outputs
// summed in one interleaved pass.  The arithmetic per output element is
// merge_head's (same weights, same four interleaved partial sums in increasing
// k, same final division), so both give identical bits.
// State (h, k) of the pair is partial index base0 + h*hs + k*stride; all
// n_states indices lie in [base0, base0 + n_states).  count <= 128.
template <class C>
__device__ __forceinline__ void merge_pair_smem(const SplitParams& p, uint8_t* smem, uint64_t* mbar_o,
                                                uint64_t* mbar_ml, size_t base0, int n_states, int count, int nh,
                                                int hs, int stride, float* out_rows, float* lse_slots) {
  constexpr int D = C::D, EPL = D / 32, W = C::kWarps, kCons = W * 32;
  constexpr int HPW = (C::G + W - 1) / W;          // heads per warp in the weights
  constexpr int IPT = (C::G * 32 + kCons - 1) / kCons;  // (head, lane slice) items per thread in the sums
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns4 = (n_states + 3) & ~3;         // keeps every array below 16-byte aligned
  float* so = reinterpret_cast<float*>(smem);  // [n_states, D]
  float* rm = so + (size_t)n_states * D;       // [n_states] m of every state, in partial order
  float* rl = rm + ns4;                        // [n_states] l likewise
  float* sw = rl + ns4;                        // [nh, 128] weights: head h, split k at h*128 + k
  float* shead = sw + nh * 128;                // [nh, 2] (max, L)
  const uint32_t obytes = (uint32_t)n_states * D * 4;
  const uint32_t mlbytes = (uint32_t)n_states * 4;
  const float* gm = p.m_part + base0;
  const float* gl = p.l_part + base0;
  const bool ml_bulk = (mlbytes & 15) == 0 && ((reinterpret_cast<uintptr_t>(gm) | reinterpret_cast<uintptr_t>(gl)) & 15) == 0;
  if (tid == 0) {
    // the ring's reads by the consumers (generic proxy) come before these async-proxy writes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (ml_bulk) {
      mbar_arrive_expect_tx(mbar_ml, 2 * mlbytes);
      bulk_load(reinterpret_cast<uint8_t*>(rm), gm, mlbytes, mbar_ml);
      bulk_load(reinterpret_cast<uint8_t*>(rl), gl, mlbytes, mbar_ml);
    }
    mbar_arrive_expect_tx(mbar_o, obytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.o_part + base0 * D);
    constexpr uint32_t kChunk = 32768;
    for (uint32_t off = 0; off < obytes; off += kChunk)
      bulk_load(reinterpret_cast<uint8_t*>(so) + off, src + off, obytes - off < kChunk ? obytes - off : kChunk, mbar_o);
  }
  bool ok = true;
  if (ml_bulk) {
    ok = mbar_wait_for(mbar_ml, 0, wait_limit(p));
  } else {
    for (int i0 = 0; i0 < n_states; i0 += 4 * kCons) {
      float mv[4], lv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kCons + tid;
        mv[u] = i < n_states ? __ldcg(gm + i) : 0.f;
        lv[u] = i < n_states ? __ldcg(gl + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kCons + tid;
        if (i < n_states) {
          rm[i] = mv[u];
          rl[i] = lv[u];
        }
      }
    }
    named_barrier(1, kCons);
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout);
    mbar_wait_for(mbar_ml, 0, wait_limit(p));  // give the copy its chance to land before the CTA leaves
  }
  if (count <= 32) {
    // One split per lane: the warp's heads reduce together (merge_max,
    // merge_weights and the warp reductions of merge_head, interleaved).
    float mk[HPW], lk[HPW], mx[HPW], wk[HPW], ls[HPW];
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      const int h = warp + i * W;
      mk[i] = -INFINITY;
      lk[i] = 0.f;
      if (h < nh && lane < count) {
        mk[i] = rm[h * hs + lane * stride];
        lk[i] = rl[h * hs + lane * stride];
      }
      mx[i] = lk[i] > 0.f ? mk[i] : -INFINITY;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < HPW; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], o));
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      wk[i] = (mx[i] != -INFINITY && lk[i] > 0.f) ? exp2f((mk[i] - mx[i]) * kLog2e) : 0.f;
      ls[i] = fmaf(wk[i], lk[i], 0.f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < HPW; ++i) ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], o);
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      const int h = warp + i * W;
      if (h < nh) {
        sw[h * 128 + lane] = wk[i];
        if (lane == 0) {
          shead[2 * h] = mx[i];
          shead[2 * h + 1] = mx[i] == -INFINITY ? 0.f : ls[i];
        }
      }
    }
  } else {
    for (int h = warp; h < nh; h += W) {
      float mk[kMergeKR], lk[kMergeKR], wk[kMergeKR];
#pragma unroll
      for (int r = 0; r < kMergeKR; ++r) {
        const int k = r * 32 + lane;
        mk[r] = -INFINITY;
        lk[r] = 0.f;
        if (k < count) {
          mk[r] = rm[h * hs + k * stride];
          lk[r] = rl[h * hs + k * stride];
        }
      }
      const float mx = warp_max(merge_max(mk, lk));
      float L = 0.f;
      if (mx != -INFINITY) {
        L = warp_sum(merge_weights(mk, lk, mx, wk));
      } else {
#pragma unroll
        for (int r = 0; r < kMergeKR; ++r) wk[r] = 0.f;
      }
#pragma unroll
      for (int r = 0; r < kMergeKR; ++r) sw[h * 128 + r * 32 + lane] = wk[r];
      if (lane == 0) {
        shead[2 * h] = mx;
        shead[2 * h + 1] = L;
      }
    }
  }
  if (!mbar_wait_for(mbar_o, 0, wait_limit(p))) {
    raise_error(p.err, kErrTimeout);
    mbar_wait_for(mbar_o, 0, wait_limit(p));  // give the copy its chance to land before the CTA leaves
  }
  named_barrier(1, kCons);
  // Item (h, j): head h, output elements [j*EPL, (j+1)*EPL).  Thread tid takes
  // items tid + i*kCons, i < IPT (one head per warp and i), all at once.  The
  // split loop has no branch, so the loads of all items and splits of a step
  // are in flight together: splits past `count` (up to the next multiple of 4)
  // read a valid state with weight 0 (sw is 0 there), and fmaf(0, v, a) == a
  // for finite v, so the sums keep merge_head's bits.  Items of heads past nh
  // read head 0 and are not stored.
  float acc[IPT][4][EPL];
  uint32_t wa[IPT], oa[IPT];  // shared addresses: the item's weights and its slice of split 0
  const uint32_t kstep = (uint32_t)stride * D * 4;  // bytes from split k to k + 1
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    const int item = tid + i * kCons;
    const int h = item >> 5, j = item & 31;
    const int hc = h < nh ? h : 0;
    wa[i] = smem_addr(sw + hc * 128);
    oa[i] = smem_addr(so) + (uint32_t)((hc * hs * D + j * EPL) * 4);
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[i][s4][e] = 0.f;
  }
  const int klast = count - 1;
  for (int k0 = 0; k0 < count; k0 += 4) {
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int k = k0 + jj;
        const float w = __uint_as_float(lds32u(wa[i] + 4 * k));
        const uint32_t va = oa[i] + (uint32_t)(k < klast ? k : klast) * kstep;
        float vv[EPL];
        if constexpr (EPL == 4) {
          const float4 x = lds128(va);
          vv[0] = x.x;
          vv[1] = x.y;
          vv[2] = x.z;
          vv[3] = x.w;
        } else {
          const uint2 x = lds64u(va);
          vv[0] = __uint_as_float(x.x);
          vv[1] = __uint_as_float(x.y);
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[i][jj][e] = fmaf(w, vv[e], acc[i][jj][e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    const int item = tid + i * kCons;
    if (item >= nh * 32) continue;
    const int h = item >> 5, j = item & 31;
    float* orow = out_rows + (size_t)h * D + j * EPL;
    const float mx = shead[2 * h], L = shead[2 * h + 1];
    float o4[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      o4[e] = mx == -INFINITY ? 0.f : (((acc[i][0][e] + acc[i][1][e]) + acc[i][2][e]) + acc[i][3][e]) / L;
    if constexpr (EPL == 4)
      *reinterpret_cast<float4*>(orow) = make_float4(o4[0], o4[1], o4[2], o4[3]);
    else
      *reinterpret_cast<float2*>(orow) = make_float2(o4[0], o4[1]);
    if (lse_slots && j == 0) lse_slots[h] = mx == -INFINITY ? -INFINITY : mx + logf(L);
  }
}

// ----------------------------------------------------------------- consumers
// Each consumer warp owns key rows [32w, 32w+32) of every stage and keeps its
// own running (m, l, O) per head.  Two engines compute a tile: the CUDA-core
// engine below (one or two heads per CTA, and fp32 caches), and MmaEngine
// (fd_split_mma.cuh) for bf16 caches with four or eight query heads per CTA,
// where q.k and p.V run on mma.sync.  Both publish the warp state the same
// way, so the merge code is shared.

template <class C, bool kFull>
__device__ __forceinline__ void pv_rows(uint32_t vbase, const uint32_t* voff, uint32_t pbase, int nv,
                                        float2 (&o)[C::G][C::kEPL / 2]) {
  constexpr int G = C::G;
  for (int t8 = 0; t8 < nv; t8 += 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = t8 + j;
      if (kFull || t < nv) {
        const uint32_t a = vbase + t * 128 + voff[j];
        float vf[C::kEPL];
        if constexpr (C::kBf16) {
          if constexpr (C::kEPL == 4) {
            const uint2 w = lds64u(a);
            vf[0] = bf16_lo(w.x);
            vf[1] = bf16_hi(w.x);
            vf[2] = bf16_lo(w.y);
            vf[3] = bf16_hi(w.y);
          } else {
            const uint32_t w = lds32u(a);
            vf[0] = bf16_lo(w);
            vf[1] = bf16_hi(w);
          }
        } else {
          if constexpr (C::kEPL == 4) {
            const float4 w = lds128(a);
            vf[0] = w.x;
            vf[1] = w.y;
            vf[2] = w.z;
            vf[3] = w.w;
          } else {
            const uint2 w = lds64u(a);
            vf[0] = __uint_as_float(w.x);
            vf[1] = __uint_as_float(w.y);
          }
        }
        const uint32_t prow = pbase + t * (G * 8);
        if constexpr (G == 1) {
          const uint2 pw = lds64u(prow);
          const float2 pp = make_float2(__uint_as_float(pw.x), __uint_as_float(pw.y));
#pragma unroll
          for (int i = 0; i < C::kEPL / 2; ++i) o[0][i] = fma2(make_float2(vf[2 * i], vf[2 * i + 1]), pp, o[0][i]);
        } else {
#pragma unroll
          for (int h = 0; h < G; h += 2) {
            const float4 pq = lds128(prow + h * 8);
            const float2 p0 = make_float2(pq.x, pq.y), p1 = make_float2(pq.z, pq.w);
#pragma unroll
            for (int i = 0; i < C::kEPL / 2; ++i) {
              const float2 v2 = make_float2(vf[2 * i], vf[2 * i + 1]);
              o[h][i] = fma2(v2, p0, o[h][i]);
              o[h + 1][i] = fma2(v2, p1, o[h + 1][i]);
            }
          }
        }
      }
    }
  }
}

// CUDA-core engine.  q.k: lane = key row, 16-byte chunks of the row, q read as
// a shared-memory broadcast.  p.V: lane = a D/32-wide slice of the output, p
// broadcast from shared memory.  m, l, O per head; m is warp-uniform.
template <class C>
struct CoreEngine {
  static constexpr int G = C::G, D = C::D, EPL = C::kEPL;
  static constexpr bool kQInSmem = false;
  float m[G], l[G];
  float2 o[G][EPL / 2];
  int32_t lim[G];  // keys each head's row may see (the piece's row limits)
  uint32_t xr, pbase, e_nb;
  uint32_t voff[8];
  int warp, lane;
  uint8_t* smem;

  __device__ __forceinline__ void setup(int warp_, int lane_, uint8_t* smem_) {
    warp = warp_;
    lane = lane_;
    smem = smem_;
    xr = lane & 7;
    pbase = smem_addr(smem) + C::kUOff + warp * 32 * G * 8;
    const int e_byte = lane * EPL * C::kEs;  // this lane's slice of a row, in bytes
    e_nb = e_byte / 128;                     // column block
    const int e_chunk = (e_byte % 128) / 16; // 16-byte chunk within the block
    const int e_in = e_byte % 16;            // byte within the chunk
#pragma unroll
    for (int j = 0; j < 8; ++j) voff[j] = ((e_chunk ^ j) << 4) + e_in;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) o[h][i] = make_float2(0.f, 0.f);
    }
  }

  __device__ __forceinline__ void begin(uint32_t, float, const RowLimits& rl) {
#pragma unroll
    for (int h = 0; h < G; ++h) lim[h] = rl(h);
  }

  __device__ __forceinline__ void tile(uint32_t kst, uint32_t vst, int nv, uint32_t qaddr, float qk_scale,
                                       int32_t tok0) {
    // ---- q.k, lane = row
    float2 acc[G][C::kAcc];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int a = 0; a < C::kAcc; ++a) acc[h][a] = make_float2(0.f, 0.f);
    const uint32_t krow = kst + (32 * warp + lane) * 128;
#pragma unroll
    for (int nb = 0; nb < C::kNB; ++nb) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int a = (nb * 8 + c) % C::kAcc;
        const uint4 kw = lds128u(krow + nb * C::kBT * 128 + ((c ^ xr) << 4));
        const int d0 = nb * (128 / C::kEs) + c * C::kChunkElems;
        if constexpr (C::kBf16) {
          const float2 k01 = make_float2(bf16_lo(kw.x), bf16_hi(kw.x));
          const float2 k23 = make_float2(bf16_lo(kw.y), bf16_hi(kw.y));
          const float2 k45 = make_float2(bf16_lo(kw.z), bf16_hi(kw.z));
          const float2 k67 = make_float2(bf16_lo(kw.w), bf16_hi(kw.w));
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float4 qa = lds128(qaddr + (h * D + d0) * 4);
            const float4 qb = lds128(qaddr + (h * D + d0 + 4) * 4);
            acc[h][a] = fma2(k01, make_float2(qa.x, qa.y), acc[h][a]);
            acc[h][a] = fma2(k23, make_float2(qa.z, qa.w), acc[h][a]);
            acc[h][a] = fma2(k45, make_float2(qb.x, qb.y), acc[h][a]);
            acc[h][a] = fma2(k67, make_float2(qb.z, qb.w), acc[h][a]);
          }
        } else {
          const float2 k01 = make_float2(__uint_as_float(kw.x), __uint_as_float(kw.y));
          const float2 k23 = make_float2(__uint_as_float(kw.z), __uint_as_float(kw.w));
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float4 qa = lds128(qaddr + (h * D + d0) * 4);
            acc[h][a] = fma2(k01, make_float2(qa.x, qa.y), acc[h][a]);
            acc[h][a] = fma2(k23, make_float2(qa.z, qa.w), acc[h][a]);
          }
        }
      }
    }
    // ---- online softmax over this warp's rows
    const int32_t key = tok0 + 32 * warp + lane;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = 0.f;
#pragma unroll
      for (int a = 0; a < C::kAcc; ++a) s += acc[h][a].x + acc[h][a].y;
      s = (lane < nv && key < lim[h]) ? s * qk_scale : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(s));
      // a head whose row has seen no key yet keeps its empty state
      const float alpha = mn == -INFINITY ? 1.f : exp2f(m[h] - mn);
      const float pr = mn == -INFINITY ? 0.f : exp2f(s - mn);
      l[h] = fmaf(l[h], alpha, pr);
      const float2 al = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) o[h][i] = make_float2(o[h][i].x * al.x, o[h][i].y * al.y);
      m[h] = mn;
      // p, duplicated as a pair, for the broadcast reads of p.V
      *reinterpret_cast<float2*>(smem + C::kUOff + (warp * 32 + lane) * G * 8 + h * 8) = make_float2(pr, pr);
    }
    __syncwarp();
    // ---- p.V, lane = output slice
    const uint32_t vbase = vst + e_nb * C::kBT * 128 + (32 * warp) * 128;
    if (nv == 32)
      pv_rows<C, true>(vbase, voff, pbase, 32, o);
    else
      pv_rows<C, false>(vbase, voff, pbase, nv, o);
    __syncwarp();
  }

  // Warp state -> merge slot `warp`: O[h][:] (unnormalised, on m[h]), m[h], l[h].
  __device__ __forceinline__ void publish(float* obuf, float* mlbuf, int) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float lw = warp_sum(l[h]);
      float* dst = obuf + (warp * G + h) * C::kObStride + lane * EPL;
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) reinterpret_cast<float2*>(dst)[i] = o[h][i];
      if (lane == 0) {
        mlbuf[(warp * G + h) * 2] = m[h];
        mlbuf[(warp * G + h) * 2 + 1] = lw;
      }
    }
  }
};

// Fused append: put the new token's K and V row (position L = len - 1 of the
// sequence, row r of its last stage) into the landed stage, in the
// 128-byte-swizzle layout the TMA boxes use (16-byte chunk c of row r sits in
// column block c/8 at chunk (c % 8) ^ (r % 8)), and, when `to_cache`, into the
// cache itself.  The owning warp loads its chunks (lane c holds chunk c) and
// looks up the cache position when the piece starts, so those loads overlap
// the piece's streaming.  Only warp r / 32 reads row r, so the warp's own
// fence and __syncwarp order the stores before its reads and before the
// stage's next TMA write.
template <class C>
struct AppendRow {
  static constexpr int kChunks = C::kRowBytes / 16;
  static_assert(kChunks <= 32, "one 16-byte chunk per lane");
  uint4 kx, vx;
  size_t dst;
  bool to_cache;

  __device__ __forceinline__ void prefetch(const SplitParams& p, int32_t b, int32_t kvh, int32_t L, int lane,
                                           bool cache_write) {
    const size_t src = ((size_t)b * p.Hkv + kvh) * C::kRowBytes;
    if (lane < kChunks) {
      kx = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.k_new) + src) + lane);
      vx = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.v_new) + src) + lane);
    }
    to_cache = cache_write;
    dst = 0;
    if (to_cache) {
      if (p.paged) {
        const int32_t page = __ldg(p.block_table + (size_t)b * p.max_pages + L / p.page_size);
        if (page < 0 || page >= p.num_pages) {
          if (lane == 0) raise_error(p.err, kErrBadIndex);
          to_cache = false;
        } else {
          dst = (((size_t)page * p.Hkv + kvh) * p.page_size + L % p.page_size) * C::kRowBytes;
        }
      } else {
        dst = (((size_t)b * p.Hkv + kvh) * p.capacity + L) * C::kRowBytes;
      }
    }
  }

  __device__ __forceinline__ void place(const SplitParams& p, uint32_t kst, uint32_t vst, int32_t r, int lane) {
    if (lane < kChunks) {
      const int c = lane;
      const uint32_t so = (uint32_t)(c >> 3) * C::kBT * 128 + (uint32_t)r * 128 + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(kst + so), "r"(kx.x), "r"(kx.y), "r"(kx.z),
                   "r"(kx.w)
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(vst + so), "r"(vx.x), "r"(vx.y), "r"(vx.z),
                   "r"(vx.w)
                   : "memory");
      if (to_cache) {
        reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + dst)[c] = kx;
        reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + dst)[c] = vx;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
  }
};

template <class C, class E>
__device__ __forceinline__ void consumer_warps(const SplitParams& p, const CtaTiles& tl, int64_t total,
                                               uint8_t* smem, volatile int* abort_flag) {
  constexpr int G = C::G, D = C::D, W = C::kWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  constexpr int kCons = W * 32;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + 2;
  float* obuf = reinterpret_cast<float*>(smem + C::kUOff);
  float* mlbuf = reinterpret_cast<float*>(smem + C::kMlOff);
  float* fin = reinterpret_cast<float*>(smem + C::kFinOff);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kFlagOff + 4);
  const uint32_t sbase = smem_addr(smem);
  const bool balanced = p.n_splits == 0;
  const bool fused = p.counters != nullptr;

  Groups gr;
  gr.g = p.g;
  gr.gpad = p.gpad;
  gr.nsub = p.nsub;
  gr.hv = p.hv;

  pdl_wait();  // before the first write (outputs, partials, counters, the cache)
  // Balanced plan: sequences with no keys own no tile; CTA b % grid writes their outputs.
  if (balanced && fused) {
    for (int32_t b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (tl.len(b) != 0) continue;
      for (int i = tid; i < p.Hq * D; i += kCons) p.out[(size_t)b * p.Hq * D + i] = 0.f;
      if (p.lse)
        for (int i = tid; i < p.Hq; i += kCons) p.lse[(size_t)b * p.Hq + i] = -INFINITY;
    }
  }

  E eng;
  eng.setup(warp, lane, smem);
  uint32_t it = 0, qi = 0;
  bool ok = true;

  // The producer announces every piece of this CTA (PieceDesc, with its q rows)
  // and then an end mark.
  const PieceDesc* desc = reinterpret_cast<const PieceDesc*>(smem + C::kDescOff);
  for (;;) {
    const uint32_t qslot = qi % C::kQBufs;
    if (!mbar_wait_for(qfull + qslot, (qi / C::kQBufs) & 1, wait_limit(p))) {
      ok = false;
      *abort_flag = 1;
      break;
    }
    const PieceDesc& d = desc[qslot];
    Piece pc;
    pc.b = d.b;
    if (pc.b < 0) break;
    pc.vkv = d.vkv;
    pc.tok_begin = d.tok_begin;
    pc.tok_end = d.tok_end;
    pc.slot = d.slot;
    pc.len = d.len;
    const int npieces = d.npieces;
    const int32_t first = d.first;  // balanced: first CTA holding this sequence
    const bool more = d.more != 0, has_q = d.has_q != 0;
    int32_t head0, nh;
    vkv_heads(gr, pc.vkv, &head0, &nh);
    const bool nonempty = pc.tok_end > pc.tok_begin;
    const int32_t pair = pc.b * p.hv + pc.vkv;
    // Does this piece hold the whole sequence?  Then it is the output.
    const bool final_here = fused && npieces == 1;
    eng.reset();
    // Fused append: the warp owning the new token's row prefetches it now.
    const bool app = p.append && nonempty && pc.tok_end == pc.len;
    const int32_t app_t0 = pc.tok_begin + (pc.tok_end - 1 - pc.tok_begin) / C::kBT * C::kBT;  // last tile
    const int32_t app_r = pc.tok_end - 1 - app_t0;                                          // its row
    AppendRow<C> arow;
    if (app && warp == (app_r >> 5))
      arow.prefetch(p, pc.b, kv_head_of_vkv(gr, pc.vkv), pc.len - 1, lane, pc.vkv % gr.nsub == 0);
    const bool run_tiles = nonempty && ok && has_q;
    const uint32_t qaddr = sbase + C::kQOff + qslot * C::kQBytes;
    if (run_tiles) {
      const RowLimits rl{head0, nh, pc.len, p.n_q, p.causal};
      eng.begin(qaddr, p.qk_scale, rl);
    }
    if constexpr (E::kQInSmem) named_barrier(1, kCons);  // every warp's share of the fragments is written
    if constexpr (C::kWide) {
      // q (if any) is in registers now and the piece is read: hand the slot back (one arrival per warp)
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty + qslot);
    }
    if (run_tiles) {
      for (int32_t t0 = pc.tok_begin; ok && t0 < pc.tok_end; t0 += C::kBT, ++it) {
        const uint32_t stage = it % C::kStages;
        if (*abort_flag || !mbar_wait_for(full + stage, (it / C::kStages) & 1, wait_limit(p))) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        const int32_t nvalid = pc.tok_end - t0 < C::kBT ? pc.tok_end - t0 : C::kBT;
        int nv = nvalid - 32 * warp;
        nv = nv < 0 ? 0 : (nv > 32 ? 32 : nv);
        if (nv > 0) {
          const uint32_t kst = sbase + stage * C::kStageBytes;
          // the new token is the last key of the sequence: this piece's last tile, row app_r
          if (app && t0 == app_t0 && warp == (app_r >> 5)) arow.place(p, kst, kst + C::kTileBytes, app_r, lane);
          eng.tile(kst, kst + C::kTileBytes, nv, qaddr, p.qk_scale, t0);
        }
        if (lane == 0) mbar_arrive(empty + stage);
      }
    }

    // ---- merge the W warp states of this piece
    named_barrier(1, kCons);  // every warp is past its last tile: the p buffers may be reused
    if constexpr (!C::kWide) {
      if (tid == 0) mbar_arrive(qempty + qslot);  // the piece's q slot and descriptor are free
    }
    ++qi;

    // kPubHeads heads per round; rounds > 1 only with sixteen heads per CTA
    constexpr int PH = C::kPubHeads;
#pragma unroll 1
    for (int r = 0; r < G / PH; ++r) {
      if (r > 0) named_barrier(1, kCons);  // the last round's readers are done with the buffers
      eng.publish(obuf, mlbuf, r);
      named_barrier(1, kCons);
      if (tid < PH) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, mlbuf[(w * PH + tid) * 2]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          // each warp state's weight exp2(m_w - M), once per head (0 for an empty state)
          const float mw = mlbuf[(w * PH + tid) * 2];
          const float sw = mw == -INFINITY ? 0.f : exp2f(mw - M);
          if (mw != -INFINITY) L = fmaf(sw, mlbuf[(w * PH + tid) * 2 + 1], L);
          mlbuf[(w * PH + tid) * 2] = sw;
        }
        fin[tid * 2] = M;
        fin[tid * 2 + 1] = L;
      }
      named_barrier(1, kCons);

      for (int idx = tid; idx < PH * D; idx += kCons) {
        const int hl = idx / D, d = idx % D;
        const int h = r * PH + hl;
        if (h >= nh) continue;
        const float M = fin[hl * 2];
        // an empty warp state has weight 0 and O = 0, and fmaf(0, 0, a) == a
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w)
          acc = fmaf(mlbuf[(w * PH + hl) * 2], obuf[(w * PH + hl) * C::kObStride + d], acc);
        if (final_here) {
          const float L = fin[hl * 2 + 1];
          p.out[((size_t)pc.b * p.Hq + head0 + h) * D + d] = M == -INFINITY ? 0.f : acc / L;
        } else if (balanced) {
          p.o_part[((size_t)pc.slot * G + h) * D + d] = acc;
        } else {
          p.o_part[(((size_t)pc.b * p.Hq + head0 + h) * p.n_splits + pc.slot) * D + d] = acc;
        }
      }
      if (tid < PH && r * PH + tid < nh) {
        const int h = r * PH + tid;
        const float M = fin[tid * 2], L = fin[tid * 2 + 1];
        const float m_nat = M == -INFINITY ? -INFINITY : M * kLn2;
        if (final_here) {
          if (p.lse) p.lse[(size_t)pc.b * p.Hq + head0 + h] = M == -INFINITY ? -INFINITY : m_nat + logf(L);
        } else {
          const size_t i = balanced ? (size_t)pc.slot * G + h
                                    : ((size_t)pc.b * p.Hq + head0 + h) * p.n_splits + pc.slot;
          p.m_part[i] = m_nat;
          p.l_part[i] = L;
        }
      }
    }

    if (fused && !final_here) {
      // The barrier orders every thread's partial stores before thread 0's
      // release; its acquire, then the barrier, orders the other pieces'
      // partials before this CTA's reads if it arrives last.
      named_barrier(1, kCons);
      if (tid == 0) *last_flag = (atomic_add_acq_rel(p.counters + pair, 1) == npieces - 1) ? 1 : 0;
      named_barrier(1, kCons);
      if (*last_flag) {
        size_t base0, stride;
        int count;
        if (balanced) {
          base0 = (size_t)(pair + first) * G;
          stride = G;
          count = npieces;
        } else {
          base0 = ((size_t)pc.b * p.Hq + head0) * p.n_splits;
          stride = 1;
          count = p.n_splits;
        }
        // Head h, split k: state base0 + h*hs + k*stride.
        const size_t hs = balanced ? 1 : (size_t)p.n_splits;
        // With no piece after this one, the ring is idle: merge out of shared memory.
        const int n_states = balanced ? count * G : nh * count;
        const bool in_smem = C::kMma && !more && !*abort_flag && count <= kMergeKR * 32 &&
                             (size_t)n_states * D * 4 + (size_t)((n_states + 3) & ~3) * 8 +
                                     (size_t)nh * (128 + 2) * 4 <=
                                 (size_t)C::kStages * C::kStageBytes;
        if (in_smem) {
          merge_pair_smem<C>(p, smem, full + 2 * C::kStages + 4, full + 2 * C::kStages + 5, base0, n_states, count,
                             nh, (int)hs, (int)stride,
                             p.out + ((size_t)pc.b * p.Hq + head0) * D,
                             p.lse ? p.lse + (size_t)pc.b * p.Hq + head0 : nullptr);
        } else {
          for (int h = warp; h < nh; h += W) {
            const GlobalPartials<D> src{p.o_part, p.m_part, p.l_part, base0 + h * hs, stride};
            merge_head<D>(src, count, p.out + ((size_t)pc.b * p.Hq + head0 + h) * D,
                          p.lse ? p.lse + (size_t)pc.b * p.Hq + head0 + h : nullptr, lane, obuf + warp * 128);
          }
        }
        if (tid == 0) p.counters[pair] = 0;  // ready for the next call
      }
    }
    named_barrier(1, kCons);  // shared merge buffers are free again
  }
  if (!ok) {
    raise_error(p.err, kErrTimeout);
    *abort_flag = 1;
  }
}

}  // namespace fdk

#include "fd_split_mma.cuh"

namespace fdk {

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fd_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kFlagOff);
  int32_t* lens = reinterpret_cast<int32_t*>(smem + C::kLenOff);
  int32_t* pre = reinterpret_cast<int32_t*>(smem + C::kPreOff);

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars + s, 1);                         // full: producer's expect_tx arrival
      mbar_init(bars + C::kStages + s, C::kWarps);    // empty: one arrival per consumer warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 2 * C::kStages + i, 1);                               // q full
      mbar_init(bars + 2 * C::kStages + 2 + i, C::kWide ? C::kWarps : 1);    // q empty
    }
    mbar_init(bars + 2 * C::kStages + 4, 1);  // the pair merge's bulk copies: partial outputs
    mbar_init(bars + 2 * C::kStages + 5, 1);  // ... and (m, l) (merge_pair_smem)
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::kWarps && (tid & 31) == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // q rows past the live heads of a group must hold finite values.
  for (int i = tid; i < C::kQBufs * C::G * C::D; i += C::kThreads)
    reinterpret_cast<float*>(smem + C::kQOff)[i] = 0.f;

  // Let the next kernel on the stream be scheduled as SMs free up.  Nothing
  // above touched global memory; with no lengths to read, the plan needs none
  // either, and each warp waits for the kernel before it (pdl_wait) only at
  // its first access, so the producer walks its plan meanwhile.
  pdl_launch_dependents();
  if (p.seq_lens != nullptr) pdl_wait();
  CtaTiles tl;
  tl.pre = pre;
  tl.ln = lens;
  tl.ul = p.max_len;
  tl.ut = ceil_div(p.max_len, kPlanTile);
  tl.uniform = 1;
  if (p.n_splits == 0 && p.seq_lens != nullptr) {
    tl.uniform = 0;
    for (int b = tid; b < p.B; b += C::kThreads) lens[b] = clamp_len(__ldg(p.seq_lens + b) + p.append, p.max_len);
    cta_sync();
    if (warp == 0) {
      const int lane = tid & 31;
      const int per = ceil_div(p.B, 32);
      const int lo = lane * per;
      const int hi = lo + per < p.B ? lo + per : p.B;
      int sum = 0;
      for (int b = lo; b < hi; ++b) sum += (int)pair_units(ceil_div(lens[b], kPlanTile), kPieceUnits);
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int run = incl - sum;
      for (int b = lo; b < hi; ++b) {
        pre[b] = run;
        run += (int)pair_units(ceil_div(lens[b], kPlanTile), kPieceUnits);
      }
      if (lane == 31) pre[p.B] = incl;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  cta_sync();
  const int64_t total = (int64_t)p.hv * tl.prefix(p.B);

  if (warp == C::kWarps)
    producer_warp<C>(&tmap_k, &tmap_v, p, tl, total, smem, abort_flag);
  else if constexpr (C::kWide)
    consumer_warps<C, MmaEngine16<C>>(p, tl, total, smem, abort_flag);
  else if constexpr (C::kMma)
    consumer_warps<C, MmaEngine<C>>(p, tl, total, smem, abort_flag);
  else
    consumer_warps<C, CoreEngine<C>>(p, tl, total, smem, abort_flag);
}

}  // namespace fdk
