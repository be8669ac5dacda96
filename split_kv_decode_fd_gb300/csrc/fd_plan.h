// fd_plan.h -- work decomposition of split-KV decode, shared by the kernels
// and by the host-side plan inspector (fd_plan_pieces).
//
// The pages give a fixed grid of (n_splits, batch*heads) blocks, each block
// taking S consecutive keys ("Kernel visualization: Flash Decoding": one
// thread block per batch, head and split; n_start = s*S).  Two decompositions
// are built here:
//
//  * explicit: exactly that grid.  Split s of (b, kv head) covers tokens
//    [s*S, min((s+1)*S, L_b)), S = 16 * ceil(ceil(max_len / n_splits) / 16).
//  * balanced ("auto"): every (b, virtual kv head) sequence is cut into tiles
//    of kPlanTile tokens; the tiles of all sequences are laid end to end in
//    (b, virtual kv head, tile) order, T tiles in total, and CTA i of G takes
//    the contiguous range [floor(i*T/G), floor((i+1)*T/G)).  A CTA range that
//    crosses sequence boundaries yields one piece per sequence it touches.
//    Every CTA therefore streams the same number of bytes (to one tile),
//    whatever the mix of lengths.
//
// A "virtual kv head" is one KV head together with a sub-group of at most
// max_group of the query heads that share it (16 for bf16 caches, whose
// tensor-core engine takes sixteen heads; 8 for fp32); when g <= max_group
// there is one sub-group per KV head.
//
// The balanced plan uses G = min(CTAs launched, T) CTAs, so that every range
// holds at least one tile and the CTAs holding one sequence are consecutive;
// extra CTAs idle.
//
// Output slots of the balanced plan: the piece of pair p (= b*HV + vkv) run by
// CTA i goes to slot p + i.  For fixed i the pairs touched are consecutive,
// for fixed p the CTAs are consecutive, and if CTA i-1 touches pair p+1 then
// CTA i starts after pair p ends, so slots never collide; at most G + P - 1
// slots are used.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define FD_HD __host__ __device__ __forceinline__
#else
#define FD_HD inline
#endif

namespace fdk {

constexpr int kPlanTile = 128;   // tokens per balancing tile
constexpr int kMaxGroupF32 = 8;   // query heads served by one CTA from one fp32 K/V read
constexpr int kMaxGroupBf16 = 16; // ... from one bf16 K/V read
constexpr int kSplitAlign = 16;  // explicit split sizes are multiples of this

FD_HD int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }
FD_HD int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

FD_HD int32_t explicit_split_size(int32_t max_len, int32_t n_splits) {
  if (max_len < 1 || n_splits < 1) return 0;
  int32_t s = ceil_div(max_len, n_splits);
  s = ceil_div(s, kSplitAlign) * kSplitAlign;
  return s < kSplitAlign ? kSplitAlign : s;
}

FD_HD int32_t clamp_len(int32_t len, int32_t max_len) {
  return len < 0 ? 0 : (len > max_len ? max_len : len);
}

// Group geometry for Hq query heads over Hkv KV heads.
struct Groups {
  int32_t g;       // query heads per KV head
  int32_t gpad;    // heads per CTA, a power of two (template parameter of the kernel)
  int32_t nsub;    // sub-groups per KV head
  int32_t hv;      // virtual KV heads per sequence = Hkv * nsub
};

FD_HD Groups make_groups(int32_t Hq, int32_t Hkv, int32_t max_group) {
  Groups r;
  r.g = Hq / Hkv;
  int32_t gp = 1;
  while (gp < r.g && gp < max_group) gp *= 2;
  r.gpad = gp;
  r.nsub = ceil_div(r.g, gp);
  r.hv = Hkv * r.nsub;
  return r;
}

// First query head and number of live heads of virtual kv head `vkv`.
FD_HD void vkv_heads(const Groups& gr, int32_t vkv, int32_t* head0, int32_t* nheads) {
  int32_t kvh = vkv / gr.nsub, sub = vkv % gr.nsub;
  *head0 = kvh * gr.g + sub * gr.gpad;
  int32_t n = gr.g - sub * gr.gpad;
  *nheads = n < gr.gpad ? n : gr.gpad;
}

FD_HD int32_t kv_head_of_vkv(const Groups& gr, int32_t vkv) { return vkv / gr.nsub; }

// CTAs that take part in the balanced plan of `total` tiles on `launched` CTAs.
FD_HD int32_t balanced_ctas(int64_t total, int32_t launched) {
  return total < (int64_t)launched ? (int32_t)total : launched;
}

// Exact floor(n / d) for 0 <= n, 0 < d; 32-bit division whenever both fit
// (a 64-bit division is a long instruction sequence on the GPU, and the plan
// is walked at the start of every CTA and of every piece).
FD_HD int64_t div_floor(int64_t n, int64_t d) {
  if (n <= 0xffffffffLL && d <= 0xffffffffLL) return (int64_t)((uint32_t)n / (uint32_t)d);
  return n / d;
}

// Balanced plan: CTA range bounds and the CTA owning a flat tile.
FD_HD int64_t range_begin(int64_t total, int32_t grid, int32_t cta) {
  return div_floor(total * (int64_t)cta, (int64_t)grid);
}

FD_HD int32_t cta_of_tile(int64_t total, int32_t grid, int64_t tile) {
  return (int32_t)div_floor((tile + 1) * (int64_t)grid - 1, total);
}

// One unit of work: a run of consecutive keys of one (b, virtual kv head).
struct Piece {
  int32_t b, vkv;
  int32_t tok_begin, tok_end;  // keys [tok_begin, tok_end), already clipped to L_b
  int32_t slot;                // balanced: output slot; explicit: split index
  int32_t len;                 // L_b, the valid length of sequence b
};

// Walk of one CTA over its tile range in the balanced plan.  `Tiles` maps a
// sequence index b to (tile_prefix(b), tiles(b), len(b)), with tile_prefix the
// number of tiles of sequences < b per virtual kv head.
template <class Tiles>
struct BalancedWalk {
  const Tiles& tl;
  int32_t B, hv, cta;
  int64_t flat, end;     // current flat tile, end of range
  int32_t b, vkv, tile;  // position of `flat`

  FD_HD BalancedWalk(const Tiles& t, int32_t B_, int32_t hv_, int64_t total, int32_t grid,
                     int32_t cta_)
      : tl(t), B(B_), hv(hv_), cta(cta_) {
    flat = range_begin(total, grid, cta);
    end = range_begin(total, grid, cta + 1);
    b = vkv = tile = 0;
    if (flat < end) locate();
  }

  // Binary search for the sequence holding `flat`, then the head and tile.
  FD_HD void locate() {
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {  // largest b with hv*prefix(b) <= flat and tiles(b) > 0
      int32_t mid = (lo + hi + 1) / 2;
      if ((int64_t)hv * tl.prefix(mid) <= flat) lo = mid; else hi = mid - 1;
    }
    b = lo;
    while (tl.tiles(b) == 0) ++b;  // empty sequences own no tiles
    int64_t off = flat - (int64_t)hv * tl.prefix(b);
    vkv = (int32_t)div_floor(off, tl.tiles(b));
    tile = (int32_t)(off - (int64_t)vkv * tl.tiles(b));
  }

  FD_HD bool done() const { return flat >= end; }

  // Current piece; then step past it.
  FD_HD Piece next() {
    Piece pc;
    int32_t nt = tl.tiles(b);
    int64_t left = end - flat;
    int32_t take = (int64_t)(nt - tile) < left ? nt - tile : (int32_t)left;
    pc.b = b;
    pc.vkv = vkv;
    pc.tok_begin = tile * kPlanTile;
    int32_t e = (tile + take) * kPlanTile;
    int32_t L = tl.len(b);
    pc.tok_end = e < L ? e : L;
    pc.len = L;
    pc.slot = (b * hv + vkv) + cta;
    flat += take;
    tile += take;
    if (tile == nt) {
      tile = 0;
      if (++vkv == hv) {
        vkv = 0;
        ++b;
        while (flat < end && tl.tiles(b) == 0) ++b;
      }
    }
    return pc;
  }
};

// Pieces of pair p = b*hv + vkv in the balanced plan: CTAs [first, last].
template <class Tiles>
FD_HD void balanced_pair_ctas(const Tiles& tl, int32_t hv, int64_t total, int32_t grid, int32_t b,
                              int32_t vkv, int32_t* first, int32_t* last) {
  int64_t f = (int64_t)hv * tl.prefix(b) + (int64_t)vkv * tl.tiles(b);
  *first = cta_of_tile(total, grid, f);
  *last = cta_of_tile(total, grid, f + tl.tiles(b) - 1);
}

}  // namespace fdk
