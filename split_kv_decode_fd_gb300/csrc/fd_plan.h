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
//  * balanced ("auto"): every (b, virtual kv head) sequence -- a "pair" -- is
//    cut into tiles of kPlanTile tokens, and the pairs are laid end to end in
//    (b, virtual kv head) order on a line of cost units: a pair costs
//    kPieceUnits (the work a CTA spends on one more piece: its merge and the
//    pipeline bubble around it, about a tile and a quarter of streaming,
//    measured) followed by kTileUnits per tile.  When all sequences have the
//    same length the pairs line up with the CTA ranges on their own and the
//    per-pair charge is left out (piece units 0).  CTA i of G takes the units
//    [floor(i*U/G), floor((i+1)*U/G)) of the U in all, and with them every tile
//    whose unit position falls inside; a range that crosses pair boundaries
//    yields one piece per pair it touches.  Every CTA therefore gets the same
//    cost (to a tile), so a CTA that meets many short sequences streams fewer
//    keys.  A tile t of a pair starting at unit v sits at unit
//    v + kPieceUnits + kTileUnits*t.
//
// A "virtual kv head" is one KV head together with a sub-group of at most
// max_group of the query heads that share it (16 for bf16 caches, whose
// tensor-core engine takes sixteen heads; 8 for fp32); when g <= max_group
// there is one sub-group per KV head.
//
// The balanced plan uses G = min(CTAs launched, U / kTileUnits) CTAs: every
// range is at least a tile's worth of units wide, so a range that lies inside
// a pair's tiles holds at least one of them and the CTAs holding one pair are
// consecutive (a CTA whose range falls between two pairs' tiles may hold none
// and idles).
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

// Exact floor(n / d) for 0 <= n, 0 < d; 32-bit division whenever both fit
// (a 64-bit division is a long instruction sequence on the GPU, and the plan
// is walked at the start of every CTA and of every piece).
FD_HD int64_t div_floor(int64_t n, int64_t d) {
  if (n <= 0xffffffffLL && d <= 0xffffffffLL) return (int64_t)((uint32_t)n / (uint32_t)d);
  return n / d;
}

// Cost units of the balanced plan (see the top of this file).
constexpr int kTileUnits = 4;
constexpr int kPieceUnits = 5;

// Units of one pair with `tiles` tiles (none for an empty sequence); `piece`
// is the plan's charge per pair (kPieceUnits, or 0 when every sequence has the
// same length: the pairs then line up with the CTA ranges as well as the
// plain split allows, and the charge would only shift work around).
FD_HD int64_t pair_units(int32_t tiles, int32_t piece) {
  return tiles > 0 ? (int64_t)kTileUnits * tiles + piece : 0;
}

// CTAs that take part in the balanced plan of `units` cost units on `launched` CTAs.
FD_HD int32_t balanced_ctas(int64_t units, int32_t launched) {
  const int64_t cap = units / kTileUnits;
  return cap < (int64_t)launched ? (int32_t)cap : launched;
}

// Balanced plan: CTA range bounds (in units) and the CTA owning a unit.
FD_HD int64_t range_begin(int64_t units, int32_t grid, int32_t cta) {
  return div_floor(units * (int64_t)cta, (int64_t)grid);
}

FD_HD int32_t cta_of_unit(int64_t units, int32_t grid, int64_t u) {
  return (int32_t)div_floor((u + 1) * (int64_t)grid - 1, units);
}

// Index of the first tile of the pair starting at unit v whose unit position
// is at or after unit r (may be past the pair's last tile).
FD_HD int32_t first_tile_at(int64_t r, int64_t v, int32_t piece) {
  const int64_t d = r - v - piece;
  return d <= 0 ? 0 : (int32_t)div_floor(d + kTileUnits - 1, kTileUnits);
}

// One unit of work: a run of consecutive keys of one (b, virtual kv head).
struct Piece {
  int32_t b, vkv;
  int32_t tok_begin, tok_end;  // keys [tok_begin, tok_end), already clipped to L_b
  int32_t slot;                // balanced: output slot; explicit: split index
  int32_t len;                 // L_b, the valid length of sequence b
};

// Walk of one CTA over its unit range in the balanced plan.  `Tiles` maps a
// sequence index b to prefix(b) (the units of the pairs of sequences < b, per
// virtual kv head), tiles(b) and len(b), and gives the plan's charge per pair
// as piece().
template <class Tiles>
struct BalancedWalk {
  const Tiles& tl;
  int32_t B, hv, cta;
  int64_t pos, end;  // current unit, end of range
  int32_t b, vkv;    // the pair holding `pos`
  int64_t v;         // its first unit

  FD_HD BalancedWalk(const Tiles& t, int32_t B_, int32_t hv_, int64_t units, int32_t grid, int32_t cta_)
      : tl(t), B(B_), hv(hv_), cta(cta_) {
    pos = range_begin(units, grid, cta);
    end = range_begin(units, grid, cta + 1);
    b = vkv = 0;
    v = 0;
    if (pos < end) locate();
  }

  FD_HD int64_t units_of(int32_t bb) const { return pair_units(tl.tiles(bb), tl.piece()); }

  // Binary search for the sequence holding `pos`, then the pair.
  FD_HD void locate() {
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {  // largest b with hv*prefix(b) <= pos
      int32_t mid = (lo + hi + 1) / 2;
      if ((int64_t)hv * tl.prefix(mid) <= pos) lo = mid; else hi = mid - 1;
    }
    b = lo;
    while (b < B - 1 && units_of(b) == 0) ++b;  // empty sequences own no units
    const int64_t base = (int64_t)hv * tl.prefix(b);
    const int64_t u = units_of(b);
    vkv = u > 0 ? (int32_t)div_floor(pos - base, u) : 0;
    v = base + (int64_t)vkv * u;
  }

  // Does the range hold units not walked yet?  (It may hold no further tile.)
  FD_HD bool done() const { return pos >= end; }

  // The next piece of the range; false when no tile is left in it.
  FD_HD bool next(Piece& pc) {
    while (pos < end) {
      const int32_t nt = tl.tiles(b);
      const int64_t pend = v + pair_units(nt, tl.piece());
      const int64_t stop = end < pend ? end : pend;
      const int32_t lo = first_tile_at(pos, v, tl.piece());
      int32_t hi = first_tile_at(stop, v, tl.piece());
      hi = hi < nt ? hi : nt;
      const int32_t cb = b, cv = vkv;
      pos = stop;
      if (pos == pend) {  // step to the next pair
        v = pend;
        if (++vkv == hv) {
          vkv = 0;
          ++b;
          while (b < B - 1 && tl.tiles(b) == 0) ++b;
        }
      }
      if (hi > lo) {
        const int32_t L = tl.len(cb);
        pc.b = cb;
        pc.vkv = cv;
        pc.tok_begin = lo * kPlanTile;
        const int32_t e = hi * kPlanTile;
        pc.tok_end = e < L ? e : L;
        pc.len = L;
        pc.slot = (cb * hv + cv) + cta;
        return true;
      }
    }
    return false;
  }
};

// Pieces of pair p = b*hv + vkv in the balanced plan: CTAs [first, last].
template <class Tiles>
FD_HD void balanced_pair_ctas(const Tiles& tl, int32_t hv, int64_t units, int32_t grid, int32_t b, int32_t vkv,
                              int32_t* first, int32_t* last) {
  const int32_t nt = tl.tiles(b);
  const int64_t v = (int64_t)hv * tl.prefix(b) + (int64_t)vkv * pair_units(nt, tl.piece());
  *first = cta_of_unit(units, grid, v + tl.piece());
  *last = cta_of_unit(units, grid, v + tl.piece() + (int64_t)kTileUnits * (nt - 1));
}

}  // namespace fdk
