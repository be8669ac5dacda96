// fd_split_mma.cuh -- tensor-core tile engine of the split kernel, for bf16
// K/V caches with four or eight query heads per CTA (GQA groups of 4 or 8, or
// larger groups taken eight heads at a time).
//
// With g heads per KV head every key costs 4*D*g flops against 4*D bytes of K
// and V, plus the widening of every bf16 element; on CUDA cores, from g = 4 on,
// that arithmetic keeps the kernel well above the time the TMA stream alone
// takes.  Here one warp handles its 32 keys of a stage with mma.sync m16n8k16
// (bf16 in, fp32 accumulate), heads on the M axis (rows >= g are idle):
//
//   q.k:  A = the g heads' q rows, split into bf16 hi (rows 0-7) and lo
//         (rows 8-15) parts with q = hi + lo to ~2^-16; B = K^T straight from the
//         swizzled stage via ldmatrix.  One MMA yields q_hi.k and q_lo.k in the
//         same thread (C rows g and g+8), whose sum is q.k to fp32 accuracy.
//   p.V:  A = p in the same hi/lo split, built in registers from the q.k
//         accumulators (the C layout of q.k is the A layout of p.V); B = V via
//         ldmatrix.trans.  O accumulates p_hi.V in rows 0-7 and p_lo.V in rows
//         8-15; the two are added when the warp publishes its state.
//
// K and V are bf16, so only q and p are split; the products are exact in fp32
// and accumulate in fp32.  The online softmax keeps a reference max per head
// and rescales only when a score rises more than kMmaTau (base 2) above it, so
// p <= 2^kMmaTau; the true max is tracked alongside and restored on publish.
#pragma once

#include <cuda_bf16.h>

#include "fd_device.cuh"

namespace fdk {

constexpr float kMmaTau = 8.0f;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// (x0, x1) = hi + lo with hi, lo in bf16; each returned as a packed pair with
// x0's part in the low half (the element order of an MMA fragment register).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 r = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

template <class C>
struct MmaEngine {
  static constexpr int D = C::D;
  static constexpr int KS = D / 16;  // k-steps of q.k
  static constexpr int NT = D / 8;   // n-tiles of p.V
  static constexpr int kRowStride = 128;
  static constexpr int kBlk = C::kBT * 128;  // bytes of one 128-byte column block of a stage tile
  static constexpr int G = C::G;
  static_assert((G == 4 || G == 8) && C::kBf16 && C::kBT == 128 && C::kWarps == 4, "MMA engine layout");

  static constexpr bool kQInSmem = false;
  uint32_t qa[KS][4];  // A fragments of q (hi rows 0-7, lo rows 8-15) for each k-step
  float o[NT][4];      // p.V accumulators: [.][0..1] from p_hi, [.][2..3] from p_lo
  float m, mt, l;      // head g of this lane's quad: reference max, true max, partial sum of p
  int32_t lim;         // keys head g's row may see
  int warp, lane, g, t;
  uint32_t kb[2], koff[KS];         // ldmatrix row address parts for K
  uint32_t vb[2], voffs[NT / 2];    // ... and for V (transposed)
  uint32_t zoff;                    // this lane's bytes of a row when clearing V rows

  __device__ __forceinline__ void setup(int warp_, int lane_, uint8_t*) {
    warp = warp_;
    lane = lane_;
    g = lane >> 2;
    t = lane & 3;
    const int mi = lane >> 3, r = lane & 7;
    // K (q.k B operand): matrix mi covers keys [8*(mi>>1), +8) and 16-byte chunk (mi&1) of the k-step
#pragma unroll
    for (int np = 0; np < 2; ++np) kb[np] = (32 * warp + 16 * np + (mi >> 1) * 8 + r) * kRowStride;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int cc = 2 * kk + (mi & 1);
      koff[kk] = (cc >> 3) * kBlk + (((cc & 7) ^ r) << 4);
    }
    // V (p.V B operand, transposed): matrix mi covers keys [8*(mi&1), +8) and d-chunk (mi>>1)
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) vb[j2] = (32 * warp + 16 * j2 + (mi & 1) * 8 + r) * kRowStride;
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int cc = 2 * np + (mi >> 1);
      voffs[np] = (cc >> 3) * kBlk + (((cc & 7) ^ r) << 4);
    }
    const int zb = lane * (D / 16);  // D/16 bytes per lane cover a 2*D-byte row
    zoff = (zb / 128) * kBlk + (zb % 128);
  }

  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    mt = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[n][j] = 0.f;
  }

  // q rows of the piece (fp32 in shared memory), times scale*log2(e), split hi/lo.
  __device__ __forceinline__ void begin(uint32_t qaddr, float qk_scale, const RowLimits& rl) {
    lim = g < G ? rl(g) : 0;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const uint32_t a = qaddr + (g * D + 16 * kk + 2 * t) * 4;
      float2 x0 = make_float2(0.f, 0.f), x1 = x0;  // rows of heads >= G stay zero
      if (g < G) {
        x0 = lds64f(a);       // d, d+1
        x1 = lds64f(a + 32);  // d+8, d+9
      }
      split_bf16x2(x0.x * qk_scale, x0.y * qk_scale, qa[kk][0], qa[kk][1]);
      split_bf16x2(x1.x * qk_scale, x1.y * qk_scale, qa[kk][2], qa[kk][3]);
    }
  }

  __device__ __forceinline__ void tile(uint32_t kst, uint32_t vst, int nv, uint32_t, float, int32_t tok0) {
    if (nv < 32) {
      // Rows past the valid keys get p = 0, but 0 * NaN is NaN: clear those V rows.
      for (int r = nv; r < 32; ++r) {
        const uint32_t a = vst + (32 * warp + r) * kRowStride + zoff;
        if constexpr (D == 128)
          asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(a), "r"(0u) : "memory");
        else
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(0u) : "memory");
      }
      // the producer's next TMA write to this stage must come after these stores
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    const bool two = nv > 16;  // second group of 16 keys holds valid keys
    // ---- q.k: S[head][key] for 32 keys, hi rows 0-7 + lo rows 8-15
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[n][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kst + kb[0] + koff[kk], b0, b1, b2, b3);
      mma_bf16_16816(sc[0], qa[kk], b0, b1);
      mma_bf16_16816(sc[1], qa[kk], b2, b3);
      if (two) {
        ldsm_x4(kst + kb[1] + koff[kk], b0, b1, b2, b3);
        mma_bf16_16816(sc[2], qa[kk], b0, b1);
        mma_bf16_16816(sc[3], qa[kk], b2, b3);
      }
    }
    // ---- online softmax for head g over the warp's keys
    float s[4][2];
    float smax = -INFINITY;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = 8 * n + 2 * t + j;
        const float v = sc[n][j] + sc[n][j + 2];
        s[n][j] = (key < nv && tok0 + 32 * warp + key < lim) ? v : -INFINITY;
        smax = fmaxf(smax, s[n][j]);
      }
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
    mt = fmaxf(mt, smax);
    if (smax > m + kMmaTau) {
      const float mn = fmaxf(m, smax);
      const float alpha = exp2f(m - mn);
      l *= alpha;
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[n][j] *= alpha;
      m = mn;
    }
    // a head whose row has seen no key yet (m = -inf) gets p = 0 for every key
    const float mref = m == -INFINITY ? 0.f : m;
    uint32_t pa[2][4];
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) {
      const float p00 = exp2f(s[2 * j2][0] - mref), p01 = exp2f(s[2 * j2][1] - mref);
      const float p10 = exp2f(s[2 * j2 + 1][0] - mref), p11 = exp2f(s[2 * j2 + 1][1] - mref);
      l += (p00 + p01) + (p10 + p11);
      split_bf16x2(p00, p01, pa[j2][0], pa[j2][1]);
      split_bf16x2(p10, p11, pa[j2][2], pa[j2][3]);
    }
    // ---- p.V
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) {
      if (j2 == 1 && !two) break;
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + vb[j2] + voffs[np], b0, b1, b2, b3);
        mma_bf16_16816(o[2 * np], pa[j2], b0, b1);
        mma_bf16_16816(o[2 * np + 1], pa[j2], b2, b3);
      }
    }
  }

  // Warp state -> merge slot `warp`, moved onto the true max of each head.
  __device__ __forceinline__ void publish(float* obuf, float* mlbuf, int) {
    const float f = m == -INFINITY ? 0.f : exp2f(m - mt);
    float ls = l + __shfl_xor_sync(0xffffffffu, l, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    if (g >= G) return;  // idle rows
    float* row = obuf + (warp * G + g) * C::kObStride + 2 * t;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2*>(row + 8 * n) = make_float2((o[n][0] + o[n][2]) * f, (o[n][1] + o[n][3]) * f);
    if (t == 0) {
      mlbuf[(warp * G + g) * 2] = mt;
      mlbuf[(warp * G + g) * 2 + 1] = ls * f;
    }
  }
};

// Sixteen heads per CTA (GQA groups of 16, or several query rows per head):
// all sixteen rows of the M axis are heads, so q and p each take two MMAs,
// one for the bf16 hi part and one for the lo part, accumulated into the same
// fp32 registers.  Lane (g, t) holds heads g (C/A rows 0-7) and g + 8 (rows
// 8-15); everything else -- stage layout, ldmatrix addressing, V-row clearing,
// lazy rescaling -- follows MmaEngine.  Per head and key the MMA work is the
// same as there; the K/V tile is read once for all sixteen heads.
template <class C>
struct MmaEngine16 {
  static constexpr int D = C::D;
  static constexpr int KS = D / 16;
  static constexpr int NT = D / 8;
  static constexpr int kRowStride = 128;
  static constexpr int kBlk = C::kBT * 128;
  static_assert(C::G == 16 && C::kBf16 && C::kBT == 128 && C::kWarps == 4, "MMA-16 engine layout");
  static_assert(KS % 4 == 0 && KS * 1024 <= C::kUBytes, "q fragments fit the publish buffer");

  static constexpr bool kQInSmem = true;  // begin() writes q's fragments to shared memory
  float o[NT][4];                 // p.V accumulators: [.][0..1] head g, [.][2..3] head g + 8
  float m[2], mt[2], l[2];        // heads g, g + 8: reference max, true max, partial sum
  int32_t lim[2];                 // keys each of the two heads' rows may see
  int32_t lim_w;                  // the least row limit of the piece's live heads, over the warp
  int warp, lane, g, t;
  uint32_t kb[2], vb[2];  // ldmatrix row addresses (K, V transposed)
  uint32_t kx, vx;        // this lane's swizzle term of the 16-byte chunk index, times 16
  uint32_t zoff;
  uint32_t fb;            // q's A fragments in shared memory: [k-step][hi, lo][lane] x 16 bytes

  // Byte offset of 16-byte chunk pair `c` (k-step or d-pair index) within a
  // swizzled row: chunk 2c + (lane bit) of block c / 4, XOR-swizzled by row.
  static __device__ __forceinline__ uint32_t chunk_off(int c, uint32_t x) {
    return (uint32_t)(c >> 2) * kBlk + (((uint32_t)(2 * (c & 3)) << 4) ^ x);
  }

  __device__ __forceinline__ void setup(int warp_, int lane_, uint8_t* smem) {
    warp = warp_;
    lane = lane_;
    g = lane >> 2;
    t = lane & 3;
    const int mi = lane >> 3, r = lane & 7;
    // K: matrix mi covers keys [8*(mi>>1), +8) and chunk (mi&1) of the k-step;
    // V (transposed): keys [8*(mi&1), +8) and d-chunk (mi>>1) of the pair
#pragma unroll
    for (int np = 0; np < 2; ++np) kb[np] = (32 * warp + 16 * np + (mi >> 1) * 8 + r) * kRowStride;
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) vb[j2] = (32 * warp + 16 * j2 + (mi & 1) * 8 + r) * kRowStride;
    kx = (uint32_t)((mi & 1) ^ r) << 4;
    vx = (uint32_t)((mi >> 1) ^ r) << 4;
    const int zb = lane * (D / 16);
    zoff = (zb / 128) * kBlk + (zb % 128);
    fb = smem_addr(smem) + C::kUOff;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      m[i] = -INFINITY;
      mt[i] = -INFINITY;
      l[i] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[n][j] = 0.f;
  }

  // q rows of the piece (fp32 in shared memory), times scale*log2(e), split
  // hi/lo into the A fragments of every k-step; the four warps convert a
  // quarter each into the publish buffer, idle until the piece ends.  The
  // caller's barrier after begin() makes all of them visible.
  __device__ __forceinline__ void begin(uint32_t qaddr, float qk_scale, const RowLimits& rl) {
    lim[0] = rl(g);
    lim[1] = rl(g + 8);
    // heads past the piece's live ones (lim 0) are never published: no bound for them
    int32_t lw = min(g < rl.nh ? lim[0] : 0x7fffffff, g + 8 < rl.nh ? lim[1] : 0x7fffffff);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) lw = min(lw, __shfl_xor_sync(0xffffffffu, lw, o));
    lim_w = lw;
#pragma unroll
    for (int j = 0; j < KS / 4; ++j) {
      const int kk = warp * (KS / 4) + j;
      const uint32_t a = qaddr + (g * D + 16 * kk + 2 * t) * 4;
      const uint32_t b = a + 8 * D * 4;  // row g + 8
      const float2 x0 = lds64f(a), x1 = lds64f(a + 32);
      const float2 y0 = lds64f(b), y1 = lds64f(b + 32);
      uint32_t h[4], l[4];
      split_bf16x2(x0.x * qk_scale, x0.y * qk_scale, h[0], l[0]);  // row g,     k 2t..
      split_bf16x2(y0.x * qk_scale, y0.y * qk_scale, h[1], l[1]);  // row g + 8, k 2t..
      split_bf16x2(x1.x * qk_scale, x1.y * qk_scale, h[2], l[2]);  // row g,     k 2t+8..
      split_bf16x2(y1.x * qk_scale, y1.y * qk_scale, h[3], l[3]);  // row g + 8, k 2t+8..
      const uint32_t f = fb + (uint32_t)kk * 1024 + lane * 16;
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(f), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(f + 512), "r"(l[0]), "r"(l[1]), "r"(l[2]),
                   "r"(l[3])
                   : "memory");
    }
  }

  __device__ __forceinline__ void qfrag(int kk, uint32_t (&h)[4], uint32_t (&l)[4]) const {
    const uint32_t f = fb + (uint32_t)kk * 1024 + lane * 16;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
                 : "r"(f));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(l[0]), "=r"(l[1]), "=r"(l[2]), "=r"(l[3])
                 : "r"(f + 512));
  }

  __device__ __forceinline__ void tile(uint32_t kst, uint32_t vst, int nv, uint32_t, float, int32_t tok0) {
    // A full stage that no head's row limit cuts (every stage but the last of
    // a piece) takes the straight-line path: no masks and no branches but the
    // rare rescale, so the compiler can overlap one key half's softmax with
    // the other half's MMAs.
    if (nv == 32 && tok0 + 32 * warp + 32 <= lim_w) {
      tile_impl<true>(kst, vst, 32, tok0);
      return;
    }
    if (nv < 32) {
      // Rows past the valid keys get p = 0, but 0 * NaN is NaN: clear those V rows.
      for (int r = nv; r < 32; ++r) {
        const uint32_t a = vst + (32 * warp + r) * kRowStride + zoff;
        if constexpr (D == 128)
          asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(a), "r"(0u) : "memory");
        else
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(0u) : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    tile_impl<false>(kst, vst, nv, tok0);
  }

  template <bool kFull>
  __device__ __forceinline__ void tile_impl(uint32_t kst, uint32_t vst, int nv, int32_t tok0) {
    const bool two = kFull || nv > 16;
    // ---- q.k: q_hi.k and q_lo.k in separate accumulators (independent MMA chains)
    float sc[4][4], sl[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[n][j] = sl[n][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t qh[4], ql[4];
      qfrag(kk, qh, ql);
      uint32_t b0, b1, b2, b3, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
      ldsm_x4(kst + kb[0] + chunk_off(kk, kx), b0, b1, b2, b3);
      if (two) ldsm_x4(kst + kb[1] + chunk_off(kk, kx), c0, c1, c2, c3);
      mma_bf16_16816(sc[0], qh, b0, b1);
      mma_bf16_16816(sc[1], qh, b2, b3);
      if (two) {
        mma_bf16_16816(sc[2], qh, c0, c1);
        mma_bf16_16816(sc[3], qh, c2, c3);
      }
      mma_bf16_16816(sl[0], ql, b0, b1);
      mma_bf16_16816(sl[1], ql, b2, b3);
      if (two) {
        mma_bf16_16816(sl[2], ql, c0, c1);
        mma_bf16_16816(sl[3], ql, c2, c3);
      }
    }
    // ---- online softmax, heads g (i = 0) and g + 8 (i = 1)
    float s[2][4][2];
    float smax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = 8 * n + 2 * t + j;
        const bool in = key < nv;
        const int32_t tok = tok0 + 32 * warp + key;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float v = sc[n][2 * i + j] + sl[n][2 * i + j];
          s[i][n][j] = (kFull || (in && tok < lim[i])) ? v : -INFINITY;
          smax[i] = fmaxf(smax[i], s[i][n][j]);
        }
      }
    float mref[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      smax[i] = fmaxf(smax[i], __shfl_xor_sync(0xffffffffu, smax[i], 1));
      smax[i] = fmaxf(smax[i], __shfl_xor_sync(0xffffffffu, smax[i], 2));
      mt[i] = fmaxf(mt[i], smax[i]);
      if (smax[i] > m[i] + kMmaTau) {
        const float mn = fmaxf(m[i], smax[i]);
        const float alpha = exp2f(m[i] - mn);
        l[i] *= alpha;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][2 * i] *= alpha;
          o[n][2 * i + 1] *= alpha;
        }
        m[i] = mn;
      }
      // a head whose row has seen no key yet (m = -inf) gets p = 0 for every key
      mref[i] = m[i] == -INFINITY ? 0.f : m[i];
    }
    // ---- per 16-key half: p as A fragments, then p.V.  a0 = (row g, keys
    // 2t..), a1 = (row g+8, keys 2t..), a2 = (row g, keys 2t+8..), a3 = (row
    // g+8, keys 2t+8..) of the half.
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) {
      if (j2 == 1 && !two) break;
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float p0 = exp2f(s[i][2 * j2][0] - mref[i]), p1 = exp2f(s[i][2 * j2][1] - mref[i]);
        const float p2 = exp2f(s[i][2 * j2 + 1][0] - mref[i]), p3 = exp2f(s[i][2 * j2 + 1][1] - mref[i]);
        l[i] += (p0 + p1) + (p2 + p3);
        split_bf16x2(p0, p1, ph[i], pl[i]);
        split_bf16x2(p2, p3, ph[2 + i], pl[2 + i]);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; np += 2) {
        uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
        ldsm_x4_t(vst + vb[j2] + chunk_off(np, vx), b0, b1, b2, b3);
        ldsm_x4_t(vst + vb[j2] + chunk_off(np + 1, vx), c0, c1, c2, c3);
        mma_bf16_16816(o[2 * np], ph, b0, b1);
        mma_bf16_16816(o[2 * np + 1], ph, b2, b3);
        mma_bf16_16816(o[2 * np + 2], ph, c0, c1);
        mma_bf16_16816(o[2 * np + 3], ph, c2, c3);
        mma_bf16_16816(o[2 * np], pl, b0, b1);
        mma_bf16_16816(o[2 * np + 1], pl, b2, b3);
        mma_bf16_16816(o[2 * np + 2], pl, c0, c1);
        mma_bf16_16816(o[2 * np + 3], pl, c2, c3);
      }
    }
  }

  // Round r publishes heads 8r..8r+7 (this lane's head g + 8r) into merge
  // slot `warp`, moved onto the true max.
  __device__ __forceinline__ void publish(float* obuf, float* mlbuf, int r) {
    const bool hi = r != 0;
    const float mi = hi ? m[1] : m[0];
    const float mti = hi ? mt[1] : mt[0];
    const float li = hi ? l[1] : l[0];
    const float f = mi == -INFINITY ? 0.f : exp2f(mi - mti);
    float ls = li + __shfl_xor_sync(0xffffffffu, li, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    float* row = obuf + (warp * 8 + g) * C::kObStride + 2 * t;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float a = hi ? o[n][2] : o[n][0];
      const float b = hi ? o[n][3] : o[n][1];
      *reinterpret_cast<float2*>(row + 8 * n) = make_float2(a * f, b * f);
    }
    if (t == 0) {
      mlbuf[(warp * 8 + g) * 2] = mti;
      mlbuf[(warp * 8 + g) * 2 + 1] = ls * f;
    }
  }
};

}  // namespace fdk
