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
  __device__ __forceinline__ void publish(float* obuf, float* mlbuf) {
    const float f = m == -INFINITY ? 0.f : exp2f(m - mt);
    float ls = l + __shfl_xor_sync(0xffffffffu, l, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    if (g >= G) return;  // idle rows
    float* row = obuf + (warp * G + g) * D + 2 * t;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2*>(row + 8 * n) = make_float2((o[n][0] + o[n][2]) * f, (o[n][1] + o[n][3]) * f);
    if (t == 0) {
      mlbuf[(warp * G + g) * 2] = mt;
      mlbuf[(warp * G + g) * 2 + 1] = ls * f;
    }
  }
};

}  // namespace fdk
