// fd_prefill.cu -- attention for many query rows per sequence (prefill, or a
// long window of new tokens), on the 5th-generation tensor cores.
//
// The rows are the last n_q tokens of each sequence, whose keys are already in
// the cache; with causal masking row i sees keys t < L_b - (n_q - 1 - i)
// (the same operation as fd_decode_rows, for windows too long to serve as
// virtual heads).  "FlashDecoding and split-KV", section "Walking through it",
// contrasts this phase -- many query rows, FlashAttention's tiling along the
// query axis -- with decode.
//
// Work item: (batch, pair of query heads of one GQA group -- or one head when
// the group size is odd --, tile of kPrefillRows = 128 query rows), taken
// longest first by one CTA per SM from a queue (a global counter).  Ten warps
// (twelve with one head per CTA: warps 2 and 3 have no role there, and the
// softmax groups are warps 4-7 and 8-11):
//   warp 0    TMA producer: 128-key K tiles and V tiles (16-row x 128-byte
//             boxes, the 128-byte swizzle), each into its own slot of a ring of
//             3 slots (6 for D = 64), shared by both heads; with one head per
//             CTA the second head's q area adds two slots;
//   warp 1    allocates all 512 TMEM columns and issues tcgen05.mma from one
//             thread, per head: S = Q K^T (M=128, N=128, K=D) into the head's
//             TMEM buffer, O += P V (M=128, N=D, K=128) into its accumulator,
//             in the order S0(j), PV1(j-1), S1(j), PV0(j), so that while one
//             head's softmax runs the tensor core works for the other head;
//   warps 2-5 and 6-9: the two heads' softmax groups.  Thread = query row =
//             TMEM lane; reads the tile's 128 scores with tcgen05.ld, masks,
//             keeps the running max and sum, writes P (bf16 hi and lo) back
//             over the same columns with tcgen05.st, rescales O in TMEM when
//             the max moves, and finally writes O / l.
// P . V takes A = P straight from TMEM.  Each head has one S buffer: S of tile
// j+1 is issued after P . V of tile j, which reads P from that buffer, and the
// tensor core runs one CTA's MMAs in issue order.  For the same reason the
// softmax may rescale O as soon as it sees S of tile j: P . V of tile j-1 was
// issued before that S, and the commit that signals S tracks it too.
// K and V are bf16, so the products are exact once q and p are bf16: q (times
// scale*log2 e) and p are split into bf16 hi + lo parts and each product is
// issued twice (hi, then lo) into the same fp32 accumulator -- two MMAs buy
// fp32-level accuracy.  The online softmax rescales lazily: the reference max
// moves only when a score exceeds it by kTau (base 2), so p <= 2^kTau; the
// softmax's arithmetic goes two keys per instruction (packed fp32), which is
// what its time per tile, and with it the steady state, depends on.
#include <cuda_bf16.h>

#include "fd_device.cuh"
#include "fd_prefill.h"

namespace fdk {
namespace {

constexpr int kM = kPrefillRows;   // query rows per CTA (TMEM lanes)
constexpr int kN = kPrefillKeys;   // keys per tile
// Threads: producer and MMA warps, then two softmax groups of four warps from
// warp kSoftmax0.  With one head per CTA two idle warps complete the first
// warpgroup, which setmaxnreg needs (measured: the two-head variant runs ~2 %
// faster without them).
template <int NG>
constexpr int kSoftmax0 = NG == 2 ? 2 : 4;
template <int NG>
constexpr int kThreads = (kSoftmax0<NG> + 8) * 32;
// Registers: the launch gives every thread kLaunchRegs (65536 / 384, rounded
// down to 8).  With one head per CTA the first warpgroup then gives registers
// back (setmaxnreg.dec) and the softmax warpgroups take them (setmaxnreg.inc),
// so that a thread holds a tile's 128 scores without spilling (measured +5 %
// there; with two heads per CTA the issuing thread's code is the one that
// matters, and it keeps the launch count).  An increase waits until the CTA's
// pool has the registers, so the split must add up exactly; the host launches
// that variant only when the compiled kernel has kLaunchRegs registers.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads<1> * kLaunchRegs, "register split exceeds the pool");
static_assert(kRegsLow + 2 * kRegsHigh <= 512, "one warp of each group per sub-partition: 16384 registers");
constexpr float kTau = 8.0f;
constexpr float kSumFast = 128.0f;  // 2^(tau - 1): see the softmax
constexpr float kLn2f = 0.6931471805599453f;
constexpr uint32_t kTmemCols = 512;  // per head (256 each): S / P at +0, O (D columns) at +128

// Shared-memory layout for head dim D (64 or 128), byte offsets from a
// 1024-aligned base.  A row of D bf16 is D/64 column blocks of 128 bytes.
template <int D>
struct PLayout {
  static constexpr int kNB = D / 64;
  static constexpr uint32_t kQhi = 0;                           // per head: [kNB][128 rows][128 B] hi, then lo
  static constexpr uint32_t kQlo = kNB * 16384u;
  static constexpr uint32_t kQGroupBytes = 2 * kQlo;
  static constexpr uint32_t kTileBytes = kNB * 16384u;          // one K or V tile: [kNB][128 rows][128 B]
  static constexpr uint32_t kBlockBytes = 16384u;               // one 128-byte column block of a tile
  static constexpr uint32_t kSlot0 = 2 * kQGroupBytes;
  // K and V tiles take one slot each, K(j) then V(j); a slot is refilled once
  // the MMAs reading it have completed.  For D = 128 three slots are what fits
  // beside the two heads' q (227 KB in all).
  static constexpr int kSlots = D == 128 ? 3 : 6;
  static constexpr uint32_t kBarOff = kSlot0 + kSlots * kTileBytes;
  // at least 116 KB, so that one CTA fits per SM: each allocates all 512 TMEM columns
  static constexpr uint32_t kSmemNeed = kBarOff + 512 + 1024;  // barriers and flags, the 1024-byte alignment
  static constexpr uint32_t kSmemAlloc = kSmemNeed > 118784u ? kSmemNeed : 118784u;
  static_assert(D == 64 || D == 128, "head dim");
  // With one head per CTA the second head's q area holds two more slots.
  static constexpr int kSlotsOneHead = kSlots + 2;
  static_assert(kSlotsOneHead <= 8, "barrier area holds 8 slots");
  static_assert(2 * kTileBytes == kQGroupBytes, "two tiles fill one head's q area");
  __device__ static uint32_t slot_off(uint32_t slot) {
    return slot < (uint32_t)kSlots ? kSlot0 + slot * kTileBytes : kQGroupBytes + (slot - kSlots) * kTileBytes;
  }
  static_assert(kSmemAlloc <= 232448, "shared memory");
};

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (sm_100 family): bits 0-13 start address >> 4,
// 16-29 leading byte offset >> 4, 32-45 stride byte offset >> 4, 46 version 1,
// 61-63 swizzle mode (2 = 128-byte swizzle).
// Built in halves: the high word (stride byte offset 1024,
// version, swizzle) is a constant here; the low word holds the start address
// and the leading byte offset, so stepping through a tile is a 32-bit add on
// the low word (addresses stay below 256 KB: the 14-bit field never carries).
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t desc_of(uint32_t lo) { return ((uint64_t)kDescHi << 32) | lo; }

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// A from tensor memory (M rows in lanes, two bf16 of K per 32-bit column).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Ties 32 registers to the point after a tcgen05.wait::ld: an empty asm that
// "modifies" them, so the compiler cannot move their uses above the wait.
__device__ __forceinline__ void reg_fence32(float* v) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                 "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]),
                 "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]),
                 "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]),
                 "+f"(v[29]), "+f"(v[30]), "+f"(v[31]));
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  reg_fence32(v);
}

// The same load without the wait: several may be in flight before one
// tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's lane, no wait.
__device__ __forceinline__ void tmem_ld64_nw(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Register count of the calling warp's role (one head per CTA only).
template <int NG, uint32_t N>
__device__ __forceinline__ void regs_dec() {
  if constexpr (NG == 1) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int NG, uint32_t N>
__device__ __forceinline__ void regs_inc() {
  if constexpr (NG == 1) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// 2^x on the special-function unit (inputs here are <= 0 or -inf).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three (the sm_100 family's three-input max: a NaN input is ignored,
// as fmaxf ignores it).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 values in one 64-bit register (x in the low half) and the sm_100
// family's packed fp32 add / subtract / multiply, which round each half as the
// scalar instruction does: one instruction for two keys in the softmax.
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// x = hi + lo in bf16 for a packed pair (p = {x0, x1}, x0's parts in the low
// halves), for q: both rounded to nearest, the residual x - hi (exact in fp32)
// by one packed subtract.
__device__ __forceinline__ void split2_rn(float x0, float x1, uint64_t p, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const uint32_t hb = *reinterpret_cast<const uint32_t*>(&h);
  float r0, r1;
  f2_unpack(f2_sub(p, f2_pack(__uint_as_float(hb << 16), __uint_as_float(hb & 0xffff0000u))), r0, r1);
  const __nv_bfloat162 r = __floats2bfloat162_rn(r0, r1);
  hi = hb;
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// x = hi + lo for a packed pair (p = {x0, x1}, x0's parts in the low
// halves), for P: hi is x truncated to bf16 (the upper 16 bits, one byte
// permute for both), the residual x - hi is exact in fp32 (one packed
// subtract) and lo is its bf16 rounding.  |lo| < 2^-7 |x| and lo is good to
// 2^-9 of itself, so hi + lo holds x to 2^-16, with an unbiased error; the
// rounding conversion of split2_rn measured 3 % slower here.
__device__ __forceinline__ void split2_trunc(float x0, float x1, uint64_t p, uint32_t& hi, uint32_t& lo) {
  const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
  hi = __byte_perm(b0, b1, 0x7632);
  float r0, r1;
  f2_unpack(f2_sub(p, f2_pack(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u))), r0, r1);
  const __nv_bfloat162 r = __floats2bfloat162_rn(r0, r1);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Byte offset of 16-byte chunk `c` (8 bf16) of row `r` in a [rows][128 B] block
// with the 128-byte swizzle (block base 1024-aligned).
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + (((c ^ r) & 7u) << 4); }

__device__ __forceinline__ int32_t row_keys(const PrefillParams& p, int32_t L, int32_t qi) {
  if (qi >= p.n_q) return 0;
  if (!p.causal) return L;
  const int32_t lim = L - (p.n_q - 1 - qi);
  return lim < 0 ? 0 : (lim > L ? L : lim);
}

// Waits of every role: false when the CTA aborts or the wait times out.  A
// phase that has already completed costs one try_wait; the abort flag is read
// only when the thread has to wait.
// limit_ns: the kernel's wait limit, used only when the phase is not complete
// at the first try.
__device__ __forceinline__ bool bar_ok(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned long long limit_ns) {
  return mbar_try_wait(bar, parity) || (!*abort_flag && mbar_wait_for(bar, parity, limit_ns));
}

__device__ __forceinline__ bool wait_ok(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned long long limit_ns) {
  const bool r = bar_ok(bar, parity, abort_flag, limit_ns);
  tc_fence_after();
  return r;
}

// Position in the K/V slot ring: use u is slot u % n in phase (u / n) & 1,
// advanced incrementally (no division on the issue path).
struct Ring {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ Ring next(uint32_t by, uint32_t n) const {
    Ring r = *this;
    r.slot += by;
    if (r.slot >= n) {
      r.slot -= n;
      r.phase ^= 1u;
    }
    return r;
  }
};

// One work item: a tile of kM query rows of one sequence for `ngroups` heads.
struct Item {
  int32_t b, h0, m0, kvh, L, n_tiles;
};

// Items in order of decreasing work (causal: the latest query rows first), so
// that the hardware, handing out CTAs in index order, starts the long ones first.
__device__ __forceinline__ Item item_of(const PrefillParams& p, int32_t idx, int32_t ngroups, int32_t n_m) {
  const int32_t hp = p.Hq / ngroups;
  const int32_t per_m = hp * p.B;
  const int32_t mi = idx / per_m, rest = idx % per_m;
  Item it;
  it.m0 = (n_m - 1 - mi) * kM;
  it.h0 = (rest % hp) * ngroups;
  it.b = rest / hp;
  it.kvh = it.h0 / p.g;
  int32_t L = p.seq_lens ? __ldg(p.seq_lens + it.b) : p.max_len;
  it.L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
  const int32_t last_row = (p.n_q - it.m0 < kM ? p.n_q - it.m0 : kM) - 1;
  const int32_t keys_max = row_keys(p, it.L, it.m0 + last_row);  // rows' limits grow with the row
  it.n_tiles = (keys_max + kN - 1) / kN;
  return it;
}

// Each CTA starts with item blockIdx.x; with fewer CTAs than items it then
// takes item gridDim.x + (a global counter's next value) until they run out.
// The producer takes the indices and hands them to the MMA thread and the
// softmax warps through two shared-memory slots, so every role walks the same
// items, and all barrier
// phases follow two running counters of the CTA: g, the key tiles processed so
// far, and f, the items with at least one tile so far.  Slot uses are numbered
// u = 2 g (K) and 2 g + 1 (V): slot u % nslots, phase u / nslots.
// NG: query heads per CTA, 2 when the GQA group size is even, else 1.
template <int D, int NG, bool kHook>
__global__ void __launch_bounds__(kThreads<NG>, 1)
    fd_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_o,
                      const PrefillParams p) {
  using Lay = PLayout<D>;
  constexpr int kD = D;
  constexpr int kNB = Lay::kNB;
  constexpr uint32_t kQhi = Lay::kQhi, kQlo = Lay::kQlo, kQGroupBytes = Lay::kQGroupBytes;
  constexpr uint32_t kBlockBytes = Lay::kBlockBytes;
  constexpr uint32_t kBarOff = Lay::kBarOff;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* kv_full = bars;        // [nslots <= 8]
  uint64_t* kv_empty = bars + 8;   // [nslots <= 8]
  // One phase per key tile and S buffer.  Neither side can get two phases
  // ahead: S into a buffer is issued only after the P that the buffer last
  // held has arrived, and that P needed the S before it.
  uint64_t* s_full = bars + 16;    // [2 buffers]
  uint64_t* p_full = bars + 18;    // [2 buffers]
  uint64_t* o_final = bars + 20;   // [2 heads]: an item's last P.V has completed
  uint64_t* drain = bars + 23;
  uint64_t* o_done = bars + 24;    // one head per CTA only: a P.V has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 208);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + 212);
  // Each head's q area has barriers of its own, so that head 0 takes its next
  // item's q while head 1 still finishes the current item (its last P.V is
  // the CTA's last MMA).
  uint64_t* q_full = bars + 34;    // [2 heads]: the item's q tiles (fp32) have landed
  uint64_t* q_ready = bars + 36;   // [2 heads]: ... and are bf16 hi / lo
  uint64_t* q_free = bars + 38;    // [2 heads]: the q area may take the next item's q
  // The item queue: the producer takes item indices from a global counter and
  // hands them to the other roles through two slots (index -1 = no more items).
  uint64_t* item_full = bars + 28;   // [2]
  uint64_t* item_empty = bars + 30;  // [2]: one arrival from the MMA thread and one per softmax warp
  volatile int32_t* item_slot = reinterpret_cast<volatile int32_t*>(smem + kBarOff + 256);  // [2]

  // Two query heads of one GQA group share an item (and every K/V tile) when
  // the group size is even: head G has S buffer G (TMEM columns 256 G) and O
  // at 256 G + 128.  Otherwise the second softmax group idles and the one head
  // alternates between both S buffers, tile by tile, so that S of tile j+1 is
  // computed while the softmax works on tile j.
  constexpr int32_t ngroups = NG;
  constexpr uint32_t nslots = NG == 2 ? (uint32_t)Lay::kSlots : (uint32_t)Lay::kSlotsOneHead;
  const int32_t n_m = (p.n_q + kM - 1) / kM;
  const int32_t n_items = n_m * (p.Hq / ngroups) * p.B;
  // persistent CTAs taking items from p.work
  const bool queue = (int32_t)gridDim.x < n_items;

  if (tid == 0) {
    for (uint32_t i = 0; i < nslots; ++i) {
      mbar_init(kv_full + i, 1);
      mbar_init(kv_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 4);
      mbar_init(o_final + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(q_ready + i, 4);
      mbar_init(q_free + i, 1);
    }
    mbar_init(drain, 1);
    mbar_init(o_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(item_full + i, 1);
      mbar_init(item_empty + i, 1 + 4 * ngroups);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_o);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every wait's limit: the default, or with the testing hook the call's
  // (the instance without the hook keeps the constant).
  const unsigned long long wl = kHook && p.wait_ns ? p.wait_ns : kWaitLimitNs;
  bool ok = true;

  // Each role sets its register count first thing, so that the compiler
  // allocates the role's code for that count.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    regs_dec<NG, kRegsLow>();
    uint32_t u = 0;   // slot uses so far
    uint32_t fq[2] = {0u, 0u};  // per head: items with key tiles whose q this warp has loaded
    uint32_t stalled = 0xffffffffu;  // the copy skipped by the testing hook
    Ring pr;          // the next use's slot
    for (uint32_t e = 0;; ++e) {
      // take the next item (longest first) and announce it; -1 ends the walk
      int32_t idx = -1;
      if (lane == 0) {
        const uint32_t sl = e & 1u;
        if (e >= 2 && ok && !bar_ok(item_empty + sl, ((e >> 1) & 1u) ^ 1u, abort_flag, wl)) ok = false;
        if (ok) {
          // the first item is the CTA's own; then, with fewer CTAs than items,
          // the next one not yet taken
          const int32_t t = e == 0 ? (int32_t)blockIdx.x
                                   : (queue ? (int32_t)gridDim.x + (int32_t)atomicAdd(p.work, 1u) : n_items);
          idx = t < n_items ? t : -1;
        }
        item_slot[sl] = idx;
        mbar_arrive(item_full + sl);
      }
      idx = __shfl_sync(0xffffffffu, idx, 0);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (idx < 0) break;
      const Item it = item_of(p, idx, ngroups, n_m);
      if (it.n_tiles > 0) {
        // the item's q tiles, fp32, into each head's q area (the softmax group
        // converts them there), once the head's previous item is done with it
#pragma unroll
        for (int G = 0; G < ngroups; ++G) {
          if (lane == 0) {
            if (ok && fq[G] > 0 && !bar_ok(q_free + G, (fq[G] - 1) & 1u, abort_flag, wl)) ok = false;
            if (ok) {
              mbar_arrive_expect_tx(q_full + G, (uint32_t)(kD * kM * 4));
#pragma unroll
              for (int blk = 0; blk < kD / 32; ++blk)
                tma_load_3d(smem + (uint32_t)G * kQGroupBytes + (uint32_t)blk * kBlockBytes, &tmap_q, q_full + G,
                            blk * 32, it.m0, it.b * p.Hq + it.h0 + G);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok) ++fq[G];
        }
      }
      for (int32_t j = 0; j < it.n_tiles && ok; ++j) {
        // lane l brings rows [16 l, 16 l + 16) of the tile: one page run when paged
        const int32_t t0 = j * kN;
        const int32_t nvalid = it.L - t0 < kN ? it.L - t0 : kN;
        const int32_t tok = t0 + 16 * lane;
        bool mine = 16 * lane < nvalid;
        int32_t row = tok, z = it.b * p.Hkv + it.kvh;
        if (p.paged && mine) {
          const int32_t page = __ldg(p.block_table + (size_t)it.b * p.max_pages + tok / p.page_size);
          if (page < 0 || page >= p.num_pages) {
            atomicOr(p.err, kErrBadIndex);
            mine = false;
          }
          row = tok % p.page_size;
          z = page * p.Hkv + it.kvh;
        }
        const unsigned issue = __ballot_sync(0xffffffffu, mine);
        for (int kv = 0; kv < 2; ++kv, ++u, pr = pr.next(1, nslots)) {
          const uint32_t slot = pr.slot;
          if (lane == 0 && !bar_ok(kv_empty + slot, pr.phase ^ 1u, abort_flag, wl)) ok = false;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (kHook && p.stall_u >= 0 && u == (uint32_t)p.stall_u) {
            // testing hook: nothing is issued for this copy, so the waits for it run
            // out (and nothing is left in flight)
            stalled = u;
            continue;
          }
          if (lane == 0) mbar_arrive_expect_tx(kv_full + slot, (uint32_t)__popc(issue) * kNB * 2048u);
          __syncwarp();
          if (mine) {
            uint8_t* dst = smem + Lay::slot_off(slot) + lane * 2048;
            const CUtensorMap* map = kv == 0 ? &tmap_k : &tmap_v;
#pragma unroll
            for (int blk = 0; blk < kNB; ++blk) tma_load_3d(dst + blk * kBlockBytes, map, kv_full + slot, blk * 64, row, z);
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
    // do not leave while this warp's copies may still be landing
    if (lane == 0) {
      const uint32_t first = u > nslots ? u - nslots : 0;
      for (uint32_t t = first; t < u; ++t)
        if (t != stalled && !mbar_wait_for(kv_full + t % nslots, (t / nslots) & 1, wl)) atomicOr(p.err, kErrTimeout);
#pragma unroll
      for (int G = 0; G < ngroups; ++G)
        if (fq[G] > 0 && !mbar_wait_for(q_full + G, (fq[G] - 1) & 1u, wl)) atomicOr(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    regs_dec<NG, kRegsLow>();
    if (lane == 0) {
      constexpr uint32_t idS = instr_desc(kM, kN, false);
      constexpr uint32_t idO = instr_desc(kM, kD, true);
      uint32_t g = 0, f = 0;
      // S = Q_G K^T into TMEM column `d_col`, for the K tile in slot `slot`:
      // D/16 k-steps, hi then lo
      auto issue_s = [=](uint32_t d_col, int G, uint32_t slot) {
        const uint32_t d = tmem + d_col;
        const uint32_t q_lo = desc_lo(sbase + (uint32_t)G * kQGroupBytes, 0);
        const uint32_t k_lo = desc_lo(sbase + Lay::slot_off(slot), 0);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int s8 = 0; s8 < kD / 16; ++s8) {
            // k-step s8: column block s8 / 4, 32 bytes into it per step
            const uint32_t a_off = ((part ? kQlo : kQhi) + (uint32_t)(s8 >> 2) * 16384u + (uint32_t)(s8 & 3) * 32u) >> 4;
            const uint32_t b_off = ((uint32_t)(s8 >> 2) * kBlockBytes + (uint32_t)(s8 & 3) * 32u) >> 4;
            umma(d, desc_of(q_lo + a_off), desc_of(k_lo + b_off), idS, (part | s8) != 0);
          }
        }
      };
      // O (TMEM column o_col) += P V, P at column p_col, for the V tile in slot
      // `slot`: 16 keys per k-step (two 8-row groups of V); k-step kk's P hi is
      // in the buffer's columns [16 kk, 16 kk + 8), its lo in the next 8
      auto issue_pv = [=](uint32_t p_col, uint32_t o_col, uint32_t slot, bool first) {
        const uint32_t v_lo = desc_lo(sbase + Lay::slot_off(slot), kBlockBytes);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            umma_tmem_a(tmem + o_col, tmem + p_col + (uint32_t)kk * 16u + (uint32_t)part * 8u,
                        desc_of(v_lo + (uint32_t)kk * (2048u >> 4)), idO, (!first || part || kk) ? 1u : 0u);
          }
        }
      };
      Ring kr;  // K of the next tile
      for (uint32_t e = 0;; ++e) {
        const uint32_t sl = e & 1u;
        if (!wait_ok(item_full + sl, (e >> 1) & 1u, abort_flag, wl)) {
          ok = false;
          break;
        }
        const int32_t idx = item_slot[sl];
        mbar_arrive(item_empty + sl);
        if (idx < 0 || !ok) break;
        const Item it = item_of(p, idx, ngroups, n_m);
        const int32_t n = it.n_tiles;
        if (n == 0) continue;  // no q_ready phase either: the softmax skips such items too
        if (!wait_ok(q_ready + 0, f & 1, abort_flag, wl)) {
          ok = false;
          break;
        }
        if (ngroups == 2) {
          Ring vprev;  // V of the previous tile
          for (int32_t j = 0; j < n; ++j) {
            const uint32_t gj = g + (uint32_t)j;
            const Ring vr = kr.next(1, nslots);  // V of this tile
            if (!wait_ok(kv_full + kr.slot, kr.phase, abort_flag, wl)) {
              ok = false;
              break;
            }
            issue_s(0, 0, kr.slot);
            umma_commit(s_full + 0);
            if (j >= 1) {
              // head 1's P.V of the previous tile, then its S of this tile
              if (!wait_ok(p_full + 1, (gj - 1) & 1, abort_flag, wl)) {
                ok = false;
                break;
              }
              issue_pv(256, 384, vprev.slot, j == 1);
              umma_commit(kv_empty + vprev.slot);
            } else if (!wait_ok(q_ready + 1, f & 1, abort_flag, wl)) {
              // head 1's q, at the item's first tile
              ok = false;
              break;
            }
            issue_s(256, 1, kr.slot);
            umma_commit(s_full + 1);
            umma_commit(kv_empty + kr.slot);
            if (!wait_ok(kv_full + vr.slot, vr.phase, abort_flag, wl) || !wait_ok(p_full + 0, gj & 1, abort_flag, wl)) {
              ok = false;
              break;
            }
            issue_pv(0, 128, vr.slot, j == 0);
            if (j == n - 1) umma_commit(o_final + 0);
            vprev = vr;
            kr = kr.next(2, nslots);
          }
          if (!ok) break;
          if (!wait_ok(p_full + 1, (g + (uint32_t)n - 1) & 1, abort_flag, wl)) {
            ok = false;
            break;
          }
          issue_pv(256, 384, vprev.slot, n == 1);
          umma_commit(kv_empty + vprev.slot);
          umma_commit(o_final + 1);
        } else {
          // one head: S(j) into buffer j % 2, then P.V of tile j-1
          Ring vprev;  // V of the previous tile
          for (int32_t j = 0; j <= n; ++j) {
            const Ring vcur = kr.next(1, nslots);
            if (j < n) {
              const uint32_t gj = g + (uint32_t)j;
              if (!wait_ok(kv_full + kr.slot, kr.phase, abort_flag, wl)) {
                ok = false;
                break;
              }
              issue_s((gj & 1) * 256u, 0, kr.slot);
              umma_commit(s_full + (gj & 1));
              umma_commit(kv_empty + kr.slot);
            }
            if (j >= 1) {
              const uint32_t gp = g + (uint32_t)j - 1;
              if (!wait_ok(kv_full + vprev.slot, vprev.phase, abort_flag, wl) ||
                  !wait_ok(p_full + (gp & 1), (gp >> 1) & 1, abort_flag, wl)) {
                ok = false;
                break;
              }
              issue_pv((gp & 1) * 256u, 128, vprev.slot, j == 1);
              umma_commit(o_done);
              umma_commit(kv_empty + vprev.slot);
              if (j == n) umma_commit(o_final + 0);
            }
            if (j < n) {
              vprev = vcur;
              kr = kr.next(2, nslots);
            }
          }
          if (!ok) break;
        }
        g += (uint32_t)n;
        ++f;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, kErrTimeout);
      }
      // every MMA this thread issued has finished before TMEM is released
      umma_commit(drain);
      if (!mbar_wait_for(drain, 0, wl)) atomicOr(p.err, kErrTimeout);
    }
  } else if (warp < kSoftmax0<NG>) {
    regs_dec<NG, kRegsLow>();  // no role
  } else if ((warp - kSoftmax0<NG>) / 4 >= ngroups) {
    regs_inc<NG, kRegsHigh>();  // the second softmax group, idle with one head per CTA
  } else {
    // ------------------------------------------------------------ softmax, head G
    regs_inc<NG, kRegsHigh>();
    const int32_t G = (warp - kSoftmax0<NG>) / 4;
    const int32_t quarter = warp & 3;
    const int32_t r = quarter * 32 + lane;  // query row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t obase = tmem + (uint32_t)G * 256u + 128u + lane_off;  // this head's O
    const bool dual = ngroups == 1;  // one head, alternating S buffers
    const uint32_t qbase = sbase + (uint32_t)G * kQGroupBytes;
    uint32_t g = 0, f = 0;
    for (uint32_t e = 0;; ++e) {
      int32_t idx = -1;
      if (lane == 0) {
        const uint32_t sl = e & 1u;
        if (bar_ok(item_full + sl, (e >> 1) & 1u, abort_flag, wl)) idx = item_slot[sl];
        mbar_arrive(item_empty + sl);
      }
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (idx < 0) break;  // every warp of the group reads the same slot, so all leave together
      const Item it = item_of(p, idx, ngroups, n_m);
      const int32_t n = it.n_tiles;
      const int32_t h = it.h0 + G;
      const int32_t qi = it.m0 + r;
      const int32_t lim = row_keys(p, it.L, qi);
      if (n > 0) {
        // The item's q rows (fp32, landed by the producer's tensor loads in
        // this head's q area as [D/32 blocks][128 rows][128 B], 128-byte
        // swizzle), times scale*log2(e), become bf16 hi / lo in the swizzled A
        // layout over the same bytes.  Row r of either layout fills row slot r
        // of each 16 KB block, so every thread converts its own row in place:
        // fp32 columns [32b, 32b+32) sit in block b, the hi of columns
        // [64h, 64h+64) in block h and their lo in block D/64 + h; a block is
        // read before it is written.  The previous item is done with this area
        // (the producer waited for the head's q_free before the loads).
        if (ok && !bar_ok(q_full + G, f & 1, abort_flag, wl)) ok = false;
        auto load32 = [&](int blk, float* v) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 x = lds128(qbase + (uint32_t)blk * kBlockBytes + swz((uint32_t)r, (uint32_t)c));
            v[4 * c] = x.x;
            v[4 * c + 1] = x.y;
            v[4 * c + 2] = x.z;
            v[4 * c + 3] = x.w;
          }
        };
        // columns [64h, 64h+64) from v[64] -> hi block h, lo block kNB + h
        const uint64_t scale2 = f2_pack(p.qk_scale, p.qk_scale);
        auto store64 = [&](int hb, const float* v) {
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            uint32_t hi0, lo0, hi1, lo1;
            const uint64_t x01 = f2_mul(f2_pack(v[c], v[c + 1]), scale2);
            const uint64_t x23 = f2_mul(f2_pack(v[c + 2], v[c + 3]), scale2);
            float x0, x1, x2, x3;
            f2_unpack(x01, x0, x1);
            f2_unpack(x23, x2, x3);
            split2_rn(x0, x1, x01, hi0, lo0);
            split2_rn(x2, x3, x23, hi1, lo1);
            const uint32_t off = (uint32_t)hb * 16384u + swz((uint32_t)r, (uint32_t)(c >> 3)) + (uint32_t)((c >> 2) & 1) * 8u;
            sts64(qbase + kQhi + off, hi0, hi1);
            sts64(qbase + kQlo + off, lo0, lo1);
          }
        };
        if constexpr (kD == 128) {
          float v[96];
          load32(0, v);
          load32(1, v + 32);
          load32(2, v + 64);
          store64(0, v);  // hi -> block 0, lo -> block 2: both read
          load32(3, v);
          float w[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            w[i] = v[64 + i];
            w[32 + i] = v[i];
          }
          store64(1, w);  // hi -> block 1, lo -> block 3: both read
        } else {
          float v[64];
          load32(0, v);
          load32(1, v + 32);
          store64(0, v);  // hi -> block 0, lo -> block 1
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready + G);
      }

      // A failed wait never leaves the loop early (the epilogue's named barrier
      // needs all 128 threads of the group): later waits are skipped, the output
      // flagged.
      float mref = -INFINITY, l = 0.f;
      for (int32_t j = 0; j < n; ++j) {
        const uint32_t gj = g + (uint32_t)j;
        const uint32_t buf = dual ? (gj & 1) : (uint32_t)G, par = dual ? (gj >> 1) & 1 : gj & 1;
        const uint32_t tbase = tmem + buf * 256u + lane_off;  // this tile's S / P
        if (ok && !bar_ok(s_full + buf, par, abort_flag, wl)) ok = false;
        tc_fence_after();
        float s[kN];
#pragma unroll
        for (int c = 0; c < kN / 64; ++c) tmem_ld64_nw(tbase + (uint32_t)c * 64u, s + 64 * c);
        tmem_wait_ld();
        // mask the keys past this row's limit (only the tiles that reach it)
        const int32_t keys_left = lim - j * kN;
        if (keys_left < kN) {
#pragma unroll
          for (int c = 0; c < kN; ++c) s[c] = c < keys_left ? s[c] : -INFINITY;
        }
        // p = 2^(s - base) and its bf16 hi / lo over the same columns, one k-step
        // (16 keys) at a time: k-step kk's hi in columns 16 kk + [0, 8), its lo in
        // 16 kk + [8, 16), two keys per column.  The whole tile's S is in
        // registers already, so the stores may overwrite any of it.  Keys go in
        // pairs through the packed fp32 instructions: four running sums, keys 4i
        // and 4i+1 into the first pair, 4i+2 and 4i+3 into the second.  Returns
        // the row's sum of p.  Warp-collective (the TMEM stores).
        auto make_p = [&](float base) -> float {
          const uint64_t base2 = f2_pack(base, base);
          uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < kN / 16; ++c) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float t0, t1;
              f2_unpack(f2_sub(f2_pack(s[16 * c + 2 * e], s[16 * c + 2 * e + 1]), base2), t0, t1);
              const float p0 = ex2(t0), p1 = ex2(t1);
              const uint64_t p2 = f2_pack(p0, p1);
              sum2[e & 1] = f2_add(sum2[e & 1], p2);
              split2_trunc(p0, p1, p2, w[e], w[8 + e]);
            }
            tmem_st16u(tbase + (uint32_t)c * 16u, w);
          }
          float sum4[4];
          f2_unpack(sum2[0], sum4[0], sum4[1]);
          f2_unpack(sum2[1], sum4[2], sum4[3]);
          return (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        };
        // The running max moves (and O and l are rescaled) only when the tile's
        // max exceeds it by more than tau.  Once a row has a finite running max,
        // P is first made with it as the base: a sum of p below 2^(tau-1) means
        // that no key came within one of tau above it, so the max would not have
        // moved and P and the sum are exactly what the max-first order gives,
        // without the 128-key max.  Otherwise (a larger or NaN sum, the first
        // keys of a row) the warp takes the max-first order, P made again.
        bool rescale = false;
        float alpha = 1.f, psum = 0.f;
        bool slow = true;
        if (__any_sync(0xffffffffu, mref != -INFINITY)) {
          psum = make_p(mref != -INFINITY ? mref : 0.f);
          slow = mref == -INFINITY || !(psum < kSumFast);
        }
        if (__any_sync(0xffffffffu, slow)) {
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < kN; c += 8)
#pragma unroll
            for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], s[c + 2 * i], s[c + 2 * i + 1]);
          const float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
          rescale = mx > mref + kTau;
          if (rescale) {
            const float mn = fmaxf(mref, mx);
            alpha = mref == -INFINITY ? 0.f : ex2(mref - mn);
            mref = mn;
          }
          psum = make_p(mref == -INFINITY ? 0.f : mref);
        }
        l = l * alpha + psum;
        // Rescaling O needs the previous tile's P.V to have finished.  With two
        // heads it was issued before this tile's S, whose completion this group
        // just saw; with one head it comes after, and o_done tells (a parity
        // wait is exact: P.V of tile g-2 was issued before this S, and that of
        // tile g needs this P).  tcgen05.ld and st are warp-collective
        // (.sync.aligned): the whole warp rescales when any of its rows must,
        // the others with alpha = 1.
        if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
          if (dual && ok && !bar_ok(o_done, (gj - 1) & 1, abort_flag, wl)) ok = false;
          tc_fence_after();
#pragma unroll 1
          for (int c4 = 0; c4 < kD / 32; ++c4) {
            float o[32];
            tmem_ld32(obase + (uint32_t)c4 * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(obase + (uint32_t)c4 * 32, o);
          }
        }
        if (G == 0 && j == n - 1 && it.L - j * kN < kN) {
          // keys past L in the last tile get p = 0, but 0 * NaN is NaN: zero those V
          // rows (head 0 does it for both: its P.V is issued first)
          const uint32_t uv = 2 * gj + 1, slot = uv % nslots;
          if (ok && !bar_ok(kv_full + slot, (uv / nslots) & 1, abort_flag, wl)) ok = false;
          const int32_t nvalid = it.L - j * kN;
          const uint32_t vt = sbase + Lay::slot_off(slot);
          const int32_t tid2 = (warp - kSoftmax0<NG>) * 32 + lane;
          constexpr int kRowChunks = kD * 2 / 16;
          for (int32_t e = tid2; e < (kN - nvalid) * kRowChunks; e += 128) {
            const uint32_t row = (uint32_t)(nvalid + e / kRowChunks), c = (uint32_t)(e % kRowChunks);
            sts128(vt + (c >> 3) * kBlockBytes + row * 128u + ((c & 7u) << 4), 0u, 0u, 0u, 0u);
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeroed V rows, if any
        tc_fence_before();
        // one arrival per warp (the barrier counts four), after the warp's own
        // lanes have stored: no barrier across the group
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + buf);
      }
      // ---- epilogue: out = O / l, lse = ln(sum of exp).  n is the same for the
      // whole CTA, so the collective loads run on every lane or none.
      if (n > 0) {
        if (ok && !bar_ok(o_final + G, f & 1, abort_flag, wl)) ok = false;
        tc_fence_after();
        // Every S MMA of the item has completed.  With one head per CTA the
        // epilogue stores its rows directly and leaves the q area alone, so the
        // next item's q may load into it while the stores run (MHA 4k -1.3 %).
        if (NG == 1 && warp == kSoftmax0<NG> + 4 * G && lane == 0) mbar_arrive(q_free + G);
      }
      const float inv = l > 0.f && ok ? 1.f / l : 0.f;
      if (NG == 2 && n > 0) {
        // O / l goes through this head's q area, free now (every S MMA of the
        // item has completed before its last P.V): [D/32 blocks][128 rows][128 B]
        // with the 128-byte swizzle, then out with tensor stores of 32 columns x
        // 128 rows, which leave the rows past n_q alone.  (Measured: 4k prompt
        // -3 %; direct stores here, even with the q area released at the last
        // MMA for the next q, +4 %.  With one head per CTA, whose CTAs are
        // short, direct stores.)
        // the row's D columns in one batch of TMEM loads, then scaled in pairs
        float o[kD];
#pragma unroll
        for (int c4 = 0; c4 < kD / 32; ++c4) tmem_ld32_nw(obase + (uint32_t)c4 * 32, o + 32 * c4);
        tmem_wait_ld();
        const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          const uint32_t blk = qbase + (uint32_t)c4 * kBlockBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int i = 32 * c4 + 4 * c;
            const uint64_t a = f2_mul(f2_pack(o[i], o[i + 1]), inv2), b = f2_mul(f2_pack(o[i + 2], o[i + 3]), inv2);
            sts128(blk + swz((uint32_t)r, (uint32_t)c), (uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b,
                   (uint32_t)(b >> 32));
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the staged rows, for the tensor stores
        named_barrier(1 + G, 128);
        if (warp == kSoftmax0<NG> + 4 * G && lane == 0) {
#pragma unroll
          for (int c4 = 0; c4 < kD / 32; ++c4)
            tma_store_3d(&tmap_o, qbase + (uint32_t)c4 * kBlockBytes, c4 * 32, it.m0, it.b * p.Hq + h);
          bulk_commit_group();
          bulk_wait_read_all();  // the q area is free again (and the CTA may exit)
          mbar_arrive(q_free + G);
        }
      } else {
        // one head per CTA (short CTAs), or an item without keys: direct stores
        float* orow = p.out + (((size_t)it.b * p.Hq + h) * p.n_q + qi) * kD;
#pragma unroll 1
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          float o[32];
          if (n > 0) {
            tmem_ld32(obase + (uint32_t)c4 * 32, o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
          if (qi < p.n_q) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(orow + c4 * 32 + i) =
                  make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
          }
        }
      }
      if (qi < p.n_q && p.lse)
        p.lse[((size_t)it.b * p.Hq + h) * p.n_q + qi] = l > 0.f ? (mref + log2f(l)) * kLn2f : -INFINITY;
      // this group's O columns are read before the next item's first P.V (which
      // needs this group's P) overwrites them
      tc_fence_before();
      g += (uint32_t)n;
      if (n > 0) ++f;
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.err, kErrTimeout);
    }
  }
  tc_fence_before();
  cta_sync();
  if (queue && tid == 0) {
    // Every CTA has taken its last index (past the end) before it counts
    // itself done; the last one returns both counters to zero for the next launch.
    __threadfence();
    if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.work, 0u);
      atomicExch(p.work + 1, 0u);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int D, int NG, bool kHook>
cudaError_t launch_prefill_t(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                             const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  static int configured = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured != dev) {
    // the setmaxnreg split assumes this launch register count: refuse any other
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fd_prefill_kernel<D, NG, kHook>);
    if (e != cudaSuccess) return e;
    if (NG == 1 && fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(fd_prefill_kernel<D, NG, kHook>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)PLayout<D>::kSmemAlloc);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const int64_t items = (int64_t)((p.n_q + kM - 1) / kM) * (p.Hq / NG) * p.B;
  if (items > 0x7FFFFFFF) return cudaErrorInvalidValue;
  static int sms = 0, sms_dev = -1;
  if (sms_dev != dev) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_dev = dev;
  }
  // One CTA per SM, each taking the next longest-first item from a global
  // counter as it finishes one, so that the next item's q and K/V load while
  // the current one ends (4k prompt: two heads per CTA -1.5 %, one head -3.7 %;
  // a CTA per item handed out by the hardware, and persistent CTAs walking a
  // fixed order, measured slower).
  const dim3 grid((unsigned)(items > sms ? sms : items));
  fd_prefill_kernel<D, NG, kHook><<<grid, kThreads<NG>, PLayout<D>::kSmemAlloc, stream>>>(tk, tv, tq, to, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(int D, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  const bool pair = p.g % 2 == 0;  // two query heads per CTA
  // the testing hook (fd_debug_stall) runs in instances of their own, so that
  // the ordinary ones keep constant wait limits and no skip test
  const bool hook = p.stall_u >= 0 || p.wait_ns != 0;
  if (D == 128) {
    if (hook)
      return pair ? launch_prefill_t<128, 2, true>(tk, tv, tq, to, p, stream)
                  : launch_prefill_t<128, 1, true>(tk, tv, tq, to, p, stream);
    return pair ? launch_prefill_t<128, 2, false>(tk, tv, tq, to, p, stream)
                : launch_prefill_t<128, 1, false>(tk, tv, tq, to, p, stream);
  }
  if (D == 64) {
    if (hook)
      return pair ? launch_prefill_t<64, 2, true>(tk, tv, tq, to, p, stream)
                  : launch_prefill_t<64, 1, true>(tk, tv, tq, to, p, stream);
    return pair ? launch_prefill_t<64, 2, false>(tk, tv, tq, to, p, stream)
                : launch_prefill_t<64, 1, false>(tk, tv, tq, to, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fdk
