// Pieces shared by the block-wise attention kernels (blockwise.cu: one CTA
// per query tile; blockwise_persist.cu: persistent CTAs for d = 64): tile
// sizes, thread layout, register split and the softmax's fp32 helpers.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "sm100_ptx.cuh"

namespace stof {
namespace bw {

constexpr int kBM = 128;  // query rows per tile (the MMA's M); key columns per OT: BN = 64 or 128
// 2 producer warps, 2 MMA-issuer warps, 8 softmax warps.  Three warps per
// SM sub-partition cap a thread at 168 registers.
constexpr int kThreads = 384;
constexpr int kStages = 3;                    // default K and V ring depth (one CTA per query tile)
constexpr float kRescaleThreshold = 8.0f;     // log2 units
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per pipeline wait

// Tiles in shared memory are 128-byte-swizzled: a matrix of R rows is stored
// as d/64 (or keys/64) atoms of R rows x 128 bytes, 8-row groups 1 KB apart.
template <int D, int BN>
struct Cfg {
  static constexpr int REGIONS = D / 64;            // swizzle atoms along d
  static constexpr int Q_BYTES = kBM * D * 2;       // the Q tile
  static constexpr int KV_BYTES = BN * D * 2;       // one K or V tile
  static constexpr int KV_ATOM = BN * 128;          // one swizzle atom of a K or V tile
  static constexpr int CHUNKS = BN / 32;            // 32-score chunks of a softmax row
  static constexpr int BITMAP_WORDS = (kBM / 8) * (BN / 8);
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// d0 = a0 * b0 + c0, d1 = a1 * b1 + c1 in one packed fp32x2 FMA
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.ftz.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// d0 += a0, d1 += a1 in one packed fp32x2 add
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 rd, {%0, %1};\n\tmov.b64 ra, {%2, %3};\n\t"
      "add.rn.ftz.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// s = -inf unless (bits & bit) != 0.  Written as a bit test and a select
// in PTX: the ternary form measured 2.4% more ALU instructions per tile.
__device__ __forceinline__ void keep_if_set(uint32_t& s, uint32_t bits, uint32_t bit) {
  asm("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t"
      "and.b32 t, %1, %2;\n\tsetp.eq.u32 p, t, 0;\n\tselp.b32 %0, %3, %0, p;\n\t}"
      : "+r"(s)
      : "r"(bits), "r"(bit), "r"(0xFF800000u));
}

// 2^x on the FMA pipe, for the exp split: x = n + f with n = rint(x)
// (adding and subtracting 1.5 * 2^23 rounds to an integer), 2^f by
// p(f) = 1 + f (c1 + f (c2 + f (c3 + f c4))), whose coefficients minimise
// the maximum relative error on [-1/2, 1/2] (Remez exchange; derived and
// checked by ex2_poly.py: at most 2.9e-6), and n added to p's exponent field.
// Exactly 1 at 0; 0 below -125, at -inf included.  For x <= 127.
__device__ __forceinline__ float ex2_fma(float x) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  const float t = x + kRound;
  const float n = t - kRound;
  const float f = x - n;
  float p = fmaf(f, 0x1.3a02ccp-7f, 0x1.c9fc46p-5f);
  p = fmaf(p, f, 0x1.ec0378p-3f);
  p = fmaf(p, f, 0x1.62e12cp-1f);
  p = fmaf(p, f, 1.f);
  const float y = __uint_as_float(__float_as_uint(p) + (__float_as_uint(t) << 23));
  return x < -125.f ? 0.f : y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ void raise_error(int64_t* err, unsigned long long bit) {
  atomicOr(reinterpret_cast<unsigned long long*>(err), bit);
}

// Register split: the kernel is launched with kLaunchRegs per thread (the
// most 384 threads can have); warpgroup 0 (producers, MMA issuers) drops to
// kProducerRegs, the two softmax warpgroups rise to kSoftmaxRegs.  The host
// refuses to launch a build whose register count is not kLaunchRegs, since
// the raise would then wait for registers that are never released.
constexpr int kLaunchRegs = 168, kProducerRegs = 56, kSoftmaxRegs = 224;
static_assert(kProducerRegs * 128 + kSoftmaxRegs * 256 <= kLaunchRegs * kThreads, "register split");
static_assert(kLaunchRegs * kThreads <= 65536, "register file");

// ---------------------------------------------------------------- per-tile softmax
// A softmax thread owns one query row of a tile (= one TMEM lane) and its
// BN = 32 * CHUNKS scores.

// The row's scores from TMEM into registers.
template <int CHUNKS>
__device__ __forceinline__ void load_scores(uint32_t tSr, uint32_t (&sr)[CHUNKS][32]) {
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc) ptx::tmem_ld32(tSr + cc * 32, sr[cc]);
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc) ptx::tmem_ld_wait(sr[cc]);
}

// The row's byte of each 8x8 inner tile of an OT (4 * CHUNKS bytes, one per
// 8 key columns) as CHUNKS words of 32 key bits.
template <int CHUNKS>
__device__ __forceinline__ void assemble_bits(const uint32_t (&nb)[CHUNKS * 4], uint32_t (&bits)[CHUNKS]) {
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc)
    bits[cc] = nb[4 * cc] | (nb[4 * cc + 1] << 8) | (nb[4 * cc + 2] << 16) | (nb[4 * cc + 3] << 24);
}

// Scores times c, in place.  Used when c = scale * log2(e) is not positive:
// the max of c*s is then not c times the max of s, and a masked score set
// to -inf before the multiply would become +inf or NaN after it.  With the
// scores pre-multiplied the softmax runs with c = 1 and masks afterwards.
template <int CHUNKS>
__device__ __forceinline__ void scale_scores(uint32_t (&sr)[CHUNKS][32], float c) {
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc)
#pragma unroll
    for (int i = 0; i < 32; ++i) sr[cc][i] = __float_as_uint(__uint_as_float(sr[cc][i]) * c);
}

// -inf at every key whose bit is clear.
template <int CHUNKS>
__device__ __forceinline__ void mask_scores(uint32_t (&sr)[CHUNKS][32], const uint32_t (&bits)[CHUNKS]) {
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc)
#pragma unroll
    for (int i = 0; i < 32; ++i) keep_if_set(sr[cc][i], bits[cc], 1u << i);
}

// Max of the row's scores (one max3 chain per 32 scores).
template <int CHUNKS>
__device__ __forceinline__ float row_max(const uint32_t (&sr)[CHUNKS][32]) {
  float m4[CHUNKS];
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc) {
    m4[cc] = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      m4[cc] = max3(m4[cc], __uint_as_float(sr[cc][i]), __uint_as_float(sr[cc][i + 1]));
      m4[cc] = max3(m4[cc], __uint_as_float(sr[cc][i + 2]), __uint_as_float(sr[cc][i + 3]));
      m4[cc] = max3(m4[cc], __uint_as_float(sr[cc][i + 4]), __uint_as_float(sr[cc][i + 5]));
      m4[cc] = max3(m4[cc], __uint_as_float(sr[cc][i + 6]), __uint_as_float(sr[cc][i + 7]));
    }
  }
  float m = m4[0];
#pragma unroll
  for (int cc = 1; cc < CHUNKS; ++cc) m = fmaxf(m, m4[cc]);
  return m;
}

// P = 2^(c s + nmu) as fp16/bf16 pairs (keys 32 cc + 2 i and + 1 in
// pk[cc][i]); returns the sum of the fp32 exponentials.  ESPLIT: one pair
// of keys in eight takes its exponentials on the FMA pipe (ex2_fma), the
// rest on the special-function unit.
template <int CHUNKS, bool BF16, bool ESPLIT = false>
__device__ __forceinline__ float exp_pack(const uint32_t (&sr)[CHUNKS][32], float c, float nmu,
                                          uint32_t (&pk)[CHUNKS][16]) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc)
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float x0, x1;
      ffma2(x0, x1, __uint_as_float(sr[cc][i]), __uint_as_float(sr[cc][i + 1]), c, c, nmu, nmu);
      const bool fma_pipe = ESPLIT && (i / 2) % 8 == 7;
      const float e0 = fma_pipe ? ex2_fma(x0) : ex2(x0), e1 = fma_pipe ? ex2_fma(x1) : ex2(x1);
      fadd2(ls[((i >> 1) & 1) * 2], ls[((i >> 1) & 1) * 2 + 1], e0, e1);
      pk[cc][i / 2] = pack2<BF16>(e0, e1);
    }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// exp_pack for one chunk of 32 scores.
template <bool BF16>
__device__ __forceinline__ float exp_pack32(const uint32_t (&sr)[32], float c, float nmu, uint32_t (&pk)[16]) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float x0, x1;
    ffma2(x0, x1, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]), c, c, nmu, nmu);
    const float e0 = ex2(x0), e1 = ex2(x1);
    fadd2(ls[((i >> 1) & 1) * 2], ls[((i >> 1) & 1) * 2 + 1], e0, e1);
    pk[i / 2] = pack2<BF16>(e0, e1);
  }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// O row (D fp32 columns at tOr) *= alpha, in TMEM.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tOr, float alpha) {
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t orr[32];
    ptx::tmem_ld32(tOr + cc * 32, orr);
    ptx::tmem_ld_wait(orr);
#pragma unroll
    for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
    ptx::tmem_st32(tOr + cc * 32, orr);
  }
}

// The row's P into TMEM (16 columns of pairs per 32 keys); complete on return.
template <int CHUNKS>
__device__ __forceinline__ void store_p(uint32_t tP, const uint32_t (&pk)[CHUNKS][16]) {
#pragma unroll
  for (int cc = 0; cc < CHUNKS; ++cc) ptx::tmem_st16(tP + cc * 16, pk[cc]);
  ptx::tmem_st_wait();
}

}  // namespace bw
}  // namespace stof
