// Row-wise masked attention kernel.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, dual-kernel strategy, row-wise kernel: meant for
// high sparsity and short sequences; Q is sliced into rows, work inside a
// row uses warp-level shuffles, and warps never synchronise with each other.
//
// GB300 design: one warp per query row (b, h, i).  The warp walks the full
// OTs, then the partial OTs, of the row's OT row.  Inside an OT only valid
// keys are visited: for a partial OT the warp turns the row's bits of the
// IT bitmaps into a list of key offsets (one shuffle scan), so masked keys
// cost nothing.  Keys are spread over groups of G = d/16 lanes; each lane
// holds 16 dimensions of q, k, v and o.  A group reduces its dot product
// with G-lane shuffles and keeps its own online softmax (running max m,
// sum l, partial o); the groups are merged once at the end of the row.
// Scores are in the log2 domain (scale * log2 e folded into q).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace stof {

namespace {

constexpr int kWarps = 8;
constexpr int kKeysPerGroup = 2;  // keys in flight per group per step

template <bool BF16>
struct Elem;
template <>
struct Elem<false> {
  using T = __half;
  using T2 = __half2;
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// 16 consecutive elements (32 bytes) -> 16 floats
template <bool BF16>
__device__ __forceinline__ void load16(const uint8_t* src, float (&x)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(src + 16));
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = Elem<BF16>::to_f2(w[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kWarps * 32) rowwise_kernel(const AttnParams p) {
  constexpr int G = D / 16;        // lanes per key
  constexpr int NG = 32 / G;       // key groups per warp
  constexpr int KSTEP = NG * kKeysPerGroup;
  __shared__ uint8_t s_list[kWarps][256];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gw = static_cast<long long>(blockIdx.x) * kWarps + warp;
  const long long n_rows_total = static_cast<long long>(p.B) * p.H * p.L;
  if (gw >= n_rows_total) return;  // warp-uniform
  const int i = static_cast<int>(gw % p.L);
  const long long bh = gw / p.L;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  const long long mrow = (b * p.stride_b + h * p.stride_h) * p.n_tr + i / p.bm;
  const int r_in_tile = i % p.bm;

  const int g = lane / G;          // key group
  const int sub = lane % G;        // 16-dim slice
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  const uint8_t* qrow = static_cast<const uint8_t*>(p.q) + gw * row_bytes + sub * 32;
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k) + bh * p.L * row_bytes + sub * 32;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v) + bh * p.L * row_bytes + sub * 32;

  float qf[16];
  load16<BF16>(qrow, qf);
#pragma unroll
  for (int t = 0; t < 16; ++t) qf[t] *= p.scale_log2;

  float m = -INFINITY, l = 0.f, o[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) o[t] = 0.f;

  // one step: up to kKeysPerGroup keys for this group (key < 0: none)
  auto step = [&](const int (&key)[kKeysPerGroup]) {
    float s[kKeysPerGroup];
    float vv[kKeysPerGroup][16];
#pragma unroll
    for (int u = 0; u < kKeysPerGroup; ++u) {
      float kf[16];
      float dot = 0.f;
      if (key[u] >= 0) {
        load16<BF16>(kbase + static_cast<size_t>(key[u]) * row_bytes, kf);
        load16<BF16>(vbase + static_cast<size_t>(key[u]) * row_bytes, vv[u]);
#pragma unroll
        for (int t = 0; t < 16; ++t) dot = fmaf(qf[t], kf[t], dot);
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) vv[u][t] = 0.f;
      }
#pragma unroll
      for (int off = G / 2; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = key[u] >= 0 ? dot : -INFINITY;
    }
    float m_new = m;
#pragma unroll
    for (int u = 0; u < kKeysPerGroup; ++u) m_new = fmaxf(m_new, s[u]);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = fast_exp2(m - m_use);  // m = -inf -> 0
    l *= alpha;
#pragma unroll
    for (int t = 0; t < 16; ++t) o[t] *= alpha;
#pragma unroll
    for (int u = 0; u < kKeysPerGroup; ++u) {
      const float pu = fast_exp2(s[u] - m_use);  // masked -> 0
      l += pu;
#pragma unroll
      for (int t = 0; t < 16; ++t) o[t] = fmaf(pu, vv[u][t], o[t]);
    }
    m = m_new;
  };

  // full OTs: every key of the tile
  const int f0 = p.full_row_ptr[mrow], f1 = p.full_row_ptr[mrow + 1];
  for (int e = f0; e < f1; ++e) {
    const int J = p.full_col_idx[e];
    if (J < 0 || J >= p.n_tc) {
      if (lane == 0) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
      continue;
    }
    const int key0 = J * p.bn;
    for (int k0 = 0; k0 < p.bn; k0 += KSTEP) {
      int key[kKeysPerGroup];
#pragma unroll
      for (int u = 0; u < kKeysPerGroup; ++u) {
        const int idx = k0 + u * NG + g;
        key[u] = idx < p.bn ? key0 + idx : -1;
      }
      step(key);
    }
  }

  // partial OTs: only the keys whose bit is set in this row
  const int itc = p.bn >> 3;
  const int wpt = (p.bm >> 3) * itc;
  const int p0 = p.part_row_ptr[mrow], p1 = p.part_row_ptr[mrow + 1];
  for (int e = p0; e < p1; ++e) {
    const int J = p.part_col_idx[e];
    if (J < 0 || J >= p.n_tc) {
      if (lane == 0) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
      continue;
    }
    // lane c (< bn/8) takes byte (r mod 8) of IT word (r/8, c): keys 8c..8c+7
    uint32_t bits = 0;
    if (lane < itc) {
      const uint64_t w =
          __ldg(reinterpret_cast<const unsigned long long*>(p.bitmaps) +
                static_cast<long long>(e) * wpt + (r_in_tile >> 3) * itc + lane);
      bits = static_cast<uint32_t>(w >> (8 * (r_in_tile & 7))) & 0xFFu;
    }
    const int cnt = __popc(bits);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int pos = incl - cnt;
    while (bits) {
      const int c = __ffs(bits) - 1;
      bits &= bits - 1;
      s_list[warp][pos++] = static_cast<uint8_t>(8 * lane + c);
    }
    __syncwarp();
    const int key0 = J * p.bn;
    for (int k0 = 0; k0 < total; k0 += KSTEP) {
      int key[kKeysPerGroup];
#pragma unroll
      for (int u = 0; u < kKeysPerGroup; ++u) {
        const int idx = k0 + u * NG + g;
        key[u] = idx < total ? key0 + s_list[warp][idx] : -1;
      }
      step(key);
    }
    __syncwarp();
  }

  // merge the NG groups: common max, rescale, sum over groups
  float m_all = m;
#pragma unroll
  for (int off = G; off < 32; off <<= 1) m_all = fmaxf(m_all, __shfl_xor_sync(0xffffffffu, m_all, off));
  const float f = (m == -INFINITY) ? 0.f : fast_exp2(m - m_all);
  l *= f;
#pragma unroll
  for (int t = 0; t < 16; ++t) o[t] *= f;
#pragma unroll
  for (int off = G; off < 32; off <<= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
    for (int t = 0; t < 16; ++t) o[t] += __shfl_xor_sync(0xffffffffu, o[t], off);
  }
  if (g == 0) {
    const float inv = l > 0.f ? 1.f / l : 0.f;  // no valid key -> 0
    uint32_t w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) w[t] = Elem<BF16>::from_f2(o[2 * t] * inv, o[2 * t + 1] * inv);
    uint8_t* orow = static_cast<uint8_t*>(p.o) + gw * row_bytes + sub * 32;
    reinterpret_cast<uint4*>(orow)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(orow)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int D, bool BF16>
cudaError_t launch_rw(const AttnParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.L;
  const long long blocks = (rows + kWarps - 1) / kWarps;
  rowwise_kernel<D, BF16><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rowwise(const AttnParams& p, bool bf16, cudaStream_t s) {
  if (p.d == 64) return bf16 ? launch_rw<64, true>(p, s) : launch_rw<64, false>(p, s);
  return bf16 ? launch_rw<128, true>(p, s) : launch_rw<128, false>(p, s);
}

}  // namespace stof
