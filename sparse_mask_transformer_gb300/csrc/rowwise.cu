// Row-wise masked attention kernel.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, dual-kernel strategy, row-wise kernel: meant for
// high sparsity and short sequences; Q is sliced into rows, work inside a
// row uses warp-level shuffles, and warps never synchronise with each other.
//
// GB300 design: one warp per query row (b, h, i).  In that regime a row has
// few valid keys and the time is a chain of dependent memory round trips,
// so the kernel keeps the chain short:
//   1. the row's four row pointers in one load (lanes 0-3);
//   2. the row's byte of every IT bitmap of its partial OTs and their column
//      indices, lane-parallel (a lane per IT column, 32 / (bn/8) OTs per
//      pass, the next pass's loads in flight while this one is listed);
//      each lane turns its byte into key indices at positions given by a
//      warp prefix sum of the popcounts, in a per-warp list in shared
//      memory, so masked keys cost nothing;
//   3. the keys (full OTs: every key of the tile; partial OTs: the list) in
//      steps of 4 keys per group of G = d/16 lanes, all K and V loads of a
//      step issued before any is used.  A lane holds 16 dimensions of q, k,
//      v and o; a group reduces its dot products with G-lane shuffles and
//      keeps its own online softmax (reference max, sum, partial o; the
//      reference is raised, and o rescaled, only when a score exceeds it by
//      more than 2^8, as in the block-wise kernel); the groups merge once
//      at the end of the row.
// Scores are in the log2 domain (scale * log2 e folded into q); everything
// after the input loads is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace stof {

namespace {

constexpr int kWarps = 4;            // query rows per CTA
constexpr int kKeysPerGroup = 4;     // keys in flight per lane group per step
constexpr int kListCap = 512;        // per-warp key list (shared memory)
constexpr float kRescaleLog2 = 8.f;  // raise the reference when a score exceeds it by more

template <bool BF16>
struct Elem;
template <>
struct Elem<false> {
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
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// 16 consecutive 16-bit elements (32 bytes), raw
struct Raw16 {
  uint4 a, b;
};
__device__ __forceinline__ Raw16 load_raw16(const uint8_t* src) {
  Raw16 r;
  r.a = __ldg(reinterpret_cast<const uint4*>(src));
  r.b = __ldg(reinterpret_cast<const uint4*>(src + 16));
  return r;
}
template <bool BF16>
__device__ __forceinline__ void widen16(const Raw16& r, float (&x)[16]) {
  const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
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
  constexpr int KPG = kKeysPerGroup;
  constexpr int STEP = NG * KPG;   // keys per warp step
  __shared__ int s_list[kWarps][kListCap];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gw = static_cast<long long>(blockIdx.x) * kWarps + warp;
  const long long n_rows_total = static_cast<long long>(p.B) * p.H * p.L;
  if (gw >= n_rows_total) return;  // warp-uniform
  const int i = static_cast<int>(gw % p.L);
  const long long bh = gw / p.L;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  const long long mrow = (b * p.stride_b + h * p.stride_h) * p.n_tr + i / p.bm;
  const int r_in_tile = i % p.bm;

  // 1. the row's pointers: lanes 0, 1 full, lanes 2, 3 partial
  int rp = 0;
  if (lane < 2) rp = __ldg(p.full_row_ptr + mrow + lane);
  else if (lane < 4) rp = __ldg(p.part_row_ptr + mrow + lane - 2);
  const int f0 = __shfl_sync(0xffffffffu, rp, 0), f1 = __shfl_sync(0xffffffffu, rp, 1);
  const int p0 = __shfl_sync(0xffffffffu, rp, 2), p1 = __shfl_sync(0xffffffffu, rp, 3);

  const int g = lane / G;          // key group
  const int sub = lane % G;        // 16-dim slice
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k) + bh * p.L * row_bytes + sub * 32;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v) + bh * p.L * row_bytes + sub * 32;

  float qf[16];
  widen16<BF16>(load_raw16(static_cast<const uint8_t*>(p.q) + gw * row_bytes + sub * 32), qf);
#pragma unroll
  for (int t = 0; t < 16; ++t) qf[t] *= p.scale_log2;

  float m_ref = -INFINITY, l = 0.f, o[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) o[t] = 0.f;

  // one step: up to KPG keys for this group (key < 0: none).  Every load is
  // issued first (a missing key reads key 0 of the head and is dropped).
  auto step = [&](const int (&key)[KPG]) {
    Raw16 kr[KPG], vr[KPG];
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
      const size_t off = static_cast<size_t>(key[u] >= 0 ? key[u] : 0) * row_bytes;
      kr[u] = load_raw16(kbase + off);
      vr[u] = load_raw16(vbase + off);
    }
    float s[KPG];
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
      float kf[16];
      widen16<BF16>(kr[u], kf);
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int t = 0; t < 16; t += 2) {
        d0 = fmaf(qf[t], kf[t], d0);
        d1 = fmaf(qf[t + 1], kf[t + 1], d1);
      }
      float dot = d0 + d1;
#pragma unroll
      for (int off = G / 2; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = key[u] >= 0 ? dot : -INFINITY;
    }
    float mx = s[0];
#pragma unroll
    for (int u = 1; u < KPG; ++u) mx = fmaxf(mx, s[u]);
    if (mx > m_ref + kRescaleLog2) {  // also the first valid key of the group
      const float alpha = fast_exp2(m_ref - mx);  // 0 when m_ref = -inf
      l *= alpha;
#pragma unroll
      for (int t = 0; t < 16; ++t) o[t] *= alpha;
      m_ref = mx;
    }
    const float mu = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
      const float pu = fast_exp2(s[u] - mu);  // no key -> 0
      float vf[16];
      widen16<BF16>(vr[u], vf);
      l += pu;
#pragma unroll
      for (int t = 0; t < 16; ++t) o[t] = fmaf(pu, vf[t], o[t]);
    }
  };

  // full OTs: every key of the tile; column indices 32 at a time
  for (int e0 = f0; e0 < f1; e0 += 32) {
    const int Jl = e0 + lane < f1 ? __ldg(p.full_col_idx + e0 + lane) : 0;
    const int n = min(32, f1 - e0);
    for (int t = 0; t < n; ++t) {
      const int J = __shfl_sync(0xffffffffu, Jl, t);
      if (J < 0 || J >= p.n_tc) {
        if (lane == 0) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
        continue;
      }
      const int key0 = J * p.bn;
      for (int k0 = 0; k0 < p.bn; k0 += STEP) {
        int key[KPG];
#pragma unroll
        for (int u = 0; u < KPG; ++u) {
          const int idx = k0 + u * NG + g;
          key[u] = idx < p.bn ? key0 + idx : -1;
        }
        step(key);
      }
    }
  }

  // partial OTs: only the keys whose bit is set in this row
  auto process_list = [&](int n) {
    __syncwarp();
    for (int k0 = 0; k0 < n; k0 += STEP) {
      int key[KPG];
#pragma unroll
      for (int u = 0; u < KPG; ++u) {
        const int idx = k0 + u * NG + g;
        key[u] = idx < n ? s_list[warp][idx] : -1;
      }
      step(key);
    }
    __syncwarp();
  };
  const int itc = p.bn >> 3;             // IT columns per OT (<= 32)
  const int opp = 32 / itc;              // OTs per pass
  const int wpt = (p.bm >> 3) * itc;     // IT words per OT
  const int c = lane % itc;
  // lane's slot of the pass starting at e0: byte (r mod 8) of IT word (r/8, c) of OT e0 + lane / itc
  auto fetch = [&](int e0, uint32_t& bits, int& J, bool& slot) {
    const int e = e0 + lane / itc;
    bits = 0;
    J = 0;
    slot = lane < opp * itc && e < p1;  // this lane has an IT column of a listed OT
    if (slot) {
      J = __ldg(p.part_col_idx + e);
      const uint8_t* bp = reinterpret_cast<const uint8_t*>(
                              p.bitmaps + static_cast<long long>(e) * wpt + (r_in_tile >> 3) * itc + c) +
                          (r_in_tile & 7);
      bits = __ldg(bp);
    }
  };
  int cnt = 0;  // keys in the list
  uint32_t bits_next = 0;
  int J_next = 0;
  bool slot_next = false;
  if (p0 < p1) fetch(p0, bits_next, J_next, slot_next);
  for (int e0 = p0; e0 < p1; e0 += opp) {
    uint32_t bits = bits_next;
    const int J = J_next;
    const bool slot = slot_next;
    if (e0 + opp < p1) fetch(e0 + opp, bits_next, J_next, slot_next);  // the next pass's loads in flight
    if (slot && (J < 0 || J >= p.n_tc)) {
      if (c == 0) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
      bits = 0;
    }
    const int nb = __popc(bits);
    int incl = nb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int pos = cnt + incl - nb;
    const int base = J * p.bn + 8 * c;
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      s_list[warp][pos++] = base + bit;
    }
    cnt += total;  // a pass adds at most 256 keys: the list never overflows
    if (cnt > kListCap - 256) {
      process_list(cnt);
      cnt = 0;
    }
  }
  if (cnt) process_list(cnt);

  // merge the NG groups: common reference, rescale, sum over groups
  float m_all = m_ref;
#pragma unroll
  for (int off = G; off < 32; off <<= 1) m_all = fmaxf(m_all, __shfl_xor_sync(0xffffffffu, m_all, off));
  const float f = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_all);
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
