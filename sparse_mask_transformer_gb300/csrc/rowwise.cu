// Row-wise masked attention kernel.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, dual-kernel strategy, row-wise kernel: meant for
// high sparsity and short sequences; Q is sliced into rows, work inside a
// row uses warp-level shuffles, and warps never synchronise with each other.
//
// GB300 design: a query row (b, h, i) is owned by LPR lanes of one warp (a
// whole warp, or a half or quarter warp for many short rows, so that more
// rows are in flight per SM); segments of a warp never wait for each other.
// In this regime a row has few valid keys and its time is a chain of
// dependent memory round trips, so the kernel keeps the chain short:
//   1. the row's four row pointers in one load;
//   2. the row's byte of every IT bitmap of its partial OTs, with the OTs'
//      column indices: the (OT, IT column) pairs of the row are numbered
//      consecutively and each lane fetches kSlotsPerLane of them per pass,
//      so one pass covers up to 8 OTs of a 128-wide tiling for a full warp
//      (the next pass's loads are in flight while this one is listed);
//      a lane turns its bytes into key indices at positions given by a
//      prefix sum of the popcounts over the row's lanes, in a per-row list
//      in shared memory, so masked keys cost nothing;
//   3. the keys (full OTs: every key of the tile; partial OTs: the list) in
//      steps of 4 keys per group of G = d/16 lanes, all K and V loads of a
//      step issued before any is used.  A lane holds 16 dimensions of q, k,
//      v and o; a group reduces its dot products with G-lane shuffles and
//      keeps its own online softmax (reference max, sum, partial o; the
//      reference is raised, and o rescaled, only when a score exceeds it by
//      more than 2^8, as in the block-wise kernel); the groups of a row
//      merge once at the end.
// Scores are in the log2 domain (scale * log2 e folded into q); everything
// after the input loads is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace stof {

namespace {

constexpr int kWarps = 4;            // warps per CTA
constexpr int kKeysPerGroup = 4;     // keys in flight per lane group per step
constexpr int kSlotsPerLane = 4;     // (OT, IT column) bytes a lane fetches per pass
constexpr int kListPerWarp = 1024;   // key list entries per warp (shared memory), split over its rows
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

// LPR: lanes per query row (32, 16 or 8).  Every loop of the kernel is
// uniform over the warp (the most OTs, slots or keys of the warp's rows; a
// row with fewer has its surplus entries masked), so all shuffles are
// whole-warp operations over LPR-lane segments and no segment waits on a
// diverged one.
template <int D, bool BF16, int LPR>
__global__ void __launch_bounds__(kWarps * 32, 5) rowwise_kernel(const AttnParams p) {
  constexpr int RPW = 32 / LPR;    // query rows per warp
  constexpr int G = D / 16;        // lanes per key
  static_assert(LPR >= G && LPR % G == 0, "a row needs at least one key group");
  constexpr int NG = LPR / G;      // key groups per row
  constexpr int KPG = kKeysPerGroup;
  constexpr int STEP = NG * KPG;   // keys per row step
  constexpr int SPL = kSlotsPerLane;
  constexpr int CAP = kListPerWarp / RPW;  // key list entries per row
  static_assert(CAP >= LPR * SPL * 8, "a pass must fit the list");
  constexpr unsigned kAll = 0xffffffffu;
  __shared__ int s_list[kWarps][kListPerWarp];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = lane / LPR, sl = lane % LPR;  // the row's segment of the warp, lane in it
  const long long gw = (static_cast<long long>(blockIdx.x) * kWarps + warp) * RPW + seg;  // query row
  const long long n_rows_total = static_cast<long long>(p.B) * p.H * p.L;
  const long long first_row = (static_cast<long long>(blockIdx.x) * kWarps + warp) * RPW;
  if (first_row >= n_rows_total) return;  // warp-uniform
  const bool live = gw < n_rows_total;    // a row past the end has no OTs and stores nothing
  const long long row = live ? gw : first_row;
  int* list = &s_list[warp][seg * CAP];
  const int i = static_cast<int>(row % p.L);
  const long long bh = row / p.L;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  const long long mrow = (b * p.stride_b + h * p.stride_h) * p.n_tr + i / p.bm;
  const int r_in_tile = i % p.bm;

  // 1. the row's pointers: lanes 0, 1 full, lanes 2, 3 partial
  int rp = 0;
  if (sl < 2) rp = __ldg(p.full_row_ptr + mrow + sl);
  else if (sl < 4) rp = __ldg(p.part_row_ptr + mrow + sl - 2);
  int f0 = __shfl_sync(kAll, rp, 0, LPR), f1 = __shfl_sync(kAll, rp, 1, LPR);
  int p0 = __shfl_sync(kAll, rp, 2, LPR), p1 = __shfl_sync(kAll, rp, 3, LPR);
  if (!live) f1 = f0, p1 = p0;

  const int g = sl / G;            // key group
  const int sub = sl % G;          // 16-dim slice
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k) + bh * p.Lk * row_bytes + sub * 32;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v) + bh * p.Lk * row_bytes + sub * 32;

  float qf[16];
  widen16<BF16>(load_raw16(static_cast<const uint8_t*>(p.q) + row * row_bytes + sub * 32), qf);
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
      for (int off = G / 2; off; off >>= 1) dot += __shfl_xor_sync(kAll, dot, off);
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

  // full OTs: every key of the tile; column indices LPR at a time
  const int nf = f1 - f0;
  const int nf_max = RPW == 1 ? nf : __reduce_max_sync(kAll, nf);
  for (int e0 = 0; e0 < nf_max; e0 += LPR) {
    int Jl = -1;
    if (e0 + sl < nf) {
      Jl = __ldg(p.full_col_idx + f0 + e0 + sl);
      if (Jl < 0 || Jl >= p.n_tc) {
        atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
        Jl = -1;
      }
    }
    const int n = min(LPR, nf_max - e0);
    for (int t = 0; t < n; ++t) {
      const int J = __shfl_sync(kAll, Jl, t, LPR);  // -1: none for this row
      for (int k0 = 0; k0 < p.bn; k0 += STEP) {
        int key[KPG];
#pragma unroll
        for (int u = 0; u < KPG; ++u) {
          const int idx = k0 + u * NG + g;
          key[u] = (J >= 0 && idx < p.bn) ? J * p.bn + idx : -1;
        }
        step(key);
      }
    }
  }

  // partial OTs: only the keys whose bit is set in this row
  auto process_list = [&](int n) {
    const int n_max = RPW == 1 ? n : __reduce_max_sync(kAll, n);
    __syncwarp();
    for (int k0 = 0; k0 < n_max; k0 += STEP) {
      int key[KPG];
#pragma unroll
      for (int u = 0; u < KPG; ++u) {
        const int idx = k0 + u * NG + g;
        key[u] = idx < n ? list[idx] : -1;
      }
      step(key);
    }
    __syncwarp();
  };
  const int itc = p.bn >> 3;                 // IT columns per OT
  const int wpt = (p.bm >> 3) * itc;         // IT words per OT
  const int nslots = (p1 - p0) * itc;        // (OT, IT column) pairs of the row
  const int nslots_max = RPW == 1 ? nslots : __reduce_max_sync(kAll, nslots);
  const uint8_t* bits_base = reinterpret_cast<const uint8_t*>(p.bitmaps) + (r_in_tile >> 3) * itc * 8 +
                             (r_in_tile & 7);
  // slot q of the row: OT p0 + q / itc, IT column q % itc; the byte of this row
  uint32_t bits_n[SPL];
  int key_n[SPL];   // first key of the slot's 8 columns
  auto fetch = [&](int q0) {
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
      const int q = q0 + j * LPR + sl;
      bits_n[j] = 0;
      key_n[j] = 0;
      if (q < nslots) {
        const int eo = q / itc, c = q - eo * itc;
        const long long e = static_cast<long long>(p0) + eo;
        const int J = __ldg(p.part_col_idx + e);
        bits_n[j] = __ldg(bits_base + (e * wpt + c) * 8);
        key_n[j] = J * p.bn + 8 * c;
        if (J < 0 || J >= p.n_tc) {
          if (c == 0) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_BAD_FORMAT);
          bits_n[j] = 0;
        }
      }
    }
  };
  int cnt = 0;  // keys in this row's list
  if (nslots_max > 0) fetch(0);
  for (int q0 = 0; q0 < nslots_max; q0 += LPR * SPL) {
    uint32_t bits[SPL];
    int key0[SPL];
    int nb = 0;
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
      bits[j] = bits_n[j];
      key0[j] = key_n[j];
      nb += __popc(bits[j]);
    }
    if (q0 + LPR * SPL < nslots_max) fetch(q0 + LPR * SPL);  // the next pass's loads in flight
    int incl = nb;
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) {
      const int y = __shfl_up_sync(kAll, incl, off, LPR);
      if (sl >= off) incl += y;
    }
    const int total = __shfl_sync(kAll, incl, LPR - 1, LPR);
    // keep every row's list within its capacity (flushed together: uniform)
    if (__any_sync(kAll, cnt + total > CAP)) {
      process_list(cnt);
      cnt = 0;
    }
    int pos = cnt + incl - nb;
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
      uint32_t bj = bits[j];
      while (bj) {
        const int bit = __ffs(bj) - 1;
        bj &= bj - 1;
        list[pos++] = key0[j] + bit;
      }
    }
    cnt += total;
  }
  if (__any_sync(kAll, cnt > 0)) process_list(cnt);

  // merge the row's NG groups: common reference, rescale, sum over groups
  float m_all = m_ref;
#pragma unroll
  for (int off = G; off < LPR; off <<= 1) m_all = fmaxf(m_all, __shfl_xor_sync(kAll, m_all, off));
  const float f = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_all);
  l *= f;
#pragma unroll
  for (int t = 0; t < 16; ++t) o[t] *= f;
#pragma unroll
  for (int off = G; off < LPR; off <<= 1) {
    l += __shfl_xor_sync(kAll, l, off);
#pragma unroll
    for (int t = 0; t < 16; ++t) o[t] += __shfl_xor_sync(kAll, o[t], off);
  }
  if (g == 0 && live) {
    const float inv = l > 0.f ? 1.f / l : 0.f;  // no valid key -> 0
    uint32_t w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) w[t] = Elem<BF16>::from_f2(o[2 * t] * inv, o[2 * t + 1] * inv);
    uint8_t* orow = static_cast<uint8_t*>(p.o) + row * row_bytes + sub * 32;
    reinterpret_cast<uint4*>(orow)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(orow)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int D, bool BF16, int LPR>
cudaError_t launch_rw(const AttnParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.L;
  const long long rows_per_cta = static_cast<long long>(kWarps) * (32 / LPR);
  const long long blocks = (rows + rows_per_cta - 1) / rows_per_cta;
  rowwise_kernel<D, BF16, LPR><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_rw_d(const AttnParams& p, cudaStream_t s) {
  const int rpw = rowwise_rows_per_warp(static_cast<long long>(p.B) * p.H * p.L, p.keys_per_row,
                                        p.listed128_per_row, p.rows_per_warp);
  // a key needs D / 16 lanes: d = 256 fits 2 rows per warp at most
  if constexpr (D / 16 <= 8) {
    if (rpw == 4) return launch_rw<D, BF16, 8>(p, s);
  } else {
    if (rpw == 4) return launch_rw<D, BF16, 16>(p, s);
  }
  if (rpw == 2) return launch_rw<D, BF16, 16>(p, s);
  return launch_rw<D, BF16, 32>(p, s);
}

}  // namespace

cudaError_t launch_rowwise(const AttnParams& p, bool bf16, cudaStream_t s) {
  switch (p.d) {
    case 32: return bf16 ? launch_rw_d<32, true>(p, s) : launch_rw_d<32, false>(p, s);
    case 64: return bf16 ? launch_rw_d<64, true>(p, s) : launch_rw_d<64, false>(p, s);
    case 128: return bf16 ? launch_rw_d<128, true>(p, s) : launch_rw_d<128, false>(p, s);
    case 256: return bf16 ? launch_rw_d<256, true>(p, s) : launch_rw_d<256, false>(p, s);
    default: return cudaErrorInvalidValue;  // the host checks d first
  }
}

}  // namespace stof
