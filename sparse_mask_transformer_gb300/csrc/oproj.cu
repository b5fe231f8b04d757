// Attention output projection with a fused epilogue, for sm_103a.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 2, operator fusion module: fusion is carried past
// the MHA layer into the operators that follow it.  The operator right after
// masked MHA in a transformer layer is the output projection with its bias
// and the residual connection:
//   y[b, l, n] = sum_{h, c} O[b, h, l, c] * W[n, h*d + c] + bias[n] + res[b, l, n]
// with O the MHA output [B][H][L][d] (heads concatenated along the
// reduction axis, as the projection sees them), W a [N][H*d] row-major
// weight and res [B][L][N].  Here it is one GEMM whose epilogue adds the
// bias and the residual and rounds once, so the projection's output is
// written once and never re-read for the additions.
//
// GB300 design: a persistent kernel, one CTA per SM, 192 threads:
//   warp 0      TMA producer: for every (128-token, 256-feature) output
//               tile and every 64-wide slice of the reduction, the O slice
//               (128 tokens of one head, 64 of its d columns, O viewed as
//               [B*H][L][d]: zeros past L) and the W slice (256 rows x 64) into a
//               four-stage ring;
//   warp 1      allocates TMEM and issues the tcgen05 MMAs (M = 128,
//               N = 256, K = 16; both operands K-major, 128-byte swizzle)
//               into one of two TMEM accumulators;
//   warps 2..5  epilogue: a thread owns one token row (= TMEM lane), reads
//               its 256 fp32 sums, adds bias and residual in fp32, rounds to
//               fp16/bf16 and stores; the accumulator then goes back to the
//               issuer, so the epilogue of one tile overlaps the MMAs of the
//               next.
// Every wait is bounded; on timeout the CTA raises STOF_DEVERR_PIPE_TIMEOUT
// in the caller's error word (if given), drains and exits.
//
// LayerNorm after the projection (stof_oproj_ln_fwd, a post-norm sublayer's
// last operator): a token's normalisation needs all N of its features, which
// span N / 256 output tiles computed by different CTAs.  The epilogue
// therefore also reduces each (token, tile) row of rounded outputs to its
// mean and sum of squared deviations (shifted by the row's first value, so
// no cancellation), written to a small workspace; a second, memory-bound
// pass merges a token's tile statistics (Chan, Golub and LeVeque's pairwise
// update) and normalises y in place: (y - mean) / sqrt(var + eps) * gamma +
// beta in fp32, rounded once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace stof {
namespace {

using namespace ptx;

constexpr int kTM = 128;     // tokens per tile (MMA M)
constexpr int kTN = 256;     // output features per tile (MMA N)
constexpr int kTK = 64;      // reduction slice per stage (one 128-byte swizzle atom)
constexpr int kStages = 4;
constexpr int kThreadsOP = 192;
constexpr int kABytes = kTM * kTK * 2;  // 16 KB
constexpr int kBBytes = kTN * kTK * 2;  // 32 KB
constexpr uint64_t kWaitNsOP = 2000000000ull;

struct alignas(1024) OpSmem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct OpParams {
  const void* bias;      // [N] or null
  const void* residual;  // [B][L][N] or null
  void* y;               // [B][L][N]
  float2* stats;         // [B*L][n_tiles] (mean, sum of squared deviations) of each tile row, or null
  int64_t* err;          // device error word or null
  int B, H, L, d, N;
  int m_tiles, n_tiles, k_blocks;
  int m_per_b;           // token tiles per batch element: ceil(L / 128)
};

struct LnParams {
  const float2* stats;   // [rows][n_tiles]
  void* y;               // [rows][N], normalised in place
  const void* gamma;     // [N] or null
  const void* beta;      // [N] or null
  float eps;
  long long rows;
  int N, n_tiles;
};

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t x) {
  if constexpr (BF16)
    return __bfloat162float(__ushort_as_bfloat16(x));
  else
    return __half2float(__ushort_as_half(x));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2f(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreadsOP, 1)
    oproj_kernel(const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmW,
                 const OpParams p) {
  extern __shared__ uint8_t smem_raw[];
  OpSmem& s = *reinterpret_cast<OpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;  // accumulator a at columns a * 256
  volatile int* abort_flag = &s.abort_flag;
  auto fail = [&]() {
    *abort_flag = 1;
    if (p.err) atomicOr(reinterpret_cast<unsigned long long*>(p.err), STOF_DEVERR_PIPE_TIMEOUT);
  };
  const int n_tiles_total = p.m_tiles * p.n_tiles;
  const int kb_per_head = p.d / kTK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmO);
      prefetch_tmap(&tmW);
      int it = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
        const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
        // token tiles are per batch element (the last may run past L: zeros there)
        const int b = mt / p.m_per_b, l0 = (mt - b * p.m_per_b) * kTM;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int st = it % kStages;
          if (it >= kStages && !mbar_wait(&s.empty[st], ((it / kStages) - 1) & 1, abort_flag, kWaitNsOP)) {
            ok = false;
            break;
          }
          const int h = kb / kb_per_head, c0 = (kb - h * kb_per_head) * kTK;
          mbar_arrive_expect_tx(&s.full[st], kABytes + kBBytes);
          tma_load_3d(s.a[st], &tmO, &s.full[st], c0, l0, b * p.H + h);
          tma_load_2d(s.b[st], &tmW, &s.full[st], kb * kTK, nt * kTN);
          issued = it + 1;
        }
      }
      if (!ok) fail();
      if (*abort_flag) {  // let the copies in flight land before exit
        for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
          mbar_wait_timeout(&s.full[i % kStages], (i / kStages) & 1, kWaitNsOP);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_f16(BF16 ? 1 : 0, 0, kTM, kTN);
    const uint64_t adesc0 = smem_desc_sw128(smem_u32(s.a[0]), 16, 1024);
    const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s.b[0]), 16, 1024);
    auto wwait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitNsOP));
    };
    int it = 0, j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x, ++j) {
      const int a = j & 1;
      // the epilogue has read this accumulator's previous tile
      if (j >= 2 && !wwait(&s.acc_empty[a], ((j >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tbase + a * kTN;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int st = it % kStages;
        if (!wwait(&s.full[st], (it / kStages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = adesc0 + static_cast<uint64_t>(st) * (kABytes / 16);
        const uint64_t bd = bdesc0 + static_cast<uint64_t>(st) * (kBBytes / 16);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk)  // 32 B per K step inside the atom
            mma_f16_ss(d_tmem, ad + kk * 2, bd + kk * 2, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&s.empty[st]);                            // stage free once these MMAs are done
          if (kb == p.k_blocks - 1) mma_commit(&s.acc_full[a]);  // the tile's sums are complete
        }
        __syncwarp();
      }
    }
    if (elect_one()) {
      if (!ok) fail();
      mma_commit(&s.drain);
      mbar_wait_timeout(&s.drain, 0, kWaitNsOP);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // token row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint16_t* bias = static_cast<const uint16_t*>(p.bias);
    const uint16_t* res = static_cast<const uint16_t*>(p.residual);
    uint16_t* y = static_cast<uint16_t*>(p.y);
    int j = 0;
    for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++j) {
      const int a = j & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&s.acc_full[a], (j >> 1) & 1, abort_flag, kWaitNsOP));
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
      const int b = mt / p.m_per_b, l = (mt - b * p.m_per_b) * kTM + r;
      const bool row_in = l < p.L;  // rows past L: computed, not read or stored
      const long long row = static_cast<long long>(b) * p.L + l;
      const int n0 = nt * kTN;
      float x0 = 0.f, s1 = 0.f, s2 = 0.f;  // LayerNorm statistics of the row's rounded outputs
#pragma unroll 1
      for (int cc = 0; cc < kTN / 32; ++cc) {
        uint32_t acc[32];
        tmem_ld32(tbase + a * kTN + lane_off + cc * 32, acc);
        tmem_ld_wait(acc);
        const int n = n0 + cc * 32;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
        if (bias) {
          const uint4* bv = reinterpret_cast<const uint4*>(bias + n);  // same address in every lane
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 t = __ldg(bv + q);
            const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * q + 2 * e] += to_f32<BF16>(static_cast<uint16_t>(w4[e] & 0xFFFFu));
              v[8 * q + 2 * e + 1] += to_f32<BF16>(static_cast<uint16_t>(w4[e] >> 16));
            }
          }
        }
        if (res && row_in) {
          const uint4* rv = reinterpret_cast<const uint4*>(res + row * p.N + n);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 t = __ldcs(rv + q);
            const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * q + 2 * e] += to_f32<BF16>(static_cast<uint16_t>(w4[e] & 0xFFFFu));
              v[8 * q + 2 * e + 1] += to_f32<BF16>(static_cast<uint16_t>(w4[e] >> 16));
            }
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) pk[q] = pack2f<BF16>(v[2 * q], v[2 * q + 1]);
        uint4* dst = reinterpret_cast<uint4*>(y + row * p.N + n);
        if (row_in) {
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        if (p.stats) {
          if (cc == 0) x0 = to_f32<BF16>(static_cast<uint16_t>(pk[0] & 0xFFFFu));
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float lo = to_f32<BF16>(static_cast<uint16_t>(pk[q] & 0xFFFFu)) - x0;
            const float hi = to_f32<BF16>(static_cast<uint16_t>(pk[q] >> 16)) - x0;
            s1 += lo + hi;
            s2 = fmaf(lo, lo, fmaf(hi, hi, s2));
          }
        }
      }
      if (p.stats && row_in)
        p.stats[row * p.n_tiles + nt] = make_float2(x0 + s1 / kTN, s2 - s1 * s1 / kTN);
      tc_fence_before();
      mbar_arrive(&s.acc_empty[a]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------- LayerNorm pass
// One warp per token row of y (N features, N % 256 == 0): the row's
// per-tile statistics (mean and sum of squared deviations of the rounded
// outputs of each 256-wide tile) are merged by Chan et al.'s pairwise
// update, then y is normalised in place: (y - mean) / sqrt(var + eps) *
// gamma + beta, in fp32, rounded once.
template <bool BF16>
__global__ void __launch_bounds__(256) layernorm_kernel(const LnParams p) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= p.rows) return;  // warp-uniform
  // merge the row's n_tiles statistics: lanes take tiles, then a shuffle tree
  float cnt = 0.f, mean = 0.f, m2 = 0.f;
  for (int t = lane; t < p.n_tiles; t += 32) {
    const float2 st = p.stats[row * p.n_tiles + t];
    const float nb = static_cast<float>(kTN);
    const float n = cnt + nb;
    const float delta = st.x - mean;
    mean += delta * (nb / n);
    m2 += st.y + delta * delta * (cnt * nb / n);
    cnt = n;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float cb = __shfl_xor_sync(0xffffffffu, cnt, off);
    const float mb = __shfl_xor_sync(0xffffffffu, mean, off);
    const float qb = __shfl_xor_sync(0xffffffffu, m2, off);
    const float n = cnt + cb;
    if (n > 0.f) {
      const float delta = mb - mean;
      mean += delta * (cb / n);
      m2 += qb + delta * delta * (cnt * cb / n);
      cnt = n;
    }
  }
  const float var = m2 / static_cast<float>(p.N);
  const float rstd = 1.f / sqrtf(var + p.eps);
  uint16_t* y = static_cast<uint16_t*>(p.y) + row * p.N;
  const uint16_t* gamma = static_cast<const uint16_t*>(p.gamma);
  const uint16_t* beta = static_cast<const uint16_t*>(p.beta);
  for (int c = lane * 8; c < p.N; c += 256) {  // 8 features (16 bytes) per lane per step
    const uint4 yv = *reinterpret_cast<const uint4*>(y + c);
    const uint4 gv = gamma ? __ldg(reinterpret_cast<const uint4*>(gamma + c)) : make_uint4(0, 0, 0, 0);
    const uint4 bv = beta ? __ldg(reinterpret_cast<const uint4*>(beta + c)) : make_uint4(0, 0, 0, 0);
    const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint16_t ys = static_cast<uint16_t>(yw[e] >> (16 * hh));
        const float g = gamma ? to_f32<BF16>(static_cast<uint16_t>(gw[e] >> (16 * hh))) : 1.f;
        const float bb = beta ? to_f32<BF16>(static_cast<uint16_t>(bw[e] >> (16 * hh))) : 0.f;
        v[hh] = fmaf((to_f32<BF16>(ys) - mean) * rstd, g, bb);
      }
      out[e] = pack2f<BF16>(v[0], v[1]);
    }
    *reinterpret_cast<uint4*>(y + c) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

template <bool BF16>
stof_status launch_op(const void* o, const void* w, const OpParams& p, cudaStream_t s) {
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t K = static_cast<uint64_t>(p.H) * p.d;
  CUtensorMap mo, mw;
  // O viewed as [B*H][L][d] (a token tile past L reads zeros); W as [N][K];
  // boxes of 64 columns (one swizzle atom)
  if (!encode_tensor_map_3d(&mo, dt, o, static_cast<uint64_t>(p.d), static_cast<uint64_t>(p.L),
                            static_cast<uint64_t>(p.B) * p.H, static_cast<uint64_t>(p.d) * 2,
                            static_cast<uint64_t>(p.L) * p.d * 2, kTK, kTM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&mw, dt, w, K, static_cast<uint64_t>(p.N), K * 2, kTK, kTN,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return STOF_ERR_CUDA;
  const size_t smem = sizeof(OpSmem) + 1024;
  auto prepare = [](const void*) {
    return record_cuda(cudaFuncSetAttribute(oproj_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(sizeof(OpSmem) + 1024))) == cudaSuccess;
  };
  if (!once_per_device(reinterpret_cast<const void*>(&oproj_kernel<BF16>), prepare, nullptr)) return STOF_ERR_CUDA;
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < device_sm_count() ? tiles : device_sm_count();
  oproj_kernel<BF16><<<grid, kThreadsOP, smem, s>>>(mo, mw, p);
  return record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}

template <bool BF16>
stof_status launch_ln(const LnParams& lp, cudaStream_t s) {
  const long long blocks = (lp.rows + 7) / 8;
  layernorm_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(lp);
  return record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}

// Argument checks shared by both entry points; fills p.
stof_status check_op(const void* o, const void* w, const void* bias, const void* residual, stof_dtype dt, int B,
                     int H, int L, int d, int N, void* y, int64_t* device_error, OpParams* p) {
  if (!o || !w || !y) return STOF_ERR_INVALID_ARG;
  if (dt != STOF_F16 && dt != STOF_BF16) return STOF_ERR_DTYPE;
  if (B < 1 || H < 1 || L < 1 || d < 1 || N < 1) return STOF_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return STOF_ERR_UNSUPPORTED;
  if (N % kTN) return STOF_ERR_SHAPE;  // any L: the last token tile of a batch element may run past it
  if (static_cast<long long>(B) * H * L >= (1ll << 31) || static_cast<long long>(B) * L * N >= (1ll << 40) ||
      static_cast<long long>(H) * d > (1 << 20))
    return STOF_ERR_SHAPE;
  auto al16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
  if (!al16(o) || !al16(w) || !al16(y) || (bias && !al16(bias)) || (residual && !al16(residual)))
    return STOF_ERR_ALIGNMENT;
  p->bias = bias;
  p->residual = residual;
  p->y = y;
  p->stats = nullptr;
  p->err = device_error;
  p->B = B;
  p->H = H;
  p->L = L;
  p->d = d;
  p->N = N;
  p->m_per_b = (L + kTM - 1) / kTM;
  p->m_tiles = B * p->m_per_b;
  p->n_tiles = N / kTN;
  p->k_blocks = H * d / kTK;
  return STOF_OK;
}

}  // namespace
}  // namespace stof

using namespace stof;

extern "C" stof_status stof_oproj_fwd(const void* o, const void* w, const void* bias, const void* residual,
                                      stof_dtype dt, int B, int H, int L, int d, int N, void* y,
                                      int64_t* device_error, void* stream) {
  OpParams p;
  const stof_status st = check_op(o, w, bias, residual, dt, B, H, L, d, N, y, device_error, &p);
  if (st != STOF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dt == STOF_BF16 ? launch_op<true>(o, w, p, s) : launch_op<false>(o, w, p, s);
}

extern "C" size_t stof_oproj_ln_workspace_bytes(int B, int L, int N) {
  if (B < 1 || L < 1 || N < 1 || N % kTN) return 0;
  return static_cast<size_t>(B) * L * (N / kTN) * sizeof(float2);
}

extern "C" stof_status stof_oproj_ln_fwd(const void* o, const void* w, const void* bias, const void* residual,
                                         const void* gamma, const void* beta, float eps, stof_dtype dt, int B,
                                         int H, int L, int d, int N, void* y, void* workspace, size_t ws_bytes,
                                         int64_t* device_error, void* stream) {
  OpParams p;
  stof_status st = check_op(o, w, bias, residual, dt, B, H, L, d, N, y, device_error, &p);
  if (st != STOF_OK) return st;
  if (!workspace || !(eps > 0.f) || !std::isfinite(eps)) return STOF_ERR_INVALID_ARG;
  if (ws_bytes < stof_oproj_ln_workspace_bytes(B, L, N)) return STOF_ERR_WORKSPACE;
  auto al16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
  if (!al16(workspace) || (gamma && !al16(gamma)) || (beta && !al16(beta))) return STOF_ERR_ALIGNMENT;
  p.stats = static_cast<float2*>(workspace);
  LnParams lp;
  lp.stats = p.stats;
  lp.y = y;
  lp.gamma = gamma;
  lp.beta = beta;
  lp.eps = eps;
  lp.rows = static_cast<long long>(B) * L;
  lp.N = N;
  lp.n_tiles = N / kTN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = dt == STOF_BF16 ? launch_op<true>(o, w, p, s) : launch_op<false>(o, w, p, s);
  if (st != STOF_OK) return st;
  return dt == STOF_BF16 ? launch_ln<true>(lp, s) : launch_ln<false>(lp, s);
}
