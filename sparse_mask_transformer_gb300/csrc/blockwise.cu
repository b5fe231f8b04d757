// Block-wise masked attention kernel for sm_103a (TMA + tcgen05 + TMEM).
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, dual-kernel strategy, block-wise kernel: Q, K and
// V are split into sub-blocks staged in shared memory by asynchronous
// copies that overlap data movement with compute; only outer tiles (OT)
// listed in the two-level format are opened, full OTs without a mask test
// and partial OTs through their 8x8 inner-tile bitmaps (same section,
// two-level storage format: exact masking).
//
// One CTA computes one 128-row query tile (b, h, OT row I) over the n OTs
// listed for its row (full OTs first):
//   warp 0      TMA producer: the Q tile once, then the K tile of every
//               listed OT into a ring of ST stages (3 by default; the tuner
//               also samples 2, and 4 at d = 64; stage t % ST is refilled
//               once S = Q K_{t-ST}^T is done);
//   warp 1      TMA producer: the V tiles into a ring of ST stages
//               (refilled once O += P_{t-ST} V_{t-ST} is done);
//   warp 2      allocates TMEM and issues the score MMAs S = Q K_t^T;
//   warp 3      issues the PV MMAs O_g += P_t V_t, P read from TMEM.
//               (Every role has a warp of its own: divergent lanes of one
//               warp are not scheduled promptly while another lane waits.)
//   warps 4..7  softmax warpgroup 0, tiles t = 0, 2, 4, ...;
//   warps 8..11 softmax warpgroup 1, tiles t = 1, 3, 5, ...
// The score MMA writes one TMEM buffer S.  Warpgroup g owns a P buffer P_g
// and an accumulator O_g in TMEM and its own running max and sum.  A thread
// owns one query row (= TMEM lane): it loads its scores into registers and
// at once hands S back, so the score MMA of the next tile (the other
// warpgroup's) runs while this one is processed.  It masks partial OTs by
// their IT bitmaps (read from global memory one tile ahead), updates its
// running max lazily (O_g is rescaled in TMEM only when the max grows by
// more than 2^8; exact, because O_g and l_g share the reference), evaluates
// exp2 in fp32 and writes P as fp16/bf16 pairs into P_g, where the PV MMA
// reads it as its A operand.  Keeping P out of shared memory leaves the
// shared-memory bandwidth to the MMA operands and the K/V copies.  The two
// warpgroups never wait for each other inside the tile loop.  At the end
// their partial results are merged:
// O = (a0 O_0 + a1 O_1) / (a0 l_0 + a1 l_1), a_g = 2^(m_g - max(m_0, m_1));
// 0 for a row without valid keys.
// TMEM columns: S [0,BN) P_0 [128,128+BN/2) P_1 [192,192+BN/2)
// O_0 [256,256+d) O_1 [256+d,256+2d).
// Q, K and V are read through per-head 3-D tensor maps ([B*H][L or Lk][d]):
// a tile that runs past a length that is not a whole number of tiles reads
// zeros there, and O rows past L are not stored.  ESPLIT instances (a tuner
// candidate) take one key pair in eight of the exponentials on the FMA pipe.
// Every pipeline wait is bounded; on timeout the CTA raises
// STOF_DEVERR_PIPE_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "blockwise_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace stof {

namespace {

using namespace ptx;
using namespace bw;

template <int D, int BN, int ST>
struct alignas(1024) Smem {
  uint8_t q[Cfg<D, BN>::Q_BYTES];
  uint8_t k[ST][Cfg<D, BN>::KV_BYTES];  // K ring, stage t % ST; at the end the warpgroups' max and sum
  uint8_t v[ST][Cfg<D, BN>::KV_BYTES];  // V ring, stage t % ST
  uint64_t q_full;
  uint64_t k_full[ST];
  uint64_t k_free[ST];
  uint64_t v_full[ST];
  uint64_t v_free[ST];
  uint64_t s_full[2];   // per warpgroup: the scores of its next tile are in S
  uint64_t s_free[2];   // per warpgroup: it has loaded its tile's scores
  uint64_t p_full[2];   // per warpgroup: P_g written
  uint64_t pv_done[2];  // per warpgroup: its last PV is done (P_g free, O_g current)
  uint64_t drain;
  uint64_t drain_qk;
  uint32_t tmem_base;
  int abort_flag;
  int fail_tile;             // 0 once a softmax thread has failed
};
static_assert(sizeof(Smem<128, 128, 3>) + 1024 <= 232448, "shared memory");
static_assert(sizeof(Smem<64, 128, 4>) + 1024 <= 232448, "shared memory");

// Barrier over `count` threads (a multiple of 32) under hardware barrier id.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// NEG: the softmax scale is not positive (the scores are multiplied by it
// before masking and the row max); a separate instance, so that the usual
// positive scale pays no test.  ESPLIT: one key pair in eight takes its
// exponentials on the FMA pipe (ex2_fma).
template <int D, int BN, bool BF16, int ST, bool NEG, bool ESPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    blockwise_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = Cfg<D, BN>;
  constexpr int kStages = ST;
  extern __shared__ uint8_t smem_raw[];
  Smem<D, BN, ST>& s = *reinterpret_cast<Smem<D, BN, ST>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                   ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: head-major, so CTAs running together stream the same head's
  // K/V through L2; inside a head the heaviest (last) OT rows first
  const int bh = static_cast<int>(blockIdx.x / p.n_tr);
  const int I = p.n_tr - 1 - static_cast<int>(blockIdx.x % p.n_tr);
  const int b = bh / p.H, h = bh % p.H;
  const long long mrow = (b * p.stride_b + h * p.stride_h) * p.n_tr + I;
  const int f0 = p.full_row_ptr[mrow];
  const int nf = p.full_row_ptr[mrow + 1] - f0;
  const int p0 = p.part_row_ptr[mrow];
  const int np = p.part_row_ptr[mrow + 1] - p0;
  const int n = nf + np;

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_free[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 128);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.pv_done[i], 1);
    }
    mbar_init(&s.drain, 1);
    mbar_init(&s.drain_qk, 1);
    s.abort_flag = 0;
    s.fail_tile = 0x7FFFFFFF;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  // S at tbase, P_g at tbase + 128 + 64 g, O_g at tbase + 256 + D g
  const uint32_t tS = tbase, tP0 = tbase + 128, tO0 = tbase + 256;
  volatile int* abort_flag = &s.abort_flag;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, STOF_DEVERR_PIPE_TIMEOUT);
  };

  // a wait whose result is the same in every lane of the warp (tcgen05.ld/st
  // and the issuers' loops are warp-collective)
  auto wwait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitNs));
  };

  // column index of the t-th listed OT of this row (full OTs first)
  auto column_of = [&](int t) {
    int J = t >= nf ? p.part_col_idx[p0 + (t - nf)] : p.full_col_idx[f0 + t];
    if (J < 0 || J >= p.n_tc) {
      raise_error(p.err, STOF_DEVERR_BAD_FORMAT);
      J = 0;
    }
    return J;
  };

  // the softmax rows (128 fp32 scores each) get the registers that the
  // producer and issuer warpgroup does not need
  if (warp < 4) {
    regs_dec<kProducerRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ K producer
      if (lane == 0 && n > 0) {  // Q, then K tiles; a row without listed OTs loads nothing
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        const int qrow = I * kBM;  // row of head bh
        mbar_arrive_expect_tx(&s.q_full, C::Q_BYTES);
#pragma unroll
        for (int r = 0; r < C::REGIONS; ++r) tma_load_3d(s.q + r * 16384, &tmQ, &s.q_full, 64 * r, qrow, bh);
        int issued = 0;
        for (int t = 0, st = 0, ph = 0; t < n; ++t) {
          // stage st = t % ST held K_{t-ST}: free once that tile's scores are done
          if (t >= kStages && !mbar_wait(&s.k_free[st], ph ^ 1, abort_flag, kWaitNs)) {
            fail();
            break;
          }
          const int krow = column_of(t) * BN;
          mbar_arrive_expect_tx(&s.k_full[st], C::KV_BYTES);
#pragma unroll
          for (int r = 0; r < C::REGIONS; ++r)
            tma_load_3d(s.k[st] + r * C::KV_ATOM, &tmK, &s.k_full[st], 64 * r, krow, bh);
          issued = t + 1;
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (*abort_flag) {  // let every copy this thread started land before exit
          mbar_wait_timeout(&s.q_full, 0, kWaitNs);
          for (int t = issued - kStages < 0 ? 0 : issued - kStages; t < issued; ++t)
            mbar_wait_timeout(&s.k_full[t % kStages], (t / kStages) & 1, kWaitNs);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ V producer
      if (lane == 0) {  // V tiles
        prefetch_tmap(&tmV);
        int issued = 0;
        for (int t = 0, st = 0, ph = 0; t < n; ++t) {
          // stage st = t % ST held V_{t-ST}: free once that tile's PV is done
          if (t >= kStages && !mbar_wait(&s.v_free[st], ph ^ 1, abort_flag, kWaitNs)) {
            fail();
            break;
          }
          const int vrow = column_of(t) * BN;
          mbar_arrive_expect_tx(&s.v_full[st], C::KV_BYTES);
#pragma unroll
          for (int r = 0; r < C::REGIONS; ++r)
            tma_load_3d(s.v[st] + r * C::KV_ATOM, &tmV, &s.v_full[st], 64 * r, vrow, bh);
          issued = t + 1;
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (*abort_flag) {
          for (int t = issued - kStages < 0 ? 0 : issued - kStages; t < issued; ++t)
            mbar_wait_timeout(&s.v_full[t % kStages], (t / kStages) & 1, kWaitNs);
        }
      }
    } else {  // warps 2 and 3
      // ------------------------------------------------------------ MMA issuers
      // Warp 2 issues the score MMAs, warp 3 the PV MMAs; each commits to its
      // own barriers (a commit tracks the issuing thread's MMAs only).  Each
      // MMA group is straight-line code.
      constexpr uint32_t idesc_qk = idesc_f16(BF16 ? 1 : 0, 0, kBM, BN);
      constexpr uint32_t idesc_pv = idesc_f16(BF16 ? 1 : 0, 1, kBM, D);
      // Descriptors are built once; a K step only adds a compile-time offset
      // (in 16-byte units) to the start-address field.  An issuing thread is
      // latency-bound, so per-MMA descriptor arithmetic would otherwise
      // throttle the tensor core.
      constexpr uint64_t kStage = C::KV_BYTES / 16;
      // The whole warp runs the loop (warp-uniform waits and descriptor
      // arithmetic, which keeps the descriptors in uniform registers); one
      // elected lane issues the MMAs and commits.
      if (warp == 2) {
        const uint64_t qdesc = smem_desc_sw128(smem_u32(s.q), 16, 1024);
        const uint64_t kdesc0 = smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
        bool ok = n == 0 || wwait(&s.q_full, 0);
        for (int t = 0, st = 0, ph = 0; ok && t < n; ++t) {
          // S is free once the previous tile's scores are loaded (by the
          // other warpgroup).  K_t is usually in place first, so that wait
          // comes first and the issue follows the hand-back of S at once.
          if (!wwait(&s.k_full[st], ph)) { ok = false; break; }
          if (t >= 1 && !wwait(&s.s_free[(t - 1) & 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kd = kdesc0 + static_cast<uint64_t>(st) * kStage;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // 32 B per K step inside an atom; Q atoms are 16 KB apart, K atoms BN * 128 B
              const uint64_t qoff = (kk >> 2) * (C::Q_BYTES / C::REGIONS / 16) + (kk & 3) * 2;
              const uint64_t koff = (kk >> 2) * (C::KV_ATOM / 16) + (kk & 3) * 2;
              mma_f16_ss(tS, qdesc + qoff, kd + koff, idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(&s.s_full[t & 1]);
            mma_commit(&s.k_free[st]);
          }
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (elect_one()) {  // the lane that issued the MMAs
          if (!ok) fail();
          mma_commit(&s.drain_qk);  // all of this thread's MMAs done before TMEM is freed
          mbar_wait_timeout(&s.drain_qk, 0, kWaitNs);
        }
      } else {
        const uint64_t vdesc0 = smem_desc_sw128(smem_u32(s.v[0]), C::KV_ATOM, 1024);
        bool ok = true;
        for (int t = 0, st = 0, ph = 0; ok && t < n; ++t) {
          const int g = t & 1;  // warpgroup, P buffer and accumulator of tile t
          // V_t is usually in place before P_t
          if (!wwait(&s.v_full[st], ph)) { ok = false; break; }
          if (!wwait(&s.p_full[g], (t >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vd = vdesc0 + static_cast<uint64_t>(st) * kStage;
          const uint32_t d_tmem = tO0 + g * D;
          const uint32_t a_tmem = tP0 + g * 64;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {  // 16 keys (8 TMEM columns of P) per K step
              // the first tile of O_g overwrites it
              mma_f16_ts(d_tmem, a_tmem + kk * 8, vd + kk * 128, idesc_pv, (t >= 2 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&s.pv_done[g]);
            mma_commit(&s.v_free[st]);
          }
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (elect_one()) {  // the lane that issued the MMAs
          if (!ok) fail();
          mma_commit(&s.drain);
          mbar_wait_timeout(&s.drain, 0, kWaitNs);
        }
      }
    }
  } else {
    regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int g = (warp - 4) >> 2;      // warpgroup: tiles t with t % 2 == g
    const int r = quarter * 32 + lane;  // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tSr = tS + lane_off;
    const uint32_t tP = tP0 + g * 64 + lane_off;
    const uint32_t tO = tO0 + g * D + lane_off;
    // NEG: the scores are multiplied by c before masking and the max, and
    // the softmax below runs with a factor of 1
    const float c = NEG ? 1.f : p.scale_log2;
    // row r of an OT's bitmaps: byte r % 8 of words (r / 8) * BN / 8 + 0 .. BN / 8 - 1
    const uint8_t* bits_row = reinterpret_cast<const uint8_t*>(p.bitmaps) + (r >> 3) * BN + (r & 7);
    uint32_t nb[BN / 8];  // bitmap bytes of this warpgroup's next partial tile, loaded a tile ahead
    auto fetch_bits = [&](int t) {
      if (t < n && t >= nf) {
        const uint8_t* src = bits_row + static_cast<long long>(p0 + (t - nf)) * (C::BITMAP_WORDS * 8);
#pragma unroll
        for (int w = 0; w < BN / 8; ++w) nb[w] = __ldg(src + w * 8);
      }
    };
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    fetch_bits(g);
    for (int t = g; ok && t < n; t += 2) {
      const int j = t >> 1;  // this warpgroup's j-th tile
      if (!wwait(&s.s_full[g], j & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[C::CHUNKS][32];
      load_scores(tSr, sr);
      tc_fence_before();
      mbar_arrive(&s.s_free[g]);  // the scores are in registers: S may be overwritten
      const bool partial = t >= nf;
      uint32_t bits[C::CHUNKS] = {};
      if (partial) assemble_bits<C::CHUNKS>(nb, bits);
      fetch_bits(t + 2);                        // the bytes of this warpgroup's next tile
      if constexpr (NEG) scale_scores(sr, p.scale_log2);
      if (partial) mask_scores(sr, bits);       // keep only the keys whose bit is set
      const float mt = row_max(sr) * c;
      float alpha = 1.f;
      if (mt > m_ref + kRescaleThreshold) {  // also the first finite max
        alpha = ex2(m_ref - mt);             // 0 when m_ref = -inf
        m_ref = mt;
      }
      const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
      l *= alpha;
      uint32_t pk[C::CHUNKS][16];
      l += exp_pack<C::CHUNKS, BF16, ESPLIT>(sr, c, nmu, pk);
      if (j > 0) {
        // P_g is rewritten and O_g rescaled once the PV of this warpgroup's
        // previous tile is done
        if (!wwait(&s.pv_done[g], (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) rescale_o<D>(tO, alpha);
      }
      store_p(tP, pk);  // P (and a rescaled O) in TMEM before the PV MMA reads them
      tc_fence_before();
      mbar_arrive(&s.p_full[g]);
    }
    // epilogue: merge the two warpgroups' partial results; warpgroup g
    // writes columns g*D/2 .. g*D/2 + D/2 - 1 of each row
    const int n_mine = n > g ? (n - 1 - g) / 2 + 1 : 0;  // tiles of this warpgroup
    const bool good = ok && (n_mine == 0 || wwait(&s.pv_done[g], (n_mine - 1) & 1));
    if (!good) atomicMin(&s.fail_tile, 0);
    // Once both warpgroups' last PVs are done, every MMA and every K copy
    // has finished: K stage 0 then carries each warpgroup's final max and
    // sum to the other.
    named_bar_sync(1, 256);
    float* xg = reinterpret_cast<float*>(s.k[0]) + g * 2 * kBM;
    if (s.fail_tile == 0x7FFFFFFF) {
      xg[r] = m_ref;
      xg[kBM + r] = l;
    }
    named_bar_sync(1, 256);
    if (s.fail_tile < 0x7FFFFFFF) {
      if (g == 0 && quarter == 0 && lane == 0) fail();
    } else {
      tc_fence_after();
      const float* x0 = reinterpret_cast<const float*>(s.k[0]);
      const float* x1 = x0 + 2 * kBM;
      const float m0 = x0[r], m1 = x1[r];
      const float m = fmaxf(m0, m1);
      const float a0 = (n > 0 && m0 != -INFINITY) ? ex2(m0 - m) : 0.f;
      const float a1 = (n > 1 && m1 != -INFINITY) ? ex2(m1 - m) : 0.f;
      const float lt = a0 * x0[kBM + r] + a1 * x1[kBM + r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float w0 = a0 * inv, w1 = a1 * inv;
      // a query tile of a padded last OT row has rows past L: computed, not stored
      const bool row_in = I * kBM + r < p.L;
      uint8_t* orow = static_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(bh) * p.L + static_cast<size_t>(I) * kBM + r) * (D * 2) + g * D;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = g * (D / 2) + cc * 32;
        uint32_t o0[32], o1[32];
        if (n > 0) {
          tmem_ld32(tO0 + lane_off + col, o0);
          tmem_ld_wait(o0);
        }
        if (n > 1) {
          tmem_ld32(tO0 + D + lane_off + col, o1);
          tmem_ld_wait(o1);
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v0 = 0.f, v1 = 0.f;
          if (n > 0) {
            v0 = w0 * __uint_as_float(o0[2 * i]);
            v1 = w0 * __uint_as_float(o0[2 * i + 1]);
          }
          if (n > 1) {
            v0 = fmaf(w1, __uint_as_float(o1[2 * i]), v0);
            v1 = fmaf(w1, __uint_as_float(o1[2 * i + 1]), v1);
          }
          w[i] = pack2<BF16>(v0, v1);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 64);
        if (row_in) {
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
// [heads][L][D] row-major 16-bit tensor (one [L][D] matrix per head, as
// Q, K and V are), box = 64 columns x box_rows rows of one head, 128-byte
// swizzle; a box that runs past row L of its head reads zeros there.
// A tensor map holds only the address, sizes, strides and box of a tensor,
// so a map made once stays right for every later call with the same key;
// the cache (round-robin over kMapCache entries) spares the driver call that
// otherwise dominates a short launch's host time.
namespace {
struct MapKey {
  int dev;
  const void* base;
  uint64_t heads, L;
  int D, box_rows;
  bool bf16;
  bool operator==(const MapKey& o) const {
    return dev == o.dev && base == o.base && heads == o.heads && L == o.L && D == o.D && box_rows == o.box_rows &&
           bf16 == o.bf16;
  }
};
struct MapEntry {
  CUtensorMap map;
  MapKey key;
  bool used;
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
}  // namespace

bool make_bw_map(CUtensorMap* m, const void* base, uint64_t heads, uint64_t L, int D, int box_rows, bool bf16) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const MapKey key{dev, base, heads, L, D, box_rows, bf16};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& e : g_maps)
      if (e.used && e.key == key) {
        *m = e.map;
        return true;
      }
  }
  if (!encode_tensor_map_3d(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base,
                            static_cast<uint64_t>(D), L, heads, static_cast<uint64_t>(D) * 2,
                            L * static_cast<uint64_t>(D) * 2, 64, static_cast<uint32_t>(box_rows),
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  e.map = *m;
  e.key = key;
  e.used = true;
  return true;
}

namespace {

template <int D, int BN, bool BF16, int ST, bool NEG, bool ESPLIT>
stof_status launch_bw(const AttnParams& p, cudaStream_t s) {
  const uint64_t heads = static_cast<uint64_t>(p.B) * p.H;
  CUtensorMap mq, mk, mv;
  if (!make_bw_map(&mq, p.q, heads, p.L, D, kBM, BF16) || !make_bw_map(&mk, p.k, heads, p.Lk, D, BN, BF16) ||
      !make_bw_map(&mv, p.v, heads, p.Lk, D, BN, BF16))
    return STOF_ERR_CUDA;
  const size_t smem = sizeof(Smem<D, BN, ST>) + 1024;
  stof_status prep = STOF_OK;
  auto prepare = [](const void* arg) {
    stof_status* st = static_cast<stof_status*>(const_cast<void*>(arg));
    if (record_cuda(cudaFuncSetAttribute(blockwise_kernel<D, BN, BF16, ST, NEG, ESPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(Smem<D, BN, ST>) + 1024))) != cudaSuccess) {
      *st = STOF_ERR_CUDA;
      return false;
    }
    cudaFuncAttributes fa;
    if (record_cuda(cudaFuncGetAttributes(&fa, blockwise_kernel<D, BN, BF16, ST, NEG, ESPLIT>)) != cudaSuccess) {
      *st = STOF_ERR_CUDA;
      return false;
    }
    if (fa.numRegs != kLaunchRegs) {  // the register split needs exactly this
      *st = STOF_ERR_UNSUPPORTED;
      return false;
    }
    return true;
  };
  if (!once_per_device(reinterpret_cast<const void*>(&blockwise_kernel<D, BN, BF16, ST, NEG, ESPLIT>), prepare, &prep))
    return prep;
  const long long grid = static_cast<long long>(p.B) * p.H * p.n_tr;
  blockwise_kernel<D, BN, BF16, ST, NEG, ESPLIT><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(mq, mk, mv, p);
  return record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}

}  // namespace

template <int D, int BN, int ST, bool ESPLIT = false>
stof_status launch_bw_t(const AttnParams& p, bool bf16, cudaStream_t s) {
  if (p.scale_log2 > 0.f)
    return bf16 ? launch_bw<D, BN, true, ST, false, ESPLIT>(p, s) : launch_bw<D, BN, false, ST, false, ESPLIT>(p, s);
  return bf16 ? launch_bw<D, BN, true, ST, true, ESPLIT>(p, s) : launch_bw<D, BN, false, ST, true, ESPLIT>(p, s);
}

namespace {
__global__ void ex2_fma_kernel(const float* x, float* y, long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    y[i] = bw::ex2_fma(x[i]);
}
}  // namespace

stof_status launch_blockwise(const AttnParams& p, bool bf16, cudaStream_t s) {
  if (p.bm != kBM || (p.bn != 64 && p.bn != 128) || (p.d != 64 && p.d != 128)) return STOF_ERR_UNSUPPORTED;
  if (static_cast<long long>(p.B) * p.H * (p.L > p.Lk ? p.L : p.Lk) >= (1ll << 31)) return STOF_ERR_SHAPE;
  // d = 64 with short query tiles (few listed OTs each): persistent CTAs that
  // overlap one query tile's start-up and finish with the next
  if (blockwise_persistent(p.d, p.variant, p.tiles_per_row)) return launch_blockwise_persist64(p, bf16, s);
  // ring depths: 3 by default; the tuner also samples 2 (and 4 at d = 64) on 128 x 128 OTs
  const int st = p.stages ? p.stages : kStages;
  if (p.softmax_wg != 0 && p.softmax_wg != 2) return STOF_ERR_UNSUPPORTED;
  if (p.exp_split) {  // sampled on 128 x 128 OTs at the default ring depth
    if (p.bn != 128 || st != kStages) return STOF_ERR_UNSUPPORTED;
    return p.d == 64 ? launch_bw_t<64, 128, 3, true>(p, bf16, s) : launch_bw_t<128, 128, 3, true>(p, bf16, s);
  }
  if (p.bn == 64) {
    if (st != kStages) return STOF_ERR_UNSUPPORTED;
    return p.d == 64 ? launch_bw_t<64, 64, 3>(p, bf16, s) : launch_bw_t<128, 64, 3>(p, bf16, s);
  }
  if (p.d == 64) {
    if (st == 2) return launch_bw_t<64, 128, 2>(p, bf16, s);
    if (st == 3) return launch_bw_t<64, 128, 3>(p, bf16, s);
    if (st == 4) return launch_bw_t<64, 128, 4>(p, bf16, s);
    return STOF_ERR_UNSUPPORTED;
  }
  if (st == 2) return launch_bw_t<128, 128, 2>(p, bf16, s);
  if (st == 3) return launch_bw_t<128, 128, 3>(p, bf16, s);
  return STOF_ERR_UNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [planes][rows][inner] with `row_bytes` between rows and `plane_bytes`
// between planes; boxes of box_inner x box_rows x 1; zeros outside.
bool encode_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t planes, uint64_t row_bytes, uint64_t plane_bytes,
                          uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {row_bytes, plane_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!count[dev] && cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    count[dev] = 1;
  return count[dev];
}

}  // namespace stof

extern "C" stof_status stof_ex2_fma(const float* x, float* y, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return STOF_ERR_INVALID_ARG;
  if (n == 0) return STOF_OK;
  const long long blocks = std::min<long long>((n + 255) / 256, 16ll * stof::device_sm_count());
  stof::ex2_fma_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return stof::record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}
