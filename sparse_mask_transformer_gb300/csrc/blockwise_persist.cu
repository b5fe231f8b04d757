// Persistent block-wise masked attention kernel for head dimension 64
// (TMA + tcgen05 + TMEM, sm_103a).
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, dual-kernel strategy, block-wise kernel (as in
// blockwise.cu): Q, K and V sub-blocks staged in shared memory by
// asynchronous copies overlapping transfer and compute; listed outer tiles
// only, full ones without a mask test, partial ones through their 8x8
// inner-tile bitmaps.
//
// With d = 64 a query tile holds few listed tiles on typical masks (4 to 30
// on the BERT, GPT-2 and Longformer shapes), so a CTA per query tile spends
// much of its life starting up (Q and first K loads before the first
// scores) and finishing (merge and store).  Here one CTA per SM takes query
// tiles ("items") from a work counter, in the order of the one-CTA-per-tile
// kernel (head-major, last OT row of a head first), and overlaps consecutive
// items: Q is double-buffered in shared memory and O in TMEM (per item
// parity), so the next item's Q and K copies, score MMAs and first PVs run
// while the previous item finishes.  The roles are those of blockwise.cu
// (warp 0 Q/K producer and item fetcher, warp 1 V producer, warp 2 score
// MMAs, warp 3 PV MMAs, warps 4-11 two softmax warpgroups); rings and
// barrier phases run on across items, and the item index travels from warp
// 0 to the other warps through a two-slot ring in shared memory.
// Tiles alternate between the two softmax warpgroups over the whole
// sequence of items (global tile T goes to warpgroup T % 2), so the first
// tile of an item goes to the warpgroup that did not take the previous
// item's last tile and can start at once.  The warpgroup that takes an
// item's last tile merges and stores the item (all d columns): the other one
// leaves its row max and sum in shared memory and moves on.
// TMEM columns: S [0,BN) P_0 [128,128+BN/2) P_1 [192,192+BN/2)
// O[item % 2][g] [256 + 128 (item % 2) + 64 g, +64).
//
// A second softmax layout (SWG = 4), one of the tuner's candidates: four
// softmax warpgroups, two per tile parity, each taking one half of a tile's
// key columns for all 128 rows (so each thread holds 64 scores, not 128,
// and 16 softmax warps share the SM instead of 8).  The two warps that hold
// the same rows of the same tile swap their halves' row max through shared
// memory (one mbarrier per pair of warps, bounded wait); both halves then
// take the same rescale decision, write their halves of P, rescale their
// halves of O and keep their own partial sums, which the epilogue adds.
// Same TMEM columns; 640 threads at 96 registers, split 32 / 112.
// The exp split (ESPLIT, another candidate) changes only the softmax's
// exponentials: one key pair in eight on the FMA pipe.
//
// Q, K and V are read through per-head 3-D tensor maps ([B*H][L or Lk][64]):
// a tile that runs past a length that is not a whole number of tiles reads
// zeros there, and O rows past L are not stored.
// The work counter lives in the format's workspace (zeroed by the encoders)
// and is zeroed again by the last CTA to finish, ready for the next launch.
// Every wait is bounded; on timeout the CTA raises STOF_DEVERR_PIPE_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "blockwise_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace stof {

namespace {

using namespace ptx;
using namespace bw;

constexpr int kD = 64;
constexpr int kDefaultRing = 4;   // default K and V ring depth (the tuner also samples 2 and 3)
// warps that read each published item: V producer, 2 issuers, the softmax warps
template <int SWG>
constexpr int kItemReaders = 3 + 4 * SWG;
// With four softmax warpgroups: 4 producer / issuer warps and 16 softmax
// warps.  Five warps per SM sub-partition cap a thread at 96 registers at
// launch; the producers drop to 32 and the softmax warps rise to 112.
constexpr int kThreads4 = 640;
constexpr int kLaunchRegs4 = 96, kProducerRegs4 = 32, kSoftmaxRegs4 = 112;
static_assert(kProducerRegs4 * 128 + kSoftmaxRegs4 * 512 <= kLaunchRegs4 * kThreads4, "register split");
static_assert(kLaunchRegs4 * kThreads4 <= 65536, "register file");
template <int SWG>
constexpr int threads_of = SWG == 4 ? kThreads4 : kThreads;

template <int BN, int kRing>
struct alignas(1024) PSmem {
  uint8_t q[2][Cfg<kD, BN>::Q_BYTES];      // per item parity
  uint8_t k[kRing][Cfg<kD, BN>::KV_BYTES];
  uint8_t v[kRing][Cfg<kD, BN>::KV_BYTES];
  uint64_t q_full[2], q_free[2];           // per Q buffer: loaded / its item's score MMAs done
  uint64_t k_full[kRing], k_free[kRing];
  uint64_t v_full[kRing], v_free[kRing];
  uint64_t s_full[2], s_free[2];           // per warpgroup
  uint64_t p_full[2], pv_done[2];          // per warpgroup
  uint64_t item_full[2], item_free[2];     // ring of work items
  uint64_t xchg[2];                        // per item parity: the max and sum for the epilogue are in
  uint64_t x_free[2];                      // per item parity: the epilogue has read them
  uint64_t o_free[2];                      // per O set: its item's epilogue is done with it
  uint64_t mx[2][4];                       // four warpgroups: per pair and row quarter, both half maxima in xm
  float xml[2][2][kBM];                    // per item parity: max, sum of the early warpgroup per row
  float xml4[2][2][2][2][kBM];             // four warpgroups: [item parity][pair][half][max, sum][row]
  float xm[2][2][2][kBM];                  // four warpgroups: [pair][tile parity][half][row], half-row max
  uint64_t drain, drain_qk;
  int item[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PSmem<128, kDefaultRing>) + 1024 <= 232448, "shared memory");

// One work item: the 128-row query tile (b, h, OT row I) and its listed OTs.
struct Item {
  int bh, I;
  int f0, nf, p0, n;
};

__device__ __forceinline__ Item decode_item(const AttnParams& p, int idx) {
  Item it;
  it.bh = idx / p.n_tr;
  it.I = p.n_tr - 1 - idx % p.n_tr;
  const int b = it.bh / p.H, h = it.bh % p.H;
  const long long mrow = (b * p.stride_b + h * p.stride_h) * p.n_tr + it.I;
  it.f0 = p.full_row_ptr[mrow];
  it.nf = p.full_row_ptr[mrow + 1] - it.f0;
  it.p0 = p.part_row_ptr[mrow];
  it.n = it.nf + (p.part_row_ptr[mrow + 1] - it.p0);
  return it;
}

// NEG: the softmax scale is not positive (see blockwise.cu).  ESPLIT: one
// key pair in eight takes its exponentials on the FMA pipe (two softmax
// warpgroups only).  SWG: softmax warpgroups, 2 or 4.
template <int BN, bool BF16, int kRing, bool NEG, bool ESPLIT, int SWG>
__global__ void __launch_bounds__(threads_of<SWG>, 1)
    blockwise_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const AttnParams p, const int n_items) {
  using C = Cfg<kD, BN>;
  static_assert(SWG == 2 || (SWG == 4 && !ESPLIT), "softmax layout");
  constexpr int HB = BN / 2;    // four warpgroups: keys per half tile
  constexpr int HCH = HB / 32;  // and 32-key chunks per half
  extern __shared__ uint8_t smem_raw[];
  PSmem<BN, kRing>& s = *reinterpret_cast<PSmem<BN, kRing>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_free[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 64 * SWG);  // every softmax thread of the tile's warpgroup(s)
      mbar_init(&s.p_full[i], 64 * SWG);
      mbar_init(&s.pv_done[i], 1);
      mbar_init(&s.item_full[i], 1);
      mbar_init(&s.item_free[i], kItemReaders<SWG>);
      mbar_init(&s.o_free[i], 2 * SWG);   // the epilogue's warps
      mbar_init(&s.xchg[i], SWG == 4 ? 16 : 4);
      mbar_init(&s.x_free[i], 2 * SWG);
      for (int q = 0; q < 4; ++q) mbar_init(&s.mx[i][q], 2);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_free[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_free[i], 1);
    }
    mbar_init(&s.drain, 1);
    mbar_init(&s.drain_qk, 1);
    s.abort_flag = 0;
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
  const uint32_t tS = tbase, tP0 = tbase + 128, tO = tbase + 256;
  volatile int* abort_flag = &s.abort_flag;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, STOF_DEVERR_PIPE_TIMEOUT);
  };
  // a wait whose result is the same in every lane of the warp
  auto wwait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitNs));
  };
  // the k-th item of this CTA, from ring slot k % 2 (whole warp)
  auto read_item = [&](int k, int& idx) {
    if (!wwait(&s.item_full[k & 1], (k >> 1) & 1)) return false;
    idx = s.item[k & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.item_free[k & 1]);
    return true;
  };
  // column index of the t-th listed OT of an item (full OTs first)
  auto column_of = [&](const Item& it, int t) {
    int J = t >= it.nf ? p.part_col_idx[it.p0 + (t - it.nf)] : p.full_col_idx[it.f0 + t];
    if (J < 0 || J >= p.n_tc) {
      raise_error(p.err, STOF_DEVERR_BAD_FORMAT);
      J = 0;
    }
    return J;
  };

  if (warp < 4) {
    regs_dec<SWG == 4 ? kProducerRegs4 : kProducerRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ Q/K producer
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        int st = 0, ph = 0, issued = 0, e = 0;  // K ring position, K tiles issued, items with tiles
        for (int k = 0;; ++k) {
          const int idx = static_cast<int>(atomicAdd(p.work, 1u));
          if (k >= 2 && !mbar_wait(&s.item_free[k & 1], ((k >> 1) & 1) ^ 1, abort_flag, kWaitNs)) {
            fail();
            break;
          }
          s.item[k & 1] = idx;
          mbar_arrive(&s.item_full[k & 1]);
          if (idx >= n_items) break;  // every reader stops at this index too
          const Item it = decode_item(p, idx);
          if (it.n == 0) continue;
          // Q buffer e % 2 held the Q of item e - 2: free once its score MMAs are done
          const int qb = e & 1;
          if (e >= 2 && !mbar_wait(&s.q_free[qb], ((e >> 1) & 1) ^ 1, abort_flag, kWaitNs)) {
            fail();
            break;
          }
          mbar_arrive_expect_tx(&s.q_full[qb], C::Q_BYTES);
          tma_load_3d(s.q[qb], &tmQ, &s.q_full[qb], 0, it.I * kBM, it.bh);
          ++e;
          bool ok = true;
          for (int t = 0; t < it.n; ++t) {
            if (issued >= kRing && !mbar_wait(&s.k_free[st], ph ^ 1, abort_flag, kWaitNs)) {
              fail();
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&s.k_full[st], C::KV_BYTES);
            tma_load_3d(s.k[st], &tmK, &s.k_full[st], 0, column_of(it, t) * BN, it.bh);
            ++issued;
            if (++st == kRing) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
        }
        if (*abort_flag) {  // let every copy this thread started land before exit
          for (int x = e - 2 < 0 ? 0 : e - 2; x < e; ++x) mbar_wait_timeout(&s.q_full[x & 1], (x >> 1) & 1, kWaitNs);
          for (int t = issued - kRing < 0 ? 0 : issued - kRing; t < issued; ++t)
            mbar_wait_timeout(&s.k_full[t % kRing], (t / kRing) & 1, kWaitNs);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ V producer
      if (lane == 0) {
        prefetch_tmap(&tmV);
        int st = 0, ph = 0, issued = 0;
        for (int k = 0;; ++k) {
          if (!mbar_wait(&s.item_full[k & 1], (k >> 1) & 1, abort_flag, kWaitNs)) {
            fail();
            break;
          }
          const int idx = s.item[k & 1];
          mbar_arrive(&s.item_free[k & 1]);
          if (idx >= n_items) break;
          const Item it = decode_item(p, idx);
          bool ok = true;
          for (int t = 0; t < it.n; ++t) {
            if (issued >= kRing && !mbar_wait(&s.v_free[st], ph ^ 1, abort_flag, kWaitNs)) {
              fail();
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&s.v_full[st], C::KV_BYTES);
            tma_load_3d(s.v[st], &tmV, &s.v_full[st], 0, column_of(it, t) * BN, it.bh);
            ++issued;
            if (++st == kRing) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
        }
        if (*abort_flag) {
          for (int t = issued - kRing < 0 ? 0 : issued - kRing; t < issued; ++t)
            mbar_wait_timeout(&s.v_full[t % kRing], (t / kRing) & 1, kWaitNs);
        }
      }
    } else {
      // ------------------------------------------------------------ MMA issuers
      // Tile t of an item belongs to warpgroup t % 2; a warpgroup's barrier
      // phases count its tiles over all items.  Descriptors are built once;
      // a K step adds a compile-time offset.  One elected lane issues.
      constexpr uint32_t idesc_qk = idesc_f16(BF16 ? 1 : 0, 0, kBM, BN);
      constexpr uint32_t idesc_pv = idesc_f16(BF16 ? 1 : 0, 1, kBM, kD);
      constexpr uint64_t kStage = C::KV_BYTES / 16;
      int st = 0, ph = 0, e = 0, c0 = 0, c1 = 0;  // ring position, items with tiles, tiles per warpgroup
      bool ok = true;
      if (warp == 2) {
        const uint64_t qdesc0 = smem_desc_sw128(smem_u32(s.q[0]), 16, 1024);
        const uint64_t kdesc0 = smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
        int pg = -1, pc = 0;  // warpgroup of the previous tile (any item) and its tile count there
        int T0 = 0;           // tiles of the items before this one
        for (int k = 0; ok; ++k) {
          int idx;
          if (!read_item(k, idx)) { ok = false; break; }
          if (idx >= n_items) break;
          const Item it = decode_item(p, idx);
          if (it.n == 0) continue;
          const int qb = e & 1;
          if (!wwait(&s.q_full[qb], (e >> 1) & 1)) { ok = false; break; }
          const uint64_t qdesc = qdesc0 + static_cast<uint64_t>(qb) * (C::Q_BYTES / 16);
          for (int t = 0; t < it.n; ++t) {
            const int g = (T0 + t) & 1;
            if (!wwait(&s.k_full[st], ph)) { ok = false; break; }
            // S is free once the previous tile's scores (of any item) are loaded
            if (pg >= 0 && !wwait(&s.s_free[pg], pc & 1)) { ok = false; break; }
            tc_fence_after();
            const uint64_t kd = kdesc0 + static_cast<uint64_t>(st) * kStage;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk) mma_f16_ss(tS, qdesc + kk * 2, kd + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
              mma_commit(&s.s_full[g]);
              mma_commit(&s.k_free[st]);
            }
            pg = g;
            pc = g ? c1++ : c0++;
            if (++st == kRing) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          if (elect_one()) mma_commit(&s.q_free[qb]);  // Q buffer qb is free once these MMAs are done
          T0 += it.n;
          ++e;
        }
        if (elect_one()) {
          if (!ok) fail();
          mma_commit(&s.drain_qk);
          mbar_wait_timeout(&s.drain_qk, 0, kWaitNs);
        }
      } else {
        const uint64_t vdesc0 = smem_desc_sw128(smem_u32(s.v[0]), C::KV_ATOM, 1024);
        int T0 = 0;
        for (int k = 0; ok; ++k) {
          int idx;
          if (!read_item(k, idx)) { ok = false; break; }
          if (idx >= n_items) break;
          const Item it = decode_item(p, idx);
          if (it.n == 0) continue;
          const int ob = e & 1;  // O set of this item
          for (int t = 0; t < it.n; ++t) {
            const int g = (T0 + t) & 1;
            if (!wwait(&s.v_full[st], ph)) { ok = false; break; }
            if (!wwait(&s.p_full[g], (g ? c1 : c0) & 1)) { ok = false; break; }
            // O set ob held item e - 2: its epilogue must be done with it
            if (t == 0 && e >= 2 && !wwait(&s.o_free[ob], ((e >> 1) & 1) ^ 1)) { ok = false; break; }
            tc_fence_after();
            const uint64_t vd = vdesc0 + static_cast<uint64_t>(st) * kStage;
            const uint32_t d_tmem = tO + ob * 128 + g * kD;
            const uint32_t a_tmem = tP0 + g * 64;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)  // the item's first tile of O_g overwrites it
                mma_f16_ts(d_tmem, a_tmem + kk * 8, vd + kk * 128, idesc_pv, (t >= 2 || kk > 0) ? 1u : 0u);
              mma_commit(&s.pv_done[g]);
              mma_commit(&s.v_free[st]);
            }
            if (g) ++c1; else ++c0;
            if (++st == kRing) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          T0 += it.n;
          ++e;
        }
        if (elect_one()) {
          if (!ok) fail();
          mma_commit(&s.drain);
          mbar_wait_timeout(&s.drain, 0, kWaitNs);
        }
      }
    }
  } else if constexpr (SWG == 4) {
    regs_inc<kSoftmaxRegs4>();
    // ------------------------------------------------------------ softmax
    const int sw = warp - 4;
    const int quarter = warp & 3;
    const int g = (sw >> 2) & 1;        // pair: tiles t with t % 2 == g
    const int hh = sw >> 3;             // key half: columns [HB hh, HB hh + HB) of each tile
    const int r = quarter * 32 + lane;  // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = NEG ? 1.f : p.scale_log2;
    const int bits_off = (r >> 3) * BN + (r & 7) + hh * (HB / 8) * 8;  // this row's byte in an OT's bitmaps
    int J = 0;   // tiles of this pair so far, all items
    int e = 0;   // items with tiles so far
    int T0 = 0;  // tiles of the items before this one
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int idx;
      if (!read_item(k, idx)) { ok = false; break; }
      if (idx >= n_items) break;
      const Item it = decode_item(p, idx);
      const int n = it.n, nf = it.nf, p0 = it.p0;
      // this thread's output row (recomputed where it is used)
      auto out_row = [&]() {
        const int bh = idx / p.n_tr, I = p.n_tr - 1 - idx % p.n_tr;
        return static_cast<uint8_t*>(p.o) +
               (static_cast<size_t>(bh) * p.L + static_cast<size_t>(I) * kBM + r) * (kD * 2);
      };
      // rows past L (a padded last OT row) are computed, not stored
      const bool row_in = (p.n_tr - 1 - idx % p.n_tr) * kBM + r < p.L;
      if (n == 0) {  // no listed tile: the rows of this query tile are 0 (a quarter of each row per warpgroup)
        if (row_in) {
          uint4* z = reinterpret_cast<uint4*>(out_row() + (2 * g + hh) * (kD / 2));
          z[0] = make_uint4(0u, 0u, 0u, 0u);
          z[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int t_first = (g ^ T0) & 1;
      const uint32_t tO_item = tO + (e & 1) * 128 + lane_off;  // this item's O set
      uint32_t nb[HB / 8];  // bitmap bytes of this half of a partial tile, loaded before its scores' wait
      auto fetch_bits = [&](int t) {
        if (t >= nf) {
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.bitmaps) + bits_off +
                               static_cast<long long>(p0 + (t - nf)) * (C::BITMAP_WORDS * 8);
#pragma unroll
          for (int w = 0; w < HB / 8; ++w) nb[w] = __ldg(src + w * 8);
        }
      };
      float m_ref = -INFINITY, l = 0.f;
      for (int t = t_first; t < n; t += 2) {
        const int j = t >> 1;  // this pair's j-th tile of the item
        fetch_bits(t);
        if (!wwait(&s.s_full[g], J & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[HCH][32];
        load_scores(tS + lane_off + hh * HB, sr);
        tc_fence_before();
        mbar_arrive(&s.s_free[g]);  // this half's scores are in registers
        const bool partial = t >= nf;
        uint32_t bits[HCH] = {};
        if (partial) assemble_bits<HCH>(nb, bits);
        if constexpr (NEG) scale_scores(sr, p.scale_log2);
        if (partial) mask_scores(sr, bits);
        // The row max over both halves: each warp leaves its half's max and
        // reads the other half's, written by the warp of the other
        // warpgroup of the pair that holds the same rows.
        const float m_half = row_max(sr);
        const int xs = J & 1;
        s.xm[g][xs][hh][r] = m_half;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.mx[g][quarter]);
        if (!wwait(&s.mx[g][quarter], J & 1)) { ok = false; break; }
        const float mt = fmaxf(m_half, s.xm[g][xs][hh ^ 1][r]) * c;
        float alpha = 1.f;
        if (mt > m_ref + kRescaleThreshold) {  // also the first finite max; the same decision in both halves
          alpha = ex2(m_ref - mt);
          m_ref = mt;
        }
        const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
        l *= alpha;
        // P_g is rewritten once the PV of this pair's previous tile (of any
        // item) is done; that also makes O_g current
        if (J > 0 && !wwait(&s.pv_done[g], (J - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        // this half's P, 32 keys at a time, and its half of a rescaled O,
        // before the PV MMA reads them
#pragma unroll
        for (int cc = 0; cc < HCH; ++cc) {
          uint32_t pk[16];
          l += exp_pack32<BF16>(sr[cc], c, nmu, pk);
          tmem_st16(tP0 + g * 64 + hh * (HB / 2) + lane_off + cc * 16, pk);
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o<kD / 2>(tO_item + g * kD + hh * (kD / 2), alpha);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&s.p_full[g]);
        ++J;
      }
      const int slot = e & 1;  // exchange slot and O set of this item
      // Every warpgroup leaves its row max and its half's sum; the pair
      // that took the item's last tile merges and stores.  The slot held
      // item e - 2's values: wait until they were read.
      if (ok && e >= 2 && !wwait(&s.x_free[slot], ((e >> 1) & 1) ^ 1)) ok = false;
      s.xml4[slot][g][hh][0][r] = m_ref;
      s.xml4[slot][g][hh][1][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.xchg[slot]);
      if (!ok) {
        if (quarter == 0 && lane == 0) fail();
        break;
      }
      if (g == ((T0 + n - 1) & 1)) {  // this pair took the item's last tile
        // O = (a_me O_me + a_ot O_ot) / (a_me l_me + a_ot l_ot) over this
        // half's kD / 2 columns, once the pair's last PV (the item's last)
        // is done and every warpgroup's max and sum are in.
        const bool good = wwait(&s.pv_done[g], (J - 1) & 1) && wwait(&s.xchg[slot], (e >> 1) & 1);
        if (!good) {
          if (quarter == 0 && lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const float mo = s.xml4[slot][g ^ 1][0][0][r];
        const float lo = s.xml4[slot][g ^ 1][0][1][r] + s.xml4[slot][g ^ 1][1][1][r];
        const float lme = s.xml4[slot][g][0][1][r] + s.xml4[slot][g][1][1][r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.x_free[slot]);
        const float m = fmaxf(m_ref, mo);
        const float a_me = m_ref != -INFINITY ? ex2(m_ref - m) : 0.f;
        const float a_ot = (n > 1 && mo != -INFINITY) ? ex2(mo - m) : 0.f;
        const float lt = a_me * lme + a_ot * lo;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float w_me = a_me * inv, w_ot = a_ot * inv;
#pragma unroll
        for (int cc = 0; cc < kD / 32; ++cc) {  // 16 columns at a time
          const uint32_t col = hh * (kD / 2) + cc * 16;
          uint32_t om[16], oo[16];
          tmem_ld16(tO_item + g * kD + col, om);
          tmem_ld_wait(om);
          if (n > 1) {  // the other pair's partial exists only with two tiles or more
            tmem_ld16(tO_item + (g ^ 1) * kD + col, oo);
            tmem_ld_wait(oo);
          }
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float v0 = w_me * __uint_as_float(om[2 * i]);
            float v1 = w_me * __uint_as_float(om[2 * i + 1]);
            if (n > 1) {
              v0 = fmaf(w_ot, __uint_as_float(oo[2 * i]), v0);
              v1 = fmaf(w_ot, __uint_as_float(oo[2 * i + 1]), v1);
            }
            w[i] = pack2<BF16>(v0, v1);
          }
          if (row_in) {
            uint4* dst = reinterpret_cast<uint4*>(out_row() + col * 2);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        // done with this item's O set: the item after next may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.o_free[slot]);
      }
      T0 += n;
      ++e;
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
    // NEG: the scores are multiplied by c before masking and the max, and
    // the softmax below runs with a factor of 1
    const float c = NEG ? 1.f : p.scale_log2;
    const uint8_t* bits_r = reinterpret_cast<const uint8_t*>(p.bitmaps) + (r >> 3) * BN + (r & 7);
    int J = 0;   // tiles of this warpgroup so far, all items
    int e = 0;   // items with tiles so far
    int T0 = 0;  // tiles of the items before this one
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int idx;
      if (!read_item(k, idx)) { ok = false; break; }
      if (idx >= n_items) break;
      const Item it = decode_item(p, idx);
      const int n = it.n, nf = it.nf;
      uint8_t* orow = static_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(it.bh) * p.L + static_cast<size_t>(it.I) * kBM + r) * (kD * 2);
      const bool row_in = it.I * kBM + r < p.L;  // rows past L (a padded last OT row): computed, not stored
      if (n == 0) {  // no listed tile: the rows of this query tile are 0
        if (row_in) {
#pragma unroll
          for (int i = 0; i < kD / 16; ++i) reinterpret_cast<uint4*>(orow + g * kD)[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      // tile t of the item is the warpgroup's iff (T0 + t) % 2 == g: tiles
      // alternate over items, so the next item's first tile goes to the
      // warpgroup that did not take this item's last one
      const int t_first = (g ^ T0) & 1;
      const int g_last = (T0 + n - 1) & 1;  // it merges and stores the item
      const uint32_t tO_item = tO + (e & 1) * 128 + lane_off;  // this item's O set
      const uint32_t tOg = tO_item + g * kD;
      uint32_t nb[BN / 8];  // bitmap bytes of this warpgroup's next partial tile, loaded a tile ahead
      auto fetch_bits = [&](int t) {
        if (t < n && t >= nf) {
          const uint8_t* src = bits_r + static_cast<long long>(it.p0 + (t - nf)) * (C::BITMAP_WORDS * 8);
#pragma unroll
          for (int w = 0; w < BN / 8; ++w) nb[w] = __ldg(src + w * 8);
        }
      };
      float m_ref = -INFINITY, l = 0.f;
      fetch_bits(t_first);
      for (int t = t_first; t < n; t += 2) {
        const int j = t >> 1;  // this warpgroup's j-th tile of the item
        if (!wwait(&s.s_full[g], J & 1)) { ok = false; break; }
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
        // P_g is rewritten once the PV of this warpgroup's previous tile (of
        // any item) is done; that also makes O_g current
        if (J > 0 && !wwait(&s.pv_done[g], (J - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o<kD>(tOg, alpha);
        store_p(tP, pk);  // P (and a rescaled O) in TMEM before the PV MMA reads them
        tc_fence_before();
        mbar_arrive(&s.p_full[g]);
        ++J;
      }
      const int slot = e & 1;  // exchange slot and O set of this item
      if (g != g_last) {
        // Hand the max and sum to the other warpgroup and go on to the next
        // item.  The slot held item e - 2's values: wait until they were read.
        if (ok && e >= 2 && !wwait(&s.x_free[slot], ((e >> 1) & 1) ^ 1)) ok = false;
        s.xml[slot][0][r] = m_ref;
        s.xml[slot][1][r] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.xchg[slot]);
        if (!ok) {
          if (quarter == 0 && lane == 0) fail();
          break;
        }
      } else {
        // Epilogue: O = (a_0 O_0 + a_1 O_1) / (a_0 l_0 + a_1 l_1) over all
        // kD columns, once this warpgroup's last PV (the item's last) is done
        // and the other warpgroup's max and sum are in.
        const bool good = ok && wwait(&s.pv_done[g], (J - 1) & 1) && wwait(&s.xchg[slot], (e >> 1) & 1);
        if (!good) {
          if (quarter == 0 && lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const float mo = s.xml[slot][0][r], lo = s.xml[slot][1][r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.x_free[slot]);
        const float m = fmaxf(m_ref, mo);
        const float a_me = m_ref != -INFINITY ? ex2(m_ref - m) : 0.f;
        const float a_ot = (n > 1 && mo != -INFINITY) ? ex2(mo - m) : 0.f;
        const float lt = a_me * l + a_ot * lo;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float w_me = a_me * inv, w_ot = a_ot * inv;
#pragma unroll
        for (int cc = 0; cc < kD / 32; ++cc) {
          uint32_t om[32], oo[32];
          tmem_ld32(tO_item + g * kD + cc * 32, om);
          tmem_ld_wait(om);
          if (n > 1) {  // the other warpgroup's partial exists only with two tiles or more
            tmem_ld32(tO_item + (g ^ 1) * kD + cc * 32, oo);
            tmem_ld_wait(oo);
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float v0 = w_me * __uint_as_float(om[2 * i]);
            float v1 = w_me * __uint_as_float(om[2 * i + 1]);
            if (n > 1) {
              v0 = fmaf(w_ot, __uint_as_float(oo[2 * i]), v0);
              v1 = fmaf(w_ot, __uint_as_float(oo[2 * i + 1]), v1);
            }
            w[i] = pack2<BF16>(v0, v1);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 64);
          if (row_in) {
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        // done with this item's O set: the item after next may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.o_free[slot]);
      }
      T0 += n;
      ++e;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // The CTA's last fetch (thread 0) is done.  The last CTA to get here sees
  // every fetch of the launch done and zeroes both counters for the next
  // launch on the stream; so the host needs no reset per call.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.work, 0u);
      atomicExch(p.work + 1, 0u);
    }
  }
}

template <int BN, bool BF16, int RING, bool NEG, bool ESPLIT, int SWG>
stof_status launch_persist(const AttnParams& p, cudaStream_t s) {
  const uint64_t heads = static_cast<uint64_t>(p.B) * p.H;
  CUtensorMap mq, mk, mv;
  if (!make_bw_map(&mq, p.q, heads, p.L, kD, kBM, BF16) || !make_bw_map(&mk, p.k, heads, p.Lk, kD, BN, BF16) ||
      !make_bw_map(&mv, p.v, heads, p.Lk, kD, BN, BF16))
    return STOF_ERR_CUDA;
  const size_t smem = sizeof(PSmem<BN, RING>) + 1024;
  stof_status prep = STOF_OK;
  auto prepare = [](const void* arg) {
    stof_status* st = static_cast<stof_status*>(const_cast<void*>(arg));
    if (record_cuda(cudaFuncSetAttribute(blockwise_persist_kernel<BN, BF16, RING, NEG, ESPLIT, SWG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(PSmem<BN, RING>) + 1024))) != cudaSuccess) {
      *st = STOF_ERR_CUDA;
      return false;
    }
    cudaFuncAttributes fa;
    if (record_cuda(cudaFuncGetAttributes(&fa, blockwise_persist_kernel<BN, BF16, RING, NEG, ESPLIT, SWG>)) != cudaSuccess) {
      *st = STOF_ERR_CUDA;
      return false;
    }
    if (fa.numRegs != (SWG == 4 ? kLaunchRegs4 : kLaunchRegs)) {  // the register split needs exactly this
      *st = STOF_ERR_UNSUPPORTED;
      return false;
    }
    return true;
  };
  if (!once_per_device(reinterpret_cast<const void*>(&blockwise_persist_kernel<BN, BF16, RING, NEG, ESPLIT, SWG>), prepare, &prep))
    return prep;
  // one resident CTA per SM, each taking items from the work counter
  const long long n_items = static_cast<long long>(p.B) * p.H * p.n_tr;
  const long long sms = device_sm_count();
  const long long grid = n_items < sms ? n_items : sms;
  blockwise_persist_kernel<BN, BF16, RING, NEG, ESPLIT, SWG><<<static_cast<unsigned>(grid), threads_of<SWG>, smem, s>>>(
      mq, mk, mv, p, static_cast<int>(n_items));
  return record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}

template <int BN, int RING, bool ESPLIT = false, int SWG = 2>
stof_status launch_persist_t(const AttnParams& p, bool bf16, cudaStream_t s) {
  if (p.scale_log2 > 0.f)
    return bf16 ? launch_persist<BN, true, RING, false, ESPLIT, SWG>(p, s)
                : launch_persist<BN, false, RING, false, ESPLIT, SWG>(p, s);
  return bf16 ? launch_persist<BN, true, RING, true, ESPLIT, SWG>(p, s)
              : launch_persist<BN, false, RING, true, ESPLIT, SWG>(p, s);
}

}  // namespace

stof_status launch_blockwise_persist64(const AttnParams& p, bool bf16, cudaStream_t s) {
  if (p.d != kD || p.bm != kBM || (p.bn != 64 && p.bn != 128)) return STOF_ERR_UNSUPPORTED;
  const int ring = p.stages ? p.stages : kDefaultRing;
  const int swg = p.softmax_wg ? p.softmax_wg : 2;
  if (swg != 2 && swg != 4) return STOF_ERR_UNSUPPORTED;
  // the exp split and four softmax warpgroups (tuner candidates, not both
  // at once) on 128 x 128 OTs at the default ring depth
  if (p.exp_split || swg == 4) {
    if (p.bn != 128 || ring != kDefaultRing || (p.exp_split && swg == 4)) return STOF_ERR_UNSUPPORTED;
    return p.exp_split ? launch_persist_t<128, kDefaultRing, true, 2>(p, bf16, s)
                       : launch_persist_t<128, kDefaultRing, false, 4>(p, bf16, s);
  }
  if (p.bn == 64) {
    if (ring != kDefaultRing) return STOF_ERR_UNSUPPORTED;
    return launch_persist_t<64, kDefaultRing>(p, bf16, s);
  }
  if (ring == 2) return launch_persist_t<128, 2>(p, bf16, s);
  if (ring == 3) return launch_persist_t<128, 3>(p, bf16, s);
  if (ring == 4) return launch_persist_t<128, 4>(p, bf16, s);
  return STOF_ERR_UNSUPPORTED;
}

}  // namespace stof
