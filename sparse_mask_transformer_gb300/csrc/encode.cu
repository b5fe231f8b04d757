// Mask encoder: dense uint8 mask -> STOF two-level format.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 1, Unified MHA module, two-level storage format:
// outer tiles (OT) are empty (skipped), full (every element valid) or
// partial (mixed); full and partial OTs are tracked by pointer arrays; each
// 8x8 inner tile (IT) of a partial OT is one uint64 bitmap.
//
// GB300 design: one pass over the mask, which is the only large stream
// (HBM-bound).  The work unit is a chunk = one OT row band x `ct`
// consecutive OTs (about 1024 mask columns).  For a chunk the encoder
//   1. packs each 8x8 IT of the chunk into a uint64 in shared memory
//      (bit 8r+c = byte (r, c) non-zero);
//   2. classifies each OT by AND / OR over its IT words;
//   3. gets the global offsets of its full and partial OTs from a
//      single-pass chained prefix sum with decoupled look-back (Merrill and
//      Garland, "Single-pass Parallel Prefix Scan with Decoupled
//      Look-back", 2016); chunks are numbered by an atomic ticket in the
//      order they are started, so every chunk it waits on is already being
//      worked on;
//   4. writes column indices, row pointers and the bitmaps of its partial
//      OTs straight into their final slots.
// Step 1 has two sources in this single-pass kernel: a dense byte mask and
// a parametric mask, whose IT words are computed from its rule (band on
// i - j, global rows and columns, block pattern) without reading any mask;
// steps 2-4 are shared.  A bit-packed mask (one byte of a row is one IT row)
// goes through three short kernels instead (further below).
// One CTA per chunk, 256 threads, at least seven CTAs per SM (eight are
// resident at the 32 registers the kernel takes) so that the loads of some
// CTAs overlap the look-back and writes of others; 16-byte (else 8-byte)
// coalesced streaming loads.  (A persistent variant that streamed
// the mask through a TMA ring with a producer warp was measured 3x slower
// on the 16k workload: one CTA per SM cannot hide each chunk's look-back.)
// Every wait on another CTA or warp is bounded; on timeout the CTA raises
// STOF_DEVERR_LOOKBACK_TIMEOUT in the device error word and finishes.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace stof {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxTilesPerChunk = 128;
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagInc = 2ull << 62;
constexpr unsigned long long kValMask = (1ull << 62) - 1;
constexpr uint64_t kLookbackTimeoutNs = 2000000000ull;

// bit c of the result = (byte c of w != 0), 4 bytes.  The msb of
// ((w & 0x7F..) + 0x7F..) | w is set iff the byte is non-zero (no carry
// crosses a byte); the multiply gathers bits 7, 15, 23, 31 into 28..31.
__device__ __forceinline__ uint32_t pack_word4(uint32_t w) {
  const uint32_t h = (((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) & 0x80808080u;
  return (h * 0x00204081u) >> 28;
}

__device__ __forceinline__ unsigned long long ld_volatile(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ void st_volatile(unsigned long long* p, unsigned long long v) {
  *reinterpret_cast<volatile unsigned long long*>(p) = v;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Per-chunk state shared by a CTA's threads.
struct ChunkState {
  unsigned long long nnz;
  unsigned long long excl;
  int nf, np;
  uint8_t cls[kMaxTilesPerChunk];
  int rank[kMaxTilesPerChunk];
  int plist[kMaxTilesPerChunk];
};

struct ChunkGeom {
  long long row;
  int cc, m, I, J0, nt, itc, itcols, bands, wpt;
  uint64_t rcp_itc, rcp_wpt;  // ceil(2^32 / itc), ceil(2^32 / wpt): see qdiv
};

// e / d for the reciprocal rcp = ceil(2^32 / d): exact while e * d < 2^32
// (with rcp = (2^32 + k) / d, 0 <= k < d, the product overshoots e / d by
// e k / (d 2^32) < 1 / d).  The encoder's divisors are at most 1024 and its
// dividends below 2^17.
__device__ __forceinline__ int qdiv(int e, uint64_t rcp) {
  return static_cast<int>((static_cast<uint64_t>(e) * rcp) >> 32);
}
__host__ __device__ __forceinline__ uint64_t reciprocal(uint32_t d) { return 0xFFFFFFFFull / d + 1; }

__device__ __forceinline__ ChunkGeom chunk_geom(const EncodeParams& p, long long chunk) {
  ChunkGeom g;
  const uint32_t c = static_cast<uint32_t>(chunk);  // chunk < n_chunks < 2^31
  const uint32_t row = c / static_cast<uint32_t>(p.cpr);
  g.row = row;
  g.cc = static_cast<int>(c - row * static_cast<uint32_t>(p.cpr));
  g.m = static_cast<int>(row / static_cast<uint32_t>(p.n_tr));
  g.I = static_cast<int>(row - static_cast<uint32_t>(g.m) * static_cast<uint32_t>(p.n_tr));
  g.J0 = g.cc * p.ct;
  g.nt = min(p.ct, p.n_tc - g.J0);
  g.itc = p.bn >> 3;
  g.itcols = g.nt * g.itc;
  g.bands = p.bm >> 3;
  g.wpt = g.bands * g.itc;
  g.rcp_itc = p.rcp_itc;
  g.rcp_wpt = p.rcp_wpt;
  return g;
}

// Phase 2: class of every OT of the chunk (0 empty, 1 full, 2 partial), one
// warp per OT.
__device__ __forceinline__ void classify(const uint64_t* words, const ChunkGeom& g, ChunkState& cs, int warp,
                                         int lane, int nwarps) {
  for (int t = warp; t < g.nt; t += nwarps) {
    uint64_t any = 0, all = ~0ull;
    for (int e = lane; e < g.wpt; e += 32) {
      const int pb = qdiv(e, g.rcp_itc), qq = e - pb * g.itc;
      const uint64_t w = words[pb * g.itcols + t * g.itc + qq];
      any |= w;
      all &= w;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      any |= __shfl_xor_sync(0xffffffffu, any, off);
      all &= __shfl_xor_sync(0xffffffffu, all, off);
    }
    if (lane == 0) cs.cls[t] = any == 0 ? 0 : (all == ~0ull ? 1 : 2);
  }
}

// Phase 3 (one warp): ranks inside the chunk and the chained prefix sum.
__device__ __forceinline__ void rank_and_lookback(const EncodeParams& p, long long chunk, const ChunkGeom& g,
                                                  ChunkState& cs, int lane) {
  int nf = 0, np = 0;
  for (int t0 = 0; t0 < g.nt; t0 += 32) {
    const int t = t0 + lane;
    const int cls = t < g.nt ? cs.cls[t] : 0;
    const unsigned bf = __ballot_sync(0xffffffffu, cls == 1);
    const unsigned bp = __ballot_sync(0xffffffffu, cls == 2);
    const unsigned lt = (1u << lane) - 1u;
    if (cls == 1) cs.rank[t] = nf + __popc(bf & lt);
    if (cls == 2) {
      const int r = np + __popc(bp & lt);
      cs.rank[t] = r;
      cs.plist[r] = t;
    }
    nf += __popc(bf);
    np += __popc(bp);
  }
  const unsigned long long agg = (static_cast<unsigned long long>(nf) << 31) | static_cast<unsigned long long>(np);
  unsigned long long excl = 0;
  if (chunk == 0) {
    if (lane == 0) st_volatile(&p.status[0], kFlagInc | agg);
  } else {
    if (lane == 0) st_volatile(&p.status[chunk], kFlagAgg | agg);
    long long top = chunk - 1;
    const uint64_t t_start = now_ns();
    bool timed_out = false;
    while (true) {
      const long long idx = top - lane;
      const unsigned long long v = idx >= 0 ? ld_volatile(&p.status[idx]) : kFlagInc;
      const unsigned long long flag = v >> 62;
      const unsigned inc = __ballot_sync(0xffffffffu, flag == 2);
      const unsigned notready = __ballot_sync(0xffffffffu, flag == 0);
      const int first_inc = inc ? __ffs(inc) - 1 : 32;
      const unsigned needed = first_inc >= 31 ? 0xffffffffu : ((2u << first_inc) - 1u);
      if ((notready & needed) && !timed_out) {
        if (now_ns() - t_start > kLookbackTimeoutNs) {
          timed_out = true;  // treat missing predecessors as empty, report
          if (lane == 0)
            atomicOr(reinterpret_cast<unsigned long long*>(&p.counts[3]),
                     static_cast<unsigned long long>(STOF_DEVERR_LOOKBACK_TIMEOUT));
        } else {
          __nanosleep(64);
        }
        continue;
      }
      unsigned long long val = (lane <= first_inc && flag != 0) ? (v & kValMask) : 0ull;
#pragma unroll
      for (int off = 16; off; off >>= 1) val += __shfl_xor_sync(0xffffffffu, val, off);
      excl += val;
      if (first_inc < 32 || timed_out) break;
      top -= 32;
    }
    if (lane == 0) st_volatile(&p.status[chunk], kFlagInc | (excl + agg));
  }
  if (lane == 0) {
    cs.excl = excl;
    cs.nf = nf;
    cs.np = np;
    if (cs.nnz) atomicAdd(reinterpret_cast<unsigned long long*>(&p.counts[2]), cs.nnz);
  }
}

// Phase 4: column indices, row pointers and bitmaps into their final slots.
__device__ __forceinline__ void write_outputs(const EncodeParams& p, long long chunk, const uint64_t* words,
                                              const ChunkGeom& g, const ChunkState& cs, int tid, int nthreads) {
  const long long ef = static_cast<long long>((cs.excl >> 31) & 0x7FFFFFFFull);
  const long long ep = static_cast<long long>(cs.excl & 0x7FFFFFFFull);
  const int nf = cs.nf, np = cs.np;
  if (g.cc == 0 && tid == 0) {
    p.full_row_ptr[g.row] = static_cast<int32_t>(ef);
    p.part_row_ptr[g.row] = static_cast<int32_t>(ep);
  }
  for (int t = tid; t < g.nt; t += nthreads) {
    const int cls = cs.cls[t];
    if (cls == 1) p.full_col_idx[ef + cs.rank[t]] = g.J0 + t;
    if (cls == 2) p.part_col_idx[ep + cs.rank[t]] = g.J0 + t;
  }
  const int total = np * g.wpt;
  for (int e = tid; e < total; e += nthreads) {
    const int r = qdiv(e, g.rcp_wpt), x = e - r * g.wpt;
    const int t = cs.plist[r];
    const int pb = qdiv(x, g.rcp_itc), qq = x - pb * g.itc;
    p.bitmaps[(ep + r) * g.wpt + x] = words[pb * g.itcols + t * g.itc + qq];
  }
  if (chunk == p.n_chunks - 1 && tid == 0) {
    p.full_row_ptr[p.n_rows] = static_cast<int32_t>(ef + nf);
    p.part_row_ptr[p.n_rows] = static_cast<int32_t>(ep + np);
    p.counts[0] = ef + nf;
    p.counts[1] = ep + np;
  }
}

// Columns c0..c0+3 of rows a, b, c, d (one byte per column in each word) to
// one word per column holding rows a, b, c, d in bytes 0..3.
__device__ __forceinline__ void transpose4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&out)[4]) {
  const uint32_t ab01 = __byte_perm(a, b, 0x5140), ab23 = __byte_perm(a, b, 0x7362);
  const uint32_t cd01 = __byte_perm(c, d, 0x5140), cd23 = __byte_perm(c, d, 0x7362);
  out[0] = __byte_perm(ab01, cd01, 0x5410);
  out[1] = __byte_perm(ab01, cd01, 0x7632);
  out[2] = __byte_perm(ab23, cd23, 0x5410);
  out[3] = __byte_perm(ab23, cd23, 0x7632);
}

// For a bit-packed mask (bit c of byte jb of a row = column 8 jb + c), one
// byte of a row is one IT row, so an IT word is the bytes of its eight rows
// in order.  A unit is VEC bytes (VEC IT columns) of 8 consecutive rows at
// src; it becomes VEC words at dst.  Returns their valid-element count.
template <int VEC>
__device__ __forceinline__ unsigned long long pack_bits_unit(const uint8_t* src, long long row_bytes,
                                                             uint64_t* dst) {
  unsigned long long nnz = 0;
  if constexpr (VEC == 1) {
    uint64_t word = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) word |= static_cast<uint64_t>(__ldcs(src + r * row_bytes)) << (8 * r);
    dst[0] = word;
    nnz += __popcll(word);
  } else {
    constexpr int G = VEC / 4;  // 4-column groups
    uint32_t x[8][G];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if constexpr (VEC == 16) {
        const uint4 t = __ldcs(reinterpret_cast<const uint4*>(src + r * row_bytes));
        x[r][0] = t.x; x[r][1] = t.y; x[r][2] = t.z; x[r][3] = t.w;
      } else {
        const uint2 t = __ldcs(reinterpret_cast<const uint2*>(src + r * row_bytes));
        x[r][0] = t.x; x[r][1] = t.y;
      }
    }
    // dst is 16-byte aligned for VEC = 8 and 16: the words go out as 16-byte stores
#pragma unroll
    for (int cg = 0; cg < G; ++cg) {
      uint32_t lo[4], hi[4];
      transpose4(x[0][cg], x[1][cg], x[2][cg], x[3][cg], lo);
      transpose4(x[4][cg], x[5][cg], x[6][cg], x[7][cg], hi);
#pragma unroll
      for (int i = 0; i < 4; ++i) nnz += __popc(lo[i]) + __popc(hi[i]);
      uint4* d4 = reinterpret_cast<uint4*>(dst + 4 * cg);
      d4[0] = make_uint4(lo[0], hi[0], lo[1], hi[1]);
      d4[1] = make_uint4(lo[2], hi[2], lo[3], hi[3]);
    }
  }
  return nnz;
}

// Phases 2-4 of a chunk whose IT words are in shared memory: the chunk's
// valid-element count, OT classes, global offsets and outputs.
__device__ __forceinline__ void finish_chunk(const EncodeParams& p, long long chunk, const ChunkGeom& g,
                                             ChunkState& cs, const uint64_t* s_words,
                                             unsigned long long local_nnz, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) local_nnz += __shfl_xor_sync(0xffffffffu, local_nnz, off);
  if (lane == 0 && local_nnz) atomicAdd(&cs.nnz, local_nnz);
  __syncthreads();
  classify(s_words, g, cs, warp, lane, kThreads / 32);
  __syncthreads();
  if (warp == 0) rank_and_lookback(p, chunk, g, cs, lane);
  __syncthreads();
  write_outputs(p, chunk, s_words, g, cs, tid, kThreads);
}

// n bytes (n <= VEC; none if n <= 0) from src into the low bytes of a uint4,
// the rest 0: the part of an IT row that lies inside the mask.
template <int VEC>
__device__ __forceinline__ uint4 load_partial(const uint8_t* src, int n) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int b = 0; b < VEC; ++b)
    if (b < n) w[b >> 2] |= static_cast<uint32_t>(src[b]) << (8 * (b & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- kernel 1
// VEC: bytes per load (16 when rows and tiles are 16-byte aligned, else 8).
// ALIGNED: mask rows start on VEC-byte boundaries, so whole units are read
// with vector loads; else byte by byte.  A mask whose sides are not whole
// OTs is encoded as its zero-padded extension: nothing outside lq x lk is
// read, and those elements count as invalid.
template <int VEC, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 7) encode_kernel(const EncodeParams p) {
  extern __shared__ uint64_t s_words[];  // [bm/8][nt * bn/8]
  __shared__ long long s_chunk;
  __shared__ ChunkState cs;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_chunk = static_cast<long long>(atomicAdd(p.ticket, 1ull));
    cs.nnz = 0;
  }
  __syncthreads();
  const long long chunk = s_chunk;
  if (chunk >= p.n_chunks) return;
  const ChunkGeom g = chunk_geom(p, chunk);
  const uint8_t* base = p.mask + (static_cast<long long>(g.m) * p.lq + static_cast<long long>(g.I) * p.bm) * p.lk +
                        static_cast<long long>(g.J0) * p.bn;

  // 1. read and pack (each unit = VEC/8 adjacent IT words of one 8-row band)
  unsigned long long local_nnz = 0;
  // a chunk wholly inside the mask, with VEC-aligned rows: vector loads;
  // else (a chunk at the lower or right edge of a padded side, or rows not
  // aligned) byte-guarded loads, one IT word per unit
  const bool interior = ALIGNED && (g.I + 1) * p.bm <= p.lq && (g.J0 + g.nt) * p.bn <= p.lk;
  if (interior) {
  constexpr int WPU = VEC / 8;                 // IT words per unit
  constexpr int kUnroll = VEC == 16 ? 1 : 2;   // units in flight per thread (128 B)
  const int upr = g.itcols / WPU;              // units per band
  const uint64_t rcp_upr = reciprocal(static_cast<uint32_t>(upr));
  const int nunits = g.bands * upr;
  for (int u0 = tid; u0 < nunits; u0 += kThreads * kUnroll) {
    uint4 v[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int w = u0 + u * kThreads;
      if (w < nunits) {
        const int pb = qdiv(w, rcp_upr), qu = w - pb * upr;
        const uint8_t* src = base + static_cast<long long>(8 * pb) * p.lk + VEC * qu;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if constexpr (VEC == 16) {
            v[u][r] = __ldcs(reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * p.lk));
          } else {
            const uint2 x = __ldcs(reinterpret_cast<const uint2*>(src + static_cast<long long>(r) * p.lk));
            v[u][r] = make_uint4(x.x, x.y, 0u, 0u);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int w = u0 + u * kThreads;
      if (w < nunits) {
        const int pb = qdiv(w, rcp_upr), qu = w - pb * upr;
#pragma unroll
        for (int h = 0; h < WPU; ++h) {
          uint64_t word = 0;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const uint32_t lo = h == 0 ? v[u][r].x : v[u][r].z;
            const uint32_t hi = h == 0 ? v[u][r].y : v[u][r].w;
            word |= static_cast<uint64_t>(pack_word4(lo) | (pack_word4(hi) << 4)) << (8 * r);
          }
          s_words[pb * g.itcols + qu * WPU + h] = word;
          local_nnz += __popcll(word);
        }
      }
    }
  }
  } else {
    const int nunits = g.bands * g.itcols;
    for (int w = tid; w < nunits; w += kThreads) {
      const int pb = w / g.itcols, qc = w - pb * g.itcols;
      const uint8_t* src = base + static_cast<long long>(8 * pb) * p.lk + 8 * qc;
      const int rows_in = min(8, p.lq - (g.I * p.bm + 8 * pb));
      const int cols_in = min(8, p.lk - (g.J0 * p.bn + 8 * qc));
      uint64_t word = 0;
      for (int r = 0; r < rows_in; ++r) {
        const uint4 x = load_partial<8>(src + static_cast<long long>(r) * p.lk, cols_in);
        word |= static_cast<uint64_t>(pack_word4(x.x) | (pack_word4(x.y) << 4)) << (8 * r);
      }
      s_words[pb * g.itcols + qc] = word;
      local_nnz += __popcll(word);
    }
  }
  finish_chunk(p, chunk, g, cs, s_words, local_nnz, tid);
}

// Phase 1 for a parametric mask (one rule per mask): every IT word is
// computed from the rule, nothing is read but the rule's small bitsets.
// Element (i, j) is valid iff band_lo <= i - j <= band_hi, or row i is a
// global row, or column j a global column, or block (i / block, j / block)
// is set.  An IT (8x8, rows and columns multiples of 8) lies in one block
// and reads one byte of each bitset.
__device__ __forceinline__ unsigned long long rule_phase(const EncodeParams& p, const ChunkGeom& g,
                                                         const RuleDev& ru, uint64_t* words, int tid) {
  unsigned long long nnz = 0;
  const long long i_base = static_cast<long long>(g.I) * p.bm;
  const long long j_base = static_cast<long long>(g.J0) * p.bn;
  const int nw = g.bands * g.itcols;
  for (int w = tid; w < nw; w += kThreads) {
    const int pb = w / g.itcols, qc = w - pb * g.itcols;
    const long long i0 = i_base + 8 * pb, j0 = j_base + 8 * qc;
    if (i0 >= p.lq || j0 >= p.lk) {  // an IT wholly in the padding of a side: invalid, nothing read
      words[pb * g.itcols + qc] = 0;
      continue;
    }
    uint32_t all_rows = 0;  // bits valid in every row of the IT
    if (ru.global_cols) all_rows |= (__ldg(ru.global_cols + (j0 >> 5)) >> (j0 & 31)) & 0xFFu;
    if (ru.blocks) {
      const long long bi = (i0 / ru.block) * ru.nbc + j0 / ru.block;
      if ((__ldg(ru.blocks + (bi >> 5)) >> (bi & 31)) & 1u) all_rows = 0xFFu;
    }
    const uint32_t grow = ru.global_rows ? (__ldg(ru.global_rows + (i0 >> 5)) >> (i0 & 31)) & 0xFFu : 0u;
    // columns j0 .. j0 + 7 inside the matrix (an edge IT of a padded side has fewer)
    const long long ncols = min(max(static_cast<long long>(p.lk) - j0, 0ll), 8ll);
    const uint32_t in_cols = ncols == 8 ? 0xFFu : (1u << ncols) - 1u;
    uint64_t word = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (i0 + r >= p.lq) break;  // rows beyond the matrix: invalid
      // band: i - band_hi <= j <= i - band_lo, as IT columns c = j - j0
      const long long clo = max(i0 + r - ru.band_hi - j0, 0ll);
      const long long chi = min(i0 + r - ru.band_lo - j0, 7ll);
      uint32_t b = clo <= chi ? ((0xFFu >> (7 - chi)) & (0xFFu << clo)) : 0u;
      b |= all_rows | ((grow >> r) & 1u ? 0xFFu : 0u);
      word |= static_cast<uint64_t>(b & in_cols) << (8 * r);
    }
    words[pb * g.itcols + qc] = word;
    nnz += __popcll(word);
  }
  return nnz;
}

__global__ void __launch_bounds__(kThreads, 7) encode_rules_kernel(const EncodeParams p,
                                                                   const __grid_constant__ RuleSet rs) {
  extern __shared__ uint64_t s_words[];  // [bm/8][nt * bn/8]
  __shared__ long long s_chunk;
  __shared__ ChunkState cs;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_chunk = static_cast<long long>(atomicAdd(p.ticket, 1ull));
    cs.nnz = 0;
  }
  __syncthreads();
  const long long chunk = s_chunk;
  if (chunk >= p.n_chunks) return;
  const ChunkGeom g = chunk_geom(p, chunk);
  const unsigned long long local_nnz = rule_phase(p, g, rs.r[g.m], s_words, tid);
  finish_chunk(p, chunk, g, cs, s_words, local_nnz, tid);
}

// ---------------------------------------------------------------- bit-packed masks
// A bit-packed mask is an eighth of the dense one, so reading it twice costs
// less than the single-pass encoder's wait for its predecessors: three short
// kernels, none waiting on another CTA.
//   1. classify: the class of every OT (and the valid-element count), per-row
//      counts of full and partial OTs;
//   2. scan: row pointers by an exclusive prefix sum of those counts;
//   3. fill: column lists and, reading the partial OTs' bytes again, their
//      IT words, straight into their final slots.
// Passes 1 and 3 give a CTA 32 consecutive OTs of one OT row band (one per
// lane, so a warp's load covers 32 * bn / 8 contiguous bytes of a row); the 8
// warps of pass 1 split the band's rows.  VEC = bytes per load.

constexpr int kGroup = 32;  // OTs per CTA in passes 1 and 3

template <int VEC>
__global__ void __launch_bounds__(kThreads) bits_classify_kernel(const EncodeParams p) {
  __shared__ uint32_t s_any[kThreads / 32][kGroup], s_all[kThreads / 32][kGroup];
  __shared__ unsigned long long s_nnz[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (p.n_tc + kGroup - 1) / kGroup;
  const long long row = blockIdx.x / ngroups;  // OT row band, mask-major
  const int J = static_cast<int>(blockIdx.x % ngroups) * kGroup + lane;
  const int m = static_cast<int>(row / p.n_tr), I = static_cast<int>(row % p.n_tr);
  const long long row_bytes = p.lk >> 3;
  const int tb = p.bn >> 3;  // bytes of one OT row
  uint32_t any = 0, all = ~0u;
  unsigned long long nnz = 0;
  // an OT reaching past a padded side: only its rows < lq and bytes < lk / 8
  // are read, and it is never full
  const bool edge_c = (J + 1) * tb > row_bytes;
  const int rows = min(p.bm, p.lq - I * p.bm);
  if (J < p.n_tc && edge_c) {
    const uint8_t* base =
        p.mask + (static_cast<long long>(m) * p.lq + static_cast<long long>(I) * p.bm) * row_bytes + static_cast<long long>(J) * tb;
    const int bytes = static_cast<int>(row_bytes - static_cast<long long>(J) * tb);
    for (int r = warp; r < rows; r += kThreads / 32)
      for (int x = 0; x < bytes; ++x) {
        const uint32_t t = __ldcs(base + r * row_bytes + x);
        any |= t;
        nnz += __popc(t);
      }
  } else if (J < p.n_tc) {
    const uint8_t* base =
        p.mask + (static_cast<long long>(m) * p.lq + static_cast<long long>(I) * p.bm) * row_bytes + static_cast<long long>(J) * tb;
#pragma unroll 4
    for (int r = warp; r < rows; r += kThreads / 32) {
      const uint8_t* src = base + r * row_bytes;
      for (int x = 0; x < tb; x += VEC) {
        if constexpr (VEC == 16) {
          const uint4 t = __ldcs(reinterpret_cast<const uint4*>(src + x));
          any |= t.x | t.y | t.z | t.w;
          all &= t.x & t.y & t.z & t.w;
          nnz += __popc(t.x) + __popc(t.y) + __popc(t.z) + __popc(t.w);
        } else if constexpr (VEC == 8) {
          const uint2 t = __ldcs(reinterpret_cast<const uint2*>(src + x));
          any |= t.x | t.y;
          all &= t.x & t.y;
          nnz += __popc(t.x) + __popc(t.y);
        } else {
          const uint32_t t = __ldcs(src + x);
          any |= t;
          all &= t | 0xFFFFFF00u;
          nnz += __popc(t);
        }
      }
    }
  }
  if (edge_c || rows < p.bm) all = 0;
  s_any[warp][lane] = any;
  s_all[warp][lane] = all;
#pragma unroll
  for (int off = 16; off; off >>= 1) nnz += __shfl_xor_sync(0xffffffffu, nnz, off);
  if (lane == 0) s_nnz[warp] = nnz;
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) {
      any |= s_any[w][lane];
      all &= s_all[w][lane];
    }
    const int cls = J >= p.n_tc ? 0 : (any == 0 ? 0 : (all == ~0u ? 1 : 2));
    if (J < p.n_tc) p.cls[row * p.n_tc + J] = static_cast<uint8_t>(cls);
    const int nf = __popc(__ballot_sync(0xffffffffu, cls == 1));
    const int np = __popc(__ballot_sync(0xffffffffu, cls == 2));
    if (lane == 0) {
      if (nf) atomicAdd(&p.rowcnt[row], nf);
      if (np) atomicAdd(&p.rowcnt[p.n_rows + row], np);
      unsigned long long t = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) t += s_nnz[w];
      if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&p.counts[2]), t);
    }
  }
}

// Pass 2, one CTA: row pointers and totals from the per-row counts.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) bits_scan_kernel(const EncodeParams p) {
  __shared__ int s_f[kScanThreads / 32], s_p[kScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry_f = 0, carry_p = 0;
  for (long long base = 0; base < p.n_rows; base += kScanThreads) {
    const long long r = base + tid;
    const int f = r < p.n_rows ? p.rowcnt[r] : 0;
    const int q = r < p.n_rows ? p.rowcnt[p.n_rows + r] : 0;
    int xf = f, xq = q;  // inclusive scans inside the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int yf = __shfl_up_sync(0xffffffffu, xf, off), yq = __shfl_up_sync(0xffffffffu, xq, off);
      if (lane >= off) {
        xf += yf;
        xq += yq;
      }
    }
    if (lane == 31) {
      s_f[warp] = xf;
      s_p[warp] = xq;
    }
    __syncthreads();
    if (warp == 0) {  // scan of the warp totals
      int wf = s_f[lane], wq = s_p[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int yf = __shfl_up_sync(0xffffffffu, wf, off), yq = __shfl_up_sync(0xffffffffu, wq, off);
        if (lane >= off) {
          wf += yf;
          wq += yq;
        }
      }
      s_f[lane] = wf;
      s_p[lane] = wq;
    }
    __syncthreads();
    const int before_f = carry_f + (warp ? s_f[warp - 1] : 0) + xf - f;
    const int before_p = carry_p + (warp ? s_p[warp - 1] : 0) + xq - q;
    if (r < p.n_rows) {
      p.full_row_ptr[r] = before_f;
      p.part_row_ptr[r] = before_p;
    }
    carry_f += s_f[kScanThreads / 32 - 1];
    carry_p += s_p[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) {
    p.full_row_ptr[p.n_rows] = carry_f;
    p.part_row_ptr[p.n_rows] = carry_p;
    p.counts[0] = carry_f;
    p.counts[1] = carry_p;
  }
}

template <int VEC>
__global__ void __launch_bounds__(kThreads) bits_fill_kernel(const EncodeParams p) {
  __shared__ int s_before[2][kThreads / 32];
  __shared__ long long s_slot[kGroup];
  __shared__ int s_plist[kGroup];
  __shared__ int s_np;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ngroups = (p.n_tc + kGroup - 1) / kGroup;
  const long long row = blockIdx.x / ngroups;
  const int J0 = static_cast<int>(blockIdx.x % ngroups) * kGroup;
  const uint8_t* crow = p.cls + row * p.n_tc;
  // full and partial OTs of this row before the group
  int bf = 0, bp = 0;
  for (int j = tid; j < J0; j += kThreads) {
    const int c = crow[j];
    bf += c == 1;
    bp += c == 2;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    bf += __shfl_xor_sync(0xffffffffu, bf, off);
    bp += __shfl_xor_sync(0xffffffffu, bp, off);
  }
  if (lane == 0) {
    s_before[0][warp] = bf;
    s_before[1][warp] = bp;
  }
  __syncthreads();
  if (warp == 0) {
    int f0 = 0, p0 = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      f0 += s_before[0][w];
      p0 += s_before[1][w];
    }
    const int J = J0 + lane;
    const int c = J < p.n_tc ? crow[J] : 0;
    const unsigned mf = __ballot_sync(0xffffffffu, c == 1), mp = __ballot_sync(0xffffffffu, c == 2);
    const unsigned lt = (1u << lane) - 1u;
    if (c == 1) p.full_col_idx[p.full_row_ptr[row] + f0 + __popc(mf & lt)] = J;
    if (c == 2) {
      const int rk = __popc(mp & lt);
      const long long e = static_cast<long long>(p.part_row_ptr[row]) + p0 + rk;
      p.part_col_idx[e] = J;
      s_slot[rk] = e;
      s_plist[rk] = J;
    }
    if (lane == 0) s_np = __popc(mp);
  }
  __syncthreads();
  // IT words of the partial OTs, read again from the mask
  const int np = s_np;
  const long long row_bytes = p.lk >> 3;
  const int tb = p.bn >> 3, bands = p.bm >> 3, upr = tb / VEC, wpt = bands * tb;
  const int m = static_cast<int>(row / p.n_tr), I = static_cast<int>(row % p.n_tr);
  const uint8_t* band0 = p.mask + (static_cast<long long>(m) * p.lq + static_cast<long long>(I) * p.bm) * row_bytes;
  const int units = np * bands * upr;
  for (int u = tid; u < units; u += kThreads) {
    const int k = u / (bands * upr), rest = u - k * (bands * upr);
    const int pb = rest / upr, qu = rest - pb * upr;
    const uint8_t* src = band0 + static_cast<long long>(8 * pb) * row_bytes + static_cast<long long>(s_plist[k]) * tb + VEC * qu;
    uint64_t* dst = p.bitmaps + s_slot[k] * wpt + pb * tb + qu * VEC;
    // rows and bytes of the unit inside the mask (fewer at the edge of a padded side)
    const int rows_in = min(8, p.lq - (I * p.bm + 8 * pb));
    const long long bytes_left = row_bytes - (static_cast<long long>(s_plist[k]) * tb + VEC * qu);
    const int bytes_in = bytes_left < VEC ? static_cast<int>(bytes_left) : VEC;
    if (rows_in == 8 && bytes_in == VEC) {
      pack_bits_unit<VEC>(src, row_bytes, dst);
    } else {
      for (int c = 0; c < VEC; ++c) {
        uint64_t word = 0;
        if (c < bytes_in)
          for (int r = 0; r < rows_in; ++r) word |= static_cast<uint64_t>(src[r * row_bytes + c]) << (8 * r);
        dst[c] = word;
      }
    }
  }
}

}  // namespace

// Mask columns per chunk of the single-pass (dense and rule) encoders.  The
// bit-packed encoder works on groups of OTs instead and ignores the chunking.
constexpr int kChunkCols = 1024;

bool encode_geometry(int n_masks, int lq, int lk, int bm, int bn, EncodeGeom* g) {
  if (n_masks < 1 || lq < 1 || lk < 1) return false;
  if (bm < 8 || bn < 8 || bm > 256 || bn > 256 || bm % 8 || bn % 8) return false;
  // a side that is not a whole number of OTs is padded to one (with invalid elements)
  g->n_tr = (lq + bm - 1) / bm;
  g->n_tc = (lk + bn - 1) / bn;
  g->n_rows = static_cast<int64_t>(n_masks) * g->n_tr;
  g->n_tiles = g->n_rows * g->n_tc;
  if (g->n_tiles >= (int64_t(1) << 31) - 1) return false;
  int ct = kChunkCols / bn;
  if (ct < 1) ct = 1;
  if (ct > kMaxTilesPerChunk) ct = kMaxTilesPerChunk;
  if (ct > g->n_tc) ct = g->n_tc;
  g->ct = ct;
  g->cpr = (g->n_tc + ct - 1) / ct;
  g->n_chunks = g->n_rows * g->cpr;
  g->words_per_tile = (bm / 8) * (bn / 8);
  g->smem_bytes = static_cast<size_t>(bm / 8) * (ct * bn / 8) * sizeof(uint64_t);
  return true;
}

WorkspaceLayout workspace_layout(const EncodeGeom& g) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  WorkspaceLayout w{};
  size_t off = 0;
  w.counts = off;                       // 4 x int64
  w.ticket = off + 32;                  // 1 x u64; off + 40: the persistent attention kernel's work counter
  w.status = off + 64;                  // n_chunks x u64
  w.status_bytes = static_cast<size_t>(g.n_chunks) * 8;
  w.rowcnt = w.status + w.status_bytes;  // 2 x n_rows x i32 (bit-packed encoder)
  w.zero_bytes = 64 + w.status_bytes + static_cast<size_t>(g.n_rows) * 8;
  off = up(w.counts + w.zero_bytes);
  w.cls = off;                          // n_tiles x u8 (bit-packed encoder)
  off = up(off + static_cast<size_t>(g.n_tiles));
  w.full_row_ptr = off;
  off = up(off + (static_cast<size_t>(g.n_rows) + 1) * 4);
  w.part_row_ptr = off;
  off = up(off + (static_cast<size_t>(g.n_rows) + 1) * 4);
  w.full_col_idx = off;
  off = up(off + static_cast<size_t>(g.n_tiles) * 4);
  w.part_col_idx = off;
  off = up(off + static_cast<size_t>(g.n_tiles) * 4);
  w.bitmaps = off;
  off = up(off + static_cast<size_t>(g.n_tiles) * g.words_per_tile * 8);
  w.total = off;
  return w;
}

// The reciprocals the kernels divide by (qdiv).
static EncodeParams with_reciprocals(const EncodeParams& p) {
  EncodeParams q = p;
  const int itc = p.bn >> 3;
  q.rcp_itc = reciprocal(static_cast<uint32_t>(itc));
  q.rcp_wpt = reciprocal(static_cast<uint32_t>((p.bm >> 3) * itc));
  return q;
}

cudaError_t launch_encode(const EncodeParams& p_in, const EncodeGeom& g, cudaStream_t s) {
  const EncodeParams p = with_reciprocals(p_in);
  // shared memory per CTA: (bm / 8) * (chunk columns / 8) words
  const unsigned grid = static_cast<unsigned>(g.n_chunks);
  const uintptr_t a = reinterpret_cast<uintptr_t>(p.mask);
  if (p.bits) {
    // a load of VEC bytes must stay inside one OT row and start aligned
    const int rb = p.lk / 8, tb = p.bn / 8;
    const int vec = (rb % 16 == 0 && tb % 16 == 0 && a % 16 == 0) ? 16 : (rb % 8 == 0 && tb % 8 == 0 && a % 8 == 0) ? 8 : 1;
    const long long groups = g.n_rows * ((g.n_tc + kGroup - 1) / kGroup);
    if (groups >= (1ll << 31)) return cudaErrorInvalidValue;
    const unsigned grid2 = static_cast<unsigned>(groups);
    if (vec == 16) bits_classify_kernel<16><<<grid2, kThreads, 0, s>>>(p);
    else if (vec == 8) bits_classify_kernel<8><<<grid2, kThreads, 0, s>>>(p);
    else bits_classify_kernel<1><<<grid2, kThreads, 0, s>>>(p);
    bits_scan_kernel<<<1, kScanThreads, 0, s>>>(p);
    if (vec == 16) bits_fill_kernel<16><<<grid2, kThreads, 0, s>>>(p);
    else if (vec == 8) bits_fill_kernel<8><<<grid2, kThreads, 0, s>>>(p);
    else bits_fill_kernel<1><<<grid2, kThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  const bool vec16 = (p.lk % 16 == 0) && (p.bn % 16 == 0) && (a % 16 == 0);
  const bool vec8 = (p.lk % 8 == 0) && (a % 8 == 0);
  if (vec16)
    encode_kernel<16, true><<<grid, kThreads, g.smem_bytes, s>>>(p);
  else if (vec8)
    encode_kernel<8, true><<<grid, kThreads, g.smem_bytes, s>>>(p);
  else
    encode_kernel<8, false><<<grid, kThreads, g.smem_bytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_encode_rules(const EncodeParams& p_in, const EncodeGeom& g, const RuleSet& rs, cudaStream_t s) {
  const EncodeParams p = with_reciprocals(p_in);
  if (g.smem_bytes > 48 * 1024 &&
      cudaFuncSetAttribute(encode_rules_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(g.smem_bytes)) != cudaSuccess)
    return cudaGetLastError();
  encode_rules_kernel<<<static_cast<unsigned>(g.n_chunks), kThreads, g.smem_bytes, s>>>(p, rs);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------
// Scratch for stof_encode_mask_noalloc(): the tile ticket (word 0) and one
// look-back status word per chunk, in a file-scope device array, so that
// callers who cannot allocate device memory can still encode.  Each GPU
// that loads the library holds these 1 MiB + 8 bytes until the process
// exits.  Host code must not use the array's name as a device address (on
// the host it names a shadow variable): the address is looked up below.
static __device__ __align__(256) unsigned long long g_noalloc_scratch[1 + kNoAllocMaxChunks];

cudaError_t noalloc_scratch_address(unsigned long long** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static unsigned long long* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {  // once per device, with that device current
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<unsigned long long*>(ptr);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace stof
