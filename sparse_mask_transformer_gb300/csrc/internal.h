// Internal declarations shared by the translation units of libstof.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "stof.h"

namespace stof {

// Remembers e (if it is an error) for stof_last_cuda_error(); returns e.
cudaError_t record_cuda(cudaError_t e);

// 2-D row-major tensor map (inner dimension contiguous, rows row_bytes
// apart) through the driver entry point; false on failure.
bool encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);
// [planes][rows][inner] tensor, boxes of box_inner x box_rows x 1 (zeros outside the tensor).
bool encode_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t planes, uint64_t row_bytes, uint64_t plane_bytes,
                          uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Runs prepare() (function attributes, checks) once per (current device, key)
// and remembers success; thread-safe.  Returns prepare()'s result, or true
// when it already succeeded on this device.
bool once_per_device(const void* key, bool (*prepare)(const void*), const void* arg);

// ---------------------------------------------------------------- encoder
// A chunk is one OT row band (bm mask rows) times `ct` consecutive OTs.
struct EncodeGeom {
  int n_tr, n_tc, ct, cpr;      // cpr = chunks per OT row
  int64_t n_rows, n_chunks, n_tiles;
  int words_per_tile;           // (bm/8) * (bn/8)
  size_t smem_bytes;            // one chunk's IT words (a CTA's dynamic shared memory per chunk buffer)
};
// False for sizes the encoder does not take.  A chunk is about 1024 mask
// columns of one OT row band (whole OTs).
bool encode_geometry(int n_masks, int lq, int lk, int bm, int bn, EncodeGeom* g);

// Workspace carve-up (byte offsets, 256-byte aligned sections).
struct WorkspaceLayout {
  size_t counts, ticket, status, status_bytes, rowcnt, zero_bytes;  // zero_bytes from `counts`
  size_t cls;
  size_t full_row_ptr, part_row_ptr, full_col_idx, part_col_idx, bitmaps, total;
};
WorkspaceLayout workspace_layout(const EncodeGeom& g);

struct EncodeParams {
  const uint8_t* mask;             // byte mask [n][lq][lk], or bit-packed [n][lq][lk / 8] if bits
  int bits;
  int lq, lk, bm, bn, n_tr, n_tc, ct, cpr;
  int64_t n_rows, n_chunks;
  int32_t* full_row_ptr;
  int32_t* full_col_idx;
  int32_t* part_row_ptr;
  int32_t* part_col_idx;
  uint64_t* bitmaps;
  int64_t* counts;                 // [0] n_full [1] n_part [2] nnz [3] error word
  unsigned long long* ticket;      // scratch, zero at launch
  unsigned long long* status;      // scratch [n_chunks], zero at launch
  uint8_t* cls;                    // bit-packed encoder: class of every OT [n_rows][n_tc]
  int32_t* rowcnt;                 // bit-packed encoder: full, then partial OT counts per row, zero at launch
  uint64_t rcp_itc, rcp_wpt;       // set by the launchers: ceil(2^32 / (bn / 8)), ceil(2^32 / IT words per OT)
};
cudaError_t launch_encode(const EncodeParams& p, const EncodeGeom& g, cudaStream_t s);

// Parametric masks (stof_encode_rules): one rule per mask, passed to the
// encoder by value in its kernel parameters.
constexpr int kMaxRules = 64;
struct RuleDev {
  long long band_lo, band_hi;      // valid if band_lo <= i - j <= band_hi
  const uint32_t* global_rows;     // bitset over query rows, or null
  const uint32_t* global_cols;     // bitset over key columns, or null
  const uint32_t* blocks;          // bitset over [lq / block][nbc] blocks, or null
  int block, nbc;                  // block edge (multiple of 8); blocks per block row
};
struct RuleSet {
  RuleDev r[kMaxRules];
};
cudaError_t launch_encode_rules(const EncodeParams& p, const EncodeGeom& g, const RuleSet& rs, cudaStream_t s);

// Scratch of stof_encode_mask_noalloc(): a static device array with room
// for the ticket and kNoAllocMaxChunks look-back words.  The address is
// looked up once per device (the current one) and cached.
constexpr long long kNoAllocMaxChunks = 131072;
cudaError_t noalloc_scratch_address(unsigned long long** out);

// ---------------------------------------------------------------- attention
struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  int B, H, L, d;                 // L: query rows per head
  int Lk;                          // keys per head (L for self-attention)
  float scale_log2;                // scale * log2(e)
  int bm, bn, n_tr, n_tc;
  int64_t stride_b, stride_h;
  const int32_t* full_row_ptr;
  const int32_t* full_col_idx;
  const int32_t* part_row_ptr;
  const int32_t* part_col_idx;
  const uint64_t* bitmaps;
  int64_t* err;                    // device error word (counts[3])
  unsigned int* work;              // work counter of the persistent kernel, in the format's workspace:
                                   // work[0] items taken, work[1] CTAs finished (both zero between launches)
  float tiles_per_row;             // mean listed OTs per OT row of the masks (synced format), else -1
  float keys_per_row;              // mean valid keys per query row (synced format), else -1
  float listed128_per_row;         // listed OT area per 128-row query tile, in 128x128 OTs (synced), else -1
  int stages;                      // block-wise K/V ring depth; 0 = the kernel's default
  int rows_per_warp;               // row-wise: query rows per warp (1, 2 or 4); 0 = automatic
  int variant;                     // block-wise: kVariantAuto, kVariantPerTile or kVariantPersistent
  int exp_split;                   // block-wise: 1 = one key pair in eight exponentiated on the FMA pipe
  int softmax_wg;                  // block-wise softmax warpgroups: 2, or 4 (persistent, d = 64); 0 = 2
};
// Block-wise kernel variants: one CTA per query tile, or persistent CTAs
// (d = 64 only); auto picks by the mean listed OTs per OT row.
constexpr int kVariantAuto = 0, kVariantPerTile = 1, kVariantPersistent = 2;
// Below this many listed OTs per OT row (mean over the masks) the d = 64
// block-wise call runs persistent CTAs.  Measured on GB300: 15% faster at 4
// to 9 OTs per query tile, 5.5% at 28, 3% slower at 64, where a CTA per
// query tile has little start-up left to hide.
constexpr float kPersistMaxTiles = 48.f;
inline bool blockwise_persistent(int d, int variant, float tiles_per_row) {
  return variant == kVariantPersistent ||
         (variant == kVariantAuto && d == 64 && tiles_per_row < kPersistMaxTiles);
}
// Ring depth a block-wise launch uses (stages = 0: the variant's default).
inline int blockwise_stages(bool persistent, int stages) { return stages ? stages : (persistent ? 4 : 3); }

// Row-wise kernel: query rows per warp.  A whole warp per row while the
// call has few rows (the GPU holds them all at once and the shortest
// dependent chain wins); for more rows with few valid keys, 2 or 4 rows per
// warp so that more rows are in flight.  A warp's loops run at the pace of
// its row with the most keys, so a mask whose keys come in blocks (few keys
// on average, many in the rows that have any) keeps one row per warp: the
// second test bounds the valid keys per (row, listed 128-column OT).
// Thresholds from kernel-only GB300 times of the three settings on 648
// short, sparse cases: within 3% of the best setting on average.
// `requested` (1, 2 or 4) overrides; negative statistics mean unknown.
constexpr long long kRowwiseFewRows = 2048;
inline int rowwise_rows_per_warp(long long rows, float keys_per_row, float listed128_per_row, int requested) {
  if (requested == 1 || requested == 2 || requested == 4) return requested;
  if (rows <= kRowwiseFewRows || keys_per_row < 0.f || listed128_per_row <= 0.f) return 1;
  const float keys_per_listed = keys_per_row / listed128_per_row;
  if (keys_per_row <= 24.f && keys_per_listed <= 32.f) return 4;
  if (keys_per_row <= 128.f && keys_per_listed <= 64.f) return 2;
  return 1;
}

// One way to run the MHA step: the kernel, the OT width it needs, the
// block-wise kernel's ring depth (0 = default) and variant, and the
// row-wise kernel's rows per warp (0 = automatic).
struct KernelChoice {
  stof_kernel kernel;
  int bn;
  int stages;
  int variant;
  int rows_per_warp;
  int exp_split;   // block-wise: 1 = one key pair in eight exponentiated on the FMA pipe
  int softmax_wg;  // block-wise softmax warpgroups: 0 (= 2), 2 or 4
};
// The candidates stof_tune() times (STOF_TUNE_CANDIDATES of them).
extern const KernelChoice kTuneCandidates[STOF_TUNE_CANDIDATES];
// The fastest cached candidate for (L, d, density bucket) among those on
// OTs of width bn; false if the cache has no such entry.
bool tuned_choice(int L, int d, double density, int bn, KernelChoice* out);
// stof_mha_fwd() with the kernel, ring depth and variant given.
stof_status mha_fwd_choice(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int L, int Lk,
                           int d, float scale, const stof_format* fmt, int64_t mask_stride_b, int64_t mask_stride_h,
                           const KernelChoice& c, void* o, void* stream);
cudaError_t launch_rowwise(const AttnParams& p, bool bf16, cudaStream_t s);
// Density bucket of the tuning cache.
int tune_density_bucket(double density);
// Returns STOF_OK or an error status (tensor-map encoding / launch).
stof_status launch_blockwise(const AttnParams& p, bool bf16, cudaStream_t s);
// The persistent block-wise kernel for d = 64 (blockwise_persist.cu).
stof_status launch_blockwise_persist64(const AttnParams& p, bool bf16, cudaStream_t s);
// TMA map of a [heads][L][D] 16-bit tensor, boxes of 64 columns x box_rows rows of
// one head (zeros past row L), 128-byte swizzle.
// Maps are kept in a small per-process cache keyed by (device, base, rows,
// D, box_rows, type), so repeated calls on the same tensors do no driver call.
bool make_bw_map(CUtensorMap* m, const void* base, uint64_t heads, uint64_t L, int D, int box_rows, bool bf16);

}  // namespace stof
