// C ABI of libstof.so: argument validation, workspace carve-up, kernel
// selection and dispatch.  The arithmetic of the method runs in the
// kernels (encode.cu, rowwise.cu, blockwise.cu); this file only checks
// arguments and launches.
//
// Method: "Accelerating Sparse Transformer Inference on GPU" (gist.science
// technical summary), Methodology 1, Unified MHA module (two-level storage
// format; row-wise and block-wise kernels; analytic kernel selection).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include <mutex>
#include <set>
#include <utility>

#include "internal.h"

using namespace stof;

namespace {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace stof {
cudaError_t record_cuda(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error = e;
  return e;
}

// Runs prepare(arg) once per (current device, key); a failed preparation is
// retried on the next call.  Guards the per-kernel function attributes, which
// are per-device state in the CUDA runtime.
bool once_per_device(const void* key, bool (*prepare)(const void*), const void* arg) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return prepare(arg);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, key})) return true;
  if (!prepare(arg)) return false;
  done.insert({dev, key});
  return true;
}

}  // namespace stof

extern "C" {

const char* stof_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

int stof_version(void) { return STOF_VERSION; }

const char* stof_status_string(stof_status s) {
  switch (s) {
    case STOF_OK: return "ok";
    case STOF_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad enum)";
    case STOF_ERR_SHAPE: return "bad shape (inconsistent sizes, not tile-divisible where required, or too large)";
    case STOF_ERR_DTYPE: return "unknown element type";
    case STOF_ERR_ALIGNMENT: return "pointer not aligned as required";
    case STOF_ERR_WORKSPACE: return "workspace too small";
    case STOF_ERR_UNSUPPORTED: return "unsupported configuration (head dim or tile size)";
    case STOF_ERR_DEVICE: return "device-side error reported by a kernel";
    case STOF_ERR_CUDA: return "CUDA runtime error";
    case STOF_ERR_NOT_SYNCED: return "format counts not synced to the host";
  }
  return "unknown status";
}

size_t stof_encode_workspace_bytes(int n_masks, int lq, int lk, int bm, int bn) {
  EncodeGeom g;
  if (!encode_geometry(n_masks, lq, lk, bm, bn, &g)) return 0;
  return workspace_layout(g).total;
}

// Encodes from a dense (bits = 0) or bit-packed (bits = 1) mask, or, with
// mask = NULL, from the rules in *rules.
static stof_status encode_impl(const uint8_t* mask, int bits, const RuleSet* rules, int n_masks, int lq, int lk,
                               int bm, int bn, void* workspace, size_t ws_bytes, stof_format* fmt, void* stream) {
  if ((!mask && !rules) || !workspace || !fmt) return STOF_ERR_INVALID_ARG;
  if (n_masks < 1 || lq < 1 || lk < 1 || bm < 1 || bn < 1) return STOF_ERR_INVALID_ARG;
  EncodeGeom g;
  if (!encode_geometry(n_masks, lq, lk, bm, bn, &g)) return STOF_ERR_SHAPE;
  if (bits && lk % 8) return STOF_ERR_SHAPE;  // a bit-packed row is lk / 8 whole bytes
  if ((mask && !aligned(mask, 8)) || !aligned(workspace, 256)) return STOF_ERR_ALIGNMENT;
  const WorkspaceLayout w = workspace_layout(g);
  if (ws_bytes < w.total) return STOF_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  stof_format f;
  std::memset(&f, 0, sizeof(f));
  f.n_masks = n_masks;
  f.lq = lq;
  f.lk = lk;
  f.bm = bm;
  f.bn = bn;
  f.n_tr = g.n_tr;
  f.n_tc = g.n_tc;
  f.synced = 0;
  f.counts_dev = reinterpret_cast<int64_t*>(ws + w.counts);
  f.scratch = ws + w.ticket;
  f.full_row_ptr = reinterpret_cast<int32_t*>(ws + w.full_row_ptr);
  f.part_row_ptr = reinterpret_cast<int32_t*>(ws + w.part_row_ptr);
  f.full_col_idx = reinterpret_cast<int32_t*>(ws + w.full_col_idx);
  f.part_col_idx = reinterpret_cast<int32_t*>(ws + w.part_col_idx);
  f.bitmaps = reinterpret_cast<uint64_t*>(ws + w.bitmaps);
  *fmt = f;

  cudaStream_t s = as_stream(stream);
  // counts, ticket and look-back state start at zero
  if (record_cuda(cudaMemsetAsync(ws + w.counts, 0, w.zero_bytes, s)) != cudaSuccess) return STOF_ERR_CUDA;
  EncodeParams p;
  p.mask = mask;
  p.bits = bits;
  p.lq = lq;
  p.lk = lk;
  p.bm = bm;
  p.bn = bn;
  p.n_tr = g.n_tr;
  p.n_tc = g.n_tc;
  p.ct = g.ct;
  p.cpr = g.cpr;
  p.n_rows = g.n_rows;
  p.n_chunks = g.n_chunks;
  p.full_row_ptr = f.full_row_ptr;
  p.full_col_idx = f.full_col_idx;
  p.part_row_ptr = f.part_row_ptr;
  p.part_col_idx = f.part_col_idx;
  p.bitmaps = f.bitmaps;
  p.counts = f.counts_dev;
  p.ticket = reinterpret_cast<unsigned long long*>(ws + w.ticket);
  p.status = reinterpret_cast<unsigned long long*>(ws + w.status);
  p.cls = ws + w.cls;
  p.rowcnt = reinterpret_cast<int32_t*>(ws + w.rowcnt);
  const cudaError_t e = rules ? launch_encode_rules(p, g, *rules, s) : launch_encode(p, g, s);
  if (record_cuda(e) != cudaSuccess) return STOF_ERR_CUDA;
  return STOF_OK;
}

stof_status stof_encode_mask(const uint8_t* mask, int n_masks, int lq, int lk, int bm, int bn,
                             void* workspace, size_t ws_bytes, stof_format* fmt, void* stream) {
  if (!mask) return STOF_ERR_INVALID_ARG;
  return encode_impl(mask, 0, nullptr, n_masks, lq, lk, bm, bn, workspace, ws_bytes, fmt, stream);
}

stof_status stof_encode_mask_bits(const uint8_t* mask_bits, int n_masks, int lq, int lk, int bm, int bn,
                                  void* workspace, size_t ws_bytes, stof_format* fmt, void* stream) {
  if (!mask_bits) return STOF_ERR_INVALID_ARG;
  return encode_impl(mask_bits, 1, nullptr, n_masks, lq, lk, bm, bn, workspace, ws_bytes, fmt, stream);
}

stof_status stof_encode_rules(const stof_mask_rule* rules, int n_masks, int lq, int lk, int bm, int bn,
                              void* workspace, size_t ws_bytes, stof_format* fmt, void* stream) {
  static_assert(STOF_MAX_RULES == kMaxRules, "rule capacity");
  if (!rules || !workspace || !fmt) return STOF_ERR_INVALID_ARG;
  if (n_masks < 1 || lq < 1 || lk < 1 || bm < 1 || bn < 1) return STOF_ERR_INVALID_ARG;
  if (n_masks > kMaxRules) return STOF_ERR_UNSUPPORTED;
  RuleSet rs;
  std::memset(&rs, 0, sizeof(rs));
  for (int m = 0; m < n_masks; ++m) {
    const stof_mask_rule& u = rules[m];
    if (!aligned(u.global_rows, 4) || !aligned(u.global_cols, 4) || !aligned(u.blocks, 4))
      return STOF_ERR_ALIGNMENT;
    if (u.blocks && (u.block < 8 || u.block % 8 != 0 || lq % u.block != 0 || lk % u.block != 0))
      return STOF_ERR_SHAPE;
    RuleDev& r = rs.r[m];
    r.band_lo = u.band_lo;
    r.band_hi = u.band_hi;
    r.global_rows = u.global_rows;
    r.global_cols = u.global_cols;
    r.blocks = u.blocks;
    r.block = u.blocks ? u.block : 8;
    r.nbc = u.blocks ? lk / u.block : 0;
  }
  return encode_impl(nullptr, 0, &rs, n_masks, lq, lk, bm, bn, workspace, ws_bytes, fmt, stream);
}

// Variant of stof_encode_mask() that allocates nothing and needs no device
// scratch from the caller: the tile ticket and look-back words live in a
// static device array of this library (see encode.cu).  Same arguments;
// the workspace receives the format, its scratch section is left unused.
stof_status stof_encode_mask_noalloc(const uint8_t* mask, int n_masks, int lq, int lk, int bm, int bn,
                                     void* workspace, size_t ws_bytes, stof_format* fmt, void* stream) {
  if (!mask || !workspace || !fmt) return STOF_ERR_INVALID_ARG;
  if (n_masks < 1 || lq < 1 || lk < 1 || bm < 1 || bn < 1) return STOF_ERR_INVALID_ARG;
  EncodeGeom g;
  if (!encode_geometry(n_masks, lq, lk, bm, bn, &g)) return STOF_ERR_SHAPE;
  if (g.n_chunks > kNoAllocMaxChunks) return STOF_ERR_SHAPE;  // beyond the static scratch
  if (!aligned(mask, 8) || !aligned(workspace, 256)) return STOF_ERR_ALIGNMENT;
  const WorkspaceLayout w = workspace_layout(g);
  if (ws_bytes < w.total) return STOF_ERR_WORKSPACE;
  unsigned long long* scratch = nullptr;
  if (record_cuda(noalloc_scratch_address(&scratch)) != cudaSuccess) return STOF_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  stof_format f;
  std::memset(&f, 0, sizeof(f));
  f.n_masks = n_masks;
  f.lq = lq;
  f.lk = lk;
  f.bm = bm;
  f.bn = bn;
  f.n_tr = g.n_tr;
  f.n_tc = g.n_tc;
  f.synced = 0;
  f.counts_dev = reinterpret_cast<int64_t*>(ws + w.counts);
  f.scratch = scratch;
  f.full_row_ptr = reinterpret_cast<int32_t*>(ws + w.full_row_ptr);
  f.part_row_ptr = reinterpret_cast<int32_t*>(ws + w.part_row_ptr);
  f.full_col_idx = reinterpret_cast<int32_t*>(ws + w.full_col_idx);
  f.part_col_idx = reinterpret_cast<int32_t*>(ws + w.part_col_idx);
  f.bitmaps = reinterpret_cast<uint64_t*>(ws + w.bitmaps);
  *fmt = f;

  cudaStream_t s = as_stream(stream);
  // the static scratch keeps the previous call's words: the workspace's
  // 64-byte header (counts and the attention kernel's counters), the ticket
  // and this call's look-back words start at zero
  if (record_cuda(cudaMemsetAsync(ws + w.counts, 0, 64, s)) != cudaSuccess) return STOF_ERR_CUDA;
  if (record_cuda(cudaMemsetAsync(scratch, 0, (static_cast<size_t>(g.n_chunks) + 1) * 8, s)) != cudaSuccess)
    return STOF_ERR_CUDA;
  EncodeParams p;
  p.mask = mask;
  p.bits = 0;
  p.lq = lq;
  p.lk = lk;
  p.bm = bm;
  p.bn = bn;
  p.n_tr = g.n_tr;
  p.n_tc = g.n_tc;
  p.ct = g.ct;
  p.cpr = g.cpr;
  p.n_rows = g.n_rows;
  p.n_chunks = g.n_chunks;
  p.full_row_ptr = f.full_row_ptr;
  p.full_col_idx = f.full_col_idx;
  p.part_row_ptr = f.part_row_ptr;
  p.part_col_idx = f.part_col_idx;
  p.bitmaps = f.bitmaps;
  p.counts = f.counts_dev;
  p.ticket = scratch;
  p.status = scratch + 1;
  p.cls = nullptr;     // used by the bit-packed encoder only
  p.rowcnt = nullptr;
  if (record_cuda(launch_encode(p, g, s)) != cudaSuccess) return STOF_ERR_CUDA;
  return STOF_OK;
}

stof_status stof_format_sync(stof_format* fmt, void* stream) {
  if (!fmt || !fmt->counts_dev) return STOF_ERR_INVALID_ARG;
  int64_t c[4] = {0, 0, 0, 0};
  cudaStream_t s = as_stream(stream);
  if (record_cuda(cudaMemcpyAsync(c, fmt->counts_dev, sizeof(c), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return STOF_ERR_CUDA;
  if (record_cuda(cudaStreamSynchronize(s)) != cudaSuccess) return STOF_ERR_CUDA;
  fmt->n_full = c[0];
  fmt->n_part = c[1];
  fmt->nnz = c[2];
  fmt->device_error = c[3];
  fmt->synced = 1;
  return c[3] ? STOF_ERR_DEVICE : STOF_OK;
}

// Analytic kernel choice ("Accelerating Sparse Transformer Inference on
// GPU", gist.science technical summary, Methodology 1: an analytical model
// chooses the row-wise or block-wise kernel from mask sparsity and
// sequence length).
//
// Predicted device time of each kernel in microseconds, linear in the work
// it does:
//   row-wise    T_row = 4.08 + 4.52e-4 R / r + 1.770e-5 K d/64 + 6.13e-5 P
//               R = query rows (heads x L) and r the kernel's rows per warp
//               (a warp's fixed cost is a few dependent memory round
//               trips), K = valid (query, key) pairs (density x L^2 x
//               heads: the K and V rows of every valid key), P = (query
//               row, listed OT) pairs (heads x L x listed OTs per query
//               tile: the bitmap bytes and column indices fetched per row);
//   block-wise  T_blk = 7.48 + 5.24e-3 T (d/64 + 1)/2 + 8.16e-3 Q
//               T = listed 128x128 OTs over all heads (each the full tile's
//               MMA and softmax work, the MMAs half as long at d = 64),
//               Q = query tiles (heads x L / 128: start-up and finish).
// The constant terms are launch and pipeline fill.  The coefficients were
// fitted to kernel-only GB300 times of both kernels (CUDA-graph replay) on
// 648 cases: L = 128 to 3072, densities 0.01 to 0.4, 1 to 64 heads, d = 64
// and 128, random, sliding-window and block-sparse masks (fitted to the 360
// cases of L = 128 to 2048 alone, it picked the faster kernel in 268 of the
// other 288).  Timed again with these coefficients, it picks the faster
// kernel in 612 of the 648 cases and costs 1.0% on average; where it
// misses, both kernels take under 30 us.  The row-wise kernel wins for high
// sparsity and few, short rows -- the regime the pages give it.
namespace {
double model_rowwise_us(double density, double L, double d, double heads, double tiles_per_row) {
  const double R = heads * L, K = density * L * L * heads, P = R * tiles_per_row;
  const double r = rowwise_rows_per_warp(static_cast<long long>(R), static_cast<float>(density * L),
                                         static_cast<float>(tiles_per_row), 0);
  return 4.08 + 4.52e-4 * R / r + 1.770e-5 * K * (d / 64.0) + 6.13e-5 * P;
}
double model_blockwise_us(double L, double d, double heads, double tiles_per_row) {
  const double n_tr = L / 128.0;
  const double T = tiles_per_row * n_tr * heads, Q = n_tr * heads;
  return 7.48 + 5.24e-3 * T * (d / 64.0 + 1.0) / 2.0 + 8.16e-3 * Q;
}
}  // namespace

stof_kernel stof_select_kernel_heads(double density, int seq_len, int head_dim, int64_t heads, double tiles_per_row) {
  if (!(density >= 0.0 && density <= 1.0) || seq_len <= 0 || head_dim <= 0 || heads <= 0)
    return STOF_KERNEL_BLOCKWISE;
  const double L = seq_len, n_tc = L / 128.0;
  // unknown or out of range: every OT of the row listed (an arbitrary mask),
  // so that the choice depends monotonically on the density
  double tpr = tiles_per_row;
  if (!(tpr >= 0.0 && tpr <= n_tc)) tpr = n_tc;
  const double t_row = model_rowwise_us(density, L, head_dim, static_cast<double>(heads), tpr);
  const double t_blk = model_blockwise_us(L, head_dim, static_cast<double>(heads), tpr);
  return t_row <= t_blk ? STOF_KERNEL_ROWWISE : STOF_KERNEL_BLOCKWISE;
}

stof_kernel stof_select_kernel(double density, int seq_len, int head_dim) {
  return stof_select_kernel_heads(density, seq_len, head_dim, 1, -1.0);
}

// OT sizes the block-wise kernel runs: 128 query rows (the MMA's M) by 64 or
// 128 key columns.
static bool blockwise_tiles(const stof_format& f) { return f.bm == 128 && (f.bn == 64 || f.bn == 128); }

static float keys_per_row(const stof_format& f) {
  return f.synced ? static_cast<float>(static_cast<double>(f.nnz) / (static_cast<double>(f.n_masks) * f.lq)) : -1.f;
}

// Listed OT area per 128-row query tile, in 128x128 OTs (synced format), else -1.
static float listed128_per_row(const stof_format& f) {
  return f.synced ? static_cast<float>(static_cast<double>(f.n_full + f.n_part) * f.bm * f.bn /
                                       (static_cast<double>(f.n_masks) * 128.0 * f.lq))
                  : -1.f;
}

static float tiles_per_row(const stof_format& f) {
  return f.synced ? static_cast<float>(static_cast<double>(f.n_full + f.n_part) /
                                       (static_cast<double>(f.n_masks) * f.n_tr))
                  : -1.f;
}

// The format and sizes agree (what a plan needs to know of a call).
// L query rows, Lk keys per head (Lk = L for self-attention).
static stof_status check_format(const stof_format* fmt, int B, int H, int L, int Lk, int d) {
  if (!fmt) return STOF_ERR_INVALID_ARG;
  if (!fmt->full_row_ptr || !fmt->full_col_idx || !fmt->part_row_ptr || !fmt->part_col_idx ||
      !fmt->bitmaps || !fmt->counts_dev)
    return STOF_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || L < 1 || Lk < 1 || d < 1) return STOF_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128 && d != 256) return STOF_ERR_UNSUPPORTED;
  if (fmt->lq != L || fmt->lk != Lk) return STOF_ERR_SHAPE;
  // the lengths need not be whole numbers of OTs: the last OT row and column are padded
  if (fmt->bm < 8 || fmt->bn < 8 || fmt->bm % 8 || fmt->bn % 8 || fmt->bm > 256 || fmt->bn > 256 ||
      fmt->n_tr != (L + fmt->bm - 1) / fmt->bm || fmt->n_tc != (Lk + fmt->bn - 1) / fmt->bn)
    return STOF_ERR_SHAPE;
  return STOF_OK;
}

// Every argument of an MHA call.
static stof_status check_call(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int L,
                              int Lk, int d, float scale, const stof_format* fmt, int64_t mask_stride_b,
                              int64_t mask_stride_h, void* o) {
  if (!q || !k || !v || !o || !fmt) return STOF_ERR_INVALID_ARG;
  if (dt != STOF_F16 && dt != STOF_BF16) return STOF_ERR_DTYPE;
  if (!std::isfinite(scale)) return STOF_ERR_INVALID_ARG;
  if (mask_stride_b < 0 || mask_stride_h < 0) return STOF_ERR_INVALID_ARG;
  const stof_status st = check_format(fmt, B, H, L, Lk, d);
  if (st != STOF_OK) return st;
  const long double max_mask = static_cast<long double>(B - 1) * mask_stride_b +
                               static_cast<long double>(H - 1) * mask_stride_h;
  if (max_mask >= fmt->n_masks) return STOF_ERR_SHAPE;
  if (static_cast<long double>(B) * H * (L > Lk ? L : Lk) >= 2147483647.0L * 8) return STOF_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return STOF_ERR_ALIGNMENT;
  return STOF_OK;
}

// What runs for `which` on this format: a forced kernel, a cached tuning
// result or the analytic model.
static stof_status plan_call(const stof_format& f, int B, int H, int L, int Lk, int d, stof_kernel which,
                             KernelChoice* c, int* source) {
  if (which != STOF_KERNEL_AUTO && which != STOF_KERNEL_ROWWISE && which != STOF_KERNEL_BLOCKWISE)
    return STOF_ERR_INVALID_ARG;
  *c = KernelChoice{which, f.bn, 0, kVariantAuto, 0, 0, 0};
  *source = STOF_PLAN_FORCED;
  const bool blk_d = d == 64 || d == 128;  // head dims of the block-wise kernels; the row-wise one takes 32-256
  if (which == STOF_KERNEL_AUTO) {
    if (!f.synced) return STOF_ERR_NOT_SYNCED;
    const double density = static_cast<double>(f.nnz) / (static_cast<double>(f.n_masks) * f.lq * f.lk);
    // a cached measurement counts only if its kernel runs on this format
    // (the block-wise kernel needs 128-row OTs)
    // (the tuner measures self-attention: its cache applies when Lk = L)
    if (L == Lk && tuned_choice(L, d, density, f.bn, c) &&
        (c->kernel == STOF_KERNEL_ROWWISE || (blockwise_tiles(f) && blk_d))) {
      *source = STOF_PLAN_TUNED;
    } else {
      *c = KernelChoice{which, f.bn, 0, kVariantAuto, 0, 0, 0};
      *source = STOF_PLAN_ANALYTIC;
      // the model's length: L, or for Lk != L the one with L * L = L * Lk valid-key positions
      const int len = L == Lk ? L : static_cast<int>(std::lround(std::sqrt(static_cast<double>(L) * Lk)));
      c->kernel = stof_select_kernel_heads(density, len, d, static_cast<int64_t>(B) * H, listed128_per_row(f));
      if (c->kernel == STOF_KERNEL_BLOCKWISE && (!blockwise_tiles(f) || !blk_d))
        c->kernel = STOF_KERNEL_ROWWISE;  // the block-wise kernel needs 128 x 64 or 128 x 128 OTs, d 64 or 128
    }
  }
  if (c->kernel == STOF_KERNEL_BLOCKWISE && (!blockwise_tiles(f) || !blk_d)) return STOF_ERR_UNSUPPORTED;
  return STOF_OK;
}

stof_status stof_mha_plan(const stof_format* fmt, int B, int H, int L, int d, stof_kernel which, stof_plan* out) {
  if (!out) return STOF_ERR_INVALID_ARG;
  stof_status st = check_format(fmt, B, H, L, L, d);
  if (st != STOF_OK) return st;
  KernelChoice c;
  int source = 0;
  st = plan_call(*fmt, B, H, L, L, d, which, &c, &source);
  if (st != STOF_OK) return st;
  out->kernel = c.kernel;
  out->source = source;
  out->persistent = 0;
  out->stages = 0;
  out->rows_per_warp = 0;
  out->exp_split = 0;
  out->softmax_warpgroups = 0;
  if (c.kernel == STOF_KERNEL_BLOCKWISE) {
    out->persistent = blockwise_persistent(d, c.variant, tiles_per_row(*fmt)) ? 1 : 0;
    out->stages = blockwise_stages(out->persistent != 0, c.stages);
    out->exp_split = c.exp_split;
    out->softmax_warpgroups = c.softmax_wg ? c.softmax_wg : 2;
  } else {
    out->rows_per_warp = rowwise_rows_per_warp(static_cast<long long>(B) * H * L, keys_per_row(*fmt),
                                               listed128_per_row(*fmt), c.rows_per_warp);
    if (d == 256 && out->rows_per_warp > 2) out->rows_per_warp = 2;  // 16 lanes per key
  }
  return STOF_OK;
}

}  // extern "C"

namespace stof {

stof_status mha_fwd_choice(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int L, int Lk,
                           int d,
                           float scale, const stof_format* fmt, int64_t mask_stride_b, int64_t mask_stride_h,
                           const KernelChoice& c, void* o, void* stream) {
  const stof_status st = check_call(q, k, v, dt, B, H, L, Lk, d, scale, fmt, mask_stride_b, mask_stride_h, o);
  if (st != STOF_OK) return st;
  if (c.kernel != STOF_KERNEL_ROWWISE && c.kernel != STOF_KERNEL_BLOCKWISE) return STOF_ERR_INVALID_ARG;
  if (c.kernel == STOF_KERNEL_BLOCKWISE && (!blockwise_tiles(*fmt) || (d != 64 && d != 128)))
    return STOF_ERR_UNSUPPORTED;
  if (c.kernel == STOF_KERNEL_ROWWISE && d == 256 && c.rows_per_warp == 4)
    return STOF_ERR_UNSUPPORTED;  // a d = 256 key needs 16 lanes: 2 rows per warp at most
  AttnParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.B = B;
  p.H = H;
  p.L = L;
  p.Lk = Lk;
  p.d = d;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.bm = fmt->bm;
  p.bn = fmt->bn;
  p.n_tr = fmt->n_tr;
  p.n_tc = fmt->n_tc;
  p.stride_b = mask_stride_b;
  p.stride_h = mask_stride_h;
  p.full_row_ptr = fmt->full_row_ptr;
  p.full_col_idx = fmt->full_col_idx;
  p.part_row_ptr = fmt->part_row_ptr;
  p.part_col_idx = fmt->part_col_idx;
  p.bitmaps = fmt->bitmaps;
  p.err = fmt->counts_dev + 3;
  // bytes 40..47 of the workspace: two words no encoder uses and every
  // encoder zeroes; the persistent kernel leaves them zero when it ends
  p.work = reinterpret_cast<unsigned int*>(fmt->counts_dev + 5);
  p.tiles_per_row = tiles_per_row(*fmt);
  p.keys_per_row = keys_per_row(*fmt);
  p.listed128_per_row = listed128_per_row(*fmt);
  p.rows_per_warp = c.rows_per_warp;
  p.stages = c.stages;
  p.variant = c.variant;
  p.exp_split = c.exp_split;
  p.softmax_wg = c.softmax_wg;
  const bool bf16 = dt == STOF_BF16;
  cudaStream_t s = as_stream(stream);
  if (c.kernel == STOF_KERNEL_ROWWISE)
    return record_cuda(launch_rowwise(p, bf16, s)) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
  return launch_blockwise(p, bf16, s);
}

}  // namespace stof

extern "C" {

stof_status stof_mha_fwd_plan(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int L, int d,
                              float scale, const stof_format* fmt, int64_t mask_stride_b, int64_t mask_stride_h,
                              const stof_plan* plan, void* o, void* stream) {
  if (!plan) return STOF_ERR_INVALID_ARG;
  if (plan->kernel != STOF_KERNEL_ROWWISE && plan->kernel != STOF_KERNEL_BLOCKWISE) return STOF_ERR_INVALID_ARG;
  if (!fmt) return STOF_ERR_INVALID_ARG;
  KernelChoice c{plan->kernel, fmt->bn, 0, kVariantAuto, 0, 0, 0};
  if (plan->kernel == STOF_KERNEL_BLOCKWISE) {
    if (plan->stages < 0 || plan->stages > 8) return STOF_ERR_INVALID_ARG;
    if (plan->exp_split != 0 && plan->exp_split != 1) return STOF_ERR_INVALID_ARG;
    const int w = plan->softmax_warpgroups;
    if (w != 0 && w != 2 && w != 4) return STOF_ERR_UNSUPPORTED;
    c.stages = plan->stages;
    c.variant = plan->persistent ? kVariantPersistent : kVariantPerTile;
    c.exp_split = plan->exp_split;
    c.softmax_wg = w;
  } else {
    const int r = plan->rows_per_warp;
    if (r != 0 && r != 1 && r != 2 && r != 4) return STOF_ERR_UNSUPPORTED;
    if (plan->exp_split != 0 || plan->softmax_warpgroups != 0) return STOF_ERR_UNSUPPORTED;
    c.rows_per_warp = r;
  }
  return mha_fwd_choice(q, k, v, dt, B, H, L, L, d, scale, fmt, mask_stride_b, mask_stride_h, c, o, stream);
}

stof_status stof_mha_fwd_cross(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H, int Lq,
                               int Lk, int d, float scale, const stof_format* fmt, int64_t mask_stride_b,
                               int64_t mask_stride_h, stof_kernel which, void* o, void* stream) {
  stof_status st = check_call(q, k, v, dt, B, H, Lq, Lk, d, scale, fmt, mask_stride_b, mask_stride_h, o);
  if (st != STOF_OK) return st;
  KernelChoice c;
  int source = 0;
  st = plan_call(*fmt, B, H, Lq, Lk, d, which, &c, &source);
  if (st != STOF_OK) return st;
  return mha_fwd_choice(q, k, v, dt, B, H, Lq, Lk, d, scale, fmt, mask_stride_b, mask_stride_h, c, o, stream);
}

stof_status stof_mha_fwd(const void* q, const void* k, const void* v, stof_dtype dt, int B, int H,
                         int L, int d, float scale, const stof_format* fmt,
                         int64_t mask_stride_b, int64_t mask_stride_h, stof_kernel which, void* o,
                         void* stream) {
  return stof_mha_fwd_cross(q, k, v, dt, B, H, L, L, d, scale, fmt, mask_stride_b, mask_stride_h, which, o, stream);
}

}  // extern "C"
