// Measured choice of the MHA step's parameters, with a result cache.
//
// "Accelerating Sparse Transformer Inference on GPU" (gist.science technical
// summary), Methodology 2, operator fusion module, two-stage tuning, stage 2
// (parameter sampling): once the operator boundaries are fixed, kernel
// parameters such as block size and pipeline stages are sampled by running
// them, and (same page, "autopilot" summary) what was measured is cached so
// that a configuration is not timed again.  For the masked MHA step the
// sampled parameters are the kernel (row-wise or block-wise), the OT width
// (64 or 128 key columns; 128 query rows), the row-wise kernel's rows per
// warp, the block-wise kernel's K/V ring depth (its pipeline stages), its
// exp split (a share of the exponentials on the FMA pipe), its softmax
// warpgroup count (2, or 4 on the persistent kernel) and, at d = 64,
// whether it runs persistent CTAs.  A result is cached under (sequence length, head dim, density
// bucket), the bucket being the density rounded to half powers of two;
// stof_mha_fwd(AUTO) runs the fastest cached candidate on the format's OT
// width.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"

namespace stof {

const KernelChoice kTuneCandidates[STOF_TUNE_CANDIDATES] = {
    // kernel, OT width, ring depth, variant, rows per warp, exp split, softmax warpgroups
    {STOF_KERNEL_ROWWISE, 128, 0, kVariantAuto, 1, 0, 0},
    {STOF_KERNEL_ROWWISE, 128, 0, kVariantAuto, 2, 0, 0},
    {STOF_KERNEL_ROWWISE, 128, 0, kVariantAuto, 4, 0, 0},
    {STOF_KERNEL_BLOCKWISE, 128, 3, kVariantPerTile, 0, 0, 0},
    {STOF_KERNEL_BLOCKWISE, 128, 2, kVariantPerTile, 0, 0, 0},
    {STOF_KERNEL_BLOCKWISE, 128, 4, kVariantPerTile, 0, 0, 0},     // d = 64 only
    {STOF_KERNEL_BLOCKWISE, 128, 4, kVariantPersistent, 0, 0, 0},  // d = 64 only
    {STOF_KERNEL_BLOCKWISE, 128, 3, kVariantPersistent, 0, 0, 0},  // d = 64 only
    {STOF_KERNEL_BLOCKWISE, 128, 2, kVariantPersistent, 0, 0, 0},  // d = 64 only
    {STOF_KERNEL_BLOCKWISE, 64, 0, kVariantAuto, 0, 0, 0},
    {STOF_KERNEL_BLOCKWISE, 128, 3, kVariantPerTile, 0, 1, 0},     // exp split
    {STOF_KERNEL_BLOCKWISE, 128, 4, kVariantPersistent, 0, 1, 0},  // exp split, d = 64 only
    {STOF_KERNEL_BLOCKWISE, 128, 4, kVariantPersistent, 0, 0, 4},  // four softmax warpgroups, d = 64 only
};

namespace {

constexpr int kTimedCalls = 3;

std::mutex g_mu;
std::map<std::tuple<int, int, int>, stof_tune_result> g_cache;

// Streams the candidates run on: the caller's stream.
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

int tune_density_bucket(double density) {
  if (!(density > 0.0)) return -61;
  const double b = std::floor(2.0 * std::log2(std::min(density, 1.0)) + 0.5);
  return static_cast<int>(std::max(-60.0, b));
}

bool tuned_choice(int L, int d, double density, int bn, KernelChoice* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  const auto it = g_cache.find(std::make_tuple(L, d, tune_density_bucket(density)));
  if (it == g_cache.end()) return false;
  const stof_tune_result& r = it->second;
  int best = -1;
  for (int i = 0; i < STOF_TUNE_CANDIDATES; ++i)
    if (r.cand_bn[i] == bn && r.cand_ms[i] > 0.f && (best < 0 || r.cand_ms[i] < r.cand_ms[best])) best = i;
  if (best < 0) return false;
  *out = kTuneCandidates[best];
  return true;
}

}  // namespace stof

using namespace stof;

extern "C" {

size_t stof_tune_workspace_bytes(int n_masks, int L) {
  size_t best = 0;
  for (const KernelChoice& c : kTuneCandidates)
    best = std::max(best, stof_encode_workspace_bytes(n_masks, L, L, 128, c.bn));
  return best;
}

stof_status stof_tune(const uint8_t* mask, int n_masks, const void* q, const void* k, const void* v,
                      stof_dtype dt, int B, int H, int L, int d, float scale, int64_t mask_stride_b,
                      int64_t mask_stride_h, void* workspace, size_t ws_bytes, void* o, stof_tune_result* out,
                      void* stream) {
  if (!mask || !q || !k || !v || !o || !workspace || !out) return STOF_ERR_INVALID_ARG;
  const size_t need = stof_tune_workspace_bytes(n_masks, L);
  if (need == 0) return STOF_ERR_SHAPE;
  if (ws_bytes < need) return STOF_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  cudaEvent_t ev[2];
  if (record_cuda(cudaEventCreate(&ev[0])) != cudaSuccess) return STOF_ERR_CUDA;
  if (record_cuda(cudaEventCreate(&ev[1])) != cudaSuccess) {
    cudaEventDestroy(ev[0]);
    return STOF_ERR_CUDA;
  }
  stof_tune_result r;
  r.kernel = STOF_KERNEL_AUTO;
  r.bn = 0;
  r.ms = -1.f;
  r.density = 0.0;
  r.stages = 0;
  r.persistent = 0;
  r.rows_per_warp = 0;
  r.exp_split = 0;
  r.softmax_warpgroups = 0;
  for (int i = 0; i < STOF_TUNE_CANDIDATES; ++i) {
    const KernelChoice& cand = kTuneCandidates[i];
    r.cand_kernel[i] = cand.kernel;
    r.cand_bn[i] = cand.bn;
    r.cand_persistent[i] = 0;
    r.cand_stages[i] = 0;
    r.cand_rows_per_warp[i] = cand.rows_per_warp;
    r.cand_exp_split[i] = cand.exp_split;
    r.cand_softmax_warpgroups[i] =
        cand.kernel == STOF_KERNEL_BLOCKWISE ? (cand.softmax_wg ? cand.softmax_wg : 2) : 0;
    r.cand_ms[i] = -1.f;
  }
  stof_status st = STOF_OK;
  for (int bn : {128, 64}) {
    stof_format fmt;
    st = stof_encode_mask(mask, n_masks, L, L, 128, bn, workspace, ws_bytes, &fmt, stream);
    if (st == STOF_OK) st = stof_format_sync(&fmt, stream);
    if (st != STOF_OK) break;
    r.density = static_cast<double>(fmt.nnz) / (static_cast<double>(n_masks) * L * L);
    const float tpr = static_cast<float>(static_cast<double>(fmt.n_full + fmt.n_part) /
                                         (static_cast<double>(fmt.n_masks) * fmt.n_tr));
    for (int i = 0; i < STOF_TUNE_CANDIDATES && st == STOF_OK; ++i) {
      const KernelChoice& cand = kTuneCandidates[i];
      if (cand.bn != bn) continue;
      if (cand.kernel == STOF_KERNEL_BLOCKWISE && (cand.variant == kVariantPersistent || cand.stages == 4) &&
          d != 64)
        continue;  // persistent CTAs and a 4-deep ring exist for d = 64 only
      st = mha_fwd_choice(q, k, v, dt, B, H, L, L, d, scale, &fmt, mask_stride_b, mask_stride_h, cand, o, stream);
      if (st == STOF_ERR_UNSUPPORTED) {  // not a candidate for these sizes
        st = STOF_OK;
        continue;
      }
      if (st != STOF_OK) break;
      if (cand.kernel == STOF_KERNEL_BLOCKWISE) {  // what the launch ran (an automatic variant resolved)
        const bool pers = blockwise_persistent(d, cand.variant, tpr);
        r.cand_persistent[i] = pers ? 1 : 0;
        r.cand_stages[i] = blockwise_stages(pers, cand.stages);
      }
      if (record_cuda(cudaEventRecord(ev[0], s)) != cudaSuccess) { st = STOF_ERR_CUDA; break; }
      for (int c = 0; c < kTimedCalls && st == STOF_OK; ++c)
        st = mha_fwd_choice(q, k, v, dt, B, H, L, L, d, scale, &fmt, mask_stride_b, mask_stride_h, cand, o, stream);
      if (st != STOF_OK) break;
      float ms = 0.f;
      if (record_cuda(cudaEventRecord(ev[1], s)) != cudaSuccess ||
          record_cuda(cudaEventSynchronize(ev[1])) != cudaSuccess ||
          record_cuda(cudaEventElapsedTime(&ms, ev[0], ev[1])) != cudaSuccess) {
        st = STOF_ERR_CUDA;
        break;
      }
      // a device-side failure of a candidate is reported, not chosen
      st = stof_format_sync(&fmt, stream);
      if (st != STOF_OK) break;
      r.cand_ms[i] = ms / kTimedCalls;
      if (r.ms < 0.f || r.cand_ms[i] < r.ms) {
        r.ms = r.cand_ms[i];
        r.kernel = cand.kernel;
        r.bn = bn;
        r.stages = r.cand_stages[i];
        r.persistent = r.cand_persistent[i];
        r.rows_per_warp = r.cand_rows_per_warp[i];
        r.exp_split = r.cand_exp_split[i];
        r.softmax_warpgroups = r.cand_softmax_warpgroups[i];
      }
    }
    if (st != STOF_OK) break;
  }
  cudaEventDestroy(ev[0]);
  cudaEventDestroy(ev[1]);
  if (st != STOF_OK) return st;
  if (r.ms < 0.f) return STOF_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_cache[std::make_tuple(L, d, tune_density_bucket(r.density))] = r;
  }
  *out = r;
  return STOF_OK;
}

int stof_tune_lookup(int L, int d, double density, stof_tune_result* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  const auto it = g_cache.find(std::make_tuple(L, d, tune_density_bucket(density)));
  if (it == g_cache.end()) return 0;
  if (out) *out = it->second;
  return 1;
}

void stof_tune_clear(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_cache.clear();
}

int stof_tune_density_bucket(double density) { return tune_density_bucket(density); }

}  // extern "C"
