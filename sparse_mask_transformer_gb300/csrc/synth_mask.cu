// Synthetic input generator (not part of the method): writes the seeded
// "causal AND Bernoulli(p) with forced diagonal" masks on the device, so a
// 16k x 16k x 32-head mask needs no 8.6 GB host buffer.
//
// Element (m, i, j) is valid iff j <= i and (j == i or (z >> 11) < threshold),
// z = SplitMix64(seed XOR (m << 48 | i << 24 | j)), where SplitMix64 is
// Sebastiano Vigna's published generator step applied to that state:
// z = x + 0x9E3779B97F4A7C15, then z ^= z >> 30, z *= 0xBF58476D1CE4E5B9,
// z ^= z >> 27, z *= 0x94D049BB133111EB, z ^= z >> 31.
// threshold = ceil(p * 2^53), so the test equals "u < p" for
// u = (z >> 11) * 2^-53.
#include <cuda_runtime.h>
#include <cstdint>

#include "stof_synth.h"

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// one thread writes 8 consecutive mask bytes of one row
__global__ void causal_bernoulli_kernel(uint8_t* out, int L, long long n_words, uint64_t seed,
                                        uint64_t threshold) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_words) return;
  const long long words_per_row = L / 8;
  const long long row = gid / words_per_row;
  const int j0 = static_cast<int>(gid % words_per_row) * 8;
  const int i = static_cast<int>(row % L);
  const uint64_t m = static_cast<uint64_t>(row / L);
  uint64_t word = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int j = j0 + c;
    uint64_t valid = 0;
    if (j == i) {
      valid = 1;
    } else if (j < i) {
      const uint64_t ctr = (m << 48) | (static_cast<uint64_t>(i) << 24) | static_cast<uint64_t>(j);
      valid = (splitmix64(seed ^ ctr) >> 11) < threshold ? 1 : 0;
    }
    word |= valid << (8 * c);
  }
  reinterpret_cast<uint64_t*>(out)[gid] = word;
}

// one thread writes 64 consecutive keys of one row as 8 bit-packed bytes
__global__ void causal_bernoulli_bits_kernel(uint8_t* out, int L, long long n_words, uint64_t seed,
                                             uint64_t threshold) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_words) return;
  const long long words_per_row = L / 64;
  const long long row = gid / words_per_row;
  const int j0 = static_cast<int>(gid % words_per_row) * 64;
  const int i = static_cast<int>(row % L);
  const uint64_t m = static_cast<uint64_t>(row / L);
  uint64_t word = 0;
  for (int c = 0; c < 64; ++c) {
    const int j = j0 + c;
    uint64_t valid = 0;
    if (j == i) {
      valid = 1;
    } else if (j < i) {
      const uint64_t ctr = (m << 48) | (static_cast<uint64_t>(i) << 24) | static_cast<uint64_t>(j);
      valid = (splitmix64(seed ^ ctr) >> 11) < threshold ? 1 : 0;
    }
    word |= valid << c;  // little-endian: byte jb holds keys 8 jb .. 8 jb + 7, lowest bit first
  }
  reinterpret_cast<uint64_t*>(out)[gid] = word;
}

// one thread packs 8 mask bytes (non-zero = valid) into one byte
__global__ void pack_bits_kernel(const uint8_t* in, uint8_t* out, long long n_out) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_out) return;
  const uint64_t w = reinterpret_cast<const uint64_t*>(in)[gid];
  uint32_t b = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) b |= ((w >> (8 * c)) & 0xFFull) != 0 ? (1u << c) : 0u;
  out[gid] = static_cast<uint8_t>(b);
}

}  // namespace

extern "C" int stof_synth_causal_bernoulli_mask_bits(uint8_t* out, int n_masks, int L, uint64_t seed,
                                                     uint64_t threshold, void* stream) {
  if (!out || n_masks < 1 || L < 64 || L % 64 || L > (1 << 24) || n_masks > (1 << 15)) return 1;
  if (reinterpret_cast<uintptr_t>(out) % 8) return 1;
  const long long n_words = static_cast<long long>(n_masks) * L * (L / 64);
  const int threads = 256;
  const long long blocks = (n_words + threads - 1) / threads;
  causal_bernoulli_bits_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      out, L, n_words, seed, threshold);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int stof_synth_pack_bits(const uint8_t* in, uint8_t* out, long long n_in, void* stream) {
  if (!in || !out || n_in < 8 || n_in % 8) return 1;
  if (reinterpret_cast<uintptr_t>(in) % 8) return 1;
  const long long n_out = n_in / 8;
  const int threads = 256;
  const long long blocks = (n_out + threads - 1) / threads;
  pack_bits_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n_out);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int stof_synth_causal_bernoulli_mask(uint8_t* out, int n_masks, int L, uint64_t seed,
                                                uint64_t threshold, void* stream) {
  if (!out || n_masks < 1 || L < 8 || L % 8 || L > (1 << 24) || n_masks > (1 << 15)) return 1;
  if (reinterpret_cast<uintptr_t>(out) % 8) return 1;
  const long long n_words = static_cast<long long>(n_masks) * L * (L / 8);
  const int threads = 256;
  const long long blocks = (n_words + threads - 1) / threads;
  causal_bernoulli_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                            reinterpret_cast<cudaStream_t>(stream)>>>(out, L, n_words, seed, threshold);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
