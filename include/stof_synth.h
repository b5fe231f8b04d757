/*
 * stof_synth.h -- synthetic input generator for tests and benchmarks
 * (libstof_synth.so).  Not part of the attention method: it only writes
 * seeded masks on the device so that very large masks need no host copy.
 */
#ifndef STOF_SYNTH_H_
#define STOF_SYNTH_H_
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* Writes uint8 out[n_masks][L][L] (device, 8-byte aligned):
 *   out[m][i][j] = (j <= i) && (j == i || (SplitMix64(seed ^ (m<<48 | i<<24 | j)) >> 11) < threshold)
 * Requires L % 8 == 0, L <= 2^24, n_masks <= 2^15.  Asynchronous on stream
 * (a cudaStream_t).  Returns 0 on success, 1 for bad arguments, 2 for a
 * launch error. */
int stof_synth_causal_bernoulli_mask(uint8_t* out, int n_masks, int L, uint64_t seed,
                                     uint64_t threshold, void* stream);

/* The same masks bit-packed: out[n_masks][L][L/8], bit c (least
 * significant first) of byte jb of row i = element (i, 8 jb + c).  Requires
 * L % 64 == 0 and the limits above. */
int stof_synth_causal_bernoulli_mask_bits(uint8_t* out, int n_masks, int L, uint64_t seed,
                                          uint64_t threshold, void* stream);

/* Packs n_in mask bytes (device, 8-byte aligned, n_in % 8 == 0; non-zero =
 * valid) into n_in / 8 bytes, least significant bit first. */
int stof_synth_pack_bits(const uint8_t* in, uint8_t* out, long long n_in, void* stream);

#ifdef __cplusplus
}
#endif
#endif
