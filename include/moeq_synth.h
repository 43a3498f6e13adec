/*
 * moeq synthetic inputs -- the device twin of the seeded generator used by the
 * tests and the benchmark (the Python module synth.py is the host twin).
 * Not part of the FFN path: it only fills buffers with seeded codes and scales
 * so that large synthetic layers (up to ~100 GB) can be built on the device.
 *
 * SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) as a counter-based generator:
 *   key    = mix64(seed * 0x9E3779B97F4A7C15 + stream)
 *   u64(i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)      (mod 2^64)
 *   mix64(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
 *             z *= 0x94D049BB133111EB; z ^= z >> 31
 * All pointers are device pointers; calls enqueue on the given stream.
 */
#ifndef MOEQ_SYNTH_H
#define MOEQ_SYNTH_H

#include <stddef.h>
#include <stdint.h>

#include "moeq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[e] = (u64(e / 16) >> (4 * (e % 16))) & ((1 << bits) - 1) for e < n;
 * n % 16 == 0, out 16-byte aligned, bits in 1..4. */
int moeq_synth_codes(uint64_t seed, uint64_t stream, int bits, size_t n, uint8_t* out,
                     moeq_stream s);

/* bits 2 or 3: fp16 bit patterns LO + (u64(i) >> 32) % (HI - LO + 1) with
 * LO = 0x068E (fp16 1e-4), HI = 0x211F (fp16 1e-2); out is uint16 [n].
 * bits 4: E8M0 bytes 114 + (u64(i) >> 32) % 7; out is uint8 [n]. */
int moeq_synth_scales(uint64_t seed, uint64_t stream, int bits, size_t n, void* out,
                      moeq_stream s);

#ifdef __cplusplus
}
#endif
#endif
