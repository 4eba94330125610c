/*
 * k3synth.h -- seeded, counter-based synthetic inputs for the routed MoE layer.
 *
 * This module holds no arithmetic of the method.  It only defines WHICH bytes and
 * numbers make up a synthetic layer, so that the CPU oracle, the tests and the
 * benchmark all see the same inputs.  Every value is a pure function of
 * (seed, tag, layer, a, b, index), so any single expert or token can be regenerated
 * alone, on the host or on the device.
 *
 * Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the 64-bit finaliser constants of Vigna's public
 * splitmix64.c).  A stream is a splitmix64 state `key`; draw i of the stream is the
 * output of step i+1 from that state, i.e. mix(key + (i+1)*GAMMA).
 *
 * Streams and their contents (canonical MXFP4 layout: per expert three matrices,
 * gate [f][d], up [f][d], down [d][f]; per matrix the nibble bytes [rows][cols/2]
 * with element 2i in the low nibble, then the E8M0 scale bytes [rows][cols/32]):
 *   tag 1  nibble bytes of (layer, expert, matrix): byte j = byte (j mod 8) of draw(j/8)
 *   tag 2  scale bytes of (layer, expert, matrix):  byte j = lo + floor(hi32(draw(j))*(hi-lo+1)/2^32)
 *   tag 3  token activations x of (layer, token, attempt): N(0,1) by Box-Muller from
 *          draws 2j and 2j+1, rounded to float32 then to bf16 (round to nearest even)
 *   tag 4  router weights W_r of (layer, expert): N(0,1)/sqrt(d), rounded to float32
 *   tag 5  hot-expert subset of (layer): partial Fisher-Yates over 0..E-1
 */
#ifndef K3SYNTH_H
#define K3SYNTH_H
#include <stdint.h>

#define K3S_GAMMA 0x9E3779B97F4A7C15ULL

#ifdef __CUDACC__
#define K3S_HD __host__ __device__
#else
#define K3S_HD
#endif

enum { K3S_TAG_NIB = 1, K3S_TAG_SCALE = 2, K3S_TAG_X = 3, K3S_TAG_WR = 4, K3S_TAG_HOT = 5 };

static inline K3S_HD uint64_t k3s_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Stream key for (seed, tag, layer, a, b); a < 2^28, b < 2^20, layer < 256. */
static inline K3S_HD uint64_t k3s_key(uint64_t seed, uint32_t tag, uint32_t layer, uint32_t a, uint32_t b) {
  uint64_t id = ((uint64_t)(tag & 0xFFu) << 56) ^ ((uint64_t)(layer & 0xFFu) << 48) ^
                ((uint64_t)(a & 0x0FFFFFFFu) << 20) ^ (uint64_t)(b & 0xFFFFFu);
  return k3s_mix(seed * K3S_GAMMA + k3s_mix(id + K3S_GAMMA));
}

static inline K3S_HD uint64_t k3s_draw(uint64_t key, uint64_t i) { return k3s_mix(key + (i + 1) * K3S_GAMMA); }

#ifdef __cplusplus
extern "C" {
#endif

/* Canonical MXFP4 bytes of experts [e0, e1) of one layer.  nib receives
 * (e1-e0) * 3*f*d/2 bytes, scl receives (e1-e0) * 3*f*d/32 bytes. */
void k3s_experts(uint64_t seed, int layer, int e0, int e1, int d, int f, int scale_lo, int scale_hi,
                 uint8_t* nib, uint8_t* scl);
/* T tokens x[T][d] as bf16 bit patterns; token t has global id t0+t and uses
 * attempt[t] (NULL = all attempts 0). */
void k3s_tokens_bf16(uint64_t seed, int layer, int t0, int T, int d, const int32_t* attempt, uint16_t* out);
/* Router weights W_r[E][d], float32. */
void k3s_router_weights(uint64_t seed, int layer, int E, int d, float* out);
/* The first n_hot entries of a seeded permutation of 0..E-1. */
void k3s_hot_experts(uint64_t seed, int layer, int E, int n_hot, int32_t* out);

#ifdef __cplusplus
}
#endif
#endif
