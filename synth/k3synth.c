/* k3synth.c -- host side of the counter-based synthetic-input generator (see k3synth.h). */
#include "k3synth.h"
#include <math.h>
#include <stddef.h>
#include <string.h>

static uint8_t scale_byte(uint64_t key, uint64_t j, int lo, int hi) {
  uint64_t r = (uint64_t)(hi - lo + 1);
  return (uint8_t)(lo + (int)(((k3s_draw(key, j) >> 32) * r) >> 32));
}

void k3s_experts(uint64_t seed, int layer, int e0, int e1, int d, int f, int scale_lo, int scale_hi,
                 uint8_t* nib, uint8_t* scl) {
  const size_t mat_nib = (size_t)f * d / 2, mat_scl = (size_t)f * d / 32;
  for (int e = e0; e < e1; ++e) {
    for (int m = 0; m < 3; ++m) {
      uint8_t* nb = nib + ((size_t)(e - e0) * 3 + m) * mat_nib;
      uint8_t* sb = scl + ((size_t)(e - e0) * 3 + m) * mat_scl;
      const uint64_t kn = k3s_key(seed, K3S_TAG_NIB, (uint32_t)layer, (uint32_t)e, (uint32_t)m);
      const uint64_t ks = k3s_key(seed, K3S_TAG_SCALE, (uint32_t)layer, (uint32_t)e, (uint32_t)m);
      const long long nwords = (long long)(mat_nib / 8);
#pragma omp parallel for schedule(static)
      for (long long w = 0; w < nwords; ++w) {
        uint64_t u = k3s_draw(kn, (uint64_t)w);
        memcpy(nb + (size_t)w * 8, &u, 8); /* little-endian: byte j%8 of draw j/8 */
      }
      for (size_t j = (size_t)nwords * 8; j < mat_nib; ++j)
        nb[j] = (uint8_t)(k3s_draw(kn, j / 8) >> (8 * (j % 8)));
#pragma omp parallel for schedule(static)
      for (long long j = 0; j < (long long)mat_scl; ++j) sb[j] = scale_byte(ks, (uint64_t)j, scale_lo, scale_hi);
    }
  }
}

static double normal_pair(uint64_t key, uint64_t j) {
  const double two53 = 9007199254740992.0;
  double u1 = ((double)(k3s_draw(key, 2 * j) >> 11) + 1.0) / two53; /* (0, 1] */
  double u2 = (double)(k3s_draw(key, 2 * j + 1) >> 11) / two53;     /* [0, 1) */
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static uint16_t f32_to_bf16_rne(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void k3s_tokens_bf16(uint64_t seed, int layer, int t0, int T, int d, const int32_t* attempt, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const uint64_t key = k3s_key(seed, K3S_TAG_X, (uint32_t)layer, (uint32_t)(t0 + t),
                                 (uint32_t)(attempt ? attempt[t] : 0));
    for (int j = 0; j < d; ++j) out[(size_t)t * d + j] = f32_to_bf16_rne((float)normal_pair(key, (uint64_t)j));
  }
}

void k3s_router_weights(uint64_t seed, int layer, int E, int d, float* out) {
  const double inv = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(static)
  for (int e = 0; e < E; ++e) {
    const uint64_t key = k3s_key(seed, K3S_TAG_WR, (uint32_t)layer, (uint32_t)e, 0);
    for (int j = 0; j < d; ++j) out[(size_t)e * d + j] = (float)(normal_pair(key, (uint64_t)j) * inv);
  }
}

void k3s_hot_experts(uint64_t seed, int layer, int E, int n_hot, int32_t* out) {
  int32_t perm[65536];
  if (E > 65536 || n_hot > E) return;
  for (int i = 0; i < E; ++i) perm[i] = i;
  const uint64_t key = k3s_key(seed, K3S_TAG_HOT, (uint32_t)layer, 0, 0);
  for (int i = 0; i < n_hot; ++i) {
    int j = i + (int)(((k3s_draw(key, (uint64_t)i) >> 32) * (uint64_t)(E - i)) >> 32);
    int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  for (int i = 0; i < n_hot; ++i) out[i] = perm[i];
}
