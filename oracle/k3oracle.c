/*
 * k3oracle.c -- THE ORACLE for the routed mixture-of-experts layer on MXFP4 experts.
 *
 * TEST INFRASTRUCTURE ONLY.  A plain, slow, obviously correct CPU restatement of
 * what the layer computes, in fp64, one scalar at a time.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Sources (the pages on the kimi-k3-in-c engine):
 *   [R1]   fiv.co.kr "kimi-k3-in-c deep dive", section "four reductions", reduction 1:
 *          experts stay MXFP4 and are multiplied on the nibbles; value =
 *          E2M1[nibble] * 2^(scale-127); 32 values share one 8-bit exponent; the
 *          E2M1 magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives; one
 *          expert holds 33,030,144 parameters in 17,547,264 bytes.
 *   [INV5] same page, table of the five invariants, row 5: the routing bias steers
 *          the selection only; the combine weights come from the unbiased sigmoid
 *          scores.
 *   [RT]   same page, "what you learn", router paragraph: sigmoid score, then the
 *          bias picks the experts, then the picked experts are mixed with the
 *          unbiased scores.
 *   [GL]   same page, glossary: MoE picks 16 of 896 experts per layer; MXFP4 is
 *          0.53125 bytes per parameter.
 *   [EX]   same page, "what you learn", the exercise paragraph: the engine has an
 *          RMSNorm kernel with an epsilon (used here only as glue between stacked
 *          layers, see k3o_residual_rmsnorm).
 * Where the pages are silent the code says READING and states the reading taken.
 * Parity unpinned: situ() (the SiTU-GLU gate, act = 1).  The pages give its ingredients and
 * its bound but no formula, so its pins check only the properties of the reading taken.
 * Every other function is pinned by tests/test_oracle_pins.py.
 *
 * Canonical expert layout (the input format of the library, defined by us):
 *   matrices gate W_g [f][d], up W_u [f][d], down W_d [d][f], in that order; per
 *   matrix the nibble bytes [rows][cols/2] then, in a separate array, the scale
 *   bytes [rows][cols/32].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decode ---- */

/* E2M1 code (4 bits) -> value.  [R1] gives the magnitudes and "their negatives".
 * READING (OCP Microscaling Formats v1.0, E2M1): bit 3 is the sign, bits 2..1 the
 * exponent with bias 1, bit 0 the mantissa; exponent 0 is subnormal (0.5*m). */
double k3o_e2m1(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E8M0 scale byte -> 2^(s-127) [R1].  READING: 255 is NaN (OCP MX v1.0). */
double k3o_e8m0(int s) { return s == 255 ? NAN : ldexp(1.0, s - 127); }

/* bf16 bit pattern -> value (exact). */
double k3o_bf16(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Element (r, c) of an MXFP4 matrix with `cols` columns.  [R1]: one scale per 32
 * values.  READING: the 32 values sharing a scale are consecutive along a row (the
 * reduction axis), and element 2i of a row sits in the low nibble of byte i. */
double k3o_mx_elem(const uint8_t* nib, const uint8_t* scl, int cols, int r, int c) {
  const uint8_t byte = nib[(size_t)r * (size_t)(cols / 2) + (size_t)(c / 2)];
  const int code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  return k3o_e2m1(code) * k3o_e8m0(scl[(size_t)r * (size_t)(cols / 32) + (size_t)(c / 32)]);
}

/* Whole matrix to fp64, row-major [rows][cols].  Used by the tests' second
 * formulation of the FFN (expand, then a library matmul). */
void k3o_decode_matrix(const uint8_t* nib, const uint8_t* scl, int rows, int cols, double* out) {
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) out[(size_t)r * cols + c] = k3o_mx_elem(nib, scl, cols, r, c);
}

/* Canonical byte sizes of one expert ([R1]: 3 matrices, 0.5 byte per value plus
 * one scale byte per 32 values). */
long long k3o_expert_nib_bytes(int d, int f) { return 3LL * f * d / 2; }
long long k3o_expert_scale_bytes(int d, int f) { return 3LL * f * d / 32; }

/* ---------------------------------------------------------------- router ---- */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

typedef struct {
  double key;
  int id;
} keyed;

/* READING (tie-break): descending key, then ascending expert id. */
static int by_key_desc(const void* pa, const void* pb) {
  const keyed* a = (const keyed*)pa;
  const keyed* b = (const keyed*)pb;
  if (a->key > b->key) return -1;
  if (a->key < b->key) return 1;
  return (a->id > b->id) - (a->id < b->id);
}

/* Router for T tokens.  [RT], [INV5], [GL]:
 *   logit[t,e] = sum_j x[t,j] * W_r[e,j]         (j ascending, fp64)
 *   sigma      = 1 / (1 + exp(-logit))
 *   key        = sigma + bias[e]                  READING: bias added after the sigmoid
 *   selection  = the k largest keys, by a full sort (brute force)
 *   w[t,i]     = sigma[idx_i] / sum_i sigma[idx_i]  READING: renormalised to sum 1,
 *                                                  no extra routed scaling factor
 * idx/w hold the picks in descending key order (READING).  logits/keys (optional,
 * [T][E]) return the fp64 intermediates. */
void k3o_router(int T, int d, int E, int k, const uint16_t* x, const float* Wr, const float* bias, int32_t* idx,
                double* w, double* logits_out, double* keys_out) {
#pragma omp parallel
  {
    keyed* all = (keyed*)malloc(sizeof(keyed) * (size_t)E);
    double* sig = (double*)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
      for (int e = 0; e < E; ++e) {
        double logit = 0.0;
        for (int j = 0; j < d; ++j) logit += k3o_bf16(x[(size_t)t * d + j]) * (double)Wr[(size_t)e * d + j];
        sig[e] = sigmoid(logit);
        all[e].key = sig[e] + (bias ? (double)bias[e] : 0.0);
        all[e].id = e;
        if (logits_out) logits_out[(size_t)t * E + e] = logit;
        if (keys_out) keys_out[(size_t)t * E + e] = all[e].key;
      }
      qsort(all, (size_t)E, sizeof(keyed), by_key_desc);
      double total = 0.0;
      for (int i = 0; i < k; ++i) total += sig[all[i].id];
      for (int i = 0; i < k; ++i) {
        idx[(size_t)t * k + i] = all[i].id;
        w[(size_t)t * k + i] = sig[all[i].id] / total;
      }
    }
    free(all);
    free(sig);
  }
}

/* ------------------------------------------------------------- bucketing ---- */

/* Token-to-expert bucketing by direct definition (the grouping that the pages'
 * MoE step implies: every expert runs on the tokens routed to it).  A pick is
 * p = t*k + slot.  counts[e] = #picks routed to e; offsets = exclusive prefix sum
 * in expert-id order (E+1 entries); perm lists, expert by expert, that expert's
 * picks in ascending p, i.e. ordered by (t, slot). */
void k3o_bucket(int T, int k, int E, const int32_t* idx, int32_t* counts, int32_t* offsets, int32_t* perm) {
  const int P = T * k;
  for (int e = 0; e < E; ++e) {
    counts[e] = 0;
    for (int p = 0; p < P; ++p)
      if (idx[p] == e) counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int pos = 0;
  for (int e = 0; e < E; ++e)
    for (int p = 0; p < P; ++p)
      if (idx[p] == e) perm[pos++] = p;
}

/* ------------------------------------------------------------ expert FFN ---- */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* SiTU-GLU gate ("kimi-k3-in-c deep dive", glossary entry SiTU-GLU: K3's activation, a
 * combination of tanh and sigmoid whose parameters beta1 = 4 and beta2 = 25 bound the gate
 * above by 100).  The pages print no formula.  READING (parity unpinned: only the bound
 * 100 = beta1 * beta2 and the two functions come from the page):
 *   situ(z) = beta1 * beta2 * sigmoid(z) * tanh(z / beta2)
 * which rises to beta1 * beta2 = 100 as z -> +inf, falls to 0 as z -> -inf, and has slope
 * beta1 / 2 at 0; h = situ(g) * u replaces silu(g) * u. */
static const double kSituBeta1 = 4.0, kSituBeta2 = 25.0;
static double situ(double z) { return kSituBeta1 * kSituBeta2 * (1.0 / (1.0 + exp(-z))) * tanh(z / kSituBeta2); }
double k3o_situ(double z) { return situ(z); }

/* Gate activation: act 0 = SwiGLU's silu, act 1 = SiTU-GLU's situ (above). */
static double gate_act(double z, int act) { return act == 1 ? situ(z) : silu(z); }

/* One expert applied to one token, with SwiGLU (the activation the layer
 * specification names; READING: no clamp, no extra scaling), or SiTU-GLU when act = 1:
 *   g_r = sum_j W_g[r,j] x_j,  u_r = sum_j W_u[r,j] x_j      (r < f, j < d)
 *   h_r = silu(g_r) * u_r,     silu(z) = z / (1 + exp(-z))     (act 0)
 *   h_r = situ(g_r) * u_r                                      (act 1)
 *   o_i = sum_r W_d[i,r] h_r                                 (i < d)
 *   a_i = sum_r |W_d[i,r] h_r|     (magnitude of the terms, for error bounds)
 * nib/scl point at the expert's canonical block (three matrices back to back).
 * h (f values) and a (d values) may be NULL. */
void k3o_expert_ffn(int d, int f, const uint8_t* nib, const uint8_t* scl, const double* x, double* h_out,
                    double* o, double* a, int act) {
  const size_t mn = (size_t)f * d / 2, ms = (size_t)f * d / 32;
  const uint8_t *ng = nib, *nu = nib + mn, *nd = nib + 2 * mn;
  const uint8_t *sg = scl, *su = scl + ms, *sd = scl + 2 * ms;
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  for (int r = 0; r < f; ++r) {
    double g = 0.0, u = 0.0;
    for (int j = 0; j < d; ++j) {
      g += k3o_mx_elem(ng, sg, d, r, j) * x[j];
      u += k3o_mx_elem(nu, su, d, r, j) * x[j];
    }
    h[r] = gate_act(g, act) * u;
    if (h_out) h_out[r] = h[r];
  }
  for (int i = 0; i < d; ++i) {
    double acc = 0.0, mag = 0.0;
    for (int r = 0; r < f; ++r) {
      const double term = k3o_mx_elem(nd, sd, f, i, r) * h[r];
      acc += term;
      mag += fabs(term);
    }
    o[i] = acc;
    if (a) a[i] = mag;
  }
  free(h);
}

/* ----------------------------------------------------------- MoE combine ---- */

/* The routed MoE output for T tokens given the router's picks.
 *   y[t,i]      = sum_{slot=0..k-1} w[t,slot] * o_{t,slot}[i]   (slot ascending)
 *   sumabs[t,i] = sum_slot |w[t,slot]| * a_{t,slot}[i] = sum of |terms| of y[t,i]
 * pick_nib[p]/pick_scl[p] point at the canonical block of the expert routed by
 * pick p = t*k + slot (the caller resolves idx to expert storage).  The expert
 * FFNs of the T*k picks are independent and run in parallel; the sums over slots
 * run in the fixed order above.  act selects the gate activation (k3o_expert_ffn). */
void k3o_moe(int T, int d, int f, int k, const uint16_t* x, const double* w, const uint8_t* const* pick_nib,
             const uint8_t* const* pick_scl, double* y, double* sumabs, int act) {
  const int P = T * k;
  double* o = (double*)malloc(sizeof(double) * (size_t)P * d);
  double* a = (double*)malloc(sizeof(double) * (size_t)P * d);
#pragma omp parallel
  {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int p = 0; p < P; ++p) {
      const int t = p / k;
      for (int j = 0; j < d; ++j) xt[j] = k3o_bf16(x[(size_t)t * d + j]);
      k3o_expert_ffn(d, f, pick_nib[p], pick_scl[p], xt, NULL, o + (size_t)p * d, a + (size_t)p * d, act);
    }
    free(xt);
  }
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < d; ++i) {
      double acc = 0.0, mag = 0.0;
      for (int slot = 0; slot < k; ++slot) {
        const size_t p = (size_t)t * k + slot;
        acc += w[p] * o[p * d + i];
        mag += fabs(w[p]) * a[p * d + i];
      }
      y[(size_t)t * d + i] = acc;
      sumabs[(size_t)t * d + i] = mag;
    }
  free(o);
  free(a);
}

/* ------------------------------------------------- glue between layers ---- */

/* Round a float to bf16, to nearest with ties to even, by its definition: keep the upper
 * 16 bits of the binary32 pattern, adding one unit of the kept part when the dropped 16
 * bits exceed half a unit, or equal half a unit and the kept part is odd.  NaN stays NaN. */
uint16_t k3o_bf16_rne(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t keep = u >> 16, drop = u & 0xffffu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1;
  return (uint16_t)keep;
}

/* Residual and pre-norm between stacked layers (the layer's output excludes the residual).
 * READING: the stacked-layer workload adds each layer's output to its input,
 *   x_next = bf16_rne(x + y), the sum taken in binary32 (the precision the kernel rounds
 *   from; the result is an integer code, so both sides decide it in the same precision);
 * and, as a transformer block does before its MoE ([EX] names the engine's RMSNorm), feeds
 * the next layer the weightless RMSNorm of x_next:
 *   x_norm = bf16_rne( x_next / sqrt( (1/d) * sum_j x_next_j^2 + eps ) ), in fp64. */
void k3o_residual_rmsnorm(int T, int d, const float* y, const uint16_t* x, double eps, uint16_t* x_next,
                          uint16_t* x_norm) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int j = 0; j < d; ++j) {
      const float sum = (float)k3o_bf16(x[(size_t)t * d + j]) + y[(size_t)t * d + j];
      const uint16_t r = k3o_bf16_rne(sum);
      x_next[(size_t)t * d + j] = r;
      const double rv = k3o_bf16(r);
      ss += rv * rv;
    }
    const double inv = 1.0 / sqrt(ss / d + eps);
    for (int j = 0; j < d; ++j)
      x_norm[(size_t)t * d + j] = k3o_bf16_rne((float)(k3o_bf16(x_next[(size_t)t * d + j]) * inv));
  }
}

/* ---------------------------------------------------------------- threads ---- */

int k3o_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void k3o_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
