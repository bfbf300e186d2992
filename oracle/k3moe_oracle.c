/*
 * k3moe_oracle.c -- plain CPU oracle for one Kimi-K3 Stable LatentMoE
 * routed-expert layer (router -> down_proj -> MXFP4 experts with SiTU-GLU ->
 * score-weighted combine -> RMSNorm -> up_proj).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file;
 * only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code with the CUDA path.
 *
 * Arithmetic is fp64 except where the method fixes another type:
 *   - tensors that cross between the layer's operations are bf16 (the model
 *     stores everything except the routed experts in bf16), so lat, h, n and
 *     y are rounded to bf16 (round to nearest even) at those points;
 *   - the routing decision is taken on fp32 keys (the precision the GPU
 *     router uses), and the routing weights are fp32 values;
 *   - SiTU-GLU is evaluated in fp64 (the model card asks for at least fp32).
 * Loops run in the order the formulas are written; no blocking or fusion.
 *
 * Sources (web pages on Kimi-K3, cited by page title and section):
 *   [kimi-k3-mlx README]  "Architecture" table: 896 routed experts, top-16,
 *       sigmoid router with aux-loss-free e_score_correction_bias; Stable
 *       LatentMoE runs experts in a 3584-d latent: down_proj -> experts ->
 *       RMSNorm -> up_proj; activation SiTU-GLU
 *       beta*tanh(g/beta)*sigmoid(g) * beta_lin*tanh(u/beta_lin), beta=4,
 *       beta_lin=25; source format MXFP4 (weight_packed u8 + e8m0
 *       weight_scale, group 32).
 *   [kimi-k3-mlx README] "Porting notes" item 1: SiTU-GLU computed in fp32.
 *   [kimi-k3-mlx README] "Tiers": MLX mxfp4 uses the identical encoding,
 *       low-bits-first codes and e8m0 scales.
 *   [kimi-k3-mlx README] "REAP" caveat: RMSNorm is applied to the combined
 *       expert output before up_proj.
 *   [K3_ARTIFACT_AUDIT] section 4.3: w1/w3 packed [3072,1792] U8 with scale
 *       [3072,112]; w2 packed [3584,1536] with scale [3584,96]; group 32.
 *   [K3_ARTIFACT_AUDIT] section 6: router weight [896,7168] bf16 and an fp32
 *       correction bias [896] per MoE layer.
 *   [kimi-k3-mlx README] "Architecture" table: 2 shared experts on every
 *       token; "Porting notes" item 3: the shared experts act on the residual,
 *       not the latent; "Parameter budget": 12.2 B shared-expert parameters
 *       (92 MoE layers x 3 x 7168 x 6144, i.e. two experts of intermediate
 *       3072).  Reading: each shared expert is a bf16 SiTU-GLU MLP; the two
 *       are summed (one MLP over their concatenated intermediate), rounded
 *       to bf16 once, and added to the routed branch's bf16 output.
 * Readings where the pages are silent (w1 = gate, w3 = up; bias used for
 * selection only; optional renormalisation and routed scaling factor; ties
 * to the lower expert id; OCP e2m1/e8m0 value tables) are the ones listed
 * in the design notes of this repository.
 *
 * Parity pins: see tests/test_oracle_pins.py (brute-force dequant against
 * an integer formula, SiTU-GLU limits, sort-based top-k, a dense all-expert
 * masked sum, work-count figures printed on the pages).  The whole layer
 * has no worked example on the pages, so the end-to-end value itself is
 * pinned only through those component checks.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int hidden, latent, n_experts, top_k, inter, group;
  double beta, beta_lin, rms_eps, routed_scaling;
  int norm_topk;
  int n_shared, shared_inter; /* shared experts (0 = none) and each one's intermediate */
  int bank2_begin;            /* 0: one bank; else experts >= bank2_begin are 2-bit affine */
} ora_dims;

/* Host arrays in checkpoint layout (experts stacked along dim 0). */
typedef struct {
  const uint16_t* router_w;   /* [E,H] bf16 */
  const float* router_bias;   /* [E] f32 */
  const uint16_t* down_proj;  /* [L,H] bf16 */
  const uint8_t* w1_packed;   /* [E,I,L/2] gate */
  const uint8_t* w1_scale;    /* [E,I,L/32] */
  const uint8_t* w3_packed;   /* [E,I,L/2] up */
  const uint8_t* w3_scale;    /* [E,I,L/32] */
  const uint8_t* w2_packed;   /* [E,L,I/2] down */
  const uint8_t* w2_scale;    /* [E,L,I/32] */
  const uint16_t* norm_w;     /* [L] bf16 */
  const uint16_t* up_proj;    /* [H,L] bf16 */
  /* shared experts, bf16, Is = n_shared * shared_inter (expert s owns
   * intermediate rows [s*shared_inter, (s+1)*shared_inter)) */
  const uint16_t* shared_w1;  /* [Is,H] gate */
  const uint16_t* shared_w3;  /* [Is,H] up */
  const uint16_t* shared_w2;  /* [H,Is] down */
  /* second bank (experts e >= bank2_begin, stored at index e - bank2_begin;
   * the MXFP4 tensors above then hold experts [0, bank2_begin) only):
   * 2-bit codes, four per byte, element j in bits 2(j%4)..2(j%4)+1 of byte
   * j/4; one bf16 scale and one bf16 bias per 64 elements of a row */
  const uint8_t* b2_w1q;      /* [E2,I,L/4] */
  const uint16_t* b2_w1s;     /* [E2,I,L/64] */
  const uint16_t* b2_w1b;     /* [E2,I,L/64] */
  const uint8_t* b2_w3q;
  const uint16_t* b2_w3s;
  const uint16_t* b2_w3b;
  const uint8_t* b2_w2q;      /* [E2,L,I/4] */
  const uint16_t* b2_w2s;     /* [E2,L,I/64] */
  const uint16_t* b2_w2b;
} ora_weights;

/* ------------------------------------------------------------------ */
/* bf16 <-> double                                                      */
/* ------------------------------------------------------------------ */

double ora_bf16_to_double(uint16_t b) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)b << 16;
  return (double)c.f;
}

/* Round a double to the nearest bf16 (ties to even), with overflow to
 * infinity and gradual underflow, directly from the double (no detour
 * through float, which could round twice). */
uint16_t ora_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);       /* a in [2^(e-1), 2^e) */
  int E = e - 1;      /* a in [2^E, 2^(E+1)) */
  if (E < -126) E = -126; /* below the normal range the spacing is 2^-133 */
  double ulp = ldexp(1.0, E - 7);
  double q = nearbyint(a / ulp); /* exact scaling; default mode rounds to even */
  double r = q * ulp;
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
  if (r < ldexp(1.0, -126)) return sign | (uint16_t)(r / ldexp(1.0, -133));
  int e2;
  double f = frexp(r, &e2); /* r = f * 2^e2, f in [0.5, 1) */
  uint16_t biased = (uint16_t)(e2 - 1 + 127);
  uint16_t mant = (uint16_t)((f * 2.0 - 1.0) * 128.0);
  return sign | (uint16_t)(biased << 7) | mant;
}

/* ------------------------------------------------------------------ */
/* MXFP4 decoding (OCP MX: e2m1 elements, e8m0 shared scale per 32)     */
/* ------------------------------------------------------------------ */

/* e2m1: bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa.
 * Exponent field 0 encodes the subnormal 0.5*m; no inf or NaN codes. */
double ora_e2m1_value(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* e8m0: an unsigned biased exponent, 2^(S-127); 0xFF is NaN. */
double ora_e8m0_value(unsigned S) {
  if (S == 255u) return NAN;
  return ldexp(1.0, (int)S - 127);
}

/* Element j of one packed row (cols elements): byte j/2 holds elements
 * 2i (low nibble) and 2i+1 (high nibble) -- "low bits first".  The scale
 * of group j/32 multiplies it. */
double ora_mxfp4_element(const uint8_t* packed_row, const uint8_t* scale_row, int j) {
  uint8_t byte = packed_row[j / 2];
  unsigned code = (j % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
  return ora_e2m1_value(code) * ora_e8m0_value(scale_row[j / 32]);
}

/* Second-bank weights (kimi-k3-mlx README, "REAP expert pruning", graded
 * mode: the top experts keep MXFP4, the middle ones go to a lower bit
 * width, in a second bank of the two-bank SwitchGLU; "Tiers": the 2-bit
 * tier stores experts at 2.50 bits per weight).  Reading: MLX affine 2-bit
 * quantisation with group 64 and a bf16 scale and bias per group (2 + 32/64
 * bits per weight), w = scale * q + bias, q in {0, 1, 2, 3}, codes packed
 * low bits first. */
double ora_affine2_element(const uint8_t* q_row, const uint16_t* s_row, const uint16_t* b_row, int j) {
  unsigned q = (q_row[j / 4] >> (2 * (j % 4))) & 3u;
  return ora_bf16_to_double(s_row[j / 64]) * (double)q + ora_bf16_to_double(b_row[j / 64]);
}

/* Dequantise a [rows, cols] MXFP4 matrix to bf16 bits (IEEE rounding of
 * the exact product, so values that overflow bf16 become infinities). */
void ora_mxfp4_dequant_bf16(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                            uint16_t* out) {
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < cols; ++j)
      out[(size_t)r * cols + j] = ora_bf16_from_double(
          ora_mxfp4_element(packed + (size_t)r * (cols / 2), scale + (size_t)r * (cols / 32), j));
}

/* ------------------------------------------------------------------ */
/* SiTU-GLU                                                             */
/* ------------------------------------------------------------------ */

double ora_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

double ora_situ_glu(double g, double u, double beta, double beta_lin) {
  return beta * tanh(g / beta) * ora_sigmoid(g) * beta_lin * tanh(u / beta_lin);
}

/* ------------------------------------------------------------------ */
/* Router: sigmoid scores, bias for selection only, top-K               */
/* ------------------------------------------------------------------ */

/* logits[e] = x . Wr[e] accumulated in fp64, then rounded to fp32 (the
 * routing decision is taken on fp32 keys). */
void ora_router_logits(const ora_dims* d, const uint16_t* x, const uint16_t* router_w,
                       float* logits) {
  for (int e = 0; e < d->n_experts; ++e) {
    double acc = 0.0;
    for (int h = 0; h < d->hidden; ++h)
      acc += ora_bf16_to_double(x[h]) * ora_bf16_to_double(router_w[(size_t)e * d->hidden + h]);
    logits[e] = (float)acc;
  }
}

/* From fp32 logits: s = sigmoid(logit) (fp32), key = s + bias (fp32 add),
 * select the K largest keys one at a time (ties to the lower expert id),
 * weights from the unbiased s, renormalised when norm_topk, times the
 * routed scaling factor, stored as fp32. */
void ora_route_from_logits(const ora_dims* d, const float* logits, const float* bias,
                           int32_t* idx, float* w, float* scores_out) {
  int E = d->n_experts, K = d->top_k;
  float* s = (float*)malloc(sizeof(float) * E);
  float* key = (float*)malloc(sizeof(float) * E);
  char* taken = (char*)calloc(E, 1);
  for (int e = 0; e < E; ++e) {
    s[e] = (float)ora_sigmoid((double)logits[e]);
    key[e] = s[e] + bias[e];
    if (scores_out) scores_out[e] = s[e];
  }
  for (int k = 0; k < K; ++k) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || key[e] > key[best]) best = e;
    }
    idx[k] = best;
    taken[best] = 1;
  }
  double sum = 0.0;
  for (int k = 0; k < K; ++k) sum += (double)s[idx[k]];
  for (int k = 0; k < K; ++k) {
    double wk = d->norm_topk ? (double)s[idx[k]] / sum : (double)s[idx[k]];
    w[k] = (float)(wk * d->routed_scaling);
  }
  free(s);
  free(key);
  free(taken);
}

/* ------------------------------------------------------------------ */
/* One token through the layer                                          */
/* ------------------------------------------------------------------ */

typedef struct {
  float* logits;     /* [E]      optional */
  uint16_t* lat;     /* [L]      optional */
  uint16_t* h;       /* [K, I]   optional, per selected expert in k order */
  double* o;         /* [K, L]   optional */
  double* c;         /* [L]      optional */
  uint16_t* n;       /* [L]      optional */
  uint16_t* hs;      /* [Is]     optional, shared experts' SiTU-GLU output */
  uint16_t* z;       /* [H]      optional, shared experts' output */
} ora_token_probe;

static void ora_forward_token(const ora_dims* d, const ora_weights* W, const uint16_t* x,
                              uint16_t* y, int32_t* idx, float* w, const ora_token_probe* p) {
  const int H = d->hidden, L = d->latent, E = d->n_experts, K = d->top_k, I = d->inter;
  float* logits = (float*)malloc(sizeof(float) * E);
  uint16_t* lat = (uint16_t*)malloc(sizeof(uint16_t) * L);
  uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * I);
  double* c = (double*)calloc(L, sizeof(double));
  uint16_t* n = (uint16_t*)malloc(sizeof(uint16_t) * L);

  /* 1. router */
  ora_router_logits(d, x, W->router_w, logits);
  ora_route_from_logits(d, logits, W->router_bias, idx, w, NULL);

  /* 2. latent down_proj: lat = bf16(Wd . x) */
  for (int l = 0; l < L; ++l) {
    double acc = 0.0;
    for (int j = 0; j < H; ++j)
      acc += ora_bf16_to_double(W->down_proj[(size_t)l * H + j]) * ora_bf16_to_double(x[j]);
    lat[l] = ora_bf16_from_double(acc);
  }

  /* 3. experts, combined in k order */
  for (int k = 0; k < K; ++k) {
    int e = idx[k];
    if (d->bank2_begin > 0 && e >= d->bank2_begin) {
      /* the second bank: 2-bit affine weights, the same arithmetic */
      const int e2 = e - d->bank2_begin;
      const uint8_t* w1q = W->b2_w1q + (size_t)e2 * I * (L / 4);
      const uint16_t* w1s = W->b2_w1s + (size_t)e2 * I * (L / 64);
      const uint16_t* w1b = W->b2_w1b + (size_t)e2 * I * (L / 64);
      const uint8_t* w3q = W->b2_w3q + (size_t)e2 * I * (L / 4);
      const uint16_t* w3s = W->b2_w3s + (size_t)e2 * I * (L / 64);
      const uint16_t* w3b = W->b2_w3b + (size_t)e2 * I * (L / 64);
      const uint8_t* w2q = W->b2_w2q + (size_t)e2 * L * (I / 4);
      const uint16_t* w2s = W->b2_w2s + (size_t)e2 * L * (I / 64);
      const uint16_t* w2b = W->b2_w2b + (size_t)e2 * L * (I / 64);
      for (int j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        for (int l = 0; l < L; ++l) {
          double a = ora_bf16_to_double(lat[l]);
          g += ora_affine2_element(w1q + (size_t)j * (L / 4), w1s + (size_t)j * (L / 64),
                                   w1b + (size_t)j * (L / 64), l) * a;
          u += ora_affine2_element(w3q + (size_t)j * (L / 4), w3s + (size_t)j * (L / 64),
                                   w3b + (size_t)j * (L / 64), l) * a;
        }
        h[j] = ora_bf16_from_double(ora_situ_glu(g, u, d->beta, d->beta_lin));
        if (p && p->h) p->h[(size_t)k * I + j] = h[j];
      }
      for (int l = 0; l < L; ++l) {
        double o = 0.0;
        for (int j = 0; j < I; ++j)
          o += ora_affine2_element(w2q + (size_t)l * (I / 4), w2s + (size_t)l * (I / 64),
                                   w2b + (size_t)l * (I / 64), j) * ora_bf16_to_double(h[j]);
        if (p && p->o) p->o[(size_t)k * L + l] = o;
        c[l] += (double)w[k] * o;
      }
      continue;
    }
    const uint8_t* w1p = W->w1_packed + (size_t)e * I * (L / 2);
    const uint8_t* w1s = W->w1_scale + (size_t)e * I * (L / 32);
    const uint8_t* w3p = W->w3_packed + (size_t)e * I * (L / 2);
    const uint8_t* w3s = W->w3_scale + (size_t)e * I * (L / 32);
    const uint8_t* w2p = W->w2_packed + (size_t)e * L * (I / 2);
    const uint8_t* w2s = W->w2_scale + (size_t)e * L * (I / 32);
    for (int j = 0; j < I; ++j) {
      double g = 0.0, u = 0.0;
      for (int l = 0; l < L; ++l) {
        double a = ora_bf16_to_double(lat[l]);
        g += ora_mxfp4_element(w1p + (size_t)j * (L / 2), w1s + (size_t)j * (L / 32), l) * a;
        u += ora_mxfp4_element(w3p + (size_t)j * (L / 2), w3s + (size_t)j * (L / 32), l) * a;
      }
      h[j] = ora_bf16_from_double(ora_situ_glu(g, u, d->beta, d->beta_lin));
      if (p && p->h) p->h[(size_t)k * I + j] = h[j];
    }
    for (int l = 0; l < L; ++l) {
      double o = 0.0;
      for (int j = 0; j < I; ++j)
        o += ora_mxfp4_element(w2p + (size_t)l * (I / 2), w2s + (size_t)l * (I / 32), j) *
             ora_bf16_to_double(h[j]);
      if (p && p->o) p->o[(size_t)k * L + l] = o;
      c[l] += (double)w[k] * o;
    }
  }

  /* 4. RMSNorm over the combined latent */
  double ms = 0.0;
  for (int l = 0; l < L; ++l) ms += c[l] * c[l];
  ms /= (double)L;
  double inv = 1.0 / sqrt(ms + d->rms_eps);
  for (int l = 0; l < L; ++l)
    n[l] = ora_bf16_from_double(c[l] * inv * ora_bf16_to_double(W->norm_w[l]));

  /* 5. latent up_proj: y = bf16(Wu . n) */
  for (int j = 0; j < H; ++j) {
    double acc = 0.0;
    for (int l = 0; l < L; ++l)
      acc += ora_bf16_to_double(W->up_proj[(size_t)j * L + l]) * ora_bf16_to_double(n[l]);
    y[j] = ora_bf16_from_double(acc);
  }

  /* 6. shared experts, on the 7168-d residual x itself (not the latent):
   *    each is a SiTU-GLU MLP; their sum is one MLP over the concatenated
   *    intermediate, gs = W1s . x, us = W3s . x, hs = bf16(SiTU(gs, us)),
   *    z = bf16(W2s . hs); the block output is y = bf16(y_routed + z). */
  if (d->n_shared > 0) {
    const int Is = d->n_shared * d->shared_inter;
    uint16_t* hs = (uint16_t*)malloc(sizeof(uint16_t) * Is);
    for (int j = 0; j < Is; ++j) {
      double gs = 0.0, us = 0.0;
      for (int i = 0; i < H; ++i) {
        double a = ora_bf16_to_double(x[i]);
        gs += ora_bf16_to_double(W->shared_w1[(size_t)j * H + i]) * a;
        us += ora_bf16_to_double(W->shared_w3[(size_t)j * H + i]) * a;
      }
      hs[j] = ora_bf16_from_double(ora_situ_glu(gs, us, d->beta, d->beta_lin));
    }
    for (int i = 0; i < H; ++i) {
      double acc = 0.0;
      for (int j = 0; j < Is; ++j)
        acc += ora_bf16_to_double(W->shared_w2[(size_t)i * Is + j]) * ora_bf16_to_double(hs[j]);
      uint16_t z = ora_bf16_from_double(acc);
      if (p && p->z) p->z[i] = z;
      y[i] = ora_bf16_from_double(ora_bf16_to_double(y[i]) + ora_bf16_to_double(z));
    }
    if (p && p->hs) memcpy(p->hs, hs, sizeof(uint16_t) * Is);
    free(hs);
  }

  if (p) {
    if (p->logits) memcpy(p->logits, logits, sizeof(float) * E);
    if (p->lat) memcpy(p->lat, lat, sizeof(uint16_t) * L);
    if (p->c) memcpy(p->c, c, sizeof(double) * L);
    if (p->n) memcpy(p->n, n, sizeof(uint16_t) * L);
  }
  free(logits);
  free(lat);
  free(h);
  free(c);
  free(n);
}

/* T tokens; tokens are independent, so they are spread over threads.
 * Optional per-token outputs are strided by token (NULL to skip):
 *   logits [T,E] f32, lat [T,L] bf16, h [T,K,I] bf16, o [T,K,L] f64,
 *   c [T,L] f64, n [T,L] bf16, hs [T,Is] bf16, z [T,H] bf16. */
void ora_forward(const ora_dims* d, const ora_weights* W, const uint16_t* x, int T, uint16_t* y,
                 int32_t* idx, float* w, float* logits, uint16_t* lat, uint16_t* h, double* o,
                 double* c, uint16_t* n, uint16_t* hs, uint16_t* z) {
  const int H = d->hidden, L = d->latent, E = d->n_experts, K = d->top_k, I = d->inter;
  const int Is = d->n_shared * d->shared_inter;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    ora_token_probe p;
    p.logits = logits ? logits + (size_t)t * E : NULL;
    p.lat = lat ? lat + (size_t)t * L : NULL;
    p.h = h ? h + (size_t)t * K * I : NULL;
    p.o = o ? o + (size_t)t * K * L : NULL;
    p.c = c ? c + (size_t)t * L : NULL;
    p.n = n ? n + (size_t)t * L : NULL;
    p.hs = hs ? hs + (size_t)t * Is : NULL;
    p.z = z ? z + (size_t)t * H : NULL;
    ora_forward_token(d, W, x + (size_t)t * H, y + (size_t)t * H, idx + (size_t)t * K,
                      w + (size_t)t * K, &p);
  }
}

/* Router only, for T tokens (used to measure the K-th/(K+1)-th key gap of
 * candidate inputs).  keys_top_out receives, per token, the K+1 largest
 * keys (s + bias, fp32) in descending order; when K == E there is no
 * (K+1)-th key and its slot holds -inf, so the gap is +inf. */
void ora_route(const ora_dims* d, const uint16_t* x, int T, const uint16_t* router_w,
               const float* bias, int32_t* idx, float* w, float* logits_out,
               float* keys_top_out) {
  const int H = d->hidden, E = d->n_experts, K = d->top_k;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    float* logits = (float*)malloc(sizeof(float) * E);
    float* s = (float*)malloc(sizeof(float) * E);
    ora_router_logits(d, x + (size_t)t * H, router_w, logits);
    ora_route_from_logits(d, logits, bias, idx + (size_t)t * K, w + (size_t)t * K, s);
    if (logits_out) memcpy(logits_out + (size_t)t * E, logits, sizeof(float) * E);
    if (keys_top_out) {
      /* K+1 largest keys, descending (selection again, ties to lower id) */
      char* taken = (char*)calloc(E, 1);
      for (int k = 0; k <= K; ++k) {
        if (k >= E) {
          keys_top_out[(size_t)t * (K + 1) + k] = -INFINITY;
          continue;
        }
        int best = -1;
        for (int e = 0; e < E; ++e) {
          if (taken[e]) continue;
          float ke = s[e] + bias[e], kb = best < 0 ? 0.f : s[best] + bias[best];
          if (best < 0 || ke > kb) best = e;
        }
        taken[best] = 1;
        keys_top_out[(size_t)t * (K + 1) + k] = s[best] + bias[best];
      }
      free(taken);
    }
    free(logits);
    free(s);
  }
}

/* Expert parallelism (Kimi-K3-Alis-MLX-Dynamic model card, "Performance"
 * and "Usage": dense weights replicated, routed experts split between two
 * machines).  Rank r holds experts [e_begin, e_begin + e_count); for every
 * token it routes over all experts (the router is replicated) and forms the
 * partial combine
 *   c_r = sum over k in k order, for selected experts in its range, of w_k o_k
 * (fp64 here).  The ranks' partials are summed (one all-reduce of [T, L];
 * RMSNorm needs the whole combine), and ora_finish applies the rest of the
 * block to the sum: RMSNorm, up_proj and the shared experts on x. */
void ora_forward_partial(const ora_dims* d, const ora_weights* W, const uint16_t* x, int T, int e_begin,
                         int e_count, double* c_out) {
  const int H = d->hidden, L = d->latent, K = d->top_k;
  double* o = (double*)malloc(sizeof(double) * (size_t)K * L);
  uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * H);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * K);
  float* w = (float*)malloc(sizeof(float) * K);
  for (int t = 0; t < T; ++t) {
    ora_token_probe p;
    memset(&p, 0, sizeof(p));
    p.o = o;
    ora_forward_token(d, W, x + (size_t)t * H, y, idx, w, &p);
    double* c = c_out + (size_t)t * L;
    for (int l = 0; l < L; ++l) c[l] = 0.0;
    for (int k = 0; k < K; ++k) {
      if (idx[k] < e_begin || idx[k] >= e_begin + e_count) continue;
      for (int l = 0; l < L; ++l) c[l] += (double)w[k] * o[(size_t)k * L + l];
    }
  }
  free(o);
  free(y);
  free(idx);
  free(w);
}

/* The block after the combine, for a given combine c [T, L]: n = bf16(c /
 * sqrt(mean(c^2) + eps) * gamma), y = bf16(Wu . n), plus the shared experts
 * of x when the dims have them (steps 4-6 of the forward, restated here
 * for a c from outside). */
void ora_finish(const ora_dims* d, const ora_weights* W, const uint16_t* x, const double* c_in, int T,
                uint16_t* y_out) {
  const int H = d->hidden, L = d->latent;
  uint16_t* n = (uint16_t*)malloc(sizeof(uint16_t) * L);
  for (int t = 0; t < T; ++t) {
    const double* c = c_in + (size_t)t * L;
    uint16_t* y = y_out + (size_t)t * H;
    double ms = 0.0;
    for (int l = 0; l < L; ++l) ms += c[l] * c[l];
    ms /= (double)L;
    double inv = 1.0 / sqrt(ms + d->rms_eps);
    for (int l = 0; l < L; ++l) n[l] = ora_bf16_from_double(c[l] * inv * ora_bf16_to_double(W->norm_w[l]));
    for (int j = 0; j < H; ++j) {
      double acc = 0.0;
      for (int l = 0; l < L; ++l)
        acc += ora_bf16_to_double(W->up_proj[(size_t)j * L + l]) * ora_bf16_to_double(n[l]);
      y[j] = ora_bf16_from_double(acc);
    }
    if (d->n_shared > 0) {
      const int Is = d->n_shared * d->shared_inter;
      const uint16_t* xt = x + (size_t)t * H;
      uint16_t* hs = (uint16_t*)malloc(sizeof(uint16_t) * Is);
      for (int j = 0; j < Is; ++j) {
        double gs = 0.0, us = 0.0;
        for (int i = 0; i < H; ++i) {
          double a = ora_bf16_to_double(xt[i]);
          gs += ora_bf16_to_double(W->shared_w1[(size_t)j * H + i]) * a;
          us += ora_bf16_to_double(W->shared_w3[(size_t)j * H + i]) * a;
        }
        hs[j] = ora_bf16_from_double(ora_situ_glu(gs, us, d->beta, d->beta_lin));
      }
      for (int i = 0; i < H; ++i) {
        double acc = 0.0;
        for (int j = 0; j < Is; ++j)
          acc += ora_bf16_to_double(W->shared_w2[(size_t)i * Is + j]) * ora_bf16_to_double(hs[j]);
        y[i] = ora_bf16_from_double(ora_bf16_to_double(y[i]) + ora_bf16_to_double(ora_bf16_from_double(acc)));
      }
      free(hs);
    }
  }
  free(n);
}

/* REAP saliency over a calibration set of T tokens (kimi-k3-mlx README,
 * "REAP expert pruning": S_j = (1/|C|) sum over x in C of g_j(x) ||e_j(x)||_2,
 * g_j the router's gate value of expert j for token x -- zero when j is not
 * selected -- and e_j(x) the expert's output).  Reading: g_j is the routing
 * weight the combine uses (topk_w) and e_j(x) is the expert output o in the
 * 3584-d latent, before the combine; |C| = T.  S [E] receives the saliency
 * and S_sum [E] (optional) the undivided sums. */
void ora_reap_saliency(const ora_dims* d, const ora_weights* W, const uint16_t* x, int T, double* S,
                       double* S_sum) {
  const int H = d->hidden, L = d->latent, E = d->n_experts, K = d->top_k;
  double* acc = (double*)calloc(E, sizeof(double));
  double* o = (double*)malloc(sizeof(double) * (size_t)K * L);
  uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * H);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * K);
  float* w = (float*)malloc(sizeof(float) * K);
  for (int t = 0; t < T; ++t) {
    ora_token_probe p;
    memset(&p, 0, sizeof(p));
    p.o = o;
    ora_forward_token(d, W, x + (size_t)t * H, y, idx, w, &p);
    for (int k = 0; k < K; ++k) {
      double ss = 0.0;
      for (int l = 0; l < L; ++l) ss += o[(size_t)k * L + l] * o[(size_t)k * L + l];
      acc[idx[k]] += (double)w[k] * sqrt(ss);
    }
  }
  for (int e = 0; e < E; ++e) {
    if (S_sum) S_sum[e] = acc[e];
    S[e] = T > 0 ? acc[e] / (double)T : 0.0;
  }
  free(acc);
  free(o);
  free(y);
  free(idx);
  free(w);
}

/* Dense all-expert masked sum: the same layer written with every expert
 * evaluated for every token and a zero weight for unselected ones.  Used
 * only as an independent formulation in the oracle's own tests. */
void ora_forward_dense_masked(const ora_dims* d, const ora_weights* W, const uint16_t* x, int T,
                              double* c_out) {
  const int H = d->hidden, L = d->latent, E = d->n_experts, K = d->top_k, I = d->inter;
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + (size_t)t * H;
    float* logits = (float*)malloc(sizeof(float) * E);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * K);
    float* wk = (float*)malloc(sizeof(float) * K);
    double* gate = (double*)calloc(E, sizeof(double));
    uint16_t* lat = (uint16_t*)malloc(sizeof(uint16_t) * L);
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * I);
    ora_router_logits(d, xt, W->router_w, logits);
    ora_route_from_logits(d, logits, W->router_bias, idx, wk, NULL);
    for (int k = 0; k < K; ++k) gate[idx[k]] = (double)wk[k];
    for (int l = 0; l < L; ++l) {
      double acc = 0.0;
      for (int j = 0; j < H; ++j)
        acc += ora_bf16_to_double(W->down_proj[(size_t)l * H + j]) * ora_bf16_to_double(xt[j]);
      lat[l] = ora_bf16_from_double(acc);
    }
    double* c = c_out + (size_t)t * L;
    for (int l = 0; l < L; ++l) c[l] = 0.0;
    for (int e = 0; e < E; ++e) {
      for (int j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        for (int l = 0; l < L; ++l) {
          double a = ora_bf16_to_double(lat[l]);
          g += ora_mxfp4_element(W->w1_packed + ((size_t)e * I + j) * (L / 2),
                                 W->w1_scale + ((size_t)e * I + j) * (L / 32), l) * a;
          u += ora_mxfp4_element(W->w3_packed + ((size_t)e * I + j) * (L / 2),
                                 W->w3_scale + ((size_t)e * I + j) * (L / 32), l) * a;
        }
        h[j] = ora_bf16_from_double(ora_situ_glu(g, u, d->beta, d->beta_lin));
      }
      for (int l = 0; l < L; ++l) {
        double o = 0.0;
        for (int j = 0; j < I; ++j)
          o += ora_mxfp4_element(W->w2_packed + ((size_t)e * L + l) * (I / 2),
                                 W->w2_scale + ((size_t)e * L + l) * (I / 32), j) *
               ora_bf16_to_double(h[j]);
        c[l] += gate[e] * o;
      }
    }
    free(logits);
    free(idx);
    free(wk);
    free(gate);
    free(lat);
    free(h);
  }
}

int ora_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
