/*
 * moe_oracle.c -- CPU oracle for the fused mixture-of-experts expert layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference leg may load this library.  It shares
 * no code, header, table or constant with the CUDA path in
 * moe_expert_layer_02_gb300/ and neither side includes or links the other.
 *
 * What it is: the plain per-token definition of the layer,
 *
 *     out[t] = sum_j w[t,j] * FFN_{idx[t,j]}(x[t]) + FFN_shared(x[t])
 *
 * written one token at a time, with every rounding step that the method itself
 * contains (per-token fp8 activation quantisation, bf16 intermediate, per-row
 * fp8 requantisation, bf16 output) emulated exactly and everything else done in
 * fp64.  Sources (page title, section):
 *   [LING]  "Optimising Ling-2.6-1T on TPU with SGLang-JAX" (Fused MoE V2 kernel):
 *           s.1 cost model (scatter -> local expert FFN -> gather; top-8 + shared),
 *           s.5 "per-channel direct_scaled_dot" (out[m,n] = (sum_k A W) * scale[n]),
 *           s.5 "activation quantisation" (dynamic per-token fp8 before scatter),
 *           s.5 "in-kernel shared expert" (dense FFN on every local token).
 *   [K3]    "Kimi K3 on the Google TPU ecosystem: feasibility analysis":
 *           s.2.4 LatentMoE block (down_proj -> experts -> RMSNorm -> up_proj,
 *           shared expert on the raw hidden; renormalised top-k),
 *           s.2.5 MXFP4 (e2m1 values, one e8m0 scale per 32 elements).
 *   [GAP]   "Implementation gaps: advanced optimisations" (sglang-jax reference),
 *           s.4 MXFP4 (two e2m1 values packed per uint8, shared e8m0 scale).
 *   Formats: OCP 8-bit floating point spec (E4M3FN) and OCP Microscaling
 *   Formats v1.0 (E2M1, E8M0).
 *
 * Readings where the pages are silent:
 *   - router logits are fp32 in one canonical order (32 strided fma chains,
 *     then a halving tree), so that top-k can be compared bit-exactly;
 *   - top-k ties go to the lower expert index; weights are the softmax over the
 *     k chosen logits (== softmax over all E, top-k, renormalise);
 *   - per-token scale s = amax/448 in fp32 (s = 1 when amax == 0); codes are
 *     e4m3(RNE, saturating) of the fp32 quotient x/s;
 *   - activation is SwiGLU, h = bf16(silu(g) * u); with act = SiTU it is
 *     h = bf16(beta * tanh(g / beta) * sigmoid(g) * u), beta = 4 [K3 s.2.6];
 *   - sigmoid routing (K3's noaux_tc, s.2.4, ungrouped, scaling factor 1):
 *     score s_e = sigmoid(logit_e), experts chosen by s_e + bias_e (the bias
 *     steers selection only), weights s_j / sum_j' s_j'.  The selection takes
 *     sigmoid in one canonical fp32 sequence (below) so that it is exact;
 *   - h is requantised per routed row to fp8 the same way as x;
 *   - the shared expert has no gate (weight 1);
 *   - LatentMoE: router on the hidden x, z = bf16(x Wd^T) quantised per token,
 *     RMSNorm (eps 1e-6, gamma given) after the routed combine, normed latent
 *     rounded to bf16, out = bf16(yn Wu^T + shared(x)); shared expert in bf16.
 *
 * Dot products of decoded fp8 (and fp8 x e2m1) values are summed in fp64; for
 * e4m3 x e4m3 every product is a multiple of 2^-18 below 2^18, so sums of up to
 * 2^13 of them are exact in fp64: the oracle's contraction is the exact one.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* Number formats                                                              */
/* ------------------------------------------------------------------------- */

/* E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa; no infinities; S.1111.111 is
 * NaN; exponent field 0 is subnormal with value m/8 * 2^-6.  Largest finite 448. */
double orc_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating to +-448 (the
 * "satfinite" convention: out-of-range finite and infinite inputs clamp). */
uint8_t orc_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a == 0.0) return sign;
  if (isinf(a) || a >= 448.0) return sign | 0x7E;
  int E;
  frexp(a, &E);       /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;      /* 2^e <= a < 2^(e+1) */
  if (e < -6) e = -6; /* below the normal range the spacing stays 2^-9 */
  double q = ldexp(1.0, e - 3);
  double n = rint(a / q); /* a/q is exact; rint rounds half to even */
  double val = n * q;
  if (val > 448.0) val = 448.0;
  if (val == 0.0) return sign;
  if (val < ldexp(1.0, -6)) return sign | (uint8_t)(val / ldexp(1.0, -9));
  frexp(val, &E);
  int e2 = E - 1;
  int m = (int)((val / ldexp(1.0, e2) - 1.0) * 8.0);
  return sign | (uint8_t)(((e2 + 7) << 3) | m);
}

/* bfloat16: the upper half of an IEEE binary32. */
double orc_bf16_decode(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double straight to bfloat16, nearest-even (no intermediate fp32). */
uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
  double a = fabs(v);
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int E;
  frexp(a, &E);
  int e = E - 1;
  if (e < -126) e = -126;
  double q = ldexp(1.0, e - 7);
  double val = rint(a / q) * q;
  if (val >= ldexp(1.0, 128)) return sign | 0x7F80;
  if (val < ldexp(1.0, -126)) return sign | (uint16_t)(val / ldexp(1.0, -133));
  frexp(val, &E);
  int e2 = E - 1;
  int m = (int)((val / ldexp(1.0, e2) - 1.0) * 128.0);
  return sign | (uint16_t)(((e2 + 127) << 7) | m);
}

/* E2M1 (OCP MX): 1 sign, 2 exponent (bias 1), 1 mantissa; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Low nibble of a packed byte = even index. */
double orc_e2m1_decode(uint8_t nib) {
  int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* E8M0 (OCP MX): unsigned exponent, value 2^(s-127); 0xFF is NaN. */
double orc_e8m0_decode(uint8_t s) {
  if (s == 0xFF) return NAN;
  return ldexp(1.0, (int)s - 127);
}

void orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_encode(v[i]);
}
void orc_bf16_from_double_array(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_bf16_from_double(v[i]);
}

/* ------------------------------------------------------------------------- */
/* A minimal pthread parallel-for over [0, n).                                 */
/* ------------------------------------------------------------------------- */
typedef void (*orc_body)(int64_t i, void* ctx);
typedef struct {
  orc_body body;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} orc_pool;

static void* orc_worker(void* arg) {
  orc_pool* p = (orc_pool*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t i = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (i >= p->n) break;
    p->body(i, p->ctx);
  }
  return NULL;
}

static void orc_parallel_for(int64_t n, int nthreads, orc_body body, void* ctx) {
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  orc_pool p = {body, ctx, n, 0, PTHREAD_MUTEX_INITIALIZER};
  if (nthreads == 1) {
    orc_worker(&p);
    return;
  }
  pthread_t th[256];
  for (int i = 0; i < nthreads; i++) pthread_create(&th[i], NULL, orc_worker, &p);
  for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
}

int orc_default_threads(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* ------------------------------------------------------------------------- */
/* S1: router logits (fp32, canonical order)                                   */
/* ------------------------------------------------------------------------- */

/* logit[e] = sum_h float(x[h]) * wr[e,h] (+ bias[e]).  Canonical order: 32
 * partial sums, partial l takes h = l, l+32, l+64, ... ascending through fmaf
 * starting from +0; then p_l += p_{l+off} for off = 16, 8, 4, 2, 1; the logit is
 * p_0, plus bias[e] as one fp32 add.  [LING s.6: routing metadata] */
static float router_logit_one(int64_t H, const uint16_t* xrow, const float* wrow) {
  float p[32];
  for (int l = 0; l < 32; l++) p[l] = 0.0f;
  int64_t h0 = 0;
  for (; h0 + 32 <= H; h0 += 32)
    for (int l = 0; l < 32; l++) p[l] = fmaf(bf16_to_float(xrow[h0 + l]), wrow[h0 + l], p[l]);
  for (int l = 0; h0 + l < H; l++) p[l] = fmaf(bf16_to_float(xrow[h0 + l]), wrow[h0 + l], p[l]);
  for (int off = 16; off >= 1; off >>= 1)
    for (int l = 0; l < off; l++) p[l] = p[l] + p[l + off];
  return p[0];
}

static void router_row(int64_t H, int64_t E, const uint16_t* xrow, const float* wr,
                       const float* bias, float* out) {
  for (int64_t e = 0; e < E; e++) {
    float v = router_logit_one(H, xrow, wr + e * H);
    if (bias) v = v + bias[e];
    out[e] = v;
  }
}

typedef struct {
  int64_t H, E;
  const uint16_t* x;
  const float* wr;
  const float* bias;
  float* logits;
} router_ctx;

static void router_body(int64_t t, void* c) {
  router_ctx* r = (router_ctx*)c;
  router_row(r->H, r->E, r->x + t * r->H, r->wr, r->bias, r->logits + t * r->E);
}

void orc_router_logits(int64_t T, int64_t H, int64_t E, const uint16_t* x, const float* wr,
                       const float* bias, float* logits, int nthreads) {
  router_ctx c = {H, E, x, wr, bias, logits};
  orc_parallel_for(T, nthreads, router_body, &c);
}

/* ------------------------------------------------------------------------- */
/* S2: top-k with renormalised softmax weights                                  */
/* ------------------------------------------------------------------------- */

/* Pick the k largest logits in descending order, ties to the lower index; the
 * weights are softmax over the chosen logits (identical to softmax over all E
 * followed by top-k and renormalisation, routed_scaling_factor 1).
 * [LING s.1 top-8 routing; K3 s.2.4 moe_renormalize] */
static void topk_row(int64_t E, int k, const float* l, int32_t* idx, double* w) {
  for (int j = 0; j < k; j++) {
    int64_t best = -1;
    for (int64_t e = 0; e < E; e++) {
      int taken = 0;
      for (int jj = 0; jj < j; jj++)
        if (idx[jj] == e) taken = 1;
      if (taken) continue;
      if (best < 0 || l[e] > l[best]) best = e;
    }
    idx[j] = (int32_t)best;
  }
  double m = (double)l[idx[0]], z = 0.0;
  for (int j = 0; j < k; j++) z += exp((double)l[idx[j]] - m);
  for (int j = 0; j < k; j++) w[j] = exp((double)l[idx[j]] - m) / z;
}

void orc_topk(int64_t T, int64_t E, int k, const float* logits, int32_t* idx, double* w) {
  for (int64_t t = 0; t < T; t++) topk_row(E, k, logits + t * E, idx + t * k, w + t * k);
}

/* Canonical fp32 exp(a) for a <= 0, written from the mathematics so that two
 * implementations following it agree bit for bit: Cody-Waite range reduction
 * a = n ln2 + r (n = rint(a log2 e), ln2 split into a 24-bit-exact head and a
 * tail, both products through fmaf), e^r by its Taylor series to r^7/7!
 * (Horner, fmaf; |r| <= 0.35 so the truncation is below 2^-26), then an exact
 * scaling by 2^n (n >= -125, so the result stays a normal number).  Inputs
 * at or below -86 (results below ~4.5e-38) give 0. */
float orc_exp_canon(float a) {
  if (!(a > -86.0f)) return 0.0f;
  if (a > 0.0f) a = 0.0f;
  const float log2e = 1.44269504f, ln2_hi = 0.693145751953125f, ln2_lo = 1.42860677e-6f;
  float n = rintf(a * log2e);
  float r = fmaf(-n, ln2_hi, a);
  r = fmaf(-n, ln2_lo, r);
  float q = 1.0f / 5040.0f;
  q = fmaf(q, r, 1.0f / 720.0f);
  q = fmaf(q, r, 1.0f / 120.0f);
  q = fmaf(q, r, 1.0f / 24.0f);
  q = fmaf(q, r, 1.0f / 6.0f);
  q = fmaf(q, r, 0.5f);
  q = fmaf(q, r, 1.0f);
  q = fmaf(q, r, 1.0f);
  union { uint32_t u; float f; } two = {(uint32_t)((int)n + 127) << 23};
  return q * two.f;
}

/* sigmoid(l) = 1 / (1 + e^-l) for l >= 0, e^l / (1 + e^l) for l < 0, with
 * u = orc_exp_canon(-|l|) and IEEE fp32 add and divide. */
float orc_sigmoid_canon(float l) {
  float u = orc_exp_canon(l >= 0.0f ? -l : l);
  return l >= 0.0f ? 1.0f / (1.0f + u) : u / (1.0f + u);
}

/* noaux_tc top-k: keys s_e + bias_e (fp32), k largest in descending order, ties
 * to the lower index; weights are the chosen (unbiased) scores renormalised.
 * [K3 s.2.4: noaux_tc + sigmoid, moe_renormalize, routed_scaling_factor 1] */
static void topk_sigmoid_row(int64_t E, int k, const float* l, const float* bias, int32_t* idx,
                             double* w) {
  float* key = (float*)malloc(sizeof(float) * (size_t)E);
  float* sc = (float*)malloc(sizeof(float) * (size_t)E);
  for (int64_t e = 0; e < E; e++) {
    sc[e] = orc_sigmoid_canon(l[e]);
    key[e] = bias ? sc[e] + bias[e] : sc[e];
  }
  for (int j = 0; j < k; j++) {
    int64_t best = -1;
    for (int64_t e = 0; e < E; e++) {
      int taken = 0;
      for (int jj = 0; jj < j; jj++)
        if (idx[jj] == e) taken = 1;
      if (taken) continue;
      if (best < 0 || key[e] > key[best]) best = e;
    }
    idx[j] = (int32_t)best;
  }
  double z = 0.0;
  for (int j = 0; j < k; j++) z += (double)sc[idx[j]];
  for (int j = 0; j < k; j++) w[j] = (double)sc[idx[j]] / z;
  free(key);
  free(sc);
}

void orc_topk_sigmoid(int64_t T, int64_t E, int k, const float* logits, const float* bias,
                      int32_t* idx, double* w) {
  for (int64_t t = 0; t < T; t++)
    topk_sigmoid_row(E, k, logits + t * E, bias, idx + t * k, w + t * k);
}

/* ------------------------------------------------------------------------- */
/* S3/S4: stable counting sort of (token, slot) pairs by expert                */
/* ------------------------------------------------------------------------- */

/* cnt[e] = #{(t,j): idx[t,j] = e}; off[e] = sum_{e'<e} cnt[e']; off[E] = T*k.
 * Row of (t,j) = off[e] + #{t' < t : e in idx[t']}; perm[t,j] = row, src[row] = t.
 * [LING s.6: per-expert counts/offsets and scatter/gather indices] */
void orc_permute(int64_t T, int64_t E, int k, const int32_t* idx, int32_t* cnt, int32_t* off,
                 int32_t* perm, int32_t* src) {
  for (int64_t e = 0; e < E; e++) cnt[e] = 0;
  for (int64_t i = 0; i < T * k; i++) cnt[idx[i]]++;
  off[0] = 0;
  for (int64_t e = 0; e < E; e++) off[e + 1] = off[e] + cnt[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int64_t e = 0; e < E; e++) fill[e] = off[e];
  for (int64_t t = 0; t < T; t++)
    for (int j = 0; j < k; j++) {
      int32_t e = idx[t * k + j];
      int32_t row = fill[e]++;
      perm[t * k + j] = row;
      src[row] = (int32_t)t;
    }
  free(fill);
}

/* Dynamic per-token fp8 quantisation [LING s.5 activation quantisation]:
 * s = amax_h |x[h]| / 448 (fp32; 1 when amax is 0), q[h] = e4m3(x[h] / s). */
static float quant_row(int64_t n, const float* v, uint8_t* q) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; i++) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int64_t i = 0; i < n; i++) q[i] = orc_e4m3_encode(v[i] / s);
  return s;
}

static float quant_row_bf16(int64_t n, const uint16_t* x, uint8_t* q) {
  float* v = (float*)malloc(sizeof(float) * (size_t)n);
  for (int64_t i = 0; i < n; i++) v[i] = bf16_to_float(x[i]);
  float s = quant_row(n, v, q);
  free(v);
  return s;
}

void orc_quant_rows(int64_t T, int64_t H, const uint16_t* x, float* scale, uint8_t* q) {
  for (int64_t t = 0; t < T; t++) scale[t] = quant_row_bf16(H, x + t * H, q + t * H);
}

/* ------------------------------------------------------------------------- */
/* S5/S6: one expert's SwiGLU FFN on one quantised row                         */
/* ------------------------------------------------------------------------- */

/* Weight formats.  FP8: w13 [2I, K] e4m3 bytes (rows 0..I-1 = W1 gate, I..2I-1
 * = W3 up), s13 [2I] fp32 per output channel; w2 [N, I] e4m3, s2 [N] fp32.
 * MXFP4: w13 [2I, K/2] packed e2m1 (low nibble = even k), s13 [2I, K/32] e8m0;
 * w2 [N, I/2], s2 [N, I/32].  K is the expert input width (H, or the latent
 * width L), N its output width (same as K). */
enum { ORC_FP8 = 0, ORC_MXFP4 = 1, ORC_FP8_BLOCK = 2 };
/* FP8_BLOCK (block-wise fp8, weight_block_size [128, 128], K3 report s.3.7):
 * w13 [2I, K] / w2 [N, I] e4m3 bytes as FP8, with one fp32 scale per 128 x 128
 * block, s13 [2I/128, K/128] and s2 [N/128, I/128]; a weight is
 * e4m3(q[n,k]) * s[n/128, k/128] and is applied inside the K-sum. */

/* Decode tables filled once from the decoders above (lookup instead of a call
 * per element; same values). */
static double tab_e4m3[256], tab_e2m1[16], tab_e8m0[256];
static pthread_once_t tab_once = PTHREAD_ONCE_INIT;
static void fill_tables(void) {
  for (int c = 0; c < 256; c++) {
    tab_e4m3[c] = orc_e4m3_decode((uint8_t)c);
    tab_e8m0[c] = orc_e8m0_decode((uint8_t)c);
  }
  for (int c = 0; c < 16; c++) tab_e2m1[c] = orc_e2m1_decode((uint8_t)c);
}

/* One weight value; srow is the row's scale row (MXFP4: e8m0 per 32 k;
 * FP8_BLOCK: fp32 per 128 k of the row's 128-row block; FP8: unused). */
static double weight_at(int fmt, const uint8_t* wrow, const void* srow, int64_t k) {
  if (fmt == ORC_FP8) return tab_e4m3[wrow[k]];
  if (fmt == ORC_FP8_BLOCK) return tab_e4m3[wrow[k]] * (double)((const float*)srow)[k / 128];
  uint8_t byte = wrow[k / 2];
  uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 15);
  return tab_e2m1[nib] * tab_e8m0[((const uint8_t*)srow)[k / 32]];
}

enum { ORC_SWIGLU = 0, ORC_SITU = 1 };

/* Gated activation times the up projection: SwiGLU silu(g) * u, or SiTU
 * beta * tanh(g / beta) * sigmoid(g) * u with beta = 4 [K3 s.2.6]. */
static double gated(int act, double g, double u) {
  if (act == ORC_SITU) return 4.0 * tanh(g / 4.0) / (1.0 + exp(-g)) * u;
  return g / (1.0 + exp(-g)) * u;
}

/* y[n] = (sum_i hq_i W2[n,i]) * s_h * s2[n] (fp8 also applies the per-channel
 * scale after the full-K sum, [LING s.5 direct_scaled_dot]); h = bf16(act(g, u))
 * with g = (sum_k xq_k W1[n,k]) * s_x * s1[n], u likewise with W3. */
static void expert_ffn(int fmt, int act, int64_t K, int64_t I, const uint8_t* xq, float sx,
                       const uint8_t* w13, const void* s13, const uint8_t* w2, const void* s2,
                       double* y, uint16_t* h_out, float* sh_out, uint8_t* hq_out) {
  int64_t rowb13 = (fmt == ORC_MXFP4) ? K / 2 : K, rows13 = (fmt == ORC_MXFP4) ? K / 32 : 0;
  int64_t rowb2 = (fmt == ORC_MXFP4) ? I / 2 : I, rows2 = (fmt == ORC_MXFP4) ? I / 32 : 0;
  double* xd = (double*)malloc(sizeof(double) * (size_t)K);
  float* hf = (float*)malloc(sizeof(float) * (size_t)I);
  uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
  uint8_t* hq = (uint8_t*)malloc((size_t)I);
  double* hd = (double*)malloc(sizeof(double) * (size_t)I);
  for (int64_t k = 0; k < K; k++) xd[k] = tab_e4m3[xq[k]];
  for (int64_t n = 0; n < I; n++) {
    const uint8_t* wg = w13 + n * rowb13;
    const uint8_t* wu = w13 + (I + n) * rowb13;
    const void *sg, *su;
    double ag = 0.0, au = 0.0;
    if (fmt == ORC_FP8) {
      sg = su = NULL;
    } else if (fmt == ORC_FP8_BLOCK) {
      sg = (const float*)s13 + (n / 128) * (K / 128);
      su = (const float*)s13 + ((I + n) / 128) * (K / 128);
    } else {
      sg = (const uint8_t*)s13 + n * rows13;
      su = (const uint8_t*)s13 + (I + n) * rows13;
    }
    for (int64_t k = 0; k < K; k++) {
      ag += xd[k] * weight_at(fmt, wg, sg, k);
      au += xd[k] * weight_at(fmt, wu, su, k);
    }
    double g = ag * (double)sx, u = au * (double)sx;
    if (fmt == ORC_FP8) {
      g *= (double)((const float*)s13)[n];
      u *= (double)((const float*)s13)[I + n];
    }
    hb[n] = orc_bf16_from_double(gated(act, g, u));
    hf[n] = bf16_to_float(hb[n]);
  }
  float s_h = quant_row(I, hf, hq);
  for (int64_t i = 0; i < I; i++) hd[i] = tab_e4m3[hq[i]];
  for (int64_t n = 0; n < K; n++) {
    const uint8_t* wr = w2 + n * rowb2;
    const void* sr = (fmt == ORC_FP8)         ? NULL
                     : (fmt == ORC_FP8_BLOCK) ? (const void*)((const float*)s2 + (n / 128) * (I / 128))
                                              : (const void*)((const uint8_t*)s2 + n * rows2);
    double acc = 0.0;
    for (int64_t i = 0; i < I; i++) acc += hd[i] * weight_at(fmt, wr, sr, i);
    double v = acc * (double)s_h;
    if (fmt == ORC_FP8) v *= (double)((const float*)s2)[n];
    y[n] = v;
  }
  if (h_out) memcpy(h_out, hb, sizeof(uint16_t) * (size_t)I);
  if (sh_out) *sh_out = s_h;
  if (hq_out) memcpy(hq_out, hq, (size_t)I);
  free(xd);
  free(hf);
  free(hb);
  free(hq);
  free(hd);
}

/* Shared expert with bf16 weights and bf16 activations (LatentMoE: shared
 * experts stay BF16 [K3 s.2.5]): sh = W2s * bf16(act(W1s x, W3s x)). */
static void shared_ffn_bf16(int act, int64_t H, int64_t Is, const uint16_t* xrow, const uint16_t* w13,
                            const uint16_t* w2, double* y) {
  double* xd = (double*)malloc(sizeof(double) * (size_t)H);
  double* hd = (double*)malloc(sizeof(double) * (size_t)Is);
  for (int64_t k = 0; k < H; k++) xd[k] = orc_bf16_decode(xrow[k]);
  for (int64_t n = 0; n < Is; n++) {
    double g = 0.0, u = 0.0;
    for (int64_t k = 0; k < H; k++) {
      g += xd[k] * orc_bf16_decode(w13[n * H + k]);
      u += xd[k] * orc_bf16_decode(w13[(Is + n) * H + k]);
    }
    hd[n] = orc_bf16_decode(orc_bf16_from_double(gated(act, g, u)));
  }
  for (int64_t m = 0; m < H; m++) {
    double acc = 0.0;
    for (int64_t i = 0; i < Is; i++) acc += hd[i] * orc_bf16_decode(w2[m * Is + i]);
    y[m] = acc;
  }
  free(xd);
  free(hd);
}

/* ------------------------------------------------------------------------- */
/* The whole layer, one token at a time                                        */
/* ------------------------------------------------------------------------- */
typedef struct {
  int64_t T, H, I, E, k, I_s, L; /* I_s = 0: no shared expert; L = 0: no latent */
  int32_t wfmt;                  /* ORC_FP8, ORC_MXFP4 or ORC_FP8_BLOCK (routed)  */
  int32_t shared_bf16;           /* shared expert weights are bf16 (else fp8)   */
  double rms_eps;
  int32_t routing;               /* 0 softmax top-k, 1 sigmoid (noaux_tc)        */
  int32_t act;                   /* ORC_SWIGLU or ORC_SITU                       */
} orc_problem;

typedef struct {
  const uint16_t* x;          /* [T, H] bf16 */
  const float* router_w;      /* [E, H] fp32 */
  const float* router_bias;   /* [E] or NULL */
  const uint8_t* w13;         /* routed, see expert_ffn */
  const void* w13_scale;
  const uint8_t* w2;
  const void* w2_scale;
  const void* sw13;           /* shared: fp8 [2I_s, H] or bf16 [2I_s, H] */
  const float* sw13_scale;    /* fp8 only: [2I_s] */
  const void* sw2;            /* fp8 [H, I_s] or bf16 [H, I_s] */
  const float* sw2_scale;     /* fp8 only: [H] */
  const uint16_t* wd;         /* latent down [L, H] bf16 */
  const uint16_t* wu;         /* latent up [H, L] bf16 */
  const uint16_t* gamma;      /* RMSNorm weight [L] bf16 */
} orc_weights;

typedef struct {
  const orc_problem* p;
  const orc_weights* w;
  const int32_t* tokens;
  double* out_f64;   /* [n, H] pre-rounding output, may be NULL */
  uint16_t* out_bf16;/* [n, H] */
  int32_t* idx_out;  /* [n, k] may be NULL */
  double* w_out;     /* [n, k] may be NULL */
} fwd_ctx;

/* Expert e's weights and scales within the [E, ...] arrays of format fmt. */
static void expert_slice(int fmt, int64_t K, int64_t I, int64_t e, const uint8_t* w13,
                         const void* s13, const uint8_t* w2, const void* s2,
                         const uint8_t** w13e, const void** s13e, const uint8_t** w2e,
                         const void** s2e) {
  int64_t rb13 = (fmt == ORC_MXFP4) ? K / 2 : K, rb2 = (fmt == ORC_MXFP4) ? I / 2 : I;
  *w13e = w13 + e * 2 * I * rb13;
  *w2e = w2 + e * K * rb2;
  if (fmt == ORC_FP8) {
    *s13e = (const float*)s13 + e * 2 * I;
    *s2e = (const float*)s2 + e * K;
  } else if (fmt == ORC_FP8_BLOCK) {
    *s13e = (const float*)s13 + e * (2 * I / 128) * (K / 128);
    *s2e = (const float*)s2 + e * (K / 128) * (I / 128);
  } else {
    *s13e = (const uint8_t*)s13 + e * 2 * I * (K / 32);
    *s2e = (const uint8_t*)s2 + e * K * (I / 32);
  }
}

/* z = bf16(x Wd^T) for one token [K3 s.2.4 routed_expert_down_proj]: each
 * product of two bf16 values is exact in fp64 and the sum is taken in fp64
 * (h ascending), then rounded once to nearest-even bf16. */
static void latent_down_row(int64_t H, int64_t L, const uint16_t* xrow, const uint16_t* wd,
                            uint16_t* z) {
  for (int64_t l = 0; l < L; l++) {
    double a = 0.0;
    for (int64_t h = 0; h < H; h++) a += orc_bf16_decode(xrow[h]) * orc_bf16_decode(wd[l * H + h]);
    z[l] = orc_bf16_from_double(a);
  }
}

typedef struct {
  int64_t H, L;
  const uint16_t* x;
  const uint16_t* wd;
  const int32_t* tokens;
  uint16_t* z;
} down_ctx;

static void down_body(int64_t i, void* c) {
  down_ctx* d = (down_ctx*)c;
  latent_down_row(d->H, d->L, d->x + (int64_t)d->tokens[i] * d->H, d->wd, d->z + i * d->L);
}

/* The LatentMoE down projection alone, for the listed tokens: z [n, L] bf16. */
void orc_latent_down(int64_t H, int64_t L, const uint16_t* x, const uint16_t* wd,
                     const int32_t* tokens, int64_t n_tokens, uint16_t* z, int nthreads) {
  down_ctx c = {H, L, x, wd, tokens, z};
  orc_parallel_for(n_tokens, nthreads, down_body, &c);
}

static void token_forward(int64_t i, void* c) {
  fwd_ctx* f = (fwd_ctx*)c;
  const orc_problem* p = f->p;
  const orc_weights* w = f->w;
  int64_t t = f->tokens[i], H = p->H, I = p->I, E = p->E;
  int k = (int)p->k;
  int64_t K = p->L > 0 ? p->L : H; /* expert input/output width */
  const uint16_t* xrow = w->x + t * H;
  float* logits = (float*)malloc(sizeof(float) * (size_t)E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* wt = (double*)malloc(sizeof(double) * (size_t)k);
  uint8_t* xq = (uint8_t*)malloc((size_t)K);
  double* acc = (double*)calloc((size_t)K, sizeof(double));
  double* y = (double*)malloc(sizeof(double) * (size_t)(K > H ? K : H));
  double* res = (double*)calloc((size_t)H, sizeof(double));

  if (p->routing == 1) { /* the bias steers selection only */
    router_row(H, E, xrow, w->router_w, NULL, logits);
    topk_sigmoid_row(E, k, logits, w->router_bias, idx, wt);
  } else {
    router_row(H, E, xrow, w->router_w, w->router_bias, logits);
    topk_row(E, k, logits, idx, wt);
  }

  float sx;
  if (p->L > 0) {
    uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)K);
    latent_down_row(H, K, xrow, w->wd, z);
    sx = quant_row_bf16(K, z, xq);
    free(z);
  } else {
    sx = quant_row_bf16(H, xrow, xq);
  }

  for (int j = 0; j < k; j++) {
    const uint8_t *w13, *w2;
    const void *s13, *s2;
    expert_slice(p->wfmt, K, I, idx[j], w->w13, w->w13_scale, w->w2, w->w2_scale, &w13, &s13,
                 &w2, &s2);
    expert_ffn(p->wfmt, p->act, K, I, xq, sx, w13, s13, w2, s2, y, NULL, NULL, NULL);
    for (int64_t n = 0; n < K; n++) acc[n] += wt[j] * y[n]; /* j ascending */
  }

  if (p->L > 0) {
    /* RMSNorm on the latent, bf16, then up_proj [K3 s.2.4] */
    double ms = 0.0;
    for (int64_t l = 0; l < K; l++) ms += acc[l] * acc[l];
    double r = 1.0 / sqrt(ms / (double)K + p->rms_eps);
    double* yn = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t l = 0; l < K; l++)
      yn[l] = orc_bf16_decode(orc_bf16_from_double(acc[l] * r * orc_bf16_decode(w->gamma[l])));
    for (int64_t h = 0; h < H; h++) {
      double a = 0.0;
      for (int64_t l = 0; l < K; l++) a += yn[l] * orc_bf16_decode(w->wu[h * K + l]);
      res[h] = a;
    }
    free(yn);
  } else {
    for (int64_t h = 0; h < H; h++) res[h] = acc[h];
  }

  if (p->I_s > 0) {
    /* shared expert, weight 1 [LING s.5 in-kernel shared expert] */
    if (p->shared_bf16) {
      shared_ffn_bf16(p->act, H, p->I_s, xrow, (const uint16_t*)w->sw13, (const uint16_t*)w->sw2,
                      y);
    } else {
      uint8_t* xqh = xq;
      float sxh = sx;
      uint8_t* tmp = NULL;
      if (p->L > 0) { /* shared path takes the raw hidden */
        tmp = (uint8_t*)malloc((size_t)H);
        sxh = quant_row_bf16(H, xrow, tmp);
        xqh = tmp;
      }
      /* an fp8 shared expert has the routed experts' fp8 format */
      expert_ffn(p->wfmt == ORC_FP8_BLOCK ? ORC_FP8_BLOCK : ORC_FP8, p->act, H, p->I_s, xqh, sxh,
                 (const uint8_t*)w->sw13, w->sw13_scale,
                 (const uint8_t*)w->sw2, w->sw2_scale, y, NULL, NULL, NULL);
      free(tmp);
    }
    for (int64_t h = 0; h < H; h++) res[h] += y[h];
  }

  for (int64_t h = 0; h < H; h++) {
    if (f->out_f64) f->out_f64[i * H + h] = res[h];
    f->out_bf16[i * H + h] = orc_bf16_from_double(res[h]);
  }
  if (f->idx_out) memcpy(f->idx_out + i * k, idx, sizeof(int32_t) * (size_t)k);
  if (f->w_out) memcpy(f->w_out + i * k, wt, sizeof(double) * (size_t)k);
  free(logits);
  free(idx);
  free(wt);
  free(xq);
  free(acc);
  free(y);
  free(res);
}

/* Full layer output for the listed tokens (any subset, any order). */
void orc_moe_forward(const orc_problem* p, const orc_weights* w, const int32_t* tokens,
                     int64_t n_tokens, double* out_f64, uint16_t* out_bf16, int32_t* idx_out,
                     double* w_out, int nthreads) {
  pthread_once(&tab_once, fill_tables);
  fwd_ctx c = {p, w, tokens, out_f64, out_bf16, idx_out, w_out};
  orc_parallel_for(n_tokens, nthreads, token_forward, &c);
}

/* ------------------------------------------------------------------------- */
/* Stage oracle for the grouped expert FFN: given expert-contiguous quantised   */
/* rows (counts per expert), y[r] = row_w[r] * FFN_{e(r)}(xq[r]).               */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t wfmt, act;
  int64_t K, I, E;
  const int32_t* off;    /* [E+1] */
  const uint8_t* xq;     /* [R, K] */
  const float* xs;       /* [R] */
  const float* row_w;    /* [R] */
  const uint8_t* w13;
  const void* w13_scale;
  const uint8_t* w2;
  const void* w2_scale;
  double* y;             /* [R, K] */
  uint16_t* h;           /* [R, I] or NULL */
  uint8_t* hq;           /* [R, I] or NULL */
  float* hs;             /* [R] or NULL */
} rows_ctx;

static void rows_body(int64_t r, void* c) {
  rows_ctx* q = (rows_ctx*)c;
  int64_t e = 0;
  while (e < q->E && q->off[e + 1] <= r) e++;
  int64_t K = q->K, I = q->I;
  const uint8_t *w13, *w2;
  const void *s13, *s2;
  expert_slice(q->wfmt, K, I, e, q->w13, q->w13_scale, q->w2, q->w2_scale, &w13, &s13, &w2, &s2);
  double* y = q->y + r * K;
  expert_ffn(q->wfmt, q->act, K, I, q->xq + r * K, q->xs[r], w13, s13, w2, s2, y, q->h ? q->h + r * I : NULL, q->hs ? q->hs + r : NULL,
             q->hq ? q->hq + r * I : NULL);
  for (int64_t n = 0; n < K; n++) y[n] *= (double)q->row_w[r];
}

void orc_expert_rows(int32_t wfmt, int32_t act, int64_t K, int64_t I, int64_t E, const int32_t* off,
                     const uint8_t* xq, const float* xs, const float* row_w, const uint8_t* w13,
                     const void* w13_scale, const uint8_t* w2, const void* w2_scale, double* y,
                     uint16_t* h, uint8_t* hq, float* hs, int nthreads) {
  pthread_once(&tab_once, fill_tables);
  rows_ctx c = {wfmt, act, K, I, E, off, xq, xs, row_w, w13, w13_scale, w2, w2_scale, y, h, hq, hs};
  orc_parallel_for(off[E], nthreads, rows_body, &c);
}

/* S7: weighted gather back to token order [LING s.1 "gather results"; s.5
 * shared expert added on every token]: out[t] = bf16(sum_j y[perm[t,j]] +
 * shared[t]) with the routing weights already inside the y rows; the sum is
 * taken in fp64 over the given bf16 values, j ascending, shared last. */
void orc_combine(int64_t T, int64_t H, int k, const uint16_t* y, const int32_t* perm,
                 const uint16_t* shared, uint16_t* out) {
  for (int64_t t = 0; t < T; t++)
    for (int64_t h = 0; h < H; h++) {
      double acc = 0.0;
      for (int j = 0; j < k; j++) acc += orc_bf16_decode(y[(int64_t)perm[t * k + j] * H + h]);
      if (shared) acc += orc_bf16_decode(shared[t * H + h]);
      out[t * H + h] = orc_bf16_from_double(acc);
    }
}
