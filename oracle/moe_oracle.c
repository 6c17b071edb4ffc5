/* CPU oracle of one DeepSeek-V4.1 MoE FFN layer forward on still-quantized
 * experts (router -> sqrt-softplus scores -> biased stable top-k -> routing
 * weights -> q8_1 activation -> Q2_K gate/up -> clipped SwiGLU -> q8_1(h) ->
 * Q3_K down -> G-weighted sum over the picks in ascending expert id -> shared
 * expert added last).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The GPU product path never
 * links, loads or calls it, and this file includes nothing from the product.
 *
 * It is plain and slow on purpose: every weight is dequantised to its exact
 * real value in f64 and every dot product is a straight f64 loop.  Lower
 * precision appears only where the method itself fixes it:
 *   - router logits are handed on as f32 (the f32-accumulated logits of the
 *     metrale moe_v41 module docs);
 *   - scores, keys and routing weights are f32 (metrale moe_v41.rs source,
 *     fn route_from_logits);
 *   - the q8_1 quantiser takes its decisions in f32 (reading C-L3);
 *   - the bf16 shared expert's h is rounded to bf16 before w2
 *     (DeepSeek V4.1 atlas page, model.py Expert.forward: w2(x.to(dtype))).
 *
 * Page references: [moe_v41 docs] = docs.metrale.ai module page
 * metrale_model_arch::moe_v41; [moe_v41.rs] = its source page;
 * [MoE atlas] = open-model-atlas "DeepSeek V4.1 · Mixture of experts"
 * (the "All 22 steps" equations, the Parameters table, the model.py
 * MoE/Gate/Expert listings and config.json).
 *
 * Readings of what the pages leave open:
 *   C-L1  Q2_K block, 84 B: scales[16] (low nibble scale, high nibble min),
 *         qs[64], fp16 d, fp16 dmin; element e = 128h + 32j + l (l < 32):
 *         q = (qs[32h + l] >> 2j) & 3, sub-block b = e / 16,
 *         w = d * (scales[b] & 15) * q - dmin * (scales[b] >> 4).
 *   C-L2  Q3_K block, 110 B: hmask[32], qs[64], scales[12], fp16 d;
 *         lo = (qs[32h + l] >> 2j) & 3, hb = (hmask[l] >> (4h + j)) & 1,
 *         q = lo - (hb ? 0 : 4); six-bit code of sub-block b: low four bits
 *         from scales[b] (b < 8) or scales[b-8] >> 4 (b >= 8), high two bits
 *         (scales[8 + b%4] >> 2*(b/4)) & 3; w = d * (code - 32) * q.
 *   C-L3  q8_1 block of 32, 36 B: fp16 d, fp16 s, int8 qs[32];
 *         amax = max |x| (f32), d = amax / 127 (f32 division),
 *         q = amax == 0 ? 0 : round-half-away(x / d) (f32 division),
 *         stored d = fp16(d), s = fp16(d * sum q) (f32 product);
 *         the dequantised value is fp16(d) * q.
 *   C-R2  score s = f32 of sqrt(log1p(exp(t))) evaluated in f64 for
 *         t = z / gate_temp (f32) <= 20, and f32 sqrt(t) above 20.
 *   C-R6  the sigmoid and softmax score functions (model.py Gate.forward)
 *         are evaluated the same way: f64 from t = f32(z / gate_temp),
 *         rounded once to f32; the softmax subtracts the largest t and sums
 *         the experts in id order; a NaN logit makes every softmax score NaN.
 *         Image tokens pick with bias_vl, and their weights stay the raw
 *         scores as for every token.
 *   C-R3  ties on equal f32 keys go to the lower expert id; picks come out in
 *         descending key order.  C-R4: a NaN key ranks below every number and
 *         is counted.
 *   C-G1  G multiplies the expert output after the down projection.
 *   C-G2  the routed outputs are summed in ascending expert id; the shared
 *         expert is added after all of them.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "moe_oracle.h"

/* ---------------------------------------------------------------- formats */

double orc_bf16_value(uint16_t b) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)b << 16;
  return (double)c.f;
}

/* f32 -> bf16, round to nearest, ties to even, as the metrale bf16_bytes
 * helper states it ([moe_v41.rs], fn bf16_bytes). */
uint16_t orc_bf16_from_f32(float v) {
  union { uint32_t u; float f; } c;
  c.f = v;
  uint32_t b = c.u;
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

double orc_f16_value(uint16_t h) {
  _Float16 v;
  memcpy(&v, &h, 2);
  return (double)v;
}

uint16_t orc_f16_from_f32(float v) {
  _Float16 h = (_Float16)v; /* IEEE conversion, round to nearest even */
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

/* ------------------------------------------------------- dequantisation */

/* Reading C-L1 (Q2_K named in [moe_v41 docs]: gate and up run on Q2_K). */
void orc_dequant_q2k(const uint8_t* blk, double* w) {
  const uint8_t* scales = blk;
  const uint8_t* qs = blk + 16;
  double d = orc_f16_value((uint16_t)(blk[80] | (blk[81] << 8)));
  double dmin = orc_f16_value((uint16_t)(blk[82] | (blk[83] << 8)));
  for (int e = 0; e < 256; ++e) {
    int h = e / 128, j = (e % 128) / 32, l = e % 32, b = e / 16;
    int q = (qs[32 * h + l] >> (2 * j)) & 3;
    int sc = scales[b] & 15, mn = scales[b] >> 4;
    w[e] = d * sc * q - dmin * mn;
  }
}

/* six-bit scale code of sub-block b of a Q3_K block (reading C-L2) */
int orc_q3k_scale_code(const uint8_t* scales12, int b) {
  int lo4 = b < 8 ? (scales12[b] & 15) : (scales12[b - 8] >> 4);
  int hi2 = (scales12[8 + b % 4] >> (2 * (b / 4))) & 3;
  return lo4 | (hi2 << 4);
}

/* Reading C-L2 (Q3_K named in [moe_v41 docs]: down runs on Q3_K). */
void orc_dequant_q3k(const uint8_t* blk, double* w) {
  const uint8_t* hmask = blk;
  const uint8_t* qs = blk + 32;
  const uint8_t* scales = blk + 96;
  double d = orc_f16_value((uint16_t)(blk[108] | (blk[109] << 8)));
  for (int e = 0; e < 256; ++e) {
    int h = e / 128, j = (e % 128) / 32, l = e % 32, b = e / 16;
    int lo = (qs[32 * h + l] >> (2 * j)) & 3;
    int hb = (hmask[l] >> (4 * h + j)) & 1;
    int q = lo - (hb ? 0 : 4);
    w[e] = d * (orc_q3k_scale_code(scales, b) - 32) * q;
  }
}

/* Row r of a [rows][cols/256 blocks] K-quant matrix, dequantised. */
static void dequant_row(int kind, const uint8_t* mat, int r, int cols, double* out) {
  int nb = cols / 256;
  size_t bb = kind == 2 ? 84 : 110;
  const uint8_t* row = mat + (size_t)r * nb * bb;
  for (int b = 0; b < nb; ++b) {
    if (kind == 2) orc_dequant_q2k(row + b * bb, out + 256 * b);
    else orc_dequant_q3k(row + b * bb, out + 256 * b);
  }
}

void orc_dequant_matrix(int kind, const uint8_t* mat, int rows, int cols, double* out) {
  for (int r = 0; r < rows; ++r) dequant_row(kind, mat, r, cols, out + (size_t)r * cols);
}

/* --------------------------------------------------------------- q8_1 */

static float round_half_away(float v) { return roundf(v); }

/* Reading C-L3 (q8_1 activations named in [moe_v41 docs]). */
void orc_quantize_q8_1(const float* x, int n, uint8_t* out) {
  for (int blk = 0; blk < n / 32; ++blk) {
    const float* xb = x + 32 * blk;
    uint8_t* ob = out + 36 * blk;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(xb[i]);
      if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    int sum = 0;
    for (int i = 0; i < 32; ++i) {
      int q = amax == 0.0f ? 0 : (int)round_half_away(xb[i] / d);
      ob[4 + i] = (uint8_t)(int8_t)q;
      sum += q;
    }
    uint16_t d16 = orc_f16_from_f32(d);
    uint16_t s16 = orc_f16_from_f32(d * (float)sum);
    ob[0] = (uint8_t)(d16 & 0xFF); ob[1] = (uint8_t)(d16 >> 8);
    ob[2] = (uint8_t)(s16 & 0xFF); ob[3] = (uint8_t)(s16 >> 8);
  }
}

/* The real values a q8_1 row stands for: fp16(d) * q. */
void orc_dequant_q8_1(const uint8_t* q8, int n, double* out) {
  for (int blk = 0; blk < n / 32; ++blk) {
    const uint8_t* b = q8 + 36 * blk;
    double d = orc_f16_value((uint16_t)(b[0] | (b[1] << 8)));
    for (int i = 0; i < 32; ++i) out[32 * blk + i] = d * (double)(int8_t)b[4 + i];
  }
}

/* ------------------------------------------------------------- routing */

/* z = x W_R^T ([MoE atlas] Router step z = x_ffn W_R; model.py Gate.forward
 * linear(x.float(), weight.float())), exact in f64 and handed on as f32. */
void orc_router_logits(const uint16_t* x, int m, const uint16_t* W, int D, int N, float* z) {
  for (int t = 0; t < m; ++t)
    for (int e = 0; e < N; ++e) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += orc_bf16_value(x[(size_t)t * D + d]) * orc_bf16_value(W[(size_t)e * D + d]);
      z[(size_t)t * N + e] = (float)acc;
    }
}

/* s = sqrt(softplus(z / gate_temp)), softplus(t) = t above 20
 * ([moe_v41.rs] fn softplus and route_from_logits; [MoE atlas] s = sqrt(softplus(z))).
 * Reading C-R2 fixes the f32 value. */
float orc_score(float z, float gate_temp) {
  float t = z / gate_temp;
  if (t > 20.0f) return (float)sqrt((double)t);
  return (float)sqrt(log1p(exp((double)t)));
}

/* The scores of one token's logits z[N] by the configuration's score function
 * ([MoE atlas] model.py Gate.forward: scores = linear(x, W) / gate_temp, then
 * softmax over the experts, sigmoid, or sqrt(softplus)).  Every step is
 * evaluated in f64 from t = f32(z / gate_temp) and rounded once to f32 (the
 * reading C-R2 extends to the other two functions); the softmax takes the
 * largest t as its shift and sums the experts in id order. */
void orc_scores(const orc_cfg* c, const float* z, float* s) {
  int N = c->n_routed;
  if (c->score_func == ORC_SCORE_SIGMOID) {
    for (int e = 0; e < N; ++e) {
      float t = z[e] / c->gate_temp;
      s[e] = (float)(1.0 / (1.0 + exp(-(double)t)));
    }
  } else if (c->score_func == ORC_SCORE_SOFTMAX) {
    double mx = -INFINITY, sum = 0.0;
    int any_nan = 0;
    for (int e = 0; e < N; ++e) {
      float t = z[e] / c->gate_temp;
      if (isnan(t)) any_nan = 1;
      else if (t > mx) mx = t;
    }
    for (int e = 0; e < N; ++e) sum += exp((double)(z[e] / c->gate_temp) - mx);
    for (int e = 0; e < N; ++e)
      s[e] = any_nan ? NAN : (float)(exp((double)(z[e] / c->gate_temp) - mx) / sum);
  } else {
    for (int e = 0; e < N; ++e) s[e] = orc_score(z[e], c->gate_temp);
  }
}

/* a ranks before b: larger key first, NaN last, equal keys by lower id */
static int ranks_before(float ka, int a, float kb, int b) {
  int na = isnan(ka), nb = isnan(kb);
  if (na != nb) return nb;
  if (!na && ka != kb) return ka > kb;
  return a < b;
}

/* One token's routing from f32 logits ([moe_v41.rs] fn route_from_logits;
 * [MoE atlas] model.py Gate.forward and the Router steps):
 * keys s + bias pick topk experts by a stable descending order; the weights
 * are the unbiased scores, divided by (sum + 1e-20) when norm_topk_prob and
 * topk > 1, then times route_scale.  Returns the number of NaN keys. */
int orc_route_token(const orc_cfg* c, const float* z, const float* bias, float* w_out, int32_t* idx_out) {
  int N = c->n_routed, k = c->topk, nan_keys = 0;
  float* s = (float*)malloc(sizeof(float) * N);
  float* key = (float*)malloc(sizeof(float) * N);
  int* order = (int*)malloc(sizeof(int) * N);
  orc_scores(c, z, s);
  for (int e = 0; e < N; ++e) {
    key[e] = s[e] + bias[e];
    if (isnan(key[e])) ++nan_keys;
    order[e] = e;
  }
  /* insertion sort: stable and plain */
  for (int i = 1; i < N; ++i) {
    int v = order[i], j = i - 1;
    while (j >= 0 && ranks_before(key[v], v, key[order[j]], order[j])) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }
  for (int i = 0; i < k; ++i) {
    idx_out[i] = order[i];
    w_out[i] = s[order[i]];
  }
  if (c->norm_topk_prob && k > 1) {
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum += w_out[i];
    sum += 1e-20f;
    for (int i = 0; i < k; ++i) w_out[i] /= sum;
  }
  for (int i = 0; i < k; ++i) w_out[i] *= c->route_scale;
  free(s); free(key); free(order);
  return nan_keys;
}

int orc_route_from_logits(const orc_cfg* c, const float* z, int m, const float* bias, float* w_out,
                          int32_t* idx_out) {
  return orc_route_from_logits_vl(c, z, m, bias, NULL, NULL, w_out, idx_out);
}

/* The same with the image-token bias: a token whose image_mask entry is
 * nonzero picks with bias_vl instead of bias ([MoE atlas] model.py
 * Gate.forward, torch.where(image_mask, bias_vl, bias)). */
int orc_route_from_logits_vl(const orc_cfg* c, const float* z, int m, const float* bias, const float* bias_vl,
                             const uint8_t* image_mask, float* w_out, int32_t* idx_out) {
  int nan_keys = 0;
  for (int t = 0; t < m; ++t) {
    const float* b = (image_mask && bias_vl && image_mask[t]) ? bias_vl : bias;
    nan_keys += orc_route_token(c, z + (size_t)t * c->n_routed, b, w_out + (size_t)t * c->topk,
                                idx_out + (size_t)t * c->topk);
  }
  return nan_keys;
}

/* ------------------------------------------------------------- SwiGLU */

/* Clipped SwiGLU ([MoE atlas] steps g' = min(g, 10), u' = clip(u, -10, 10),
 * a = g' sigma(g'), h = a * u'; model.py Expert.forward clamps only when
 * swiglu_limit > 0). */
double orc_swiglu(double g, double u, double limit, int* clipped) {
  if (limit > 0) {
    if (g > limit) { g = limit; if (clipped) ++*clipped; }
    if (u > limit) { u = limit; if (clipped) ++*clipped; }
    if (u < -limit) { u = -limit; if (clipped) ++*clipped; }
  }
  double sig = 1.0 / (1.0 + exp(-g));
  return g * sig * u;
}

/* ------------------------------------------------------------- experts */

/* One routed expert on one token ([MoE atlas] Routed expert steps;
 * [moe_v41 docs]: gate/up on Q2_K, down on Q3_K, activations as q8_1).
 * xq8 is q8_1(x) ([D/32] blocks); E receives h W2 in f64. */
void orc_expert_kquant(const orc_cfg* c, const uint8_t* xq8, const uint8_t* w1, const uint8_t* w3,
                       const uint8_t* w2, double* E, int* clipped) {
  int D = c->dim, I = c->inter;
  double* xh = (double*)malloc(sizeof(double) * D);
  double* row = (double*)malloc(sizeof(double) * (D > I ? D : I));
  float* h = (float*)malloc(sizeof(float) * I);
  uint8_t* hq8 = (uint8_t*)malloc((size_t)36 * (I / 32));
  double* hh = (double*)malloc(sizeof(double) * I);
  orc_dequant_q8_1(xq8, D, xh);
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0;
    dequant_row(2, w1, r, D, row);
    for (int d = 0; d < D; ++d) g += row[d] * xh[d];
    dequant_row(2, w3, r, D, row);
    for (int d = 0; d < D; ++d) u += row[d] * xh[d];
    h[r] = (float)orc_swiglu(g, u, c->swiglu_limit, clipped);
  }
  /* the SwiGLU output goes to q8_1 before the Q3_K down projection
   * ([moe_v41.rs] Kernels: swiglu_q8, and the h_q8 scratch) */
  orc_quantize_q8_1(h, I, hq8);
  orc_dequant_q8_1(hq8, I, hh);
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    dequant_row(3, w2, d, I, row);
    for (int j = 0; j < I; ++j) acc += row[j] * hh[j];
    E[d] = acc;
  }
  free(xh); free(row); free(h); free(hq8); free(hh);
}

/* The bf16 shared expert on one token: the same clipped SwiGLU FFN with no
 * routing weight ([MoE atlas] Shared expert steps); h is rounded to bf16
 * before w2 (model.py Expert.forward casts to the input dtype). */
void orc_shared_bf16(const orc_cfg* c, const uint16_t* x, const uint16_t* w1, const uint16_t* w3,
                     const uint16_t* w2, double* S, int* clipped) {
  int D = c->dim, I = c->inter;
  double* hb = (double*)malloc(sizeof(double) * I);
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0;
    for (int d = 0; d < D; ++d) {
      double xv = orc_bf16_value(x[d]);
      g += orc_bf16_value(w1[(size_t)r * D + d]) * xv;
      u += orc_bf16_value(w3[(size_t)r * D + d]) * xv;
    }
    float h = (float)orc_swiglu(g, u, c->swiglu_limit, clipped);
    hb[r] = orc_bf16_value(orc_bf16_from_f32(h));
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += orc_bf16_value(w2[(size_t)d * I + j]) * hb[j];
    S[d] = acc;
  }
  free(hb);
}

/* --------------------------------------------------------------- layer */

typedef struct {
  const orc_cfg* c;
  const orc_layer* L;
  const int32_t* tokens;
  int n_tok;
  double* out;
  float* topk_w;
  int32_t* topk_idx;
  int next;            /* shared cursor */
  pthread_mutex_t mu;
  int status;
  int nan_keys;
  int clipped;
} layer_job;

static int token_forward(const orc_cfg* c, const orc_layer* L, int t, double* out, float* w, int32_t* idx,
                         int* nan_keys, int* clipped) {
  int D = c->dim, N = c->n_routed, k = c->topk;
  const uint16_t* xt = L->x + (size_t)t * D;
  float* z = (float*)malloc(sizeof(float) * N);
  if (L->given_logits) memcpy(z, L->given_logits + (size_t)t * N, sizeof(float) * N);
  else orc_router_logits(xt, 1, L->router_w, D, N, z);
  const float* bias = (L->image_mask && L->bias_vl && L->image_mask[t]) ? L->bias_vl : L->bias;
  *nan_keys += orc_route_token(c, z, bias, w, idx);
  free(z);

  float* xf = (float*)malloc(sizeof(float) * D);
  uint8_t* xq8 = (uint8_t*)malloc((size_t)36 * (D / 32));
  for (int d = 0; d < D; ++d) xf[d] = (float)orc_bf16_value(xt[d]);
  orc_quantize_q8_1(xf, D, xq8);

  double* y = (double*)calloc((size_t)D, sizeof(double));
  double* E = (double*)malloc(sizeof(double) * D);
  /* routed experts in ascending expert id ([MoE atlas] model.py MoE.forward
   * loops i upward; [moe_v41.rs] rows grouped by ascending expert id) */
  int status = 0;
  for (int e = 0; e < N && !status; ++e) {
    int slot = -1;
    for (int i = 0; i < k; ++i)
      if (idx[i] == e) slot = i;
    if (slot < 0) continue;
    const uint8_t* w1 = L->experts[3 * e + 0];
    const uint8_t* w3 = L->experts[3 * e + 1];
    const uint8_t* w2 = L->experts[3 * e + 2];
    if (!w1 || !w3 || !w2) { status = ORC_ERR_MISSING_EXPERT; break; }
    orc_expert_kquant(c, xq8, w1, w3, w2, E, clipped);
    double g = (double)w[slot];
    for (int d = 0; d < D; ++d) y[d] += g * E[d];
  }
  if (!status) {
    /* the shared expert, added last ([moe_v41 docs] shared_side: added after
     * the routed experts; [MoE atlas] Delta = y_routed + y_shared) */
    if (L->shared_kind == ORC_SHARED_BF16)
      orc_shared_bf16(c, xt, (const uint16_t*)L->sh1, (const uint16_t*)L->sh3, (const uint16_t*)L->sh2, E, clipped);
    else
      orc_expert_kquant(c, xq8, (const uint8_t*)L->sh1, (const uint8_t*)L->sh3, (const uint8_t*)L->sh2, E, clipped);
    for (int d = 0; d < D; ++d) out[d] = y[d] + E[d];
  }
  free(xf); free(xq8); free(y); free(E);
  return status;
}

static void* layer_worker(void* p) {
  layer_job* J = (layer_job*)p;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int i = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (i >= J->n_tok) break;
    int t = J->tokens ? J->tokens[i] : i;
    int nan_keys = 0, clipped = 0;
    int st = token_forward(J->c, J->L, t, J->out + (size_t)i * J->c->dim, J->topk_w + (size_t)i * J->c->topk,
                           J->topk_idx + (size_t)i * J->c->topk, &nan_keys, &clipped);
    pthread_mutex_lock(&J->mu);
    if (st && !J->status) J->status = st;
    J->nan_keys += nan_keys;
    J->clipped += clipped;
    pthread_mutex_unlock(&J->mu);
  }
  return NULL;
}

/* One layer for the listed token rows (all m when tokens is NULL).  Row i of
 * out / topk_w / topk_idx belongs to token tokens[i].  Tokens are independent,
 * so they are spread over nthreads threads; the arithmetic of one token never
 * depends on the thread count. */
int orc_moe_layer(const orc_cfg* c, const orc_layer* L, const int32_t* tokens, int n_tok, double* out,
                  float* topk_w, int32_t* topk_idx, int nthreads, orc_stats* stats) {
  if (c->dim % 256 || c->inter % 256 || c->topk < 1 || c->topk > c->n_routed) return ORC_ERR_ARG;
  layer_job J;
  memset(&J, 0, sizeof J);
  J.c = c; J.L = L; J.tokens = tokens; J.n_tok = n_tok; J.out = out; J.topk_w = topk_w; J.topk_idx = topk_idx;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, layer_worker, &J);
  layer_worker(&J);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  if (stats) { stats->nan_keys = J.nan_keys; stats->clipped = J.clipped; }
  return J.status;
}

/* ------------------------------------------------------ brute-force mode */

/* The whole layer a second way, for small inputs: every matrix of every
 * expert (and the shared expert) is first dequantised to a dense f64 array,
 * then the layer runs as textbook dense loops over all tokens at once.  The
 * selection here takes k rounds of "the best remaining expert" (largest key,
 * NaN last, lower id on equal keys) instead of a sort; the routed sum visits
 * the experts in ascending id through a [m, N] weight matrix that is zero
 * where a token did not pick.  Same formulas as orc_moe_layer ([MoE atlas]
 * Router / Routed expert / Shared expert steps; [moe_v41.rs]
 * route_from_logits), composed independently; the two must agree to
 * rounding of the f64 sums.  Memory: 8 * (3 * N * D * I + 3 * D * I) bytes. */
int orc_moe_layer_dense(const orc_cfg* c, const orc_layer* L, int m, double* out, float* topk_w,
                        int32_t* topk_idx) {
  const int D = c->dim, I = c->inter, N = c->n_routed, k = c->topk;
  if (D % 256 || I % 256 || k < 1 || k > N) return ORC_ERR_ARG;
  for (int e = 0; e < N; ++e)
    for (int j = 0; j < 3; ++j)
      if (!L->experts[3 * e + j]) return ORC_ERR_MISSING_EXPERT;
  const size_t DI = (size_t)D * I;
  double* W1 = (double*)malloc(sizeof(double) * DI * N);
  double* W3 = (double*)malloc(sizeof(double) * DI * N);
  double* W2 = (double*)malloc(sizeof(double) * DI * N);
  double* S1 = (double*)malloc(sizeof(double) * DI);
  double* S3 = (double*)malloc(sizeof(double) * DI);
  double* S2 = (double*)malloc(sizeof(double) * DI);
  double* X = (double*)malloc(sizeof(double) * (size_t)m * D);   /* bf16 x, exact */
  double* XQ = (double*)malloc(sizeof(double) * (size_t)m * D);  /* q8_1(x) values */
  float* Z = (float*)malloc(sizeof(float) * (size_t)m * N);
  double* G = (double*)calloc((size_t)m * N, sizeof(double));   /* routing weight, 0 = not picked */
  /* 1. every matrix, dense */
  for (int e = 0; e < N; ++e) {
    orc_dequant_matrix(2, L->experts[3 * e + 0], I, D, W1 + DI * e);
    orc_dequant_matrix(2, L->experts[3 * e + 1], I, D, W3 + DI * e);
    orc_dequant_matrix(3, L->experts[3 * e + 2], D, I, W2 + DI * e);
  }
  if (L->shared_kind == ORC_SHARED_BF16) {
    for (size_t i = 0; i < DI; ++i) {
      S1[i] = orc_bf16_value(((const uint16_t*)L->sh1)[i]);
      S3[i] = orc_bf16_value(((const uint16_t*)L->sh3)[i]);
      S2[i] = orc_bf16_value(((const uint16_t*)L->sh2)[i]);
    }
  } else {
    orc_dequant_matrix(2, (const uint8_t*)L->sh1, I, D, S1);
    orc_dequant_matrix(2, (const uint8_t*)L->sh3, I, D, S3);
    orc_dequant_matrix(3, (const uint8_t*)L->sh2, D, I, S2);
  }
  /* 2. activations: bf16 values and their q8_1 values */
  {
    float* xf = (float*)malloc(sizeof(float) * D);
    uint8_t* q8 = (uint8_t*)malloc((size_t)36 * (D / 32));
    for (int t = 0; t < m; ++t) {
      for (int d = 0; d < D; ++d) {
        X[(size_t)t * D + d] = orc_bf16_value(L->x[(size_t)t * D + d]);
        xf[d] = (float)X[(size_t)t * D + d];
      }
      orc_quantize_q8_1(xf, D, q8);
      orc_dequant_q8_1(q8, D, XQ + (size_t)t * D);
    }
    free(xf); free(q8);
  }
  /* 3. logits: Z = X W_R^T (f64 sums handed on as f32), unless given */
  for (int t = 0; t < m; ++t)
    for (int e = 0; e < N; ++e) {
      if (L->given_logits) { Z[(size_t)t * N + e] = L->given_logits[(size_t)t * N + e]; continue; }
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += X[(size_t)t * D + d] * orc_bf16_value(L->router_w[(size_t)e * D + d]);
      Z[(size_t)t * N + e] = (float)acc;
    }
  /* 4. selection by k rounds of the best remaining key, then the weights */
  {
    float* s = (float*)malloc(sizeof(float) * N);
    float* key = (float*)malloc(sizeof(float) * N);
    char* taken = (char*)malloc((size_t)N);
    for (int t = 0; t < m; ++t) {
      const float* b = (L->image_mask && L->bias_vl && L->image_mask[t]) ? L->bias_vl : L->bias;
      orc_scores(c, Z + (size_t)t * N, s);
      for (int e = 0; e < N; ++e) { key[e] = s[e] + b[e]; taken[e] = 0; }
      float* w = topk_w + (size_t)t * k;
      int32_t* ix = topk_idx + (size_t)t * k;
      for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < N; ++e) {
          if (taken[e]) continue;
          if (best < 0) { best = e; continue; }
          int en = isnan(key[e]), bn = isnan(key[best]);
          if (en) continue;                               /* NaN never beats anything */
          if (bn || key[e] > key[best]) best = e;         /* ids ascend: equal keys keep the lower */
        }
        taken[best] = 1;
        ix[i] = best;
        w[i] = s[best];
      }
      /* renormalised over the picks (in pick order, f32) when asked and k > 1 */
      const int renorm = c->norm_topk_prob != 0 && k >= 2;
      float denom = 0.0f;
      for (int i = 0; i < k && renorm; ++i) denom += w[i];
      denom = denom + 1e-20f;
      for (int i = 0; i < k; ++i) {
        if (renorm) w[i] = w[i] / denom;
        w[i] *= c->route_scale;
        G[(size_t)t * N + ix[i]] = (double)w[i];
      }
    }
    free(s); free(key); free(taken);
  }
  /* 5. dense expert FFNs; y[t] = sum over e ascending of G[t, e] E_e[t],
   *    then the shared expert */
  {
    double* hv = (double*)malloc(sizeof(double) * I);
    float* hf = (float*)malloc(sizeof(float) * I);
    uint8_t* hq = (uint8_t*)malloc((size_t)36 * (I / 32));
    for (int t = 0; t < m; ++t) {
      double* o = out + (size_t)t * D;
      const double* xq = XQ + (size_t)t * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int e = 0; e <= N; ++e) {          /* e == N: the shared expert */
        const int shared = e == N;
        if (!shared && G[(size_t)t * N + e] == 0.0) continue;
        const double* A1 = shared ? S1 : W1 + DI * e;
        const double* A3 = shared ? S3 : W3 + DI * e;
        const double* A2 = shared ? S2 : W2 + DI * e;
        const int bf = shared && L->shared_kind == ORC_SHARED_BF16;
        const double* xin = bf ? X + (size_t)t * D : xq;
        for (int r = 0; r < I; ++r) {
          double g = 0.0, u = 0.0;
          for (int d = 0; d < D; ++d) {
            g += A1[(size_t)r * D + d] * xin[d];
            u += A3[(size_t)r * D + d] * xin[d];
          }
          hf[r] = (float)orc_swiglu(g, u, c->swiglu_limit, NULL);
        }
        if (bf) {
          for (int r = 0; r < I; ++r) hv[r] = orc_bf16_value(orc_bf16_from_f32(hf[r]));
        } else {
          orc_quantize_q8_1(hf, I, hq);
          orc_dequant_q8_1(hq, I, hv);
        }
        const double gw = shared ? 1.0 : G[(size_t)t * N + e];
        for (int d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int j = 0; j < I; ++j) acc += A2[(size_t)d * I + j] * hv[j];
          o[d] += gw * acc;
        }
      }
    }
    free(hv); free(hf); free(hq);
  }
  free(W1); free(W3); free(W2); free(S1); free(S3); free(S2); free(X); free(XQ); free(Z); free(G);
  return ORC_OK;
}

/* ------------------------------------------------- requantisation flips */

/* Reading C-F1.  h is requantised twice in the method: to q8_1 before a
 * K-quant down projection ([moe_v41.rs] swiglu_q8) and to bf16 before the
 * bf16 shared expert's w2 ([MoE atlas] model.py Expert.forward).  Both are
 * decisions taken on an f32 h, and an implementation that accumulates g and
 * u in f32 holds them only to within some multiple of 2^-24 sum |terms|.
 * Where the exact h lies that close to a rounding boundary, either side of
 * the boundary is a result of the method.  orc_flip_candidates lists, for
 * one token, each requantised value that a g' in [g - kappa sum|a x|,
 * g + kappa sum|a x|] and a u' in the like interval of u can change, with
 * the change it makes to the token's output:
 *   kind 0  a q8_1 code of h (the block's scale as the oracle has it),
 *   kind 1  a q8_1 block scale: the block's largest |h| moved far enough to
 *           give another fp16(d); every code of the block taken again,
 *   kind 2  a bf16 value of the bf16 shared expert's h.
 * meta[4 c] = {slot (k: the shared expert), kind, element or block, the
 * alternative code, fp16 bits of d, or bf16 bits}; delta[c D ..] = the
 * output change (routing weight included; the shared expert's weight is 1).
 * Candidates whose change stays below min_change in every output element
 * are left out.  Returns the number of candidates; only the first max_c are
 * written. */

typedef struct {
  int slot, kind, index, alt;
  int j0, n;           /* output change: sum over i < n of coef[i] * W2[:, j0 + i] */
  double coef[32];
} flip_cand;

typedef struct {
  flip_cand* v;
  int n, cap;
} flip_list;

static flip_cand* flip_push(flip_list* L) {
  if (L->n == L->cap) {
    L->cap = L->cap ? 2 * L->cap : 64;
    L->v = (flip_cand*)realloc(L->v, sizeof(flip_cand) * (size_t)L->cap);
  }
  flip_cand* f = &L->v[L->n++];
  memset(f, 0, sizeof(*f));
  return f;
}

/* The smallest and largest swiglu over g' in [g - dg, g + dg], u' in
 * [u - du, u + du]: for a fixed g' the value is linear in the clamped u', and
 * for a fixed u' silu(min(g', limit)) has its one minimum at g*, the root
 * of 1 + g (1 - sigma(g)) = 0 (the derivative of g sigma(g) over sigma(g)). */
static void swiglu_range(double g, double u, double dg, double du, double limit, float* lo, float* hi) {
  const double gstar = -1.2784645427610738;
  double gs[3] = {g - dg, g + dg, gstar};
  int ng = (gstar > g - dg && gstar < g + dg) ? 3 : 2;
  double us[2] = {u - du, u + du};
  float mn = 0.0f, mx = 0.0f;
  int first = 1;
  for (int a = 0; a < ng; ++a)
    for (int b = 0; b < 2; ++b) {
      float v = (float)orc_swiglu(gs[a], us[b], limit, NULL);
      if (first || v < mn) mn = v;
      if (first || v > mx) mx = v;
      first = 0;
    }
  *lo = mn;
  *hi = mx;
}

static int q8_code(float v, float d, float amax) {
  int q = amax == 0.0f ? 0 : (int)round_half_away(v / d);
  return q > 127 ? 127 : (q < -127 ? -127 : q);
}

/* The q8_1 candidates of one K-quant expert on one token (xh: q8_1(x) values). */
static void flips_kquant(const orc_cfg* c, const double* xh, const uint8_t* w1, const uint8_t* w3, double G, int slot,
                         double kappa, flip_list* F) {
  int D = c->dim, I = c->inter;
  double* row = (double*)malloc(sizeof(double) * D);
  double* row3 = (double*)malloc(sizeof(double) * D);
  float* h = (float*)malloc(sizeof(float) * I);
  float* lo = (float*)malloc(sizeof(float) * I);
  float* hi = (float*)malloc(sizeof(float) * I);
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0, sg = 0.0, su = 0.0;
    dequant_row(2, w1, r, D, row);
    dequant_row(2, w3, r, D, row3);
    for (int d = 0; d < D; ++d) {
      g += row[d] * xh[d];
      u += row3[d] * xh[d];
      sg += fabs(row[d] * xh[d]);
      su += fabs(row3[d] * xh[d]);
    }
    h[r] = (float)orc_swiglu(g, u, c->swiglu_limit, NULL);
    swiglu_range(g, u, kappa * sg, kappa * su, c->swiglu_limit, &lo[r], &hi[r]);
  }
  for (int b = 0; b < I / 32; ++b) {
    const float* hb = h + 32 * b;
    float amax = 0.0f, alo = 0.0f, ahi = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(hb[i]);
      if (a > amax) amax = a;
      float l = lo[32 * b + i], u = hi[32 * b + i];
      float mn = (l <= 0.0f && u >= 0.0f) ? 0.0f : fminf(fabsf(l), fabsf(u));
      float mx = fmaxf(fabsf(l), fabsf(u));
      if (mn > alo) alo = mn;
      if (mx > ahi) ahi = mx;
    }
    const float d = (amax / 127.0f);  /* the q8_1 rule, reading C-L3 */
    uint16_t d16 = orc_f16_from_f32(d);
    double dv = orc_f16_value(d16);
    int q[32];
    for (int i = 0; i < 32; ++i) q[i] = q8_code(hb[i], d, amax);
    for (int i = 0; i < 32; ++i) {
      int qa = q8_code(lo[32 * b + i], d, amax), qb = q8_code(hi[32 * b + i], d, amax);
      for (int qq = qa; qq <= qb; ++qq) {
        if (qq == q[i]) continue;
        flip_cand* f = flip_push(F);
        f->slot = slot; f->kind = 0; f->index = 32 * b + i; f->alt = qq;
        f->j0 = 32 * b + i; f->n = 1;
        f->coef[0] = G * (double)(qq - q[i]) * dv;
      }
    }
    float ends[2] = {alo, ahi};
    uint16_t seen = d16;
    for (int e = 0; e < 2; ++e) {
      float d2 = ends[e] / 127.0f;
      uint16_t b16 = orc_f16_from_f32(d2);
      if (b16 == d16 || b16 == seen) continue;
      seen = b16;
      double dv2 = orc_f16_value(b16);
      flip_cand* f = flip_push(F);
      f->slot = slot; f->kind = 1; f->index = b; f->alt = b16;
      f->j0 = 32 * b; f->n = 32;
      int any = 0;
      for (int i = 0; i < 32; ++i) {
        int q2 = q8_code(hb[i], d2, ends[e]);
        f->coef[i] = G * ((double)q2 * dv2 - (double)q[i] * dv);
        any |= f->coef[i] != 0.0;
      }
      if (!any) --F->n;
    }
  }
  free(row); free(row3); free(h); free(lo); free(hi);
}

/* bf16 bits as an integer in value order (-0 and +0 alike). */
static int bf16_key(uint16_t b) { return (b & 0x8000u) ? -(int)(b & 0x7FFFu) : (int)b; }

enum { BF16_SPAN = 16 };

/* The bf16 candidates of the bf16 shared expert on one token. */
static void flips_bf16(const orc_cfg* c, const uint16_t* x, const uint16_t* w1, const uint16_t* w3, int slot,
                       double kappa, flip_list* F) {
  int D = c->dim, I = c->inter;
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0, sg = 0.0, su = 0.0;
    for (int d = 0; d < D; ++d) {
      double xv = orc_bf16_value(x[d]);
      double a = orc_bf16_value(w1[(size_t)r * D + d]) * xv, b = orc_bf16_value(w3[(size_t)r * D + d]) * xv;
      g += a; u += b; sg += fabs(a); su += fabs(b);
    }
    float h = (float)orc_swiglu(g, u, c->swiglu_limit, NULL);
    float lo, hi;
    swiglu_range(g, u, kappa * sg, kappa * su, c->swiglu_limit, &lo, &hi);
    /* every bf16 value between those of the window's ends (bf16 bits in
     * value order: the sign-magnitude key); a window over more than
     * BF16_SPAN values (h near 0) gives its two ends only */
    uint16_t hb = orc_bf16_from_f32(h);
    int k0 = bf16_key(orc_bf16_from_f32(lo)), k1 = bf16_key(orc_bf16_from_f32(hi)), kh = bf16_key(hb);
    for (int key = k0; key <= k1; ++key) {
      if (key == kh || (k1 - k0 > BF16_SPAN && key != k0 && key != k1)) continue;
      uint16_t alt = key < 0 ? (uint16_t)(0x8000 | -key) : (uint16_t)key;
      flip_cand* f = flip_push(F);
      f->slot = slot; f->kind = 2; f->index = r; f->alt = alt;
      f->j0 = r; f->n = 1;
      f->coef[0] = orc_bf16_value(alt) - orc_bf16_value(hb);
    }
  }
}

/* Row d of an expert's W2 as f64 values. */
static void w2_row(int kquant, const void* w2, int d, int I, double* row) {
  if (kquant) dequant_row(3, (const uint8_t*)w2, d, I, row);
  else
    for (int j = 0; j < I; ++j) row[j] = orc_bf16_value(((const uint16_t*)w2)[(size_t)d * I + j]);
}

/* The change of one candidate in the output element whose W2 row is `row`. */
static double flip_change(const flip_cand* f, const double* row) {
  double s = 0.0;
  for (int i = 0; i < f->n; ++i) s += f->coef[i] * row[f->j0 + i];
  return s;
}

/* Candidates [from, F->n) of one expert: those whose output change reaches
 * min_change in some element stay (the others are dropped from F), and the
 * output changes of the ones among the first max_c overall are written.
 * Two passes over the rows of W2: the largest change of each, then the
 * changes. */
static void flip_deltas(const orc_cfg* c, flip_list* F, int from, int max_c, int kquant, const void* w2,
                        double min_change, double* delta) {
  int D = c->dim, I = c->inter, n = F->n - from;
  if (n <= 0) return;
  double* row = (double*)malloc(sizeof(double) * I);
  double* big = (double*)calloc((size_t)n, sizeof(double));
  for (int d = 0; d < D; ++d) {
    w2_row(kquant, w2, d, I, row);
    for (int k = 0; k < n; ++k) {
      double s = fabs(flip_change(&F->v[from + k], row));
      if (s > big[k]) big[k] = s;
    }
  }
  int kept = from;
  for (int k = 0; k < n; ++k)
    if (big[k] >= min_change && big[k] > 0.0) F->v[kept++] = F->v[from + k];
  F->n = kept;
  int to = F->n < max_c ? F->n : max_c;
  if (from < to) {
    for (int d = 0; d < D; ++d) {
      w2_row(kquant, w2, d, I, row);
      for (int k = from; k < to; ++k) delta[(size_t)k * D + d] = flip_change(&F->v[k], row);
    }
  }
  free(row); free(big);
}

int orc_flip_candidates(const orc_cfg* c, const orc_layer* L, int t, const float* w, const int32_t* idx,
                        double kappa, double min_change, int max_c, int32_t* meta, double* delta) {
  int D = c->dim, k = c->topk;
  const uint16_t* xt = L->x + (size_t)t * D;
  float* xf = (float*)malloc(sizeof(float) * D);
  uint8_t* xq8 = (uint8_t*)malloc((size_t)36 * (D / 32));
  double* xh = (double*)malloc(sizeof(double) * D);
  for (int d = 0; d < D; ++d) xf[d] = (float)orc_bf16_value(xt[d]);
  orc_quantize_q8_1(xf, D, xq8);
  orc_dequant_q8_1(xq8, D, xh);
  flip_list F = {0};
  int status = 0;
  for (int s = 0; s <= k && !status; ++s) {
    int from = F.n;
    if (s < k) {
      const uint8_t* const* ex = L->experts + 3 * idx[s];
      if (!ex[0] || !ex[1] || !ex[2]) { status = -ORC_ERR_MISSING_EXPERT; break; }
      flips_kquant(c, xh, ex[0], ex[1], (double)w[s], s, kappa, &F);
      flip_deltas(c, &F, from, max_c, 1, ex[2], min_change, delta);
    } else if (L->shared_kind == ORC_SHARED_KQUANT) {
      flips_kquant(c, xh, (const uint8_t*)L->sh1, (const uint8_t*)L->sh3, 1.0, s, kappa, &F);
      flip_deltas(c, &F, from, max_c, 1, L->sh2, min_change, delta);
    } else {
      flips_bf16(c, xt, (const uint16_t*)L->sh1, (const uint16_t*)L->sh3, s, kappa, &F);
      flip_deltas(c, &F, from, max_c, 0, L->sh2, min_change, delta);
    }
  }
  int n = status ? status : F.n;
  for (int i = 0; i < F.n && i < max_c && !status; ++i) {
    meta[4 * i + 0] = F.v[i].slot;
    meta[4 * i + 1] = F.v[i].kind;
    meta[4 * i + 2] = F.v[i].index;
    meta[4 * i + 3] = F.v[i].alt;
  }
  free(F.v); free(xf); free(xq8); free(xh);
  return n;
}
