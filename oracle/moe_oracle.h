/* CPU oracle of the DeepSeek-V4.1 MoE FFN on still-quantized experts.
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  Shares no code with the GPU path. */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

typedef struct {
  int32_t dim, inter, n_routed, topk;
  float gate_temp;
  int32_t norm_topk_prob;
  float route_scale, swiglu_limit;
  int32_t score_func;              /* ORC_SCORE_*: the Gate's score function */
} orc_cfg;

/* [MoE atlas] model.py Gate.forward: score_func "sqrtsoftplus" (the default),
 * "sigmoid" or "softmax" over the experts */
enum { ORC_SCORE_SQRTSOFTPLUS = 0, ORC_SCORE_SIGMOID = 1, ORC_SCORE_SOFTMAX = 2 };

enum { ORC_SHARED_BF16 = 0, ORC_SHARED_KQUANT = 1 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_MISSING_EXPERT = 2 };

typedef struct {
  const uint16_t* x;               /* bf16 [m, dim] */
  const uint16_t* router_w;        /* bf16 [n_routed, dim] */
  const float* bias;               /* f32 [n_routed] */
  const float* given_logits;       /* optional f32 [m, n_routed]: skip the router */
  const uint8_t* const* experts;   /* [n_routed * 3] host pointers {w1, w3, w2}; NULL = absent */
  int32_t shared_kind;
  const void* sh1;                 /* bf16 [inter, dim] or Q2_K */
  const void* sh3;                 /* bf16 [inter, dim] or Q2_K */
  const void* sh2;                 /* bf16 [dim, inter] or Q3_K */
  const float* bias_vl;            /* optional f32 [n_routed]: the bias of image tokens */
  const uint8_t* image_mask;       /* optional [m]: nonzero for tokens inside an image span */
} orc_layer;

typedef struct {
  int32_t nan_keys;
  int32_t clipped;
} orc_stats;

double orc_bf16_value(uint16_t b);
uint16_t orc_bf16_from_f32(float v);
double orc_f16_value(uint16_t h);
uint16_t orc_f16_from_f32(float v);
void orc_dequant_q2k(const uint8_t* blk, double* w);
void orc_dequant_q3k(const uint8_t* blk, double* w);
int orc_q3k_scale_code(const uint8_t* scales12, int b);
void orc_dequant_matrix(int kind, const uint8_t* mat, int rows, int cols, double* out);
void orc_quantize_q8_1(const float* x, int n, uint8_t* out);
void orc_dequant_q8_1(const uint8_t* q8, int n, double* out);
void orc_router_logits(const uint16_t* x, int m, const uint16_t* W, int D, int N, float* z);
float orc_score(float z, float gate_temp);
void orc_scores(const orc_cfg* c, const float* z, float* s);
int orc_route_token(const orc_cfg* c, const float* z, const float* bias, float* w_out, int32_t* idx_out);
int orc_route_from_logits(const orc_cfg* c, const float* z, int m, const float* bias, float* w_out,
                          int32_t* idx_out);
int orc_route_from_logits_vl(const orc_cfg* c, const float* z, int m, const float* bias, const float* bias_vl,
                             const uint8_t* image_mask, float* w_out, int32_t* idx_out);
double orc_swiglu(double g, double u, double limit, int* clipped);
void orc_expert_kquant(const orc_cfg* c, const uint8_t* xq8, const uint8_t* w1, const uint8_t* w3,
                       const uint8_t* w2, double* E, int* clipped);
void orc_shared_bf16(const orc_cfg* c, const uint16_t* x, const uint16_t* w1, const uint16_t* w3,
                     const uint16_t* w2, double* S, int* clipped);
/* Requantisation alternatives of one token (reading C-F1 in moe_oracle.c):
 * meta [max_c][4], delta [max_c][dim]; returns the count (or -status). */
int orc_flip_candidates(const orc_cfg* c, const orc_layer* L, int t, const float* w, const int32_t* idx,
                        double kappa, double min_change, int max_c, int32_t* meta, double* delta);
int orc_moe_layer(const orc_cfg* c, const orc_layer* L, const int32_t* tokens, int n_tok, double* out,
                  float* topk_w, int32_t* topk_idx, int nthreads, orc_stats* stats);
/* Brute-force mode for small inputs: dense f64 matrices up front, textbook
 * loops over all m tokens (no token subset, no threads). */
int orc_moe_layer_dense(const orc_cfg* c, const orc_layer* L, int m, double* out, float* topk_w,
                        int32_t* topk_idx);

#endif
