// Parameter blocks and host launchers shared by the kernel files and the
// C-ABI file.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {

struct SelectParams {
  const float* logits;  // [m, N]
  const float* bias;    // [N]
  const float* bias_vl;        // [N] or NULL: the bias of image tokens
  const uint8_t* image_mask;   // [m] or NULL: nonzero marks an image token
  int m, N, k, norm, score_func;
  float gate_temp, route_scale;
  float* topk_w;
  int* topk_idx;
  Ctrl* ctrl;
};

struct RouteParams {
  const uint16_t* x;         // bf16 [m, D]
  const uint16_t* router_w;  // bf16 [N, D]
  const float* bias;
  const float* bias_vl;      // [N] or NULL
  const uint8_t* image_mask; // [m] or NULL
  int m, D, N, k, norm, score_func;
  float gate_temp, route_scale;
  float* logits;             // [m, N]
  float* topk_w;
  int* topk_idx;
  uint8_t* xq8;              // q8_1 blocks [m][D/32]
  int* xu;                   // unit layout [m][...]
  Ctrl* ctrl;
};

struct DecodeParams {
  int m, D, I, N, k, norm, score_func;
  float gate_temp, route_scale, swiglu_limit;
  int shared_kind;
  const uint16_t* x;         // bf16 [m, D]
  const uint16_t* router_w;  // bf16 [N, D]
  const float* bias;         // [N]
  const float* bias_vl;      // [N] or NULL: the bias of image tokens
  const uint8_t* image_mask; // [m] or NULL: nonzero marks an image token
  const unsigned long long* expert_ptrs;  // [N][3]
  const uint8_t* sh1;
  const uint8_t* sh3;
  const uint8_t* sh2;
  float* logits;             // [m, N]
  float2* sk;                // (fast score, fast key) [m, N]
  float* topk_w;             // [m, k]
  int* topk_idx;             // [m, k]
  int* xu;                   // unit layout of q8_1(x) (when not kept in shared memory)
  int* hu;                   // unit layout of q8_1(h), one per vector (pairs, then shared tokens)
  uint8_t* shh;              // bf16 shared expert: h [m, I] bf16
  int shvec0;                // first vector index of the shared expert's tokens
  float* out;                // f32 [m, D]
  Ctrl* ctrl;
  unsigned long long timeout_ns;
  // shared-memory plan of the launch (set by launch_decode_layer); a cache
  // offset of 0 means "not cached, read from global memory"
  uint32_t sm_ctl, sm_plan, sm_items, item_bytes, sm_sel, sm_xb, sm_ep, ep_bytes, sm_x, sm_hr, sm_hs, sm_bias,
      smem_bytes;
};

struct PrefillParams {
  int m, D, I, N, k, norm, score_func;
  float gate_temp, route_scale, swiglu_limit;
  int shared_kind;
  const uint16_t* x;         // bf16 [m, D]
  const uint16_t* router_w;  // bf16 [N, D]
  const float* bias;         // [N]
  const float* bias_vl;      // [N] or NULL
  const uint8_t* image_mask; // [m] or NULL
  const unsigned long long* expert_ptrs;  // [N][3]
  const uint8_t* sh1;
  const uint8_t* sh3;
  const uint8_t* sh2;
  float* logits;             // [m, N]
  float* topk_w;             // [m, k]
  int* topk_idx;             // [m, k]
  float* out;                // f32 [m, D]
  Ctrl* ctrl;
  uint8_t* pw;               // the workspace's prefill region
  PrefillLayout L;
  unsigned long long timeout_ns;
};

// Configuration checks every entry point starts with: MOE_OK, or MOE_ERR_ARG
// for a value out of the ranges include/moe_v41.h states.
inline int check_cfg(const moe_v41_cfg* c) {
  if (!c) return MOE_ERR_ARG;
  if (c->dim < 256 || c->dim > 7680 || c->dim % 256) return MOE_ERR_ARG;
  if (c->inter < 256 || c->inter > 7680 || c->inter % 256) return MOE_ERR_ARG;
  if (c->n_routed < 1 || c->n_routed > MAX_N) return MOE_ERR_ARG;
  if (c->topk < 1 || c->topk > MAX_TOPK || c->topk > c->n_routed) return MOE_ERR_ARG;
  if (!(c->gate_temp > 0.0f)) return MOE_ERR_ARG;
  if (c->max_tokens < 1 || c->max_tokens > 65536) return MOE_ERR_ARG;
  if (c->path < MOE_PATH_AUTO || c->path > MOE_PATH_PREFILL) return MOE_ERR_ARG;
  if (c->score_func < MOE_SCORE_SQRTSOFTPLUS || c->score_func > MOE_SCORE_SOFTMAX) return MOE_ERR_ARG;
  return MOE_OK;
}

// One launch of the persistent exact down GEMM of the routed experts (k_prefill_kq.cu).
struct KqLaunch {
  const void* bh;                       // q8_1(h) as fp16 hi / lo parts [b_rows][K]
  const void* bl;
  int b_rows;
  const int4* tiles;                    // two int4 per tile: (expert, row tile, first pair, pairs <= PF_TNQ),
                                        // the address of the tile's first W2 row
  const int* n_tiles;                   // device count of tiles
  int K, a_row_bytes, out_ld;
  float* out_e;                         // E f32 [pair][out_ld]
  unsigned* status;
  unsigned long long timeout_ns;
  unsigned grid;                        // persistent blocks (one per SM)
};
int launch_kq_gemm(const KqLaunch& L, cudaStream_t s);

// A tensor map of a row-major matrix of 16-bit values [rows][cols] (cols a
// multiple of 64, row pitch a multiple of 16 bytes), read in boxes of 64
// values x box_rows rows into 128-byte-swizzled shared memory; rows past the
// end read zeros.
bool make_map_b16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);

int launch_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, void* q8, cudaStream_t s);
int launch_select(const SelectParams& p, cudaStream_t s);
int launch_route_decode(const RouteParams& p, cudaStream_t s);
int launch_decode_layer(const DecodeParams& p, int num_sms, cudaStream_t s);
bool decode_fits(int D, int I);
int launch_prefill(const PrefillParams& p, cudaStream_t s);
int launch_prefill_route(const PrefillParams& p, cudaStream_t s);
int prefill_launches(int shared_kind);
size_t decode_smem_bytes();

// The routing of m tokens with k picks per token (k may differ from
// cfg->topk; 1 <= k <= min(MAX_TOPK, n_routed)) into the workspace's pred
// region: *idx_out receives its device address ([m, k] int32, the weights
// follow the ids).  The router kernel and order are those of moe_v41_route.
int route_topk(const moe_v41_cfg* cfg, int k, const void* x, int m, const void* router_w, const float* bias,
               int32_t** idx_out, void* ws, size_t ws_bytes, cudaStream_t s);

}  // namespace moe
