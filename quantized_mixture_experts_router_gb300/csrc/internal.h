// Parameter blocks and host launchers shared by the kernel files and the
// C-ABI file.
#pragma once

#include "common.cuh"

namespace moe {

struct SelectParams {
  const float* logits;  // [m, N]
  const float* bias;    // [N]
  int m, N, k, norm;
  float gate_temp, route_scale;
  float* topk_w;
  int* topk_idx;
  Ctrl* ctrl;
};

struct RouteParams {
  const uint16_t* x;         // bf16 [m, D]
  const uint16_t* router_w;  // bf16 [N, D]
  const float* bias;
  int m, D, N, k, norm;
  float gate_temp, route_scale;
  float* logits;             // [m, N]
  float* topk_w;
  int* topk_idx;
  uint8_t* xq8;              // q8_1 blocks [m][D/32]
  int* xu;                   // unit layout [m][...]
  DecodePlan* plan;          // nullptr: routing only
  const unsigned long long* expert_ptrs;
  Ctrl* ctrl;
};

struct DecodeParams {
  int m, D, I, k;
  float swiglu_limit;
  int shared_kind;
  const uint8_t* sh1;
  const uint8_t* sh3;
  const uint8_t* sh2;
  const uint16_t* x;     // bf16 [m, D]
  const int* xu;         // unit layout of q8_1(x)
  int* hu;               // unit layout of q8_1(h), one vector per pair
  uint8_t* shh;          // shared h: bf16 [m, I] or unit layout per token
  const DecodePlan* plan;
  float* out;            // f32 [m, D]
  Ctrl* ctrl;
  unsigned long long timeout_ns;
};

int launch_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, void* q8, cudaStream_t s);
int launch_select(const SelectParams& p, cudaStream_t s);
int launch_route_decode(const RouteParams& p, cudaStream_t s);
int launch_decode_experts(const DecodeParams& p, int num_sms, cudaStream_t s);

}  // namespace moe
