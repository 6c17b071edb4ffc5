// bf16 dot products with f32 accumulation in one fixed order, shared by the
// fused decode kernel's router rows and the standalone router kernel, so that
// both produce bit-identical logits for the same x and router rows (the
// selection of a separate route call then equals the forward's own).
//
// Order of one row (`chunks` 16-byte chunks of 8 bf16 values): lane l takes
// chunks l, l + 64, l + 128, ... into accumulator pair a and chunks l + 32,
// l + 96, ... into pair b; within a chunk the low halves go to .x and the
// high halves to .y in element order; the lane's value is
// (a.x + a.y) + (b.x + b.y), and the warp sums the lanes with an xor
// butterfly (offsets 16, 8, 4, 2, 1).
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// c + a*b for the low (hi = 0) or high bf16 halves of a and b, with one f32
// rounding: the mixed-precision fma takes the bf16 operands directly, the same
// result as fmaf on the widened values without the two unpacking instructions.
__device__ __forceinline__ float fma_bf16(uint32_t a, uint32_t b, float c, int hi) {
  unsigned short al, ah, bl, bh;
  asm("mov.b32 {%0, %1}, %2;" : "=h"(al), "=h"(ah) : "r"(a));
  asm("mov.b32 {%0, %1}, %2;" : "=h"(bl), "=h"(bh) : "r"(b));
  if (hi) asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(ah), "h"(bh));
  else asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(al), "h"(bl));
  return c;
}

// 8 bf16 products into two accumulators (two independent FMA chains)
__device__ __forceinline__ void dot8(float2& acc, const uint4& w, const uint4& x) {
  acc.x = fma_bf16(w.x, x.x, acc.x, 0); acc.y = fma_bf16(w.x, x.x, acc.y, 1);
  acc.x = fma_bf16(w.y, x.y, acc.x, 0); acc.y = fma_bf16(w.y, x.y, acc.y, 1);
  acc.x = fma_bf16(w.z, x.z, acc.x, 0); acc.y = fma_bf16(w.z, x.z, acc.y, 1);
  acc.x = fma_bf16(w.w, x.w, acc.x, 0); acc.y = fma_bf16(w.w, x.w, acc.y, 1);
}

// the lane's share of one row, combined as the order above states
__device__ __forceinline__ float lane_total(const float2& a, const float2& b) { return (a.x + a.y) + (b.x + b.y); }

}  // namespace moe
