// Routing kernels: the q8_1 activation quantiser (plain q8_1 blocks and the
// unit layout the K-quant dots read), the router GEMV for up to eight tokens
// with the selection done on the device by the grid's last block, and the
// selection alone from given logits (one warp per token).
//
// Method: metrale moe_v41 module docs / moe_v41.rs source (route_from_logits:
// scores sqrt(softplus(logit / gate_temp)), keys score + bias, stable
// descending order with ties to the lower id, weights the unbiased scores
// renormalised when norm_topk_prob and topk > 1, times route_scale);
// DeepSeek V4.1 atlas "Mixture of experts", model.py Gate.forward (sigmoid
// and softmax scores; bias_vl for image tokens).
#include "internal.h"
#include "bf16dot.cuh"
#include "select.cuh"

namespace moe {

// Standalone quantiser: rows x cols (bf16 or f32) -> q8_1 blocks.
__global__ void k_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, uint8_t* q8) {
  const int nblk = cols / 32;
  const long total = (long)rows * nblk;
  const int lane = threadIdx.x & 31;
  for (long w = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; w < total;
       w += ((long)gridDim.x * blockDim.x) >> 5) {
    const long r = w / nblk;
    const int qb = (int)(w % nblk);
    const long e = r * cols + (long)qb * 32 + lane;
    float v = x_is_f32 ? reinterpret_cast<const float*>(x)[e]
                       : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[e]);
    q8_block_warp(v, qb, q8 + (size_t)r * nblk * Q8_B, nullptr);
  }
}

__global__ void k_select(SelectParams p) {
  extern __shared__ __align__(16) float sel_scratch[];
  const int warps = (gridDim.x * blockDim.x) >> 5;
  float* scratch = sel_scratch + (size_t)(threadIdx.x >> 5) * (select_scratch_bytes(p.N) / 4);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < p.m; t += warps)
    route_token_warp(p.logits + (size_t)t * p.N, nullptr, token_bias(p.bias, p.bias_vl, p.image_mask, t), p.N, p.k,
                     p.gate_temp, p.score_func, p.norm, p.route_scale, p.topk_w + (size_t)t * p.k,
                     p.topk_idx + (size_t)t * p.k, &p.ctrl->status, scratch);
}

// ---------------------------------------------- router + selection (m <= 8)
// Warps 0..N-1 (over the grid) compute one router row each for all m tokens;
// the remaining warps quantise x.  The last block to finish selects the
// experts of every token (moe_v41_route).
__global__ void __launch_bounds__(256) k_route_decode(RouteParams p) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int chunks = p.D / 8;  // 16-B chunks of a bf16 row
  if (gw < p.N) {
    // the fused decode kernel's order (bf16dot.cuh): same logits, bit for bit
    const uint4* wrow = reinterpret_cast<const uint4*>(p.router_w + (size_t)gw * p.D);
    float2 a[DECODE_MAX_M], b[DECODE_MAX_M];
#pragma unroll
    for (int t = 0; t < DECODE_MAX_M; ++t) a[t] = b[t] = make_float2(0.f, 0.f);
#pragma unroll 1
    for (int ch = lane; ch < chunks; ch += 64) {
      const bool two = ch + 32 < chunks;
      const uint4 w0 = __ldg(wrow + ch);
      const uint4 w1 = two ? __ldg(wrow + ch + 32) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int t = 0; t < DECODE_MAX_M; ++t) {
        if (t < p.m) {
          const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
          dot8(a[t], w0, __ldg(xr + ch));
          if (two) dot8(b[t], w1, __ldg(xr + ch + 32));
        }
      }
    }
#pragma unroll
    for (int t = 0; t < DECODE_MAX_M; ++t) {
      const float z = warp_sum(lane_total(a[t], b[t]));
      if (lane == 0 && t < p.m) p.logits[(size_t)t * p.N + gw] = z;
    }
  } else {
    // q8_1 of x: one warp per q8_1 block
    const int nq = p.D / 32;
    const int wq = gw - p.N;
    if (wq < p.m * nq) {
      const int t = wq / nq, qb = wq % nq;
      const float v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.x)[(size_t)t * p.D + qb * 32 + lane]);
      q8_block_warp(v, qb, p.xq8 + (size_t)t * nq * Q8_B, p.xu + (size_t)t * (unit_bytes(p.D) / 4));
    }
  }

  // ---- last block: selection and grouping
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&p.ctrl->route_arrive, 1u);
    s_last = (prev == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) {
    p.ctrl->route_arrive = 0u;  // ready for the next call
  }
  extern __shared__ __align__(16) float sel_scratch[];
  const int warp = threadIdx.x >> 5;
  if (warp < p.m)
    route_token_warp(p.logits + (size_t)warp * p.N, nullptr, token_bias(p.bias, p.bias_vl, p.image_mask, warp), p.N,
                     p.k, p.gate_temp, p.score_func, p.norm, p.route_scale, p.topk_w + (size_t)warp * p.k,
                     p.topk_idx + (size_t)warp * p.k, &p.ctrl->status,
                     sel_scratch + (size_t)warp * (select_scratch_bytes(p.N) / 4));
}

// ------------------------------------------------------------- launchers
int launch_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, void* q8, cudaStream_t s) {
  const long warps = (long)rows * (cols / 32);
  long blocks = (warps * 32 + 255) / 256;
  if (blocks > 152L * 16) blocks = 152L * 16;
  if (blocks < 1) blocks = 1;
  k_quantize_q8_1<<<(unsigned)blocks, 256, 0, s>>>(x, x_is_f32, rows, cols, (uint8_t*)q8);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_select(const SelectParams& p, cudaStream_t s) {
  constexpr int WPB = 4;  // warps (tokens) per block
  const size_t smem = WPB * select_scratch_bytes(p.N);
  long blocks = ((long)p.m + WPB - 1) / WPB;
  if (blocks > 152L * 16) blocks = 152L * 16;
  k_select<<<(unsigned)blocks, WPB * 32, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_route_decode(const RouteParams& p, cudaStream_t s) {
  const long warps = (long)p.N + (long)p.m * (p.D / 32);
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  const size_t smem = (size_t)p.m * select_scratch_bytes(p.N);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k_route_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  k_route_decode<<<blocks, 256, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
