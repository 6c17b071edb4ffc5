// Routing kernels: the q8_1 activation quantiser (plain q8_1 blocks and the
// unit layout the K-quant dots read), the router GEMV for up to eight tokens
// with the selection done on the device by the grid's last block, and the
// selection alone from given logits (one warp per token).
//
// Method: metrale moe_v41 module docs / moe_v41.rs source (route_from_logits:
// scores sqrt(softplus(logit / gate_temp)), keys score + bias, stable
// descending order with ties to the lower id, weights the unbiased scores
// renormalised when norm_topk_prob and topk > 1, times route_scale);
// DeepSeek V4.1 atlas "Mixture of experts", model.py Gate.forward.
#include "internal.h"

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

// ------------------------------------------------------------- selection
// Order-preserving 64-bit key: larger = ranks first.  NaN ranks below every
// number; equal keys rank by lower expert id.  -0 and +0 are equal keys.
__device__ __forceinline__ unsigned long long rank_key(float key, int id) {
  uint32_t u;
  if (key != key) {
    u = 0u;
  } else {
    key = key + 0.0f;  // -0 -> +0
    u = __float_as_uint(key);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Score with every step correctly rounded or evaluated in f64 and rounded
// once: t = z / T (f32); t > 20: sqrt(t) (f32); else f32(sqrt(log1p(exp(t)))) in f64.
__device__ __forceinline__ float score_exact(float z, float T) {
  const float t = __fdiv_rn(z, T);
  if (t > 20.0f) return __fsqrt_rn(t);
  return __double2float_rn(sqrt(log1p(exp((double)t))));
}

// The same in f32 with the accurate single-precision functions: within a few
// ulp of score_exact; used only to find the candidates near the cut.
__device__ __forceinline__ float score_fast(float z, float T) {
  const float t = __fdiv_rn(z, T);
  if (t > 20.0f) return __fsqrt_rn(t);
  return __fsqrt_rn(log1pf(expf(t)));
}

constexpr int SEL_PER_LANE = MAX_N / 32;

// One token's routing by one warp.  The top k are found on f32 keys first;
// every expert whose f32 key lies within delta of the k-th is re-scored with
// score_exact, and the picks are taken among those on the exact keys.  With
// |fast - exact| <= eps for every key and delta >= 2 eps, every exact top-k
// expert is among the candidates, so the picks equal the exact selection.
__device__ void route_token_warp(const float* __restrict__ z, const float* __restrict__ bias, int N, int k,
                                 float T, int norm, float route_scale, float* w_out, int* idx_out, unsigned* status) {
  const int lane = threadIdx.x & 31;
  float kf[SEL_PER_LANE];
  bool any_nan = false;
#pragma unroll
  for (int i = 0; i < SEL_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float key = -INFINITY;
    if (e < N) {
      key = __fadd_rn(score_fast(z[e], T), bias[e]);
      any_nan |= (key != key);
    }
    kf[i] = key;
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) atomicOr(status, (unsigned)MOE_STATUS_NAN_KEY);
  // k-th largest fast key (rank keys, ties by id); taken entries masked out
  uint32_t taken = 0;
  unsigned long long kth = 0;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0;
#pragma unroll
    for (int i = 0; i < SEL_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < N && !(taken >> i & 1u)) {
        const unsigned long long rk = rank_key(kf[i], e);
        best = rk > best ? rk : best;
      }
    }
    best = warp_max_u64(best);
    kth = best;
    const int win = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
  }
  // candidate threshold from the k-th fast key
  const int kth_id = (int)(0xFFFFFFFFu - (uint32_t)(kth & 0xFFFFFFFFu));
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < SEL_PER_LANE; ++i)
    if (i == (kth_id >> 5)) mine = kf[i];
  const float kth_key = __shfl_sync(0xffffffffu, mine, kth_id & 31);
  const bool kth_nan = kth_key != kth_key;
  const float delta = 0x1.0p-10f * fmaxf(1.0f, fabsf(kth_key));
  const float thresh = kth_key - delta;
  // exact keys of the candidates
  float se[SEL_PER_LANE];
  uint32_t cand = 0;
#pragma unroll
  for (int i = 0; i < SEL_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    se[i] = 0.f;
    if (e < N && (kth_nan || !(kf[i] < thresh))) {
      cand |= 1u << i;
      se[i] = score_exact(z[e], T);
      kf[i] = __fadd_rn(se[i], bias[e]);
    }
  }
  float picked_s[MAX_TOPK];
  int picked_id[MAX_TOPK];
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < SEL_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (cand >> i & 1u) {
        // rank keys are distinct (the id is in the low word) and never 0,
        // so a NaN candidate still beats "no candidate left"
        const unsigned long long rk = rank_key(kf[i], e);
        if (rk > best) {
          best = rk;
          bs = se[i];
        }
      }
    }
    const unsigned long long wmax = warp_max_u64(best);
    const int win = (int)(0xFFFFFFFFu - (uint32_t)(wmax & 0xFFFFFFFFu));
    const float ws = __shfl_sync(0xffffffffu, bs, win & 31);
    if ((win & 31) == lane) cand &= ~(1u << (win >> 5));
    if (r < MAX_TOPK) {
      picked_s[r] = ws;
      picked_id[r] = win;
    }
  }
  if (lane == 0) {
    float w[MAX_TOPK];
    for (int r = 0; r < k; ++r) w[r] = picked_s[r];
    if (norm && k > 1) {
      float sum = 0.f;
      for (int r = 0; r < k; ++r) sum = __fadd_rn(sum, w[r]);
      sum = __fadd_rn(sum, 1e-20f);
      for (int r = 0; r < k; ++r) w[r] = __fdiv_rn(w[r], sum);
    }
    for (int r = 0; r < k; ++r) {
      w_out[r] = __fmul_rn(w[r], route_scale);
      idx_out[r] = picked_id[r];
    }
  }
}

__global__ void k_select(SelectParams p) {
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < p.m; t += warps)
    route_token_warp(p.logits + (size_t)t * p.N, p.bias, p.N, p.k, p.gate_temp, p.norm, p.route_scale,
                     p.topk_w + (size_t)t * p.k, p.topk_idx + (size_t)t * p.k, &p.ctrl->status);
}

// --------------------------------------------- decode router + selection
// Warps 0..N-1 (over the grid) compute one router row each for all m tokens;
// the remaining warps quantise x.  The last block to finish selects the
// experts of every token and groups the (expert, token) pairs by ascending
// expert id into the decode plan.
__global__ void __launch_bounds__(256) k_route_decode(RouteParams p) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int chunks = p.D / 8;  // 16-B chunks of a bf16 row
  if (gw < p.N) {
    const uint4* wrow = reinterpret_cast<const uint4*>(p.router_w + (size_t)gw * p.D);
    float acc[DECODE_MAX_M];
#pragma unroll
    for (int t = 0; t < DECODE_MAX_M; ++t) acc[t] = 0.f;
    for (int c0 = 0; c0 < chunks; c0 += 32 * 8) {
      uint4 wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        wv[i] = c < chunks ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c >= chunks) break;
        const float w0 = bf16lo(wv[i].x), w1 = bf16hi(wv[i].x), w2 = bf16lo(wv[i].y), w3 = bf16hi(wv[i].y);
        const float w4 = bf16lo(wv[i].z), w5 = bf16hi(wv[i].z), w6 = bf16lo(wv[i].w), w7 = bf16hi(wv[i].w);
#pragma unroll
        for (int t = 0; t < DECODE_MAX_M; ++t) {
          if (t < p.m) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D) + c);
            float a = acc[t];
            a = fmaf(w0, bf16lo(xv.x), a); a = fmaf(w1, bf16hi(xv.x), a);
            a = fmaf(w2, bf16lo(xv.y), a); a = fmaf(w3, bf16hi(xv.y), a);
            a = fmaf(w4, bf16lo(xv.z), a); a = fmaf(w5, bf16hi(xv.z), a);
            a = fmaf(w6, bf16lo(xv.w), a); a = fmaf(w7, bf16hi(xv.w), a);
            acc[t] = a;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < DECODE_MAX_M; ++t) {
      float a = acc[t];
#pragma unroll
      for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0 && t < p.m) p.logits[(size_t)t * p.N + gw] = a;
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
    p.ctrl->ticket_gu = 0u;
    p.ctrl->ticket_dn = 0u;
  }
  const int warp = threadIdx.x >> 5;
  if (warp < p.m)
    route_token_warp(p.logits + (size_t)warp * p.N, p.bias, p.N, p.k, p.gate_temp, p.norm, p.route_scale,
                     p.topk_w + (size_t)warp * p.k, p.topk_idx + (size_t)warp * p.k, &p.ctrl->status);
  __syncthreads();
  if (!p.plan) return;
  // group the m*k pairs by (expert, token): rank of each pair among all
  __shared__ int s_e[MAXP], s_t[MAXP], s_first[MAXP], s_sorted_e[MAXP];
  __shared__ float s_w[MAXP];
  const int P = p.m * p.k;
  const int i = threadIdx.x;
  int e = 0, t = 0;
  float w = 0.f;
  if (i < P) {
    t = i / p.k;
    e = __ldcg(p.topk_idx + i);
    w = __ldcg(p.topk_w + i);
  }
  __syncthreads();
  if (i < P) { s_e[i] = e; s_t[i] = t; s_w[i] = w; }
  __syncthreads();
  DecodePlan* plan = p.plan;
  if (i < P) {
    int rank = 0;
    for (int q = 0; q < P; ++q)
      rank += (s_e[q] < e) || (s_e[q] == e && s_t[q] < t);
    plan->pair_tok[rank] = t;
    plan->pair_w[rank] = w;
    s_sorted_e[rank] = e;
  }
  __syncthreads();
  if (i < P) s_first[i] = (i == 0 || s_sorted_e[i - 1] != s_sorted_e[i]) ? 1 : 0;
  __syncthreads();
  if (i < P && s_first[i]) {
    int slot = 0;
    for (int q = 0; q < i; ++q) slot += s_first[q];
    const int ex = s_sorted_e[i];
    plan->exp_id[slot] = ex;
    plan->exp_off[slot] = i;
    unsigned long long ptr[3];
    bool bad = false;
    for (int j = 0; j < 3; ++j) {
      ptr[j] = p.expert_ptrs ? p.expert_ptrs[(size_t)ex * 3 + j] : 0ull;
      bad |= (ptr[j] == 0ull) || (ptr[j] & 255ull);
    }
    if (bad) atomicOr(&p.ctrl->status, (unsigned)MOE_STATUS_MISSING_EXPERT);
    for (int j = 0; j < 3; ++j) plan->exp_ptr[slot][j] = bad ? 0ull : ptr[j];
  }
  if (i == 0) {
    int n = 0;
    for (int q = 0; q < P; ++q) n += s_first[q];
    plan->n_exp = n;
    plan->n_pairs = P;
    plan->exp_off[n] = P;
  }
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
  long blocks = ((long)p.m * 32 + 255) / 256;
  if (blocks > 152L * 8) blocks = 152L * 8;
  k_select<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_route_decode(const RouteParams& p, cudaStream_t s) {
  const long warps = (long)p.N + (long)p.m * (p.D / 32);
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  k_route_decode<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
