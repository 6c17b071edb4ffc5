// Routing selection for one token by one warp (shared by the router kernels).
//
// Method: metrale moe_v41.rs source, fn route_from_logits (scores
// sqrt(softplus(logit / gate_temp)) with softplus(t) = t above 20, keys
// score + bias, stable descending order with ties to the lower id, weights
// the unbiased scores, divided by (sum + 1e-20) when norm_topk_prob and
// topk > 1, then times route_scale); DeepSeek V4.1 atlas "Mixture of
// experts", model.py Gate.forward.
#pragma once

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------- selection
// Order-preserving 64-bit key: larger = ranks first.  NaN ranks below every
// number; equal keys rank by lower expert id.  -0 and +0 are equal keys.
static __device__ __forceinline__ unsigned long long rank_key(float key, int id) {
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

static __device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Score with every step correctly rounded or evaluated in f64 and rounded
// once: t = z / T (f32); t > 20: sqrt(t) (f32); else f32(sqrt(log1p(exp(t)))) in f64.
static __device__ __forceinline__ float score_exact(float z, float T) {
  const float t = __fdiv_rn(z, T);
  if (t > 20.0f) return __fsqrt_rn(t);
  return __double2float_rn(sqrt(log1p(exp((double)t))));
}

// The same in f32 with the accurate single-precision functions: within a few
// ulp of score_exact; used only to find the candidates near the cut.
static __device__ __forceinline__ float score_fast(float z, float T) {
  const float t = __fdiv_rn(z, T);
  if (t > 20.0f) return __fsqrt_rn(t);
  return __fsqrt_rn(log1pf(expf(t)));
}

constexpr int SEL_PER_LANE = MAX_N / 32;

// One token's routing by one warp.
//
// Every key is first computed in f32 with the accurate single-precision
// functions (score_fast).  Its distance to the exact key (score_exact + bias,
// the value the method defines) is at most eps = 2^-18 (S + K), S and K the
// largest |score| and |key| of the token: expf and log1pf are within 2 ulp,
// sqrt halves the relative error, and each of the two roundings adds half an
// ulp.  When the fast top-k is separated by more than 2 eps from every
// neighbour it is the exact top-k in the exact order, and no f64 work is
// done.  Otherwise every expert within 2 eps of the k-th fast key is
// re-scored with score_exact (one candidate per lane per pass) and the picks
// are taken on the exact keys: the exact top-k is always inside that set.
// Weights use the scores of the path taken (fast scores differ from the exact
// ones by < 2^-20 relative).
static __device__ __noinline__ void route_token_warp(const float* __restrict__ z, const float* __restrict__ bias, int N, int k,
                                 float T, int norm, float route_scale, float* w_out, int* idx_out, unsigned* status) {
  const int lane = threadIdx.x & 31;
  float kf[SEL_PER_LANE], sf[SEL_PER_LANE];
  bool any_nan = false;
  float smax = 0.f, kmax = 0.f;
#pragma unroll
  for (int i = 0; i < SEL_PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float key = -INFINITY, sc = 0.f;
    if (e < N) {
      sc = score_fast(__ldcg(z + e), T);
      key = __fadd_rn(sc, __ldg(bias + e));
      any_nan |= (key != key);
      if (key == key) {
        smax = fmaxf(smax, fabsf(sc));
        kmax = fmaxf(kmax, fabsf(key));
      }
    }
    kf[i] = key;
    sf[i] = sc;
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) atomicOr(status, (unsigned)MOE_STATUS_NAN_KEY);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  const float eps = 0x1.0p-18f * (smax + kmax) + 0x1.0p-126f;

  // fast top-(k+1) in rank order (ties by id)
  uint32_t taken = 0;
  float prev_key = 0.f;
  bool resolved = true;
  int picked_id[MAX_TOPK];
  float picked_s[MAX_TOPK];
  float kth_key = 0.f;
  const int rounds = k < N ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    unsigned long long best = 0;
    float bk = 0.f, bs = 0.f;
#pragma unroll
    for (int i = 0; i < SEL_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < N && !(taken >> i & 1u)) {
        const unsigned long long rk = rank_key(kf[i], e);
        if (rk > best) { best = rk; bk = kf[i]; bs = sf[i]; }
      }
    }
    const unsigned long long wmax = warp_max_u64(best);
    const int win = (int)(0xFFFFFFFFu - (uint32_t)(wmax & 0xFFFFFFFFu));
    const float wk = __shfl_sync(0xffffffffu, bk, win & 31);
    const float ws = __shfl_sync(0xffffffffu, bs, win & 31);
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    // neighbouring keys must be separated by more than 2 eps (NaN never is)
    if (r > 0 && !(prev_key - wk > 2.0f * eps)) resolved = false;
    prev_key = wk;
    if (r < k) {
      picked_id[r] = win;
      picked_s[r] = ws;
      kth_key = wk;
    }
  }

  if (!resolved) {
    // exact keys for every expert within 2 eps of the k-th fast key
    const bool kth_nan = kth_key != kth_key;
    const float thresh = kth_key - 2.0f * eps;
    uint32_t pend = 0;
#pragma unroll
    for (int i = 0; i < SEL_PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < N && (kth_nan || !(kf[i] < thresh))) pend |= 1u << i;
    }
    uint32_t cand = pend;
    float se[SEL_PER_LANE];
#pragma unroll
    for (int i = 0; i < SEL_PER_LANE; ++i) se[i] = 0.f;
    // one candidate per lane per pass
    while (__any_sync(0xffffffffu, pend != 0)) {
      const int i = pend ? __ffs(pend) - 1 : -1;
      float v = 0.f;
      if (i >= 0) {
        const int e = lane + 32 * i;
        v = score_exact(__ldcg(z + e), T);
        pend &= pend - 1;
      }
#pragma unroll
      for (int q = 0; q < SEL_PER_LANE; ++q)
        if (q == i) { se[q] = v; kf[q] = __fadd_rn(v, __ldg(bias + lane + 32 * q)); }
    }
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0;
      float bs = 0.f;
#pragma unroll
      for (int i = 0; i < SEL_PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (cand >> i & 1u) {
          // rank keys are never 0, so a NaN candidate still beats "none left"
          const unsigned long long rk = rank_key(kf[i], e);
          if (rk > best) { best = rk; bs = se[i]; }
        }
      }
      const unsigned long long wmax = warp_max_u64(best);
      const int win = (int)(0xFFFFFFFFu - (uint32_t)(wmax & 0xFFFFFFFFu));
      picked_s[r] = __shfl_sync(0xffffffffu, bs, win & 31);
      picked_id[r] = win;
      if ((win & 31) == lane) cand &= ~(1u << (win >> 5));
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

}  // namespace moe
