// Routing selection for one token by one warp (shared by the router kernels).
//
// Method: metrale moe_v41.rs source, fn route_from_logits (scores
// sqrt(softplus(logit / gate_temp)) with softplus(t) = t above 20, keys
// score + bias, stable descending order with ties to the lower id, weights
// the unbiased scores, divided by (sum + 1e-20) when norm_topk_prob and
// topk > 1, then times route_scale); DeepSeek V4.1 atlas "Mixture of
// experts", model.py Gate.forward (the sigmoid and softmax score functions,
// and bias_vl in place of the bias for image tokens).
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

// The bias a token's keys use: bias_vl for an image token (image_mask[t]
// nonzero), else bias.  bias_vl or image_mask NULL: every token uses bias.
static __device__ __forceinline__ const float* token_bias(const float* bias, const float* bias_vl,
                                                          const uint8_t* image_mask, int t) {
  return (bias_vl && image_mask && __ldg(image_mask + t)) ? bias_vl : bias;
}

// Score with every step correctly rounded or evaluated in f64 and rounded
// once, from t = z / T (f32):
//   sqrt(softplus): t > 20: sqrt(t) (f32); else f32(sqrt(log1p(exp(t)))) in f64;
//   sigmoid: f32(1 / (1 + exp(-t))) in f64.
static __device__ __forceinline__ float score_exact(float z, float T, int sf) {
  const float t = __fdiv_rn(z, T);
  if (sf == MOE_SCORE_SIGMOID) return __double2float_rn(1.0 / (1.0 + exp(-(double)t)));
  if (t > 20.0f) return __fsqrt_rn(t);
  return __double2float_rn(sqrt(log1p(exp((double)t))));
}

// The same in f32 with the accurate single-precision functions: within a few
// ulp of score_exact; used only to find the candidates near the cut.
// Sigmoid: expf (2 ulp), one add and one division (half an ulp each) give at
// most 3 ulp of the score, inside the bound route_token_warp assumes.
static __device__ __forceinline__ float score_fast(float z, float T, int sf) {
  const float t = __fdiv_rn(z, T);
  if (sf == MOE_SCORE_SIGMOID) return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-t)));
  if (t > 20.0f) return __fsqrt_rn(t);
  return __fsqrt_rn(log1pf(expf(t)));
}

// Routing weights from the picks: lane r < k holds pick r (id, score).  The
// sum runs in pick order (every lane computes it), then lane r writes weight
// r: score / (sum + 1e-20) when norm and k > 1, times route_scale.
static __device__ __forceinline__ void write_picks(int my_id, float my_s, int k, int norm, float route_scale,
                                                   float* w_out, int* idx_out, int* pick_id, float* pick_w) {
  const int lane = threadIdx.x & 31;
  float sum = 0.f;
#pragma unroll 1
  for (int q = 0; q < k; ++q) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_s, q));
  sum = __fadd_rn(sum, 1e-20f);
  if (lane < k) {
    const float wv = __fmul_rn(norm && k > 1 ? __fdiv_rn(my_s, sum) : my_s, route_scale);
    w_out[lane] = wv;
    idx_out[lane] = my_id;
    if (pick_id) {
      pick_id[lane] = my_id;
      pick_w[lane] = wv;
    }
  }
  __syncwarp();
}

// Scratch one warp needs in shared memory for one token: 3 * N words,
// rounded up to 16 bytes so that consecutive warps' scratch stays aligned
// (the softmax path keeps N doubles at its start).
__host__ __device__ inline size_t select_scratch_bytes(int N) { return ((size_t)3 * N * 4 + 15) & ~(size_t)15; }

// One token's routing with softmax scores, by one warp, exactly as defined:
// t = z / T in f32 for every expert, the shift = the largest t that is not
// NaN, exp(t - shift) in f64, their sum in expert-id order (one lane), each
// score f32(exp(t - shift) / sum); a NaN t makes every score NaN.  Keys are
// score + bias; the picks take k rounds of the warp's largest rank key.
// scratch: select_scratch_bytes(N) bytes, 8-byte aligned (N doubles, then
// N key words).
static __device__ __noinline__ void route_token_softmax(const float* __restrict__ z, const float* __restrict__ bias,
                                                        int N, int k, float T, int norm, float route_scale,
                                                        float* w_out, int* idx_out, unsigned* status,
                                                        float* scratch, int* pick_id, float* pick_w) {
  const int lane = threadIdx.x & 31;
  double* ex = reinterpret_cast<double*>(scratch);
  float* skey = scratch + 2 * N;
  bool t_nan = false;
  float mx = -INFINITY;
  for (int e = lane; e < N; e += 32) {
    const float t = __fdiv_rn(__ldcg(z + e), T);
    if (t != t) t_nan = true;
    else mx = fmaxf(mx, t);
  }
  t_nan = __any_sync(0xffffffffu, t_nan);
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  for (int e = lane; e < N; e += 32) ex[e] = exp((double)__fdiv_rn(__ldcg(z + e), T) - (double)mx);
  __syncwarp();
  double sum = 0.0;
  if (lane == 0) {
#pragma unroll 8
    for (int e = 0; e < N; ++e) sum += ex[e];
  }
  sum = __shfl_sync(0xffffffffu, sum, 0);
  bool any_nan = false;
  for (int e = lane; e < N; e += 32) {
    const float sc = t_nan ? __int_as_float(0x7fc00000) : __double2float_rn(ex[e] / sum);
    const float key = __fadd_rn(sc, __ldg(bias + e));
    any_nan |= (key != key);
    skey[e] = key;
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) atomicOr(status, (unsigned)MOE_STATUS_NAN_KEY);
  __syncwarp();
  uint32_t taken = 0;  // bit i: expert lane + 32 i picked
  int my_id = 0;       // lane r < k: pick r
  float my_s = 0.f;
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0;
    for (int e = lane, i = 0; e < N; e += 32, ++i) {
      if (!(taken >> i & 1u)) {
        const unsigned long long rk = rank_key(skey[e], e);
        best = rk > best ? rk : best;
      }
    }
    const int win = (int)(0xFFFFFFFFu - (uint32_t)(warp_max_u64(best) & 0xFFFFFFFFu));
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == r) {
      my_id = win;
      my_s = t_nan ? __int_as_float(0x7fc00000) : __double2float_rn(ex[win] / sum);
    }
  }
  write_picks(my_id, my_s, k, norm, route_scale, w_out, idx_out, pick_id, pick_w);
}

// One token's routing by one warp.
//
// Every key is first computed in f32 with the accurate single-precision
// functions (score_fast).  Its distance to the exact key (score_exact + bias,
// the value the method defines) is at most eps = 2^-18 (S + K), S and K the
// largest |score| and |key| of the token: expf and log1pf are within 2 ulp,
// sqrt halves the relative error, and each of the two roundings adds half an
// ulp (the sigmoid's bound is 3 ulp of the score).  sf selects the score
// function (MOE_SCORE_*); the softmax has no separable fast form and is
// evaluated exactly by route_token_softmax (sk is then not read).  When the fast top-k is separated by more than 2 eps from every
// neighbour it is the exact top-k in the exact order, and no f64 work is
// done.  Otherwise every expert within 2 eps of the k-th fast key is
// re-scored with score_exact (one candidate per lane) and the picks are taken
// on the exact keys: the exact top-k is always inside that set.  Weights use
// the scores of the path taken (fast scores are within 2^-20 relative).
// scratch: select_scratch_bytes(N) bytes of shared memory for this warp.
// sk (may be NULL): the (score_fast, fast key) pairs already computed for this
// token, exactly as below.  pick_id / pick_w (may be NULL): shared-memory
// copies of the picks.
static __device__ __noinline__ void route_token_warp(const float* __restrict__ z, const float2* __restrict__ sk,
                                                     const float* __restrict__ bias, int N, int k, float T, int sf,
                                                     int norm, float route_scale, float* w_out, int* idx_out,
                                                     unsigned* status, float* scratch, int* pick_id = nullptr,
                                                     float* pick_w = nullptr) {
  if (sf == MOE_SCORE_SOFTMAX) {
    route_token_softmax(z, bias, N, k, T, norm, route_scale, w_out, idx_out, status, scratch, pick_id, pick_w);
    return;
  }
  const int lane = threadIdx.x & 31;
  float* skey = scratch;
  float* ssc = scratch + N;
  int* slist = reinterpret_cast<int*>(scratch + 2 * N);
  bool any_nan = false;
  float smax = 0.f, kmax = 0.f;
  for (int e = lane; e < N; e += 32) {
    float sc, key;
    if (sk) {
      const float2 v = __ldcg(sk + e);
      sc = v.x;
      key = v.y;
    } else {
      sc = score_fast(__ldcg(z + e), T, sf);
      key = __fadd_rn(sc, __ldg(bias + e));
    }
    any_nan |= (key != key);
    if (key == key) {
      smax = fmaxf(smax, fabsf(sc));
      kmax = fmaxf(kmax, fabsf(key));
    }
    skey[e] = key;
    ssc[e] = sc;
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) atomicOr(status, (unsigned)MOE_STATUS_NAN_KEY);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  __syncwarp();
  const float eps = 0x1.0p-18f * (smax + kmax) + 0x1.0p-126f;

  // fast top-(k+1) in rank order (ties by id); taken entries: bit i of the
  // lane's mask stands for expert lane + 32 i
  uint32_t taken = 0;
  float prev_key = 0.f, kth_key = 0.f;
  bool resolved = true;
  int my_id = 0;  // lane r < k: pick r
  float my_s = 0.f;
  const int rounds = k < N ? k + 1 : k;
#pragma unroll 1
  for (int r = 0; r < rounds; ++r) {
    unsigned long long best = 0;
    for (int e = lane, i = 0; e < N; e += 32, ++i) {
      if (!(taken >> i & 1u)) {
        const unsigned long long rk = rank_key(skey[e], e);
        best = rk > best ? rk : best;
      }
    }
    const unsigned long long wmax = warp_max_u64(best);
    const int win = (int)(0xFFFFFFFFu - (uint32_t)(wmax & 0xFFFFFFFFu));
    const float wk = skey[win];
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    // neighbouring keys must be separated by more than 2 eps (NaN never is)
    if (r > 0 && !(prev_key - wk > 2.0f * eps)) resolved = false;
    prev_key = wk;
    if (r < k) {
      if (lane == r) {
        my_id = win;
        my_s = ssc[win];
      }
      kth_key = wk;
    }
  }

  if (!resolved) {
    // candidates: every expert within 2 eps of the k-th fast key
    const bool kth_nan = kth_key != kth_key;
    const float thresh = kth_key - 2.0f * eps;
    int nc = 0;
    for (int base = 0; base < N; base += 32) {
      const int e = base + lane;
      const bool c = e < N && (kth_nan || !(skey[e] < thresh));
      const unsigned bal = __ballot_sync(0xffffffffu, c);
      if (c) slist[nc + __popc(bal & ((1u << lane) - 1u))] = e;
      nc += __popc(bal);
    }
    __syncwarp();
    for (int c = lane; c < nc; c += 32) {
      const int e = slist[c];
      const float sx = score_exact(__ldcg(z + e), T, sf);
      ssc[e] = sx;
      skey[e] = __fadd_rn(sx, __ldg(bias + e));
    }
    __syncwarp();
    uint32_t used = 0;  // bit c of lane's mask: candidate lane + 32 c taken
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0;
      for (int c = lane, i = 0; c < nc; c += 32, ++i) {
        if (!(used >> i & 1u)) {
          // rank keys are never 0, so a NaN candidate still beats "none left"
          const int e = slist[c];
          const unsigned long long rk = rank_key(skey[e], e);
          best = rk > best ? rk : best;
        }
      }
      const unsigned long long wmax = warp_max_u64(best);
      const int win = (int)(0xFFFFFFFFu - (uint32_t)(wmax & 0xFFFFFFFFu));
      if (lane == r) {
        my_id = win;
        my_s = ssc[win];
      }
      for (int c = lane, i = 0; c < nc; c += 32, ++i)
        if (slist[c] == win) used |= 1u << i;
    }
  }
  __syncwarp();
  write_picks(my_id, my_s, k, norm, route_scale, w_out, idx_out, pick_id, pick_w);
}

// The same routing with up to 12 keys per lane held in registers (N <= 384),
// for the latency-critical single-warp use: every load is issued before any
// is used, and the picks travel by shuffles.  sk: the fast (score, key) pairs
// of score function sf (not the softmax, which has none).
// Falls back to route_token_warp (shared-memory scratch, exact re-scoring)
// when the fast keys do not separate the picks.  Same results.
static __device__ __noinline__ void route_token_warp_r12(const float* __restrict__ z, const float2* __restrict__ sk,
                                                         const float* __restrict__ bias, int N, int k, float T, int sf,
                                                         int norm, float route_scale, float* w_out, int* idx_out,
                                                         unsigned* status, float* scratch, int* pick_id,
                                                         float* pick_w) {
  constexpr int PL = 12;
  const int lane = threadIdx.x & 31;
  float kf[PL], sc[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    const float2 v = e < N ? __ldcg(sk + e) : make_float2(0.f, 0.f);
    sc[i] = v.x;
    kf[i] = v.y;
  }
  bool any_nan = false;
  float smax = 0.f, kmax = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    if (lane + 32 * i < N) {
      any_nan |= (kf[i] != kf[i]);
      if (kf[i] == kf[i]) {
        smax = fmaxf(smax, fabsf(sc[i]));
        kmax = fmaxf(kmax, fabsf(kf[i]));
      }
    }
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) atomicOr(status, (unsigned)MOE_STATUS_NAN_KEY);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  const float eps = 0x1.0p-18f * (smax + kmax) + 0x1.0p-126f;
  float prev_key = 0.f;
  bool resolved = true;
  int my_id = 0;  // lane r < k: pick r
  float my_s = 0.f;
  const int rounds = k < N ? k + 1 : k;
  // order-preserving key bits (the high word of rank_key), computed once; the
  // scores go to the scratch by expert id, read back for the picks
  uint32_t ku[PL];
  uint32_t live = 0;  // bit i: entry i exists and is not taken
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    ku[i] = (uint32_t)(rank_key(kf[i], 0) >> 32);
    if (lane + 32 * i < N) {
      live |= 1u << i;
      scratch[lane + 32 * i] = sc[i];
    }
  }
  __syncwarp();
#pragma unroll 1
  for (int r = 0; r < rounds; ++r) {
    // the lane's best untaken key, ties to the lower index (the lower id):
    // a branch-free tree maximum of (key bits, 255 - index), 0 = no entry
    unsigned long long v[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i)
      v[i] = (live >> i & 1u) ? (((unsigned long long)ku[i] << 32) | (unsigned long long)(255 - i)) : 0ull;
#pragma unroll
    for (int w = 1; w < PL; w <<= 1)
#pragma unroll
      for (int i = 0; i + w < PL; i += 2 * w) v[i] = v[i] > v[i + w] ? v[i] : v[i + w];
    const bool has = v[0] != 0ull;
    const uint32_t best = (uint32_t)(v[0] >> 32);
    const int bi = 255 - (int)(v[0] & 255ull);
    // the warp's largest key, then the lowest id among the lanes holding it
    // (a lane with nothing left offers no id; NaN keys, bits 0, still win
    // over nothing)
    const uint32_t top = __reduce_max_sync(0xffffffffu, has ? best : 0u);
    const uint32_t cand = (has && best == top) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    // the winner's key from its bits (the inverse of rank_key's map)
    const float wk = __uint_as_float((top & 0x80000000u) ? (top & 0x7FFFFFFFu) : ~top);
    if ((win & 31) == lane) live &= ~(1u << (win >> 5));
    if (r > 0 && !(prev_key - wk > 2.0f * eps)) resolved = false;
    prev_key = wk;
    if (r < k && lane == r) {
      my_id = win;
      my_s = scratch[win];
    }
  }
  if (!resolved) {
    route_token_warp(z, sk, bias, N, k, T, sf, norm, route_scale, w_out, idx_out, status, scratch, pick_id,
                     pick_w);
    return;
  }
  write_picks(my_id, my_s, k, norm, route_scale, w_out, idx_out, pick_id, pick_w);
}

}  // namespace moe
