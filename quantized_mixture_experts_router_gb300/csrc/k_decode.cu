// Decode path (m <= 8): one fused persistent kernel per layer call.
//
// One block per SM: a producer warp and NCW consumer warps around a ring of
// shared-memory stages.  The producer takes tickets from one counter and
// streams each task's raw weight rows into the ring with 1-D bulk copies
// (cp.async.bulk, completing on the stage's mbarrier); every stage is taken
// and finished by a single consumer warp, so there are no block-wide
// barriers.  Tickets run in dependency order:
//   q8_1(x) | router rows | shared gate/up | routed gate/up | shared down | routed down
// A task that needs earlier results (the plan, q8_1(x), the h vectors) waits
// on a counter with a bounded spin; the producer never waits for results, so
// weight bytes keep streaming while the consumers catch up.  Results that
// span several tasks are finished by the task that completes them (the last
// arriver on a counter): the selection after the last router rows, q8_1(h)
// after the last 4-row slice of a 32-row group, and the ordered combine
// y = sum_{ascending expert} G_i E_i + S after the last part of an 8-row
// output group.  Every such sum runs in a fixed order, so results do not
// depend on timing.
//
// Method: DeepSeek V4.1 atlas "Mixture of experts" (Router, Routed expert and
// Shared expert steps: g' = min(g, L), u' = clip(u, -L, L), h = g' sigmoid(g') u',
// y = sum G_i E_i + y_shared); metrale moe_v41 module docs and moe_v41.rs
// (Q2_K gate/up, Q3_K down, q8_1 activations, swiglu_q8, the shared expert
// added after the routed experts).
#include "internal.h"
#include "select.cuh"

namespace moe {

namespace {

constexpr int NCW = 6;                 // consumer warps
constexpr int NTH = (NCW + 1) * 32;    // + producer warp
constexpr int SB = 16384;              // bytes per ring stage
constexpr int NST = 12;                // ring stages
constexpr int GR = 4;                  // rows of W1 and of W3 per gate/up stage
constexpr int DG = 8;                  // output rows per down group
constexpr int Q8_CHUNK = 32;           // q8_1 blocks per q8 task

enum : int { K_STOP = 0, K_Q8, K_ROUTER, K_SHGU_B, K_SHGU_Q, K_RTGU, K_SHDN_B, K_SHDN_Q, K_RTDN };

struct Task {
  int kind, a, b, c;
};

struct SmemCtl {
  Task task[NST];
  unsigned long long full[NST];
  unsigned long long empty[NST];
  unsigned next;  // consumer grab counter
};

constexpr size_t RING = (size_t)NST * SB + 16;
constexpr size_t SMEM_BYTES = RING + sizeof(SmemCtl);

__device__ __forceinline__ uint8_t* ring() {
  extern __shared__ __align__(128) uint8_t dyn[];
  return dyn;
}
__device__ __forceinline__ SmemCtl& ctl() {
  extern __shared__ __align__(128) uint8_t dyn[];
  return *reinterpret_cast<SmemCtl*>(dyn + RING);
}

// ----------------------------------------------------------- counters
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *p >= target.  false after the deadline (status set).
__device__ __forceinline__ bool wait_count(const unsigned* p, unsigned target, uint64_t deadline, unsigned* status) {
  uint32_t spins = 0;
  while (ld_acquire(p) < target) {
    __nanosleep(64);
    if ((++spins & 15u) == 0 && globaltimer_ns() > deadline) {
      atomicOr(status, (unsigned)MOE_STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Publish this warp's global writes, then add 1 to *p; returns the old value
// (lane 0's, broadcast).
__device__ __forceinline__ unsigned warp_signal(unsigned* p) {
  __threadfence();
  __syncwarp();
  unsigned old = 0;
  if ((threadIdx.x & 31) == 0) old = atomicAdd(p, 1u);
  return __shfl_sync(0xffffffffu, old, 0);
}

// ------------------------------------------------------------ the plan
struct Sizes {
  int n_q8, n_router, rrows, n_shgu, shgu_target, gtiles, shdn_parts, sdr, groups;
  bool shq;  // shared expert in K-quant blocks
};

__device__ __forceinline__ Sizes sizes_of(const DecodeParams& p) {
  Sizes z;
  const int q8_per_tok = (p.D / 32 + Q8_CHUNK - 1) / Q8_CHUNK;
  z.n_q8 = p.m * q8_per_tok;
  z.rrows = 1;
  z.n_router = p.N;
  z.gtiles = p.I / GR;
  z.shq = p.shared_kind != MOE_SHARED_BF16;
  z.n_shgu = z.shq ? z.gtiles : 2 * p.I;
  z.shgu_target = z.shq ? z.gtiles : p.I;  // bf16: one count per finished (gate, up) row pair
  int sdr = SB / (2 * p.I);
  sdr = sdr >= 8 ? 8 : sdr >= 4 ? 4 : sdr >= 2 ? 2 : 1;
  z.sdr = sdr;
  z.shdn_parts = z.shq ? 1 : DG / sdr;
  z.groups = p.D / DG;
  return z;
}

// Ticket -> task.  Routed tasks need n_exp; -1 means "wait for the plan".
__device__ __forceinline__ Task decode_ticket(unsigned t, const Sizes& z, int n_exp) {
  Task k{K_STOP, 0, 0, 0};
  if (t < (unsigned)z.n_q8) { k.kind = K_Q8; k.a = (int)t; return k; }
  t -= z.n_q8;
  if (t < (unsigned)z.n_router) { k.kind = K_ROUTER; k.a = (int)t * z.rrows; return k; }
  t -= z.n_router;
  if (t < (unsigned)z.n_shgu) {
    if (z.shq) { k.kind = K_SHGU_Q; k.a = (int)t * GR; }
    else { k.kind = K_SHGU_B; k.a = (int)t >> 1; k.b = (int)t & 1; }
    return k;
  }
  t -= z.n_shgu;
  if (n_exp < 0) { k.kind = -1; return k; }
  const unsigned n_rtgu = (unsigned)n_exp * z.gtiles;
  if (t < n_rtgu) { k.kind = K_RTGU; k.a = (int)(t / z.gtiles); k.b = (int)(t % z.gtiles) * GR; return k; }
  t -= n_rtgu;
  const unsigned n_shdn = (unsigned)z.groups * z.shdn_parts;
  if (t < n_shdn) {
    k.kind = z.shq ? K_SHDN_Q : K_SHDN_B;
    k.a = (int)(t / z.shdn_parts);
    k.b = (int)(t % z.shdn_parts);
    return k;
  }
  t -= n_shdn;
  const unsigned n_rtdn = (unsigned)z.groups * n_exp;
  if (t < n_rtdn) { k.kind = K_RTDN; k.a = (int)(t / n_exp); k.b = (int)(t % n_exp); return k; }
  return k;
}

// ---------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void dot8(float& acc, const uint4& w, const uint4& x) {
  acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc); acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc); acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc); acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc); acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
}

// activation unit from memory written in this kernel (L2, not the
// non-coherent read-only path)
__device__ __forceinline__ void load_unit_cg(XUnit& x, const int4* p) {
  int4 v0 = __ldcg(p + 0), v1 = __ldcg(p + 1), v2 = __ldcg(p + 2), v3 = __ldcg(p + 3);
  int4 v4 = __ldcg(p + 4), v5 = __ldcg(p + 5);
  x.q[0] = v0.x; x.q[1] = v0.y; x.q[2] = v0.z; x.q[3] = v0.w;
  x.q[4] = v1.x; x.q[5] = v1.y; x.q[6] = v1.z; x.q[7] = v1.w;
  x.q[8] = v2.x; x.q[9] = v2.y; x.q[10] = v2.z; x.q[11] = v2.w;
  x.q[12] = v3.x; x.q[13] = v3.y; x.q[14] = v3.z; x.q[15] = v3.w;
  x.dq[0] = __int_as_float(v4.x); x.dq[1] = __int_as_float(v4.y);
  x.dq[2] = __int_as_float(v4.z); x.dq[3] = __int_as_float(v4.w);
  x.s16[0] = v5.x; x.s16[1] = v5.y; x.s16[2] = v5.z; x.s16[3] = v5.w;
}

// ------------------------------------------------------------- the plan
// Selection for every token and grouping of the (expert, token) pairs by
// ascending expert id; run by the one warp that finished the router.
__device__ void build_plan(const DecodeParams& p) {
  const int lane = threadIdx.x & 31;
  for (int t = 0; t < p.m; ++t)
    route_token_warp(p.logits + (size_t)t * p.N, p.bias, p.N, p.k, p.gate_temp, p.norm, p.route_scale,
                     p.topk_w + (size_t)t * p.k, p.topk_idx + (size_t)t * p.k, &p.ctrl->status);
  __syncwarp();
  __threadfence();
  DecodePlan* plan = p.plan_w;
  const int P = p.m * p.k;
  // rank of pair i among all pairs by (expert, token); each lane handles i = lane + 32 j
  int sorted_e_local[MAXP / 32];
  for (int j = 0; j < MAXP / 32; ++j) sorted_e_local[j] = 0;
  for (int i = lane; i < P; i += 32) {
    const int e = __ldcg(p.topk_idx + i), t = i / p.k;
    int rank = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = __ldcg(p.topk_idx + q), tq = q / p.k;
      rank += (eq < e) || (eq == e && tq < t);
    }
    plan->pair_tok[rank] = t;
    plan->pair_w[rank] = __ldcg(p.topk_w + i);
    plan->exp_id[rank] = e;  // scratch: the expert of each sorted pair (rewritten below)
  }
  __syncwarp();
  __threadfence();
  // distinct experts: first pair of each run
  int n_first_before = 0;
  for (int base = 0; base < P; base += 32) {
    const int i = base + lane;
    int e = -1, first = 0;
    if (i < P) {
      e = __ldcg(&plan->exp_id[i]);
      first = (i == 0) || (__ldcg(&plan->exp_id[i - 1]) != e);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, first);
    const int slot = n_first_before + __popc(bal & ((1u << lane) - 1u));
    sorted_e_local[base / 32] = first ? (slot | (e << 8)) : -1;
    n_first_before += __popc(bal);
  }
  __syncwarp();
  // now rewrite exp_id / exp_off / pointers (exp_id[] was used as scratch)
  for (int base = 0; base < P; base += 32) {
    const int i = base + lane;
    const int v = sorted_e_local[base / 32];
    if (i < P && v >= 0) {
      const int slot = v & 255, e = v >> 8;
      plan->exp_off[slot] = i;
      unsigned long long ptr[3];
      bool bad = false;
      for (int j = 0; j < 3; ++j) {
        ptr[j] = p.expert_ptrs[(size_t)e * 3 + j];
        bad |= (ptr[j] == 0ull) || (ptr[j] & 255ull);
      }
      if (bad) atomicOr(&p.ctrl->status, (unsigned)MOE_STATUS_MISSING_EXPERT);
      for (int j = 0; j < 3; ++j) plan->exp_ptr[slot][j] = bad ? 0ull : ptr[j];
      // exp_id written after every lane has read the scratch values
    }
  }
  __syncwarp();
  __threadfence();
  for (int base = 0; base < P; base += 32) {
    const int i = base + lane;
    const int v = sorted_e_local[base / 32];
    if (i < P && v >= 0) plan->exp_id[v & 255] = v >> 8;
  }
  __syncwarp();
  // each token's pairs in ascending expert id
  for (int i = lane; i < P; i += 32) {
    const int t = __ldcg(&plan->pair_tok[i]);
    int r = 0;
    for (int q = 0; q < i; ++q) r += __ldcg(&plan->pair_tok[q]) == t;
    plan->tok_pairs[t][r] = i;
  }
  if (lane == 0) {
    plan->n_exp = n_first_before;
    plan->n_pairs = P;
    plan->exp_off[n_first_before] = P;
  }
  __syncwarp();
}

// ------------------------------------------------------------- tasks
struct Ctx {
  const DecodeParams& p;
  const Sizes& z;
  uint64_t deadline;
  // flags cached per warp once a counter has been seen complete
  bool q8_ok, plan_ok, shgu_ok, rtgu_ok;
};

__device__ __forceinline__ const DecodePlan* plan_r(const DecodeParams& p) { return p.plan_w; }

// q8_1 of x for Q8_CHUNK blocks of one token
__device__ void task_q8(Ctx& c, int task) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int per_tok = (p.D / 32 + Q8_CHUNK - 1) / Q8_CHUNK;
  const int t = task / per_tok, b0 = (task % per_tok) * Q8_CHUNK;
  const int nb = p.D / 32;
  for (int qb = b0; qb < b0 + Q8_CHUNK && qb < nb; ++qb) {
    const float v = __bfloat162float(
        reinterpret_cast<const __nv_bfloat16*>(p.x)[(size_t)t * p.D + (size_t)qb * 32 + lane]);
    q8_block_warp(v, qb, p.xq8 + (size_t)t * nb * Q8_B, p.xu + (size_t)t * (unit_bytes(p.D) / 4));
  }
  warp_signal(&p.ctrl->q8_done);
}

// rows [r0, r0+rows) of the router against every token; the warp that
// finishes the last router task builds the plan
__device__ void task_router(Ctx& c, const uint8_t* stage, int r0) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int chunks = p.D / 8;
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  for (int t = 0; t < p.m; ++t) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
    float acc = 0.f;
    for (int ch = lane; ch < chunks; ch += 32) dot8(acc, w[ch], __ldg(xr + ch));
    acc = warp_sum(acc);
    if (lane == 0) p.logits[(size_t)t * p.N + r0] = acc;
  }
  const unsigned old = warp_signal(&p.ctrl->router_done);
  if (old == (unsigned)c.z.n_router - 1) {
    __threadfence();
    build_plan(p);
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      p.ctrl->router_done = 0u;
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.ctrl->route_ready), "r"(1u) : "memory");
    }
  }
}

// one row of the bf16 shared gate (mat 0) or up (mat 1) projection; the
// second of the pair to finish forms h = SwiGLU(g, u), rounded to bf16
__device__ void task_shgu_b(Ctx& c, const uint8_t* stage, int row, int mat) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int chunks = p.D / 8;
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  float* gu = p.shgu;
  for (int t = 0; t < p.m; ++t) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
    float acc = 0.f;
    for (int ch = lane; ch < chunks; ch += 32) dot8(acc, w[ch], __ldg(xr + ch));
    acc = warp_sum(acc);
    if (lane == 0) gu[((size_t)t * 2 + mat) * p.I + row] = acc;
  }
  const unsigned old = warp_signal(p.cnt + cnt_shpair(p.I) + row);
  if (old == 1u) {
    __threadfence();
    if (lane < p.m) {
      const float g = __ldcg(gu + ((size_t)lane * 2 + 0) * p.I + row);
      const float u = __ldcg(gu + ((size_t)lane * 2 + 1) * p.I + row);
      reinterpret_cast<__nv_bfloat16*>(p.shh)[(size_t)lane * p.I + row] =
          __float2bfloat16_rn(swiglu_f32(g, u, p.swiglu_limit));
    }
    if (lane == 0) p.cnt[cnt_shpair(p.I) + row] = 0u;
    warp_signal(&p.ctrl->shgu_done);
  }
}

// GR rows of W1 (stage offset 0) and W3 (offset GR*rb) in Q2_K against the
// q8_1(x) units of the vector's tokens: half-warp 0 takes W1, half-warp 1 W3,
// each lane 1/16 of the units of every row.  h of the GR rows goes to hf;
// the slice completing a 32-row group quantises it to q8_1 units.
__device__ void task_gateup_q(Ctx& c, const uint8_t* stage, int slot, int r0) {
  const DecodeParams& p = c.p;
  const DecodePlan* plan = plan_r(p);
  const int lane = threadIdx.x & 31, half = lane >> 4, l = lane & 15;
  const int rb = (p.D / QK) * Q2K_B;
  const int U = p.D / 64;
  const bool shared = slot < 0;
  int pair0 = 0, ntok = p.m, vec0;
  bool present = true;
  if (!shared) {
    pair0 = __ldcg(&plan->exp_off[slot]);
    ntok = __ldcg(&plan->exp_off[slot + 1]) - pair0;
    present = __ldcg(&plan->exp_ptr[slot][0]) != 0ull;
    vec0 = pair0;
  } else {
    vec0 = p.shvec0;
  }
  if (!c.q8_ok) c.q8_ok = wait_count(&p.ctrl->q8_done, (unsigned)c.z.n_q8, c.deadline, &p.ctrl->status);
  const uint8_t* base = stage + (size_t)half * GR * rb;
  const size_t xs = unit_bytes(p.D) / 16;
  for (int tt = 0; tt < ntok && present; ++tt) {
    const int tok = shared ? tt : __ldcg(&plan->pair_tok[pair0 + tt]);
    const int4* xb = reinterpret_cast<const int4*>(p.xu) + (size_t)tok * xs;
    float acc[GR];
#pragma unroll
    for (int r = 0; r < GR; ++r) acc[r] = 0.f;
    for (int u = l; u < U; u += 16) {
      XUnit xr;
      load_unit_cg(xr, xb + u * 6);
      const uint8_t* ub = base + (u >> 2) * Q2K_B;
#pragma unroll
      for (int r = 0; r < GR; ++r) acc[r] += q2k_unit_dot(ub + (size_t)r * rb, u & 3, xr);
    }
#pragma unroll
    for (int r = 0; r < GR; ++r) {
#pragma unroll
      for (int o = 8; o; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
    }
    // lane 0 holds g, lane 16 holds u
    float* hv = p.hf + (size_t)(vec0 + tt) * p.I + r0;
#pragma unroll
    for (int r = 0; r < GR; ++r) {
      const float u = __shfl_sync(0xffffffffu, acc[r], 16);
      if (lane == 0) hv[r] = swiglu_f32(acc[r], u, p.swiglu_limit);
    }
  }
  // group of 32 rows complete?
  const int grp = r0 / 32;
  const int hidx = (shared ? MAXP : slot) * (p.I / 32) + grp;
  const unsigned old = warp_signal(p.cnt + cnt_hgrp(p.I) + hidx);
  if (old == 32u / GR - 1u) {
    __threadfence();
    for (int tt = 0; tt < ntok && present; ++tt) {
      const float v = __ldcg(p.hf + (size_t)(vec0 + tt) * p.I + grp * 32 + lane);
      q8_block_warp(v, grp, nullptr, p.hu + (size_t)(vec0 + tt) * (unit_bytes(p.I) / 4));
    }
    if (lane == 0) p.cnt[cnt_hgrp(p.I) + hidx] = 0u;
  }
  warp_signal(shared ? &p.ctrl->shgu_done : &p.ctrl->rtgu_done);
}

// finish output group g if this part was its last
__device__ void maybe_combine(Ctx& c, int g) {
  const DecodeParams& p = c.p;
  const DecodePlan* plan = plan_r(p);
  const int lane = threadIdx.x & 31;
  const int n_exp = __ldcg(&plan->n_exp);
  const unsigned parts = (unsigned)(n_exp + c.z.shdn_parts);
  const unsigned old = warp_signal(p.cnt + cnt_dgrp(p.I) + g);
  if (old != parts - 1u) return;
  __threadfence();
  for (int q = lane; q < p.m * DG; q += 32) {
    const int t = q / DG, d = g * DG + q % DG;
    float acc = 0.f;
    for (int i = 0; i < p.k; ++i) {
      const int pr = __ldcg(&plan->tok_pairs[t][i]);
      acc = fmaf(__ldcg(&plan->pair_w[pr]), __ldcg(p.ep + (size_t)pr * p.D + d), acc);
    }
    acc += __ldcg(p.sp + (size_t)t * p.D + d);
    p.out[(size_t)t * p.D + d] = acc;
  }
  if (lane == 0) p.cnt[cnt_dgrp(p.I) + g] = 0u;
}

// 8 rows of a Q3_K down matrix (stage) against h units: lane = (row, 1/4 of
// the units); results to ep (routed pairs, unweighted) or sp (shared)
__device__ void task_down_q(Ctx& c, const uint8_t* stage, int g, int slot) {
  const DecodeParams& p = c.p;
  const DecodePlan* plan = plan_r(p);
  const int lane = threadIdx.x & 31, row = lane >> 2, q = lane & 3;
  const int rb2 = (p.I / QK) * Q3K_B;
  const int U2 = p.I / 64;
  const bool shared = slot < 0;
  int pb = 0, pe = p.m;
  bool present = true;
  if (!shared) {
    pb = __ldcg(&plan->exp_off[slot]);
    pe = __ldcg(&plan->exp_off[slot + 1]);
    present = __ldcg(&plan->exp_ptr[slot][2]) != 0ull;
  }
  const size_t hs = unit_bytes(p.I) / 16;
  const uint8_t* rowp = stage + (size_t)row * rb2;
  for (int pi = pb; pi < pe; ++pi) {
    const int vec = shared ? p.shvec0 + pi : pi;
    float acc = 0.f;
    if (present) {
      const int4* hb = reinterpret_cast<const int4*>(p.hu) + (size_t)vec * hs;
      for (int u = q; u < U2; u += 4) {
        XUnit hr;
        load_unit_cg(hr, hb + u * 6);
        acc += q3k_unit_dot(rowp + (u >> 2) * Q3K_B, u & 3, hr);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (q == 0) {
      if (shared) p.sp[(size_t)pi * p.D + g * DG + row] = acc;
      else p.ep[(size_t)pi * p.D + g * DG + row] = acc;
    }
  }
  maybe_combine(c, g);
}

// rows of the bf16 shared down matrix against h (bf16 [m, I]) -> sp
__device__ void task_down_b(Ctx& c, const uint8_t* stage, int g, int part) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int rows = c.z.sdr;
  const int chunks = p.I / 8;
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  for (int t = 0; t < p.m; ++t) {
    const uint4* hr = reinterpret_cast<const uint4*>(p.shh) + (size_t)t * chunks;
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.f;
    for (int ch = lane; ch < chunks; ch += 32) {
      const uint4 hv = __ldcg(hr + ch);
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < rows) dot8(acc[r], w[r * chunks + ch], hv);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r < rows) {
        const float s = warp_sum(acc[r]);
        if (lane == 0) p.sp[(size_t)t * p.D + g * DG + part * rows + r] = s;
      }
    }
  }
  maybe_combine(c, g);
}

// ================================================================ kernel
__global__ void __launch_bounds__(NTH, 1) k_decode_layer(const __grid_constant__ DecodeParams p) {
  SmemCtl& S = ctl();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(reinterpret_cast<uint64_t*>(&S.full[i]), 1);
      mbar_init(reinterpret_cast<uint64_t*>(&S.empty[i]), 1);
    }
    S.next = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Sizes z = sizes_of(p);

  if (warp == NCW) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t n = 0;  // stages issued
      int n_exp = -1;
      int stops = 0;
      bool ok = true;
      while (ok && stops < NCW) {
        Task k;
        if (stops > 0) {
          k.kind = K_STOP;
        } else {
          const unsigned t = atomicAdd(&p.ctrl->ticket, 1u);
          k = decode_ticket(t, z, n_exp);
          if (k.kind == -1) {
            ok = wait_count(&p.ctrl->route_ready, 1u, deadline, &p.ctrl->status);
            if (!ok) break;
            n_exp = __ldcg(&p.plan_w->n_exp);
            k = decode_ticket(t, z, n_exp);
          }
        }
        const uint32_t slot = n % NST, use = n / NST;
        if (use > 0 && !mbar_wait_bounded(reinterpret_cast<uint64_t*>(&S.empty[slot]), (use - 1) & 1u, deadline,
                                          &p.ctrl->status)) {
          ok = false;
          break;
        }
        uint8_t* dst = ring() + (size_t)slot * SB;
        const uint8_t *a = nullptr, *b = nullptr;
        uint32_t bytes = 0, boff = 0;
        const int rb = (p.D / QK) * Q2K_B, rb2 = (p.I / QK) * Q3K_B;
        switch (k.kind) {
          case K_ROUTER:
            a = reinterpret_cast<const uint8_t*>(p.router_w) + (size_t)k.a * 2 * p.D;
            bytes = (uint32_t)(2 * p.D * z.rrows);
            break;
          case K_SHGU_B:
            a = (k.b ? p.sh3 : p.sh1) + (size_t)k.a * 2 * p.D;
            bytes = (uint32_t)(2 * p.D);
            break;
          case K_SHGU_Q:
            a = p.sh1 + (size_t)k.a * rb;
            b = p.sh3 + (size_t)k.a * rb;
            bytes = (uint32_t)(GR * rb);
            boff = bytes;
            break;
          case K_RTGU: {
            const unsigned long long w1 = __ldcg(&p.plan_w->exp_ptr[k.a][0]);
            const unsigned long long w3 = __ldcg(&p.plan_w->exp_ptr[k.a][1]);
            if (w1 && w3) {
              a = reinterpret_cast<const uint8_t*>(w1) + (size_t)k.b * rb;
              b = reinterpret_cast<const uint8_t*>(w3) + (size_t)k.b * rb;
              bytes = (uint32_t)(GR * rb);
              boff = bytes;
            }
            break;
          }
          case K_SHDN_B:
            a = p.sh2 + (size_t)(k.a * DG + k.b * z.sdr) * 2 * p.I;
            bytes = (uint32_t)(2 * p.I * z.sdr);
            break;
          case K_SHDN_Q:
            a = p.sh2 + (size_t)k.a * DG * rb2;
            bytes = (uint32_t)(DG * rb2);
            break;
          case K_RTDN: {
            const unsigned long long w2 = __ldcg(&p.plan_w->exp_ptr[k.b][2]);
            if (w2) {
              a = reinterpret_cast<const uint8_t*>(w2) + (size_t)k.a * DG * rb2;
              bytes = (uint32_t)(DG * rb2);
            }
            break;
          }
          default:
            break;
        }
        S.task[slot] = k;
        mbar_arrive_expect_tx(reinterpret_cast<uint64_t*>(&S.full[slot]), a ? (b ? 2u * bytes : bytes) : 0u);
        if (a) bulk_g2s(dst, a, bytes, reinterpret_cast<uint64_t*>(&S.full[slot]));
        if (a && b) bulk_g2s(dst + boff, b, bytes, reinterpret_cast<uint64_t*>(&S.full[slot]));
        ++n;
        if (k.kind == K_STOP) ++stops;
      }
      if (!ok) {
        // let the copies already issued land before the block can exit
        const uint64_t d2 = globaltimer_ns() + p.timeout_ns;
        for (uint32_t i = n > (uint32_t)NST ? n - NST : 0u; i < n; ++i)
          mbar_wait_bounded(reinterpret_cast<uint64_t*>(&S.full[i % NST]), (i / NST) & 1u, d2, &p.ctrl->status);
      }
    }
  } else {
    // --------------------------------------------------------- consumers
    Ctx c{p, z, deadline, false, false, false, false};
    for (;;) {
      unsigned n = 0;
      if (lane == 0) n = atomicAdd(&S.next, 1u);
      n = __shfl_sync(0xffffffffu, n, 0);
      const uint32_t slot = n % NST;
      bool got = true;
      if (lane == 0)
        got = mbar_wait_bounded(reinterpret_cast<uint64_t*>(&S.full[slot]), (n / NST) & 1u, deadline,
                                &p.ctrl->status);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      const Task k = S.task[slot];
      if (k.kind == K_STOP) break;
      const uint8_t* st = ring() + (size_t)slot * SB;
      switch (k.kind) {
        case K_Q8: task_q8(c, k.a); break;
        case K_ROUTER: task_router(c, st, k.a); break;
        case K_SHGU_B: task_shgu_b(c, st, k.a, k.b); break;
        case K_SHGU_Q: task_gateup_q(c, st, -1, k.a); break;
        case K_RTGU: task_gateup_q(c, st, k.a, k.b); break;
        case K_SHDN_B:
        case K_SHDN_Q:
          if (!c.shgu_ok)
            c.shgu_ok = wait_count(&p.ctrl->shgu_done, (unsigned)z.shgu_target, deadline, &p.ctrl->status);
          if (k.kind == K_SHDN_B) task_down_b(c, st, k.a, k.b);
          else task_down_q(c, st, k.a, -1);
          break;
        case K_RTDN:
          if (!c.rtgu_ok) {
            const int n_exp = __ldcg(&p.plan_w->n_exp);
            c.rtgu_ok = wait_count(&p.ctrl->rtgu_done, (unsigned)(n_exp * z.gtiles), deadline, &p.ctrl->status);
          }
          task_down_q(c, st, k.a, k.b);
          break;
        default: break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(reinterpret_cast<uint64_t*>(&S.empty[slot]));
    }
  }
  // the last block out resets the call-wide counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&p.ctrl->exit_count, 1u);
    if (old == gridDim.x - 1) {
      p.ctrl->ticket = 0u;
      p.ctrl->q8_done = 0u;
      p.ctrl->route_ready = 0u;
      p.ctrl->shgu_done = 0u;
      p.ctrl->rtgu_done = 0u;
      p.ctrl->router_done = 0u;
      __threadfence();
      p.ctrl->exit_count = 0u;
    }
  }
}

}  // namespace

size_t decode_smem_bytes() { return SMEM_BYTES; }

bool decode_fits(int D, int I) {
  const int rb = (D / QK) * Q2K_B, rb2 = (I / QK) * Q3K_B;
  return 2 * GR * rb <= SB && DG * rb2 <= SB && 2 * D <= SB && 2 * I <= SB && D % DG == 0;
}

int launch_decode_layer(const DecodeParams& p, int num_sms, cudaStream_t s) {
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(k_decode_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_dev = dev;
  }
  k_decode_layer<<<num_sms, NTH, SMEM_BYTES, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
