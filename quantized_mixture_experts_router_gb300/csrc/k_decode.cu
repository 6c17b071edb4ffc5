// Decode path (m <= 8): one fused persistent kernel per layer call.
//
// One block per SM: a producer warp and NCW consumer warps around a ring of
// NST shared-memory stages.  The producer takes ITEMS by ticket, in dependency
// order
//   q8_1(x) | router rows | shared gate/up | routed gate/up | down groups
// and streams each item's raw weight rows into the ring as stages with 1-D
// bulk copies (cp.async.bulk, completing on the stage's mbarrier).  Each stage
// is one TASK, taken and finished by a single consumer warp; the warps of the
// block share an item through a small shared-memory state (a task counter and
// a result buffer), and the warp finishing an item's last task completes it:
//   router item   -> counts it; after the last one, selection and the plan
//   gate/up item  -> SwiGLU is done per task; the 32-row group of h goes to
//                    q8_1 units (metrale's fused swiglu_q8 step)
//   down item     -> y = sum over the picked experts in ascending id of
//                    G_i E_i, then the shared expert, written to out
// so a device-scope fence is paid once per item, not per task.  Waits on
// results of other blocks (q8_1(x), the plan, the h vectors) are bounded
// spins; the producer never waits for results, so weight bytes keep
// streaming while consumers catch up.  Every sum runs in a fixed order, so
// results do not depend on timing.  q8_1(x) and the h vectors are copied
// into shared memory once per block (when they fit) with bulk copies.
//
// Method: DeepSeek V4.1 atlas "Mixture of experts" (Router, Routed expert and
// Shared expert steps: g' = min(g, L), u' = clip(u, -L, L), h = g' sigmoid(g') u',
// y = sum G_i E_i + y_shared); metrale moe_v41 module docs and moe_v41.rs
// (Q2_K gate/up, Q3_K down, q8_1 activations, the shared expert added after
// the routed experts).
#include "internal.h"
#include "select.cuh"

namespace moe {

namespace {

constexpr int NCW = 8;               // consumer warps
constexpr int W_PROD = NCW;          // the producer warp
constexpr int W_PLAN = NCW + 1;      // the planner warp: this block's copy of the routing
constexpr int NTH = (NCW + 2) * 32;
constexpr int SB = 20480;            // bytes per ring stage
constexpr int NST = 8;               // ring stages
constexpr int NIS = 4;               // item state slots
constexpr int GR = 4;                // rows of W1 and of W3 per gate/up stage
constexpr int GT = 32;               // rows per gate/up item (one q8_1 block of h)
constexpr int DG = 8;                // output rows per down item
constexpr int RR = 2;                // router rows per router item (one stage)
constexpr int SHP = 8;               // shared bf16 (gate, up) row pairs per item
constexpr int Q8B = 32;              // q8_1 blocks per q8 item (one per lane)
constexpr int SDR = 4;               // shared bf16 down rows per stage

enum : int { K_STOP = 0, K_Q8, K_ROUTER, K_SHGU_B, K_GU_Q, K_DN_SHB, K_DN_SHQ, K_DN_RT };
enum : int { I_Q8 = 0, I_ROUTER, I_SHGU_B, I_GU, I_DN };
// shared-memory copies: x (bf16), routed h units, shared h, q8_1(x) units, expert pointer table, bias
enum : int { CB_XB = 0, CB_HR, CB_HS, CB_XU, CB_EP, CB_BIAS, N_CB };

struct Hdr {
  int kind, slot, a, b;
};

struct Item {
  int kind, a, b, pad;
  unsigned remaining;
};

struct Ctl {
  Hdr hdr[NST];
  Item item[NIS];
  unsigned long long full[NST];
  unsigned long long empty[NST];
  unsigned long long item_done[NIS];
  unsigned long long pbar;        // the block's plan is built
  unsigned long long cbar[N_CB];  // shared-memory copies: see CB_*
  unsigned cstate[N_CB];          // 0 empty, 1 being filled
  unsigned next;               // consumer grab counter
};

__device__ __forceinline__ uint8_t* smem_base() {
  extern __shared__ __align__(128) uint8_t dyn[];
  return dyn;
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
    __nanosleep(100);
    if ((++spins & 15u) == 0 && globaltimer_ns() > deadline) {
      atomicOr(status, (unsigned)MOE_STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint64_t* bar(unsigned long long& b) { return reinterpret_cast<uint64_t*>(&b); }

// ------------------------------------------------------------- sizes
struct Sizes {
  int n_q8, n_router, n_shgu, gt, dn_sh_parts;
  bool shq;
};

__device__ __forceinline__ Sizes sizes_of(const DecodeParams& p) {
  Sizes z;
  z.n_q8 = (p.m * (p.D / 32) + Q8B - 1) / Q8B;
  z.n_router = (p.N + RR - 1) / RR;
  z.shq = p.shared_kind != MOE_SHARED_BF16;
  z.gt = p.I / GT;
  z.n_shgu = z.shq ? z.gt : (p.I + SHP - 1) / SHP;
  z.dn_sh_parts = z.shq ? 1 : DG / SDR;
  return z;
}

// Ticket -> item.  Items past the shared gate/up need n_exp; kind -1 asks
// the caller to wait for the plan, kind -2 means no work is left.
__device__ __forceinline__ Item decode_ticket(unsigned t, const Sizes& z, int groups, int n_exp) {
  Item it{-2, 0, 0, 0, 0};
  if (t < (unsigned)z.n_q8) { it.kind = I_Q8; it.a = (int)t; return it; }
  t -= z.n_q8;
  if (t < (unsigned)z.n_router) { it.kind = I_ROUTER; it.a = (int)t; return it; }
  t -= z.n_router;
  if (t < (unsigned)z.n_shgu) {
    if (z.shq) { it.kind = I_GU; it.a = -1; it.b = (int)t; }
    else { it.kind = I_SHGU_B; it.a = (int)t; }
    return it;
  }
  t -= z.n_shgu;
  if (n_exp < 0) { it.kind = -1; return it; }
  const unsigned n_rtgu = (unsigned)n_exp * z.gt;
  if (t < n_rtgu) { it.kind = I_GU; it.a = (int)(t / z.gt); it.b = (int)(t % z.gt); return it; }
  t -= n_rtgu;
  if (t < (unsigned)groups) { it.kind = I_DN; it.a = (int)t; return it; }
  return it;
}

// ---------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 8 bf16 products into two accumulators (two independent FMA chains)
__device__ __forceinline__ void dot8(float2& acc, const uint4& w, const uint4& x) {
  acc.x = fmaf(bf16lo(w.x), bf16lo(x.x), acc.x); acc.y = fmaf(bf16hi(w.x), bf16hi(x.x), acc.y);
  acc.x = fmaf(bf16lo(w.y), bf16lo(x.y), acc.x); acc.y = fmaf(bf16hi(w.y), bf16hi(x.y), acc.y);
  acc.x = fmaf(bf16lo(w.z), bf16lo(x.z), acc.x); acc.y = fmaf(bf16hi(w.z), bf16hi(x.z), acc.y);
  acc.x = fmaf(bf16lo(w.w), bf16lo(x.w), acc.x); acc.y = fmaf(bf16hi(w.w), bf16hi(x.w), acc.y);
}

// an activation unit: from shared memory, or (written by other blocks in
// this kernel) from L2 without the non-coherent read-only path
__device__ __forceinline__ void load_unit(XUnit& x, const int4* p, bool in_smem) {
  int4 v[6];
  if (in_smem) {
#pragma unroll
    for (int i = 0; i < 6; ++i) v[i] = p[i];
  } else {
#pragma unroll
    for (int i = 0; i < 6; ++i) v[i] = __ldcg(p + i);
  }
  x.q[0] = v[0].x; x.q[1] = v[0].y; x.q[2] = v[0].z; x.q[3] = v[0].w;
  x.q[4] = v[1].x; x.q[5] = v[1].y; x.q[6] = v[1].z; x.q[7] = v[1].w;
  x.q[8] = v[2].x; x.q[9] = v[2].y; x.q[10] = v[2].z; x.q[11] = v[2].w;
  x.q[12] = v[3].x; x.q[13] = v[3].y; x.q[14] = v[3].z; x.q[15] = v[3].w;
  x.dq[0] = __int_as_float(v[4].x); x.dq[1] = __int_as_float(v[4].y);
  x.dq[2] = __int_as_float(v[4].z); x.dq[3] = __int_as_float(v[4].w);
  x.s16[0] = v[5].x; x.s16[1] = v[5].y; x.s16[2] = v[5].z; x.s16[3] = v[5].w;
}

// ------------------------------------------------------------- context
struct Ctx {
  const DecodeParams& p;
  const Sizes& z;
  Ctl& C;
  uint64_t deadline;
  int n_exp;  // -1 until the warp has read the plan
  bool x_ok, rt_ok, sh_ok, plan_ok, xb_ok;
};

// Wait (once per warp) for the copy of x that the producer started at launch.
__device__ __forceinline__ void need_xb(Ctx& c) {
  if (c.p.sm_xb && !c.xb_ok) {
    if ((threadIdx.x & 31) == 0) mbar_wait_bounded(bar(c.C.cbar[CB_XB]), 0u, c.deadline, &c.p.ctrl->status);
    __syncwarp();
    c.xb_ok = true;
  }
}

// The block's shared-memory copy of the plan (bulk-copied by the producer once
// the plan exists); the first use by a warp waits for the copy.
__device__ __forceinline__ const DecodePlan* splan(Ctx& c) {
  if (!c.plan_ok) {
    if ((threadIdx.x & 31) == 0) mbar_wait_bounded(bar(c.C.pbar), 0u, c.deadline, &c.p.ctrl->status);
    __syncwarp();
    c.plan_ok = true;
  }
  return reinterpret_cast<const DecodePlan*>(smem_base() + c.p.sm_plan);
}

__device__ __forceinline__ int plan_n_exp(Ctx& c) {
  if (c.n_exp < 0) c.n_exp = splan(c)->n_exp;
  return c.n_exp;
}

// Bounded wait of a whole warp on a global counter (lane 0 spins).
__device__ __forceinline__ bool warp_wait(Ctx& c, bool& done_flag, const unsigned* ctr, unsigned target) {
  if (!done_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_count(ctr, target, c.deadline, &c.p.ctrl->status);
    done_flag = __shfl_sync(0xffffffffu, ok, 0);
  }
  return done_flag;
}

// Shared-memory copy of a region written by other blocks, made once per block
// (which = CB_HR, CB_HS or CB_XU).  The first warp to need it
// waits for the producing counter, then bulk-copies it; every warp waits on
// the copy's mbarrier.
__device__ void ensure_cache(Ctx& c, int which, const unsigned* counter, unsigned target, const void* src,
                             uint32_t bytes, uint32_t dst_off) {
  if ((threadIdx.x & 31) == 0) {
    if (atomicCAS(&c.C.cstate[which], 0u, 1u) == 0u) {
      wait_count(counter, target, c.deadline, &c.p.ctrl->status);
      asm volatile("fence.proxy.async;" ::: "memory");
      mbar_arrive_expect_tx(bar(c.C.cbar[which]), bytes);
      bulk_g2s(smem_base() + dst_off, src, bytes, bar(c.C.cbar[which]));
    }
    mbar_wait_bounded(bar(c.C.cbar[which]), 0u, c.deadline, &c.p.ctrl->status);
  }
  __syncwarp();
}

// ------------------------------------------------------------- the plan
// Selection for every token and grouping of the (expert, token) pairs by
// ascending expert id, into this block's shared-memory plan; run by the
// planner warp of every block once all router rows are done (every block
// computes the same plan; block 0 also writes the routing outputs).  Under
// full load every dependent global round trip costs microseconds, so the
// plan never goes through global memory.
__device__ void build_plan(Ctx& c) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  float* scratch = reinterpret_cast<float*>(smem_base() + p.sm_sel);
  int* pk_id = reinterpret_cast<int*>(smem_base() + p.sm_sel + select_scratch_bytes(p.N));
  float* pk_w = reinterpret_cast<float*>(pk_id + MAXP);
  int* s_e = pk_id + 2 * MAXP;  // expert of each sorted position
  int* s_t = pk_id + 3 * MAXP;  // token of each sorted position
  const bool writer = blockIdx.x == 0;
  for (int t = 0; t < p.m; ++t) {
    float* wo = writer ? p.topk_w + (size_t)t * p.k : pk_w + t * p.k;
    int* io = writer ? p.topk_idx + (size_t)t * p.k : pk_id + t * p.k;
    if (p.N <= 384)
      route_token_warp_r12(p.logits + (size_t)t * p.N, p.sk + (size_t)t * p.N, p.bias, p.N, p.k, p.gate_temp,
                           p.norm, p.route_scale, wo, io, &p.ctrl->status, scratch, pk_id + t * p.k, pk_w + t * p.k);
    else
      route_token_warp(p.logits + (size_t)t * p.N, p.sk + (size_t)t * p.N, p.bias, p.N, p.k, p.gate_temp, p.norm,
                       p.route_scale, wo, io, &p.ctrl->status, scratch, pk_id + t * p.k, pk_w + t * p.k);
  }
  // the expert pointer table: the block's copy when there is one
  const unsigned long long* eptr = p.expert_ptrs;
  if (p.ep_bytes) {
    mbar_wait_bounded(bar(c.C.cbar[CB_EP]), 0u, c.deadline, &p.ctrl->status);
    __syncwarp();
  }
  const unsigned long long* eptr_s = reinterpret_cast<const unsigned long long*>(smem_base() + p.sm_ep);
  __syncwarp();
  DecodePlan* plan = reinterpret_cast<DecodePlan*>(smem_base() + p.sm_plan);
  const int P = p.m * p.k;
  for (int i = lane; i < P; i += 32) {
    const int e = pk_id[i], t = i / p.k;
    int rank = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = pk_id[q], tq = q / p.k;
      rank += (eq < e) || (eq == e && tq < t);
    }
    s_e[rank] = e;
    s_t[rank] = t;
    plan->pair_tok[rank] = t;
    plan->pair_w[rank] = pk_w[i];
  }
  __syncwarp();
  int n_exp = 0;
  for (int base = 0; base < P; base += 32) {
    const int i = base + lane;
    const bool first = i < P && (i == 0 || s_e[i - 1] != s_e[i]);
    const unsigned bal = __ballot_sync(0xffffffffu, first);
    if (first) {
      const int slot = n_exp + __popc(bal & ((1u << lane) - 1u));
      const int e = s_e[i];
      plan->exp_id[slot] = e;
      plan->exp_off[slot] = i;
      unsigned long long ptr[3];
      bool bad = false;
      for (int j = 0; j < 3; ++j) {
        const size_t w = (size_t)e * 3 + j;
        ptr[j] = (w + 1) * 8 <= p.ep_bytes ? eptr_s[w] : eptr[w];
      }
      for (int j = 0; j < 3; ++j) bad |= (ptr[j] == 0ull) || (ptr[j] & 255ull);
      if (bad && writer) atomicOr(&p.ctrl->status, (unsigned)MOE_STATUS_MISSING_EXPERT);
      for (int j = 0; j < 3; ++j) plan->exp_ptr[slot][j] = bad ? 0ull : ptr[j];
    }
    n_exp += __popc(bal);
  }
  // each token's pairs in ascending expert id
  for (int i = lane; i < P; i += 32) {
    const int t = s_t[i];
    int r = 0;
    for (int q = 0; q < i; ++q) r += s_t[q] == t;
    plan->tok_pairs[t][r] = i;
  }
  if (lane == 0) {
    plan->n_exp = n_exp;
    plan->n_pairs = P;
    plan->exp_off[n_exp] = P;
  }
  __syncwarp();
}

// ------------------------------------------------------------- tasks
__device__ __forceinline__ float* item_buf(const DecodeParams& p, int slot) {
  return reinterpret_cast<float*>(smem_base() + p.sm_items + (size_t)slot * p.item_bytes);
}

// q8_1 of x into global units: Q8B of the m*D/32 blocks, one per thread
__device__ void task_q8(Ctx& c, int it) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int nb = p.D / 32;
  const int total = p.m * nb;
  for (int g = it * Q8B + lane; g < it * Q8B + Q8B && g < total; g += 32) {
    const int t = g / nb, qb = g % nb;
    q8_block_thread(p.x + (size_t)t * p.D + (size_t)qb * 32, qb, p.xu + (size_t)t * (unit_bytes(p.D) / 4));
  }
}

// x of token t as uint4 chunks: the shared-memory copy when there is one
__device__ __forceinline__ uint4 x_chunk(const DecodeParams& p, int t, int ch) {
  if (p.sm_xb) return reinterpret_cast<const uint4*>(smem_base() + p.sm_xb)[(size_t)t * (p.D / 8) + ch];
  return __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D) + ch);
}

// router rows r0, r0+1 against every token -> logits
__device__ void task_router(Ctx& c, const uint8_t* stage, int r0) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int chunks = p.D / 8;
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  const int rows = min(RR, p.N - r0);
  need_xb(c);
  if (p.sm_bias && (threadIdx.x & 31) == 0) mbar_wait_bounded(bar(c.C.cbar[CB_BIAS]), 0u, c.deadline, &p.ctrl->status);
  __syncwarp();
  const float* bias = p.sm_bias ? reinterpret_cast<const float*>(smem_base() + p.sm_bias) : p.bias;
  for (int t = 0; t < p.m; ++t) {
    float2 a0[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, a1[2] = {a0[0], a0[0]};
    for (int ch = lane, i = 0; ch < chunks; ch += 32, ++i) {
      const uint4 xv = x_chunk(p, t, ch);
      dot8(a0[i & 1], w[ch], xv);
      if (rows > 1) dot8(a1[i & 1], w[chunks + ch], xv);
    }
    const float s0 = warp_sum((a0[0].x + a0[0].y) + (a0[1].x + a0[1].y));
    const float s1 = warp_sum((a1[0].x + a1[0].y) + (a1[1].x + a1[1].y));
    // the logit, and the fast score and key the selection starts from
    if (lane < rows) {
      const float z = lane == 0 ? s0 : s1;
      const int e = r0 + lane;
      const float sc = score_fast(z, p.gate_temp);
      p.logits[(size_t)t * p.N + e] = z;
      p.sk[(size_t)t * p.N + e] = make_float2(sc, __fadd_rn(sc, bias[e]));
    }
  }
}

// one (gate, up) row pair of the bf16 shared expert: h = SwiGLU(g, u) -> bf16
__device__ void task_shgu_b(Ctx& c, const uint8_t* stage, int row) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int chunks = p.D / 8;
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  need_xb(c);
  for (int t = 0; t < p.m; ++t) {
    float2 ga[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, ua[2] = {ga[0], ga[0]};
    for (int ch = lane, i = 0; ch < chunks; ch += 32, ++i) {
      const uint4 xv = x_chunk(p, t, ch);
      dot8(ga[i & 1], w[ch], xv);
      dot8(ua[i & 1], w[chunks + ch], xv);
    }
    const float g = warp_sum((ga[0].x + ga[0].y) + (ga[1].x + ga[1].y));
    const float u = warp_sum((ua[0].x + ua[0].y) + (ua[1].x + ua[1].y));
    if (lane == 0)
      reinterpret_cast<__nv_bfloat16*>(p.shh)[(size_t)t * p.I + row] =
          __float2bfloat16_rn(swiglu_f32(g, u, p.swiglu_limit));
  }
}

// GR rows of W1 (stage offset 0) and of W3 (offset GR*rb) in Q2_K against the
// q8_1(x) units of the item's tokens: half-warp 0 takes W1, half-warp 1 W3,
// each lane 1/16 of the units of every row.  h of the rows -> item buffer.
__device__ void task_gu_q(Ctx& c, const uint8_t* stage, int slot, int stg, float* ib) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31, half = lane >> 4, l = lane & 15;
  const int rb = (p.D / QK) * Q2K_B;
  const int U = p.D / 64;
  const bool shared = slot < 0;
  int pair0 = 0, ntok = p.m;
  const DecodePlan* plan = shared ? nullptr : splan(c);
  if (!shared) {
    pair0 = plan->exp_off[slot];
    ntok = plan->exp_off[slot + 1] - pair0;
    if (plan->exp_ptr[slot][0] == 0ull) return;
  }
  const bool xs = p.sm_x != 0;
  if (xs) ensure_cache(c, CB_XU, &p.ctrl->q8_done, (unsigned)c.z.n_q8, p.xu, (uint32_t)(p.m * unit_bytes(p.D)), p.sm_x);
  else warp_wait(c, c.x_ok, &p.ctrl->q8_done, (unsigned)c.z.n_q8);
  const uint8_t* base = stage + (size_t)half * GR * rb;
  const size_t xstride = unit_bytes(p.D) / 16;
  const int4* xall = xs ? reinterpret_cast<const int4*>(smem_base() + p.sm_x) : reinterpret_cast<const int4*>(p.xu);
  for (int tt = 0; tt < ntok; ++tt) {
    const int tok = shared ? tt : plan->pair_tok[pair0 + tt];
    const int4* xb = xall + (size_t)tok * xstride;
    float acc[GR];
#pragma unroll
    for (int r = 0; r < GR; ++r) acc[r] = 0.f;
    for (int u = l; u < U; u += 16) {
      XUnit xr;
      load_unit(xr, xb + u * 6, xs);
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
#pragma unroll
    for (int r = 0; r < GR; ++r) {
      const float u = __shfl_sync(0xffffffffu, acc[r], 16);
      if (lane == 0) ib[(stg * GR + r) * p.m + tt] = swiglu_f32(acc[r], u, p.swiglu_limit);
    }
  }
}

// 8 rows of a Q3_K down matrix (stage) against h units: lane = (row, 1/4 of
// the units).  Routed: E of each pair of the slot -> item buffer (unweighted);
// shared (slot < 0): the shared expert's rows.
__device__ void task_dn_q(Ctx& c, const uint8_t* stage, int slot, float* ib) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31, row = lane >> 2, q = lane & 3;
  const int rb2 = (p.I / QK) * Q3K_B;
  const int U2 = p.I / 64;
  const bool shared = slot < 0;
  const int P = p.m * p.k;
  const size_t hstride = unit_bytes(p.I) / 16;
  int pb = 0, pe = p.m;
  bool present = true, hs;
  const int4* hbase;
  if (!shared) {
    const DecodePlan* plan = splan(c);
    pb = plan->exp_off[slot];
    pe = plan->exp_off[slot + 1];
    present = plan->exp_ptr[slot][2] != 0ull;
    const unsigned target = (unsigned)(plan_n_exp(c) * c.z.gt);
    hs = p.sm_hr != 0;
    if (hs) {
      ensure_cache(c, CB_HR, &p.ctrl->rtgu_done, target, p.hu, (uint32_t)(P * unit_bytes(p.I)), p.sm_hr);
      hbase = reinterpret_cast<const int4*>(smem_base() + p.sm_hr);
    } else {
      warp_wait(c, c.rt_ok, &p.ctrl->rtgu_done, target);
      hbase = reinterpret_cast<const int4*>(p.hu);
    }
  } else {
    hs = p.sm_hs != 0;
    const unsigned target = (unsigned)c.z.n_shgu;
    if (hs) {
      ensure_cache(c, CB_HS, &p.ctrl->shgu_done, target, p.hu + (size_t)p.shvec0 * (unit_bytes(p.I) / 4),
                   (uint32_t)(p.m * unit_bytes(p.I)), p.sm_hs);
      hbase = reinterpret_cast<const int4*>(smem_base() + p.sm_hs);
    } else {
      warp_wait(c, c.sh_ok, &p.ctrl->shgu_done, target);
      hbase = reinterpret_cast<const int4*>(p.hu) + (size_t)p.shvec0 * hstride;
    }
  }
  const uint8_t* rowp = stage + (size_t)row * rb2;
  for (int pi = pb; pi < pe; ++pi) {
    float acc = 0.f;
    if (present) {
      const int4* hb = hbase + (size_t)pi * hstride;
      for (int u = q; u < U2; u += 4) {
        XUnit hr;
        load_unit(hr, hb + u * 6, hs);
        acc += q3k_unit_dot(rowp + (u >> 2) * Q3K_B, u & 3, hr);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (q == 0) {
      if (shared) ib[(P + pi) * DG + row] = acc;
      else ib[pi * DG + row] = acc;
    }
  }
}

// SDR rows of the bf16 shared down matrix against h (bf16 [m, I]) -> item buffer
__device__ void task_dn_b(Ctx& c, const uint8_t* stage, int part, float* ib) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  const int chunks = p.I / 8;
  const int P = p.m * p.k;
  const bool hs = p.sm_hs != 0;
  const uint4* hbase;
  if (hs) {
    ensure_cache(c, CB_HS, &p.ctrl->shgu_done, (unsigned)c.z.n_shgu, p.shh, (uint32_t)(p.m * 2 * p.I), p.sm_hs);
    hbase = reinterpret_cast<const uint4*>(smem_base() + p.sm_hs);
  } else {
    warp_wait(c, c.sh_ok, &p.ctrl->shgu_done, (unsigned)c.z.n_shgu);
    hbase = reinterpret_cast<const uint4*>(p.shh);
  }
  const uint4* w = reinterpret_cast<const uint4*>(stage);
  for (int t = 0; t < p.m; ++t) {
    const uint4* hr = hbase + (size_t)t * chunks;
    float2 acc[SDR];
#pragma unroll
    for (int r = 0; r < SDR; ++r) acc[r] = make_float2(0.f, 0.f);
    for (int ch = lane; ch < chunks; ch += 32) {
      const uint4 hv = hs ? hr[ch] : __ldcg(hr + ch);
#pragma unroll
      for (int r = 0; r < SDR; ++r) dot8(acc[r], w[r * chunks + ch], hv);
    }
#pragma unroll
    for (int r = 0; r < SDR; ++r) {
      const float s = warp_sum(acc[r].x + acc[r].y);
      if (lane == 0) ib[(P + t) * DG + part * SDR + r] = s;
    }
  }
}

// ------------------------------------------------------- item completion
__device__ void complete_item(Ctx& c, const Item& it, float* ib) {
  const DecodeParams& p = c.p;
  const int lane = threadIdx.x & 31;
  switch (it.kind) {
    case I_Q8:
      __threadfence();
      if (lane == 0) atomicAdd(&p.ctrl->q8_done, 1u);
      break;
    case I_ROUTER:
      __threadfence();
      if (lane == 0) atomicAdd(&p.ctrl->router_done, 1u);
      break;
    case I_SHGU_B:
      __threadfence();
      if (lane == 0) atomicAdd(&p.ctrl->shgu_done, 1u);
      break;
    case I_GU: {
      // q8_1 of the item's 32 rows of h, per token
      const bool shared = it.a < 0;
      int ntok = p.m, vec0 = p.shvec0;
      bool present = true;
      if (!shared) {
        const DecodePlan* plan = splan(c);
        vec0 = plan->exp_off[it.a];
        ntok = plan->exp_off[it.a + 1] - vec0;
        present = plan->exp_ptr[it.a][0] != 0ull;
      }
      for (int tt = 0; tt < ntok && present; ++tt)
        q8_block_warp(ib[lane * p.m + tt], it.b, nullptr, p.hu + (size_t)(vec0 + tt) * (unit_bytes(p.I) / 4));
      __threadfence();
      if (lane == 0) atomicAdd(shared ? &p.ctrl->shgu_done : &p.ctrl->rtgu_done, 1u);
      break;
    }
    case I_DN: {
      // y = sum over the token's pairs in ascending expert id of G E, then + S
      const DecodePlan* plan = splan(c);
      const int P = p.m * p.k;
      for (int qd = lane; qd < p.m * DG; qd += 32) {
        const int t = qd / DG, r = qd % DG;
        float acc = 0.f;
        for (int i = 0; i < p.k; ++i) {
          const int pr = plan->tok_pairs[t][i];
          acc = fmaf(plan->pair_w[pr], ib[pr * DG + r], acc);
        }
        acc += ib[(P + t) * DG + r];
        p.out[(size_t)t * p.D + it.a * DG + r] = acc;
      }
      break;
    }
    default:
      break;
  }
}

// ================================================================ kernel
__global__ void __launch_bounds__(NTH, 1) k_decode_layer(const __grid_constant__ DecodeParams p) {
  Ctl& C = *reinterpret_cast<Ctl*>(smem_base() + p.sm_ctl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(C.full[i]), 1);
      mbar_init(bar(C.empty[i]), 1);
    }
    for (int i = 0; i < NIS; ++i) mbar_init(bar(C.item_done[i]), 1);
    mbar_init(bar(C.pbar), 1);
    for (int i = 0; i < N_CB; ++i) {
      mbar_init(bar(C.cbar[i]), 1);
      C.cstate[i] = 0u;
    }
    C.next = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  const Sizes z = sizes_of(p);
  const int groups = p.D / DG;

  if (warp == W_PLAN) {
    // ----------------------------------------------------------- planner
    // Wait for every router row of the call, then build this block's plan.
    // On a timeout the plan is left empty (no routed expert work) so the
    // block still finishes; the status word already says why.
    Ctx c{p, z, C, deadline, -1, false, false, false, false, false};
    bool ok = true;
    if (lane == 0) ok = wait_count(&p.ctrl->router_done, (unsigned)z.n_router, deadline, &p.ctrl->status);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      build_plan(c);
    } else if (lane == 0) {
      DecodePlan* plan = reinterpret_cast<DecodePlan*>(smem_base() + p.sm_plan);
      plan->n_exp = 0;
      plan->n_pairs = 0;
      plan->exp_off[0] = 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C.pbar));
  } else if (warp == W_PROD) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      // x and the expert pointer table are inputs of the call: copy them to
      // shared memory at once
      if (p.sm_xb) {
        const uint32_t xbytes = (uint32_t)(p.m * 2 * p.D);
        mbar_arrive_expect_tx(bar(C.cbar[CB_XB]), xbytes);
        bulk_g2s(smem_base() + p.sm_xb, p.x, xbytes, bar(C.cbar[CB_XB]));
      }
      if (p.ep_bytes) {
        mbar_arrive_expect_tx(bar(C.cbar[CB_EP]), p.ep_bytes);
        bulk_g2s(smem_base() + p.sm_ep, p.expert_ptrs, p.ep_bytes, bar(C.cbar[CB_EP]));
      }
      if (p.sm_bias) {
        mbar_arrive_expect_tx(bar(C.cbar[CB_BIAS]), (uint32_t)(p.N * 4));
        bulk_g2s(smem_base() + p.sm_bias, p.bias, (uint32_t)(p.N * 4), bar(C.cbar[CB_BIAS]));
      }
      uint32_t n = 0;  // stages issued
      uint32_t j = 0;  // items started
      int n_exp = -1;
      bool ok = true;
      const int rb = (p.D / QK) * Q2K_B, rb2 = (p.I / QK) * Q3K_B;
      unsigned t_next = atomicAdd(&p.ctrl->ticket, 1u);
      for (;;) {
        const unsigned t = t_next;
        Item it = decode_ticket(t, z, groups, n_exp);
        if (it.kind == -1) {
          // the block's plan, built by the planner warp
          if (!(ok = mbar_wait_bounded(bar(C.pbar), 0u, deadline, &p.ctrl->status))) break;
          n_exp = reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan)->n_exp;
          it = decode_ticket(t, z, groups, n_exp);
        }
        if (it.kind == -2) break;
        t_next = atomicAdd(&p.ctrl->ticket, 1u);  // the next ticket is in flight while this item streams
        int ns;
        switch (it.kind) {
          case I_Q8: ns = 1; break;
          case I_ROUTER: ns = 1; break;
          case I_SHGU_B: ns = min(SHP, p.I - it.a * SHP); break;
          case I_GU: ns = GT / GR; break;
          default: ns = z.dn_sh_parts + n_exp; break;
        }
        const uint32_t islot = j % NIS;
        if (j >= (uint32_t)NIS &&
            !(ok = mbar_wait_bounded(bar(C.item_done[islot]), (j / NIS - 1) & 1u, deadline, &p.ctrl->status)))
          break;
        it.remaining = (unsigned)ns;
        C.item[islot] = it;
        for (int s = 0; s < ns; ++s) {
          const uint32_t slot = n % NST, use = n / NST;
          if (use > 0 && !(ok = mbar_wait_bounded(bar(C.empty[slot]), (use - 1) & 1u, deadline, &p.ctrl->status)))
            break;
          Hdr h{K_STOP, (int)islot, 0, 0};
          const uint8_t *a = nullptr, *b = nullptr;
          uint32_t bytes = 0, boff = 0;
          switch (it.kind) {
            case I_Q8:
              h.kind = K_Q8; h.a = it.a;
              break;
            case I_ROUTER: {
              const int r0 = it.a * RR;
              h.kind = K_ROUTER; h.a = r0;
              a = reinterpret_cast<const uint8_t*>(p.router_w) + (size_t)r0 * 2 * p.D;
              bytes = (uint32_t)(min(RR, p.N - r0) * 2 * p.D);
              break;
            }
            case I_SHGU_B: {
              const int row = it.a * SHP + s;
              h.kind = K_SHGU_B; h.a = row;
              a = p.sh1 + (size_t)row * 2 * p.D;
              b = p.sh3 + (size_t)row * 2 * p.D;
              bytes = (uint32_t)(2 * p.D);
              boff = bytes;
              break;
            }
            case I_GU: {
              const int r0 = it.b * GT + s * GR;
              h.kind = K_GU_Q; h.a = it.a; h.b = s;
              const uint8_t *w1, *w3;
              if (it.a < 0) {
                w1 = p.sh1; w3 = p.sh3;
              } else {
                const DecodePlan* sp = reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan);
                w1 = reinterpret_cast<const uint8_t*>(sp->exp_ptr[it.a][0]);
                w3 = reinterpret_cast<const uint8_t*>(sp->exp_ptr[it.a][1]);
              }
              if (w1 && w3) {
                a = w1 + (size_t)r0 * rb;
                b = w3 + (size_t)r0 * rb;
                bytes = (uint32_t)(GR * rb);
                boff = bytes;
              }
              break;
            }
            default: {  // I_DN: shared parts first, then the experts in ascending id
              const int d0 = it.a * DG;
              if (s < z.dn_sh_parts) {
                if (z.shq) {
                  h.kind = K_DN_SHQ;
                  a = p.sh2 + (size_t)d0 * rb2;
                  bytes = (uint32_t)(DG * rb2);
                } else {
                  h.kind = K_DN_SHB; h.a = s;
                  a = p.sh2 + (size_t)(d0 + s * SDR) * 2 * p.I;
                  bytes = (uint32_t)(SDR * 2 * p.I);
                }
              } else {
                const int e = s - z.dn_sh_parts;
                h.kind = K_DN_RT; h.a = e;
                const unsigned long long w2 =
                    reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan)->exp_ptr[e][2];
                if (w2) {
                  a = reinterpret_cast<const uint8_t*>(w2) + (size_t)d0 * rb2;
                  bytes = (uint32_t)(DG * rb2);
                }
              }
              break;
            }
          }
          C.hdr[slot] = h;
          uint8_t* dst = smem_base() + (size_t)slot * SB;
          mbar_arrive_expect_tx(bar(C.full[slot]), a ? (b ? 2u * bytes : bytes) : 0u);
          if (a) bulk_g2s(dst, a, bytes, bar(C.full[slot]));
          if (a && b) bulk_g2s(dst + boff, b, bytes, bar(C.full[slot]));
          ++n;
        }
        if (!ok) break;
        ++j;
      }
      if (ok) {
        // one stop per consumer warp
        for (int s = 0; s < NCW; ++s) {
          const uint32_t slot = n % NST, use = n / NST;
          if (use > 0 && !(ok = mbar_wait_bounded(bar(C.empty[slot]), (use - 1) & 1u, deadline, &p.ctrl->status)))
            break;
          C.hdr[slot] = Hdr{K_STOP, 0, 0, 0};
          mbar_arrive(bar(C.full[slot]));
          ++n;
        }
      }
      if (!ok) {
        // let the copies already issued land before the block can exit
        const uint64_t d2 = globaltimer_ns() + p.timeout_ns;
        for (uint32_t i = n > (uint32_t)NST ? n - NST : 0u; i < n; ++i)
          mbar_wait_bounded(bar(C.full[i % NST]), (i / NST) & 1u, d2, &p.ctrl->status);
      }
    }
  } else {
    // --------------------------------------------------------- consumers
    Ctx c{p, z, C, deadline, -1, false, false, false, false, false};
    for (;;) {
      unsigned n = 0;
      if (lane == 0) n = atomicAdd(&C.next, 1u);
      n = __shfl_sync(0xffffffffu, n, 0);
      const uint32_t slot = n % NST;
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(bar(C.full[slot]), (n / NST) & 1u, deadline, &p.ctrl->status);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      const Hdr h = C.hdr[slot];
      if (h.kind == K_STOP) break;
      const uint8_t* st = smem_base() + (size_t)slot * SB;
      float* ib = item_buf(p, h.slot);
      switch (h.kind) {
        case K_Q8: task_q8(c, h.a); break;
        case K_ROUTER: task_router(c, st, h.a); break;
        case K_SHGU_B: task_shgu_b(c, st, h.a); break;
        case K_GU_Q: task_gu_q(c, st, h.a, h.b, ib); break;
        case K_DN_SHB: task_dn_b(c, st, h.a, ib); break;
        case K_DN_SHQ: task_dn_q(c, st, -1, ib); break;
        case K_DN_RT: task_dn_q(c, st, h.a, ib); break;
        default: break;
      }
      // release the stage, then count the task against its item
      __syncwarp();
      __threadfence_block();
      unsigned left = 0;
      if (lane == 0) {
        mbar_arrive(bar(C.empty[slot]));
        left = atomicSub(&C.item[h.slot].remaining, 1u);
      }
      left = __shfl_sync(0xffffffffu, left, 0);
      if (left == 1u) {
        __threadfence_block();
        const Item it = C.item[h.slot];
        complete_item(c, it, ib);
        __syncwarp();
        __threadfence_block();
        if (lane == 0) mbar_arrive(bar(C.item_done[h.slot]));
      }
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
      p.ctrl->router_done = 0u;
      p.ctrl->shgu_done = 0u;
      p.ctrl->rtgu_done = 0u;
      __threadfence();
      p.ctrl->exit_count = 0u;
    }
  }
}

constexpr size_t SMEM_MAX = 232448;  // 227 KB of dynamic shared memory per block

size_t a16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory plan of one launch; the caches only where they fit.
bool plan_smem(DecodeParams& p) {
  size_t off = (size_t)NST * SB + 16;
  p.sm_ctl = (uint32_t)off;
  off = a16(off + sizeof(Ctl));
  p.sm_plan = (uint32_t)off;
  off = a16(off + sizeof(DecodePlan));
  const size_t P = (size_t)p.m * p.k;
  const size_t gu = (size_t)GT * p.m * 4, dn = (P + p.m) * DG * 4;
  p.item_bytes = (uint32_t)a16(gu > dn ? gu : dn);
  p.sm_items = (uint32_t)off;
  off += (size_t)NIS * p.item_bytes;
  p.sm_sel = (uint32_t)off;
  off = a16(off + select_scratch_bytes(p.N) + (size_t)4 * MAXP * 4);  // selection, picks, sorted pairs
  if (off > SMEM_MAX) return false;
  auto try_cache = [&](size_t bytes) -> uint32_t {
    if (off + bytes > SMEM_MAX) return 0u;
    const uint32_t o = (uint32_t)off;
    off = a16(off + bytes);
    return o;
  };
  p.sm_xb = try_cache((size_t)p.m * 2 * p.D);
  const size_t ep = ((size_t)p.N * 24) & ~size_t(15);  // bulk copies move multiples of 16 bytes
  p.sm_ep = try_cache(ep);
  p.ep_bytes = p.sm_ep ? (uint32_t)ep : 0u;
  p.sm_x = try_cache((size_t)p.m * unit_bytes(p.D));
  p.sm_hr = try_cache(P * unit_bytes(p.I));
  p.sm_hs = try_cache(p.shared_kind == MOE_SHARED_BF16 ? (size_t)p.m * 2 * p.I : (size_t)p.m * unit_bytes(p.I));
  // the bias, when a bulk copy can move it (16-B aligned, a multiple of 16 bytes)
  p.sm_bias = (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0 && (p.N * 4) % 16 == 0 ? try_cache((size_t)p.N * 4) : 0u;
  p.smem_bytes = (uint32_t)off;
  return true;
}

}  // namespace

bool decode_fits(int D, int I) {
  const int rb = (D / QK) * Q2K_B, rb2 = (I / QK) * Q3K_B;
  return 2 * GR * rb <= SB && DG * rb2 <= SB && RR * 2 * D <= SB && 4 * D <= SB && SDR * 2 * I <= SB &&
         D % DG == 0 && I % GT == 0;
}

int launch_decode_layer(const DecodeParams& p_in, int num_sms, cudaStream_t s) {
  DecodeParams p = p_in;
  if (!plan_smem(p)) return MOE_ERR_ARG;
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(k_decode_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MAX) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_dev = dev;
  }
  k_decode_layer<<<num_sms, NTH, p.smem_bytes, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
