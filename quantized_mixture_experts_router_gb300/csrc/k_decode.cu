// Decode path (m <= 8): one fused persistent kernel per layer call.
//
// One block per SM: a producer warp, a planner warp and NCW consumer warps
// (NPAIR pairs) around a ring of NST shared-memory stages.  The producer takes ITEMS by
// ticket from four streams: first
//   q8_1(x) | router rows | shared gate/up
// then routed gate/up items as soon as its block's plan exists, shared down
// items while it does not (and when the routed gate/up items run out), and
// the routed down items last, and streams each item's raw weight rows into the ring as stages with 1-D
// bulk copies (cp.async.bulk, completing on the stage's mbarrier).  Each stage
// is one TASK, taken and finished by a pair of consumer warps (each does half
// of the stage's rows); the pairs of the block share an item through a small
// shared-memory state (a task counter and a result buffer), and the pair
// finishing an item's last task completes it:
//   router item   -> counts it; the planner warp of every block then selects
//                    the experts and groups the pairs into its own plan
//   gate/up item  -> SwiGLU is done per task; the 32-row group of h goes to
//                    q8_1 units (metrale's fused swiglu_q8 step)
//   shared down   -> y_shared of 8 output rows, written to out
//   routed down   -> y = sum over the picked experts in ascending id of
//                    G_i E_i, then + y_shared read back from out
// so a device-scope fence is paid once per item, not per task.  Waits on
// results of other blocks (q8_1(x), the plan, the h vectors) are bounded
// spins; the producer never waits for results, so weight bytes keep
// streaming while consumers catch up.  Every sum runs in a fixed order, so
// results do not depend on timing.  q8_1(x) and the h vectors are copied
// into shared memory once per block (when they fit) with bulk copies.
//
// Code layout: the SM's instruction cache holds a few tens of KB, and warps
// of one SM run different task kinds at once; a miss costs a trip to L2,
// which under the full streaming load takes microseconds.  So every task kind
// is one out-of-line routine with rolled loops, called from a single site,
// and the readiness of inputs is a block-level bit in shared memory.
//
// Method: DeepSeek V4.1 atlas "Mixture of experts" (Router, Routed expert and
// Shared expert steps: g' = min(g, L), u' = clip(u, -L, L), h = g' sigmoid(g') u',
// y = sum G_i E_i + y_shared); metrale moe_v41 module docs and moe_v41.rs
// (Q2_K gate/up, Q3_K down, q8_1 activations, the shared expert added after
// the routed experts).
#include <algorithm>

#include "internal.h"
#include "bf16dot.cuh"
#include "select.cuh"

namespace moe {

namespace {

constexpr int NCW = 16;              // consumer warps
constexpr int NPAIR = NCW / 2;       // consumer pairs: a stage is one task of a pair of warps
constexpr int W_PROD = NCW;          // the producer warp
constexpr int W_PLAN = NCW + 1;      // the planner warp: this block's copy of the routing
constexpr int NTH = (NCW + 2) * 32;
constexpr int SB = 13440;            // bytes per ring stage (4 + 4 Q2_K rows of 5120)
constexpr int NST = 12;              // ring stages: NPAIR in work plus the copies in flight
constexpr int NIS = 4;               // item state slots
constexpr int GR = 4;                // rows of W1 and of W3 per gate/up stage
constexpr int GT = 32;               // rows per gate/up item (one q8_1 block of h)
constexpr int DG = 8;                // output rows per down item
constexpr int RR = 1;                // router rows per router item (one stage)
constexpr int SHP = 8;               // shared bf16 (gate, up) row pairs per item, one row per stage
constexpr int Q8B = 32;              // q8_1 blocks per q8 item (one per lane)
constexpr int SDR = 2;               // shared bf16 down rows per stage
constexpr int UB = UNIT_WORDS * 4;   // bytes of one activation unit
// the producer ends the ring with one stop stage per consumer; a stop stage
// is never released, so all of them must fit in the ring at once
static_assert(NPAIR <= NST, "more consumer pairs than ring stages");
static_assert(GR == 4 && RR == 1 && SDR == 2, "the row routines are instantiated for these row counts");
static_assert(SB % 16 == 0, "stages start on 16-byte boundaries");

enum : int { K_STOP = 0, K_Q8, K_ROUTER, K_SHGU_B, K_GU_Q, K_DN_SHB, K_DN_SHQ, K_DN_RT, K_LOCAL };
enum : int { I_Q8 = 0, I_ROUTER, I_SHGU_B, I_GU, I_SHDN, I_DN, I_LOCAL };
// shared-memory copies: x (bf16), routed h units, shared h, q8_1(x) units, expert pointer table, bias
enum : int { CB_XB = 0, CB_HR, CB_HS, CB_XU, CB_EP, CB_BIAS, N_CB };
// block-level readiness of the inputs a task reads (bits of Ctl::rdy)
enum : unsigned { RQ_XB = 1u, RQ_BIAS = 2u, RQ_XU = 4u, RQ_HR = 8u, RQ_HS = 16u, RQ_PLAN = 32u, RQ_SHDN = 64u };

struct Hdr {
  int kind, slot, a, b;
  unsigned seq;  // the stage sequence number this header belongs to
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
  unsigned next;                  // consumer grab counter
  unsigned rdy;                   // RQ_* bits: inputs ready for every warp of the block
  unsigned xq;                    // consumer warps done with their share of q8_1(x)
  unsigned sink;                  // status bits of the planner's warm-up pass (discarded)
  unsigned pair_n[NPAIR];         // the stage each pair works on (written by its leader)
  unsigned pair_ok[NPAIR];        // 0: the leader's wait for the stage failed
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

__device__ __forceinline__ unsigned ld_acquire_cta(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.cta.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
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
  // with a shared-memory copy of q8_1(x) the planner warp of every block
  // quantises x itself; otherwise q8 items write it to global memory
  z.n_q8 = p.sm_x ? 0 : (p.m * (p.D / 32) + Q8B - 1) / Q8B;
  z.n_router = (p.N + RR - 1) / RR;
  z.shq = p.shared_kind != MOE_SHARED_BF16;
  z.gt = p.I / GT;
  z.n_shgu = z.shq ? z.gt : (p.I + SHP - 1) / SHP;
  z.dn_sh_parts = z.shq ? 1 : DG / SDR;
  return z;
}

// Ticket streams of the producer and the item a ticket stands for; kind -2
// when the stream is exhausted.  The routed streams need n_exp >= 0.
enum : int { S_MAIN = 0, S_SHDN, S_GU, S_DN, N_STREAMS };

__device__ __forceinline__ Item decode_ticket(int stream, unsigned t, const Sizes& z, int groups, int n_exp) {
  Item it{-2, 0, 0, 0, 0};
  switch (stream) {
    case S_MAIN:
      if (t < (unsigned)z.n_q8) { it.kind = I_Q8; it.a = (int)t; return it; }
      t -= z.n_q8;
      if (t < (unsigned)z.n_router) { it.kind = I_ROUTER; it.a = (int)t; return it; }
      t -= z.n_router;
      if (t < (unsigned)z.n_shgu) {
        if (z.shq) { it.kind = I_GU; it.a = -1; it.b = (int)t; }
        else { it.kind = I_SHGU_B; it.a = (int)t; }
      }
      return it;
    case S_SHDN:
      if (t < (unsigned)groups) { it.kind = I_SHDN; it.a = (int)t; }
      return it;
    case S_GU:
      if (t < (unsigned)(n_exp * z.gt)) { it.kind = I_GU; it.a = (int)(t / z.gt); it.b = (int)(t % z.gt); }
      return it;
    default:
      if (n_exp > 0 && t < (unsigned)groups) { it.kind = I_DN; it.a = (int)t; }
      return it;
  }
}

// 16 bytes of an activation vector: from the block's shared-memory copy (S,
// byte offset so + off), else from global memory through L2 (the vector may
// have been written by other blocks of this kernel)
template <bool S>
__device__ __forceinline__ uint4 vld(uint32_t so, const uint8_t* g, uint32_t off) {
  if constexpr (S) return *reinterpret_cast<const uint4*>(smem_base() + so + off);
  else return __ldcg(reinterpret_cast<const uint4*>(g + off));
}

template <bool S>
__device__ __forceinline__ void load_unit(XUnit& x, uint32_t so, const uint8_t* g, uint32_t off) {
  uint4 v[6];
#pragma unroll
  for (int i = 0; i < 6; ++i) v[i] = vld<S>(so, g, off + 16u * i);
  x.q[0] = (int)v[0].x; x.q[1] = (int)v[0].y; x.q[2] = (int)v[0].z; x.q[3] = (int)v[0].w;
  x.q[4] = (int)v[1].x; x.q[5] = (int)v[1].y; x.q[6] = (int)v[1].z; x.q[7] = (int)v[1].w;
  x.q[8] = (int)v[2].x; x.q[9] = (int)v[2].y; x.q[10] = (int)v[2].z; x.q[11] = (int)v[2].w;
  x.q[12] = (int)v[3].x; x.q[13] = (int)v[3].y; x.q[14] = (int)v[3].z; x.q[15] = (int)v[3].w;
  x.dq[0] = __uint_as_float(v[4].x); x.dq[1] = __uint_as_float(v[4].y);
  x.dq[2] = __uint_as_float(v[4].z); x.dq[3] = __uint_as_float(v[4].w);
  x.s16[0] = (int)v[5].x; x.s16[1] = (int)v[5].y; x.s16[2] = (int)v[5].z; x.s16[3] = (int)v[5].w;
}

// ------------------------------------------------------ row dot routines
// R rows of bf16 weights (stage offset w, row stride rs bytes) dotted with
// one bf16 vector of `chunks` 16-byte chunks (chunks a multiple of 32).
// Every lane returns the R sums.
template <int R, bool S>
__device__ __noinline__ float4 bf16_rows_dot(uint32_t w, uint32_t rs, uint32_t vs, const uint8_t* vg, int chunks) {
  const int lane = threadIdx.x & 31;
  const uint8_t* sw = smem_base() + w;
  float2 a[R], b[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a[r] = b[r] = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int ch = lane; ch < chunks; ch += 64) {
    const uint4 v0 = vld<S>(vs, vg, 16u * ch);
#pragma unroll
    for (int r = 0; r < R; ++r) dot8(a[r], *reinterpret_cast<const uint4*>(sw + r * rs + 16u * ch), v0);
    if (ch + 32 < chunks) {
      const uint4 v1 = vld<S>(vs, vg, 16u * (ch + 32));
#pragma unroll
      for (int r = 0; r < R; ++r) dot8(b[r], *reinterpret_cast<const uint4*>(sw + r * rs + 16u * (ch + 32)), v1);
    }
  }
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < R; ++r) o[r] = warp_sum(lane_total(a[r], b[r]));
  return make_float4(o[0], o[1], o[2], o[3]);
}

// nr (at most four) Q2_K rows (stage offset w, row stride rb) against one
// q8_1(x) vector in the unit layout, by a half-warp (16 lanes, 1/16 of the
// units each).  Every lane of the half returns the sums (rows past nr: 0).
template <bool S>
__device__ __noinline__ float4 q2k_rows4_dot(uint32_t w, uint32_t rb, int nr, int U, uint32_t xs, const uint8_t* xg) {
  const int l = threadIdx.x & 15;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 1
  for (int u = l; u < U; u += 16) {
    XUnit xr;
    load_unit<S>(xr, xs, xg, (uint32_t)u * UB);
    const uint8_t* blk = smem_base() + w + (u >> 2) * Q2K_B;
    const int c = u & 3;
    // one copy of the unit dot in the loop body (a smaller instruction footprint)
#pragma unroll 1
    for (int r = 0; r < nr; ++r) {
      const float d = q2k_unit_dot(blk + r * rb, c, xr);
      a0 += r == 0 ? d : 0.f;
      a1 += r == 1 ? d : 0.f;
      a2 += r == 2 ? d : 0.f;
      a3 += r == 3 ? d : 0.f;
    }
  }
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    a3 += __shfl_xor_sync(0xffffffffu, a3, o);
  }
  return make_float4(a0, a1, a2, a3);
}

// One Q3_K row (stage offset rowp) against one q8_1(h) vector, by the eight
// lanes of a row group (1/8 of the units each); the eight lanes return the sum.
template <bool S>
__device__ __noinline__ float q3k_row_dot(uint32_t rowp, int U2, uint32_t hs, const uint8_t* hg) {
  const int q = threadIdx.x & 7;
  float acc = 0.f;
#pragma unroll 1
  for (int u = q; u < U2; u += 8) {
    XUnit hr;
    load_unit<S>(hr, hs, hg, (uint32_t)u * UB);
    acc += q3k_unit_dot(smem_base() + rowp + (u >> 2) * Q3K_B, u & 3, hr);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  return acc;
}

// ------------------------------------------------------------- readiness
// Copy of a region written by other blocks into shared memory, made once per
// block: the first warp to need it waits for the producing counter, then
// bulk-copies it; every warp waits on the copy's mbarrier.  Without a copy
// (dst 0) the counter itself is waited for.  Lane 0 only.
__device__ void fill_or_wait(Ctl& C, int which, const unsigned* counter, unsigned target, const void* src,
                             uint32_t bytes, uint32_t dst, uint64_t deadline, unsigned* status) {
  if (!dst) {
    wait_count(counter, target, deadline, status);
    return;
  }
  if (atomicCAS(&C.cstate[which], 0u, 1u) == 0u) {
    wait_count(counter, target, deadline, status);
    asm volatile("fence.proxy.async;" ::: "memory");
    mbar_arrive_expect_tx(bar(C.cbar[which]), bytes);
    bulk_g2s(smem_base() + dst, src, bytes, bar(C.cbar[which]));
  }
  mbar_wait_bounded(bar(C.cbar[which]), 0u, deadline, status);
}

// Returns once the inputs in `bits` (RQ_*) are ready.  The first warp of the
// block to need one waits for it and publishes the bit (release at block
// scope after its own acquire), so later warps pay one shared-memory load.
// After a timeout the bit is published anyway (the status word says why).
__device__ __noinline__ void require(const DecodeParams& p, Ctl& C, unsigned bits, uint64_t deadline) {
  if ((threadIdx.x & 31) == 0) {
    const unsigned have = ld_acquire_cta(&C.rdy);
    unsigned need = bits & ~have;
    unsigned* st = &p.ctrl->status;
    while (need) {
      const unsigned bit = need & (0u - need);
      need &= need - 1u;
      const Sizes z = sizes_of(p);
      switch (bit) {
        case RQ_XB:
          if (p.sm_xb) mbar_wait_bounded(bar(C.cbar[CB_XB]), 0u, deadline, st);
          break;
        case RQ_BIAS:
          if (p.sm_bias) mbar_wait_bounded(bar(C.cbar[CB_BIAS]), 0u, deadline, st);
          break;
        case RQ_PLAN:
          mbar_wait_bounded(bar(C.pbar), 0u, deadline, st);
          break;
        case RQ_XU:
          if (p.sm_x) {
            // every consumer warp quantises its share of x at launch
            uint32_t spins = 0;
            while (ld_acquire_cta(&C.xq) < (unsigned)NCW) {
              __nanosleep(64);
              if ((++spins & 15u) == 0 && globaltimer_ns() > deadline) {
                atomicOr(st, (unsigned)MOE_STATUS_TIMEOUT);
                break;
              }
            }
          } else {
            wait_count(&p.ctrl->q8_done, (unsigned)z.n_q8, deadline, st);
          }
          break;
        case RQ_HR: {
          mbar_wait_bounded(bar(C.pbar), 0u, deadline, st);
          const DecodePlan* plan = reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan);
          fill_or_wait(C, CB_HR, &p.ctrl->rtgu_done, (unsigned)(plan->n_exp * z.gt), p.hu,
                       (uint32_t)(p.m * p.k * unit_bytes(p.I)), p.sm_hr, deadline, st);
          break;
        }
        case RQ_HS:
          if (z.shq)
            fill_or_wait(C, CB_HS, &p.ctrl->shgu_done, (unsigned)z.n_shgu,
                         p.hu + (size_t)p.shvec0 * (unit_bytes(p.I) / 4), (uint32_t)(p.m * unit_bytes(p.I)), p.sm_hs,
                         deadline, st);
          else
            fill_or_wait(C, CB_HS, &p.ctrl->shgu_done, (unsigned)z.n_shgu, p.shh, (uint32_t)(p.m * 2 * p.I),
                         p.sm_hs, deadline, st);
          break;
        case RQ_SHDN:
          wait_count(&p.ctrl->shdn_done, (unsigned)(p.D / DG), deadline, st);
          break;
        default:
          break;
      }
      __threadfence_block();
      atomicOr(&C.rdy, bit);
    }
  }
  __syncwarp();
}

__device__ __forceinline__ const DecodePlan* plan_of(const DecodeParams& p) {
  return reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan);
}

// ------------------------------------------------------------- the plan
// Selection for every token and grouping of the (expert, token) pairs by
// ascending expert id, into this block's shared-memory plan; run by the
// planner warp of every block once all router rows are done (every block
// computes the same plan; block 0 also writes the routing outputs).  Under
// full load every dependent global round trip costs microseconds, so the
// plan never goes through global memory.
// dry: the warm-up pass on whatever the workspace holds (the previous call's
// keys): it writes only this block's shared-memory plan, which the real pass
// overwrites before the plan barrier, and its status bits go to a sink.
__device__ __noinline__ void build_plan(const DecodeParams& p, Ctl& C, uint64_t deadline, bool dry) {
  const uint32_t sel = p.sm_sel, plan_off = p.sm_plan;
  const int lane = threadIdx.x & 31;
  float* scratch = reinterpret_cast<float*>(smem_base() + sel);
  int* pk_id = reinterpret_cast<int*>(smem_base() + sel + select_scratch_bytes(p.N));
  float* pk_w = reinterpret_cast<float*>(pk_id + MAXP);
  int* s_e = pk_id + 2 * MAXP;  // expert of each sorted position
  int* s_t = pk_id + 3 * MAXP;  // token of each sorted position
  const bool writer = !dry && blockIdx.x == 0;
  unsigned* status = dry ? &C.sink : &p.ctrl->status;
#pragma unroll 1
  for (int t = 0; t < p.m; ++t) {
    float* wo = writer ? p.topk_w + (size_t)t * p.k : pk_w + t * p.k;
    int* io = writer ? p.topk_idx + (size_t)t * p.k : pk_id + t * p.k;
    const float* bt = token_bias(p.bias, p.bias_vl, p.image_mask, t);
    if (p.N <= 384 && p.score_func != MOE_SCORE_SOFTMAX)
      route_token_warp_r12(p.logits + (size_t)t * p.N, p.sk + (size_t)t * p.N, bt, p.N, p.k, p.gate_temp,
                           p.score_func, p.norm, p.route_scale, wo, io, status, scratch, pk_id + t * p.k,
                           pk_w + t * p.k);
    else
      route_token_warp(p.logits + (size_t)t * p.N, p.sk + (size_t)t * p.N, bt, p.N, p.k, p.gate_temp, p.score_func,
                       p.norm, p.route_scale, wo, io, status, scratch, pk_id + t * p.k, pk_w + t * p.k);
  }
  // the expert pointer table: the block's copy when there is one
  const unsigned long long* eptr = p.expert_ptrs;
  const uint32_t ep_bytes = dry ? 0u : p.ep_bytes;  // the copy may still be in flight during the warm-up
  if (ep_bytes) {
    mbar_wait_bounded(bar(C.cbar[CB_EP]), 0u, deadline, &p.ctrl->status);
    __syncwarp();
  }
  const unsigned long long* eptr_s = reinterpret_cast<const unsigned long long*>(smem_base() + p.sm_ep);
  __syncwarp();
  DecodePlan* plan = reinterpret_cast<DecodePlan*>(smem_base() + plan_off);
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
        ptr[j] = (w + 1) * 8 <= ep_bytes ? eptr_s[w] : eptr[w];
      }
      for (int j = 0; j < 3; ++j) bad |= (ptr[j] == 0ull) || (ptr[j] & 255ull);
      if (bad && writer) atomicOr(status, (unsigned)MOE_STATUS_MISSING_EXPERT);
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
__device__ __noinline__ void task_q8(const DecodeParams& p, int it) {
  const int lane = threadIdx.x & 31;
  const int nb = p.D / 32;
  const int total = p.m * nb;
  const int g = it * Q8B + lane;
  if (g < total) {
    const int t = g / nb, qb = g % nb;
    q8_block_thread(p.x + (size_t)t * p.D + (size_t)qb * 32, qb, p.xu + (size_t)t * (unit_bytes(p.D) / 4));
  }
}

// q8_1 of x into the block's shared-memory unit layout: q8_1 blocks first,
// first + stride, ... of all tokens, one per thread
__device__ __noinline__ void quantize_x_smem(const DecodeParams& p, int first, int stride) {
  const int nb = p.D / 32;
  const uint16_t* xs = p.sm_xb ? reinterpret_cast<const uint16_t*>(smem_base() + p.sm_xb) : p.x;
#pragma unroll 1
  for (int g = first; g < p.m * nb; g += stride) {
    const int t = g / nb, qb = g % nb;
    q8_block_thread(xs + (size_t)t * p.D + (size_t)qb * 32, qb,
                    reinterpret_cast<int*>(smem_base() + p.sm_x + (size_t)t * unit_bytes(p.D)));
  }
}

// Block-local work, one task per consumer pair issued after the block's
// router rows: each warp quantises share `part` (of NCW) of q8_1(x) into
// shared memory.  All consumer warps run the code at once, so its
// instruction-cache misses are paid once per SM, not per warp.
__device__ __noinline__ void task_local(const DecodeParams& p, Ctl& C, int part, uint64_t deadline) {
  // part: this warp's share, 0 .. NCW - 1
  const int lane = threadIdx.x & 31;
  if (p.sm_x) {
    require(p, C, RQ_XB, deadline);
    quantize_x_smem(p, part * 32 + lane, NCW * 32);
    __syncwarp();
    __threadfence_block();
    if (lane == 0) atomicAdd(&C.xq, 1u);
  }
}

// router row e (stage offset st) against every token -> the logit and the
// fast (score, key) pair the selection starts from (none for the softmax,
// whose scores need every logit)
__device__ __noinline__ void task_router(const DecodeParams& p, Ctl& C, uint32_t st, int e, uint64_t deadline) {
  const int lane = threadIdx.x & 31;
  require(p, C, RQ_XB | RQ_BIAS, deadline);
  const float* bias = p.sm_bias ? reinterpret_cast<const float*>(smem_base() + p.sm_bias) : p.bias;
#pragma unroll 1
  for (int t = 0; t < p.m; ++t) {
    const float4 s = p.sm_xb ? bf16_rows_dot<1, true>(st, 0u, p.sm_xb + 2u * t * p.D, nullptr, p.D / 8)
                             : bf16_rows_dot<1, false>(st, 0u, 0u,
                                                       reinterpret_cast<const uint8_t*>(p.x + (size_t)t * p.D), p.D / 8);
    if (lane == 0) {
      p.logits[(size_t)t * p.N + e] = s.x;
      if (p.score_func != MOE_SCORE_SOFTMAX) {
        // image tokens key on bias_vl (read from global memory)
        const float* bt = (p.bias_vl && p.image_mask && __ldg(p.image_mask + t)) ? p.bias_vl : bias;
        const float sc = score_fast(s.x, p.gate_temp, p.score_func);
        p.sk[(size_t)t * p.N + e] = make_float2(sc, __fadd_rn(sc, bt[e]));
      }
    }
  }
}

// one gate (which 0) or up (which 1) row of the bf16 shared expert against
// every token -> item buffer slot (pair s of the item, which, token); the
// item's completion applies SwiGLU
__device__ __noinline__ void task_shgu_b(const DecodeParams& p, Ctl& C, uint32_t st, int s, int which, float* ib,
                                         uint64_t deadline) {
  const int lane = threadIdx.x & 31;
  require(p, C, RQ_XB, deadline);
#pragma unroll 1
  for (int t = 0; t < p.m; ++t) {
    const float4 r = p.sm_xb ? bf16_rows_dot<1, true>(st, 0u, p.sm_xb + 2u * t * p.D, nullptr, p.D / 8)
                             : bf16_rows_dot<1, false>(st, 0u, 0u,
                                                       reinterpret_cast<const uint8_t*>(p.x + (size_t)t * p.D), p.D / 8);
    if (lane == 0) ib[(size_t)(2 * s + which) * p.m + t] = r.x;
  }
}

// Rows 2 part, 2 part + 1 of the stage's GR rows of W1 (stage offset 0) and of
// W3 (offset GR*rb) in Q2_K against the q8_1(x) units of the item's tokens
// (part: this warp's half of the pair's task): half-warp 0 takes W1,
// half-warp 1 W3.  h of the rows -> item buffer.
__device__ __noinline__ void task_gu_q(const DecodeParams& p, Ctl& C, uint32_t st, int slot, int stg, float* ib,
                                       int part, uint64_t deadline) {
  const int lane = threadIdx.x & 31, half = lane >> 4;
  const uint32_t rb = (p.D / QK) * Q2K_B;
  const int U = p.D / 64;
  const bool shared = slot < 0;
  int pair0 = 0, ntok = p.m;
  const DecodePlan* plan = plan_of(p);
  if (!shared) {
    require(p, C, RQ_PLAN, deadline);
    pair0 = plan->exp_off[slot];
    ntok = plan->exp_off[slot + 1] - pair0;
    if (plan->exp_ptr[slot][0] == 0ull) return;
  }
  require(p, C, RQ_XU, deadline);
  const uint32_t w = st + (uint32_t)half * GR * rb + (uint32_t)(2 * part) * rb;
  const uint32_t xstride = unit_bytes(p.D);
#pragma unroll 1
  for (int tt = 0; tt < ntok; ++tt) {
    const int tok = shared ? tt : plan->pair_tok[pair0 + tt];
    const float4 a = p.sm_x ? q2k_rows4_dot<true>(w, rb, 2, U, p.sm_x + (uint32_t)tok * xstride, nullptr)
                            : q2k_rows4_dot<false>(w, rb, 2, U, 0u,
                                                   reinterpret_cast<const uint8_t*>(p.xu) + (size_t)tok * xstride);
    // lanes 0..15 hold the W1 sums, lanes 16..31 the W3 sums
    const float u0 = __shfl_sync(0xffffffffu, a.x, 16), u1 = __shfl_sync(0xffffffffu, a.y, 16);
    if (lane == 0) {
      float* o = ib + ((size_t)stg * GR + 2 * part) * p.m + tt;
      o[0] = swiglu_f32(a.x, u0, p.swiglu_limit);
      o[p.m] = swiglu_f32(a.y, u1, p.swiglu_limit);
    }
  }
}

// Rows 4 part .. 4 part + 3 of the stage's DG rows of a Q3_K down matrix (stage
// offset st; part: this warp's half of the pair's task) against h units: lane =
// (row, 1/8 of the units).  Routed (slot >= 0): E of each pair of the slot ->
// item buffer row pair*DG (unweighted); shared (slot < 0): the shared
// expert's rows -> item buffer row t*DG.
__device__ __noinline__ void task_dn_q(const DecodeParams& p, Ctl& C, uint32_t st, int slot, float* ib,
                                       int part, uint64_t deadline) {
  const int lane = threadIdx.x & 31, row = 4 * part + (lane >> 3), q = lane & 7;
  const uint32_t rb2 = (p.I / QK) * Q3K_B;
  const int U2 = p.I / 64;
  const uint32_t hstride = unit_bytes(p.I);
  int pb = 0, pe = p.m;
  bool present = true;
  uint32_t hs;
  const uint8_t* hg;
  if (slot >= 0) {
    require(p, C, RQ_PLAN | RQ_HR, deadline);
    const DecodePlan* plan = plan_of(p);
    pb = plan->exp_off[slot];
    pe = plan->exp_off[slot + 1];
    present = plan->exp_ptr[slot][2] != 0ull;
    hs = p.sm_hr;
    hg = reinterpret_cast<const uint8_t*>(p.hu);
  } else {
    require(p, C, RQ_HS, deadline);
    hs = p.sm_hs;
    hg = reinterpret_cast<const uint8_t*>(p.hu) + (size_t)p.shvec0 * hstride;
  }
  const uint32_t rowp = st + (uint32_t)row * rb2;
#pragma unroll 1
  for (int pi = pb; pi < pe; ++pi) {
    const int v = slot >= 0 ? pi : pi - pb;  // vector index within the source
    float acc = 0.f;
    if (present)
      acc = hs ? q3k_row_dot<true>(rowp, U2, hs + (uint32_t)v * hstride, nullptr)
               : q3k_row_dot<false>(rowp, U2, 0u, hg + (size_t)v * hstride);
    if (q == 0) ib[(size_t)pi * DG + row] = acc;
  }
}

// Row `half` (this warp's half of the pair's task) of the stage's SDR rows of
// the bf16 shared down matrix, part `part` of the group, against h (bf16
// [m, I]) -> item buffer
__device__ __noinline__ void task_dn_b(const DecodeParams& p, Ctl& C, uint32_t st, int part, float* ib,
                                       int half, uint64_t deadline) {
  const int lane = threadIdx.x & 31;
  require(p, C, RQ_HS, deadline);
#pragma unroll 1
  for (int t = 0; t < p.m; ++t) {
    const uint32_t row = st + (uint32_t)half * 2u * p.I;
    const float4 s = p.sm_hs ? bf16_rows_dot<1, true>(row, 0u, p.sm_hs + 2u * t * p.I, nullptr, p.I / 8)
                             : bf16_rows_dot<1, false>(row, 0u, 0u, p.shh + (size_t)t * 2 * p.I, p.I / 8);
    if (lane == 0) ib[(size_t)t * DG + part * SDR + half] = s.x;
  }
}

// An L2 policy that makes the lines a load brings in the first to be evicted:
// for data read once per call (expert weights), so that the call's small,
// reused data (instructions, activations, counters) keeps its place in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy (l2_evict_first_policy)
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// ------------------------------------------------------- item completion
__device__ __noinline__ void complete_item(const DecodeParams& p, Ctl& C, Item it, float* ib, uint64_t deadline) {
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
    case I_SHGU_B: {
      // h = SwiGLU(g, u) of the item's rows, per token -> bf16
      const int row0 = it.a * SHP, ns = min(SHP, p.I - row0);
#pragma unroll 1
      for (int q = lane; q < ns * p.m; q += 32) {
        const int s = q / p.m, t = q % p.m;
        const float g = ib[(size_t)(2 * s) * p.m + t], u = ib[(size_t)(2 * s + 1) * p.m + t];
        reinterpret_cast<__nv_bfloat16*>(p.shh)[(size_t)t * p.I + row0 + s] =
            __float2bfloat16_rn(swiglu_f32(g, u, p.swiglu_limit));
      }
      __threadfence();
      if (lane == 0) atomicAdd(&p.ctrl->shgu_done, 1u);
      break;
    }
    case I_GU: {
      // q8_1 of the item's 32 rows of h, per token
      const bool shared = it.a < 0;
      int ntok = p.m, vec0 = p.shvec0;
      bool present = true;
      if (!shared) {
        require(p, C, RQ_PLAN, deadline);
        const DecodePlan* plan = plan_of(p);
        vec0 = plan->exp_off[it.a];
        ntok = plan->exp_off[it.a + 1] - vec0;
        present = plan->exp_ptr[it.a][0] != 0ull;
      }
#pragma unroll 1
      for (int tt = 0; tt < ntok && present; ++tt)
        q8_block_warp(ib[lane * p.m + tt], it.b, nullptr, p.hu + (size_t)(vec0 + tt) * (unit_bytes(p.I) / 4));
      __threadfence();
      if (lane == 0) atomicAdd(shared ? &p.ctrl->shgu_done : &p.ctrl->rtgu_done, 1u);
      break;
    }
    case I_SHDN: {
      // y_shared of the group's rows -> out (the routed down item adds to it)
#pragma unroll 1
      for (int qd = lane; qd < p.m * DG; qd += 32) {
        const int t = qd / DG, r = qd % DG;
        p.out[(size_t)t * p.D + it.a * DG + r] = ib[t * DG + r];
      }
      __threadfence();
      if (lane == 0) atomicAdd(&p.ctrl->shdn_done, 1u);
      break;
    }
    case I_DN: {
      // y = sum over the token's pairs in ascending expert id of G E, then
      // + y_shared (every shared down item finished long before; the wait is
      // bounded all the same)
      require(p, C, RQ_PLAN | RQ_SHDN, deadline);
      const DecodePlan* plan = plan_of(p);
#pragma unroll 1
      for (int qd = lane; qd < p.m * DG; qd += 32) {
        const int t = qd / DG, r = qd % DG;
        float acc = 0.f;
#pragma unroll 1
        for (int i = 0; i < p.k; ++i) {
          const int pr = plan->tok_pairs[t][i];
          acc = fmaf(plan->pair_w[pr], ib[pr * DG + r], acc);
        }
        float* o = p.out + (size_t)t * p.D + it.a * DG + r;
        *o = acc + __ldcg(o);
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
  // Programmatic dependent launch: the next launch on the stream may start
  // its blocks as this grid's blocks exit, and this grid touches no global
  // memory before the previous launch has completed (the wait below).  Both
  // are no-ops for a launch without the attribute.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(C.full[i]), 1);
      mbar_init(bar(C.empty[i]), 1);
      C.hdr[i].seq = 0xFFFFFFFFu;
    }
    for (int i = 0; i < NIS; ++i) mbar_init(bar(C.item_done[i]), 1);
    mbar_init(bar(C.pbar), 1);
    for (int i = 0; i < N_CB; ++i) {
      mbar_init(bar(C.cbar[i]), 1);
      C.cstate[i] = 0u;
    }
    C.next = 0u;
    C.rdy = 0u;
    C.xq = 0u;
    C.sink = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
  const Sizes z = sizes_of(p);
  const int groups = p.D / DG;

  if (warp == W_PLAN) {
    // ----------------------------------------------------------- planner
    // Wait for every router row of the call, then build this block's plan.
    // On a timeout the plan is left empty (no routed expert work) so the
    // block still finishes; the status word already says why.
    // The selection and plan code runs once per call, so its instructions are
    // never cached when the routing is ready, and under the weight stream an
    // instruction-cache miss costs about a microsecond: run it once on stale
    // inputs while the router rows are computed.
    build_plan(p, C, deadline, true);
    bool ok = true;
    if (lane == 0) ok = wait_count(&p.ctrl->router_done, (unsigned)z.n_router, deadline, &p.ctrl->status);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      build_plan(p, C, deadline, false);
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
    // Lane 0 takes the tickets and picks the next item; the lanes then issue
    // the item's stages in parallel (lane l: stages l, l + 32, ... of the
    // item), each waiting only for its own ring slot, so that the ticket and
    // item logic is paid once per item rather than once per stage.
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
    }
    // every weight byte is read once per call: its lines go first when L2 needs room
    const uint64_t evict_first = l2_evict_first_policy();
    uint32_t n = 0;  // stages issued
    uint32_t j = 0;  // items started
    bool ok = true;
    const int rb = (p.D / QK) * Q2K_B, rb2 = (p.I / QK) * Q3K_B;
    const DecodePlan* splan = reinterpret_cast<const DecodePlan*>(smem_base() + p.sm_plan);
    // ticket state, used by lane 0 only
    int n_exp = -1;
    bool local_done = false;
    unsigned* const ctr[N_STREAMS] = {&p.ctrl->ticket, &p.ctrl->ticket_sh, &p.ctrl->ticket_gu, &p.ctrl->ticket_dn};
    bool exhausted[N_STREAMS] = {false, false, false, false};
    // the stream to take the next ticket from: -1 nothing left, N_STREAMS
    // wait for the plan first
    // Before the plan exists, shared down items are taken only once the
    // shared h is complete: their tasks would otherwise hold ring stages
    // while they wait, and the routed gate/up items could not get in.
    bool sh_ready = false;
    auto shared_ready = [&]() -> bool {
      if (!sh_ready) sh_ready = ld_acquire(&p.ctrl->shgu_done) >= (unsigned)z.n_shgu;
      return sh_ready;
    };
    auto choose = [&]() -> int {
      if (!exhausted[S_MAIN]) return S_MAIN;
      if (n_exp < 0 && mbar_try_wait(bar(C.pbar), 0u)) n_exp = splan->n_exp;
      if (n_exp >= 0 && !exhausted[S_GU]) return S_GU;
      if (!exhausted[S_SHDN] && (n_exp >= 0 || shared_ready())) return S_SHDN;
      if (n_exp < 0) return N_STREAMS;
      return exhausted[S_DN] ? -1 : S_DN;
    };
    // one ticket is taken ahead, so that its atomic is in flight while
    // the current item streams
    int ps = -1;
    unsigned pt = 0;
    for (;;) {
      // --- lane 0: the next item (kind -1: none left, -3: stop on an error)
      Item it{-1, 0, 0, 0, 0};
      int ns = 0;
      if (lane == 0) {
        for (;;) {
          if (ps < 0) {
            const int sel = choose();
            if (sel < 0) break;
            if (sel == N_STREAMS) {
              // wait for the plan, or for the shared h while shared down items are left
              uint32_t spins = 0;
              for (;;) {
                if (mbar_try_wait(bar(C.pbar), 0u)) {
                  n_exp = splan->n_exp;
                  break;
                }
                if (!exhausted[S_SHDN] && shared_ready()) break;
                __nanosleep(200);
                if ((++spins & 15u) == 0 && globaltimer_ns() > deadline) {
                  atomicOr(&p.ctrl->status, (unsigned)MOE_STATUS_TIMEOUT);
                  it.kind = -3;
                  break;
                }
              }
              if (it.kind == -3) break;
              continue;
            }
            ps = sel;
            pt = atomicAdd(ctr[sel], 1u);
          }
          Item t = decode_ticket(ps, pt, z, groups, n_exp);
          if (t.kind == -2) {
            exhausted[ps] = true;
            ps = -1;
            continue;
          }
          // the block-local item goes in before the block's first item past the router rows
          if (!local_done && t.kind != I_Q8 && t.kind != I_ROUTER) {
            local_done = true;
            t = Item{I_LOCAL, 0, 0, 0, 0};  // the ticket stays taken for the next round
          } else {
            const int sel = choose();
            ps = (sel >= 0 && sel < N_STREAMS) ? sel : -1;
            if (ps >= 0) pt = atomicAdd(ctr[ps], 1u);
          }
          it = t;
          break;
        }
        if (it.kind >= 0) {
          switch (it.kind) {
            case I_Q8: ns = 1; break;
            case I_ROUTER: ns = 1; break;
            case I_SHGU_B: ns = 2 * min(SHP, p.I - it.a * SHP); break;
            case I_GU: ns = GT / GR; break;
            case I_SHDN: ns = z.dn_sh_parts; break;
            case I_LOCAL: ns = NPAIR; break;
            default: ns = n_exp; break;
          }
          const uint32_t islot = j % NIS;
          if (j >= (uint32_t)NIS &&
              !mbar_wait_bounded(bar(C.item_done[islot]), (j / NIS - 1) & 1u, deadline, &p.ctrl->status)) {
            it.kind = -3;
          } else {
            it.remaining = (unsigned)ns;
            C.item[islot] = it;
          }
        }
      }
      it.kind = __shfl_sync(0xffffffffu, it.kind, 0);
      if (it.kind < 0) {
        ok = it.kind != -3;
        break;
      }
      it.a = __shfl_sync(0xffffffffu, it.a, 0);
      it.b = __shfl_sync(0xffffffffu, it.b, 0);
      ns = __shfl_sync(0xffffffffu, ns, 0);
      __syncwarp();  // the item state (lane 0) before any of its stages
      // --- the lanes: the item's stages, in rounds of at most NST (one per
      // ring slot).  A round starts once the previous one is issued, so the
      // empty barrier a lane waits on is at most one phase behind the use
      // it waits for (its parity alone then identifies that use).
      const uint32_t islot = j % NIS;
      bool lane_ok = true;
      for (int base = 0; base < ns; base += NST) {
        __syncwarp();
        const int s = base + lane;
        if (lane >= NST || s >= ns || !lane_ok) continue;
        const uint32_t sn = n + (uint32_t)s, slot = sn % NST, use = sn / NST;
        if (use > 0 && !mbar_wait_bounded(bar(C.empty[slot]), (use - 1) & 1u, deadline, &p.ctrl->status)) {
          lane_ok = false;
          continue;
        }
        Hdr h{K_STOP, (int)islot, 0, 0, sn};
        const uint8_t *a = nullptr, *b = nullptr;
        uint32_t bytes = 0, boff = 0;
        switch (it.kind) {
          case I_Q8:
            h.kind = K_Q8; h.a = it.a;
            break;
          case I_LOCAL:
            h.kind = K_LOCAL; h.a = s;
            break;
          case I_ROUTER: {
            const int r0 = it.a * RR;
            h.kind = K_ROUTER; h.a = r0;
            a = reinterpret_cast<const uint8_t*>(p.router_w) + (size_t)r0 * 2 * p.D;
            bytes = (uint32_t)(min(RR, p.N - r0) * 2 * p.D);
            break;
          }
          case I_SHGU_B: {
            const int row = it.a * SHP + s / 2;
            h.kind = K_SHGU_B; h.a = s / 2; h.b = s & 1;
            a = ((s & 1) ? p.sh3 : p.sh1) + (size_t)row * 2 * p.D;
            bytes = (uint32_t)(2 * p.D);
            break;
          }
          case I_GU: {
            const int r0 = it.b * GT + s * GR;
            h.kind = K_GU_Q; h.a = it.a; h.b = s;
            const uint8_t *w1, *w3;
            if (it.a < 0) {
              w1 = p.sh1; w3 = p.sh3;
            } else {
              w1 = reinterpret_cast<const uint8_t*>(splan->exp_ptr[it.a][0]);
              w3 = reinterpret_cast<const uint8_t*>(splan->exp_ptr[it.a][1]);
            }
            if (w1 && w3) {
              a = w1 + (size_t)r0 * rb;
              b = w3 + (size_t)r0 * rb;
              bytes = (uint32_t)(GR * rb);
              boff = bytes;
            }
            break;
          }
          case I_SHDN: {  // the shared expert's rows of the group
            const int d0 = it.a * DG;
            if (z.shq) {
              h.kind = K_DN_SHQ;
              a = p.sh2 + (size_t)d0 * rb2;
              bytes = (uint32_t)(DG * rb2);
            } else {
              h.kind = K_DN_SHB; h.a = s;
              a = p.sh2 + (size_t)(d0 + s * SDR) * 2 * p.I;
              bytes = (uint32_t)(SDR * 2 * p.I);
            }
            break;
          }
          default: {  // I_DN: expert s of the plan (ascending id), the group's rows
            const int d0 = it.a * DG;
            h.kind = K_DN_RT; h.a = s;
            const unsigned long long w2 = splan->exp_ptr[s][2];
            if (w2) {
              a = reinterpret_cast<const uint8_t*>(w2) + (size_t)d0 * rb2;
              bytes = (uint32_t)(DG * rb2);
            }
            break;
          }
        }
        C.hdr[slot] = h;
        uint8_t* dst = smem_base() + (size_t)slot * SB;
        mbar_arrive_expect_tx(bar(C.full[slot]), a ? (b ? 2u * bytes : bytes) : 0u);
        if (a) bulk_g2s_hint(dst, a, bytes, bar(C.full[slot]), evict_first);
        if (a && b) bulk_g2s_hint(dst + boff, b, bytes, bar(C.full[slot]), evict_first);
      }
      ok = __all_sync(0xffffffffu, lane_ok);
      n += (uint32_t)ns;
      if (!ok) break;
      ++j;
    }
    if (lane == 0) {
      if (ok) {
        // one stop per consumer pair
        for (int s = 0; s < NPAIR; ++s) {
          const uint32_t slot = n % NST, use = n / NST;
          if (use > 0 && !(ok = mbar_wait_bounded(bar(C.empty[slot]), (use - 1) & 1u, deadline, &p.ctrl->status)))
            break;
          C.hdr[slot] = Hdr{K_STOP, 0, 0, 0, n};
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
    // Warps 2i and 2i + 1 form pair i and work on one stage together: the
    // leader takes the stage and waits for it, both run their half of the
    // task, and after the pair's named barrier the leader releases the stage
    // and counts the task (completing the item when it was the last).  Both
    // warps leave the loop at the same stage, so the pair's barrier never
    // waits for a warp that is gone.
    const int pair = warp >> 1, pw = warp & 1, pbar_id = 1 + pair;
    for (;;) {
      if (pw == 0) {
        unsigned n = 0;
        if (lane == 0) n = atomicAdd(&C.next, 1u);
        n = __shfl_sync(0xffffffffu, n, 0);
        const uint32_t slot = n % NST;
        // A consumer can be more than one ring turn ahead of the stage it took
        // (copies land out of order), where the parity of the full barrier
        // alone would also match the stage's previous use: wait first until the
        // producer has written this stage's header, then for the barrier.
        bool got = true;
        if (lane == 0) {
          const volatile unsigned* seq = &C.hdr[slot].seq;
          uint32_t spins = 0;
          while (*seq != n) {
            __nanosleep(32);
            if ((++spins & 15u) == 0 && globaltimer_ns() > deadline) {
              atomicOr(&p.ctrl->status, (unsigned)MOE_STATUS_TIMEOUT);
              got = false;
              break;
            }
          }
          if (got) got = mbar_wait_bounded(bar(C.full[slot]), (n / NST) & 1u, deadline, &p.ctrl->status);
          C.pair_n[pair] = n;
          C.pair_ok[pair] = got ? 1u : 0u;
        }
        __syncwarp();
      }
      named_bar_sync(pbar_id, 64);
      const unsigned n = *reinterpret_cast<volatile unsigned*>(&C.pair_n[pair]);
      if (!*reinterpret_cast<volatile unsigned*>(&C.pair_ok[pair])) break;
      const uint32_t slot = n % NST;
      const Hdr h = C.hdr[slot];
      if (h.kind == K_STOP) break;
      const uint32_t st = slot * (uint32_t)SB;
      float* ib = item_buf(p, h.slot);
      switch (h.kind) {
        case K_Q8: if (pw == 0) task_q8(p, h.a); break;
        case K_ROUTER: if (pw == 0) task_router(p, C, st, h.a, deadline); break;
        case K_SHGU_B: if (pw == 0) task_shgu_b(p, C, st, h.a, h.b, ib, deadline); break;
        case K_LOCAL: task_local(p, C, 2 * h.a + pw, deadline); break;
        case K_GU_Q: task_gu_q(p, C, st, h.a, h.b, ib, pw, deadline); break;
        case K_DN_SHB: task_dn_b(p, C, st, h.a, ib, pw, deadline); break;
        case K_DN_SHQ:
        case K_DN_RT: task_dn_q(p, C, st, h.kind == K_DN_RT ? h.a : -1, ib, pw, deadline); break;
        default: break;
      }
      // both halves are done with the stage: release it, then count the task
      __syncwarp();
      __threadfence_block();
      named_bar_sync(pbar_id, 64);
      if (pw == 0) {
        unsigned left = 0;
        if (lane == 0) {
          mbar_arrive(bar(C.empty[slot]));
          left = atomicSub(&C.item[h.slot].remaining, 1u);
        }
        left = __shfl_sync(0xffffffffu, left, 0);
        if (left == 1u) {
          __threadfence_block();
          const Item it = C.item[h.slot];
          complete_item(p, C, it, ib, deadline);
          __syncwarp();
          __threadfence_block();
          if (lane == 0) mbar_arrive(bar(C.item_done[h.slot]));
        }
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
      p.ctrl->ticket_sh = 0u;
      p.ctrl->ticket_gu = 0u;
      p.ctrl->ticket_dn = 0u;
      p.ctrl->q8_done = 0u;
      p.ctrl->router_done = 0u;
      p.ctrl->shgu_done = 0u;
      p.ctrl->rtgu_done = 0u;
      p.ctrl->shdn_done = 0u;
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
  const size_t gu = (size_t)GT * p.m * 4, dn = (P + p.m) * DG * 4, sg = (size_t)2 * SHP * p.m * 4;
  p.item_bytes = (uint32_t)a16(std::max(std::max(gu, dn), sg));
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
  return 2 * GR * rb <= SB && DG * rb2 <= SB && RR * 2 * D <= SB && 2 * D <= SB && SDR * 2 * I <= SB &&
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
  // programmatic stream serialisation: the block set-up of this call
  // overlaps the tail of the previous launch on the stream
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)num_sms);
  lc.blockDim = dim3(NTH);
  lc.dynamicSmemBytes = p.smem_bytes;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, k_decode_layer, p) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
