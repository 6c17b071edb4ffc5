// Decode path (m <= 8): the picked experts and the shared expert.
//
// Two persistent kernels, one CTA per SM, each a producer warp plus ten
// consumer warps around a ring of shared-memory stages:
//  - the producer takes work items by atomic ticket and streams each item's
//    raw weight rows into the ring with 1-D bulk copies (cp.async.bulk,
//    completing on an mbarrier), running ahead of the consumers;
//  - the consumers dot the rows with the activations held in the unit layout.
// gate/up: routed items are (distinct expert, 32 rows of W1 and W3); the
//   SwiGLU (DeepSeek V4.1 atlas "Mixture of experts": g' = min(g, L),
//   u' = clip(u, -L, L), h = g' sigmoid(g') u') and q8_1(h) are fused at the
//   end of the item (metrale moe_v41.rs names the fused swiglu_q8 step);
//   shared bf16 items write h rounded to bf16.
// down: items are 8 output rows; their stages are the W2 rows of every
//   distinct expert in ascending id, then the shared expert's, and the
//   consumers keep y += G_i E_i in that order, add the shared expert last and
//   write the rows out (the atlas's y_routed + y_shared; the metrale docs:
//   the shared expert is added after the routed experts).
#include "internal.h"

namespace moe {
namespace {

constexpr int NCW = 10;            // consumer warps
constexpr int NCT = NCW * 32;      // consumer threads
constexpr int NTH = NCT + 32;      // + producer warp
constexpr int STAGE = 40960;       // bytes per ring stage
constexpr int NST = 4;             // ring stages
constexpr int GU_ROWS = 8;         // rows of W1 (and of W3) per gate/up stage
constexpr int GU_TILE = 32;        // rows per routed gate/up item = one q8_1 block of h
constexpr int SH_ITEM_STAGES = 4;  // stages per shared bf16 gate/up item
constexpr int DN_ROWS = 8;         // output rows per down item
constexpr int PBUF = 16 * 120;     // partial sums: rows x units (units <= 7680/64)

struct Hdr {
  int item, stage, nstage, arg;
};

struct Smem {
  Hdr hdr[NST];
  Hdr cur;
  unsigned long long full[NST];
  unsigned long long empty[NST];
  float pbuf[PBUF];
  float red[NCW][16];
  float gacc[GU_TILE][DECODE_MAX_M];
  float uacc[GU_TILE][DECODE_MAX_M];
  float acc[DN_ROWS][DECODE_MAX_M];
  float stash[16][DECODE_MAX_M];
};

constexpr size_t RING_BYTES = (size_t)NST * STAGE + 16;
constexpr size_t SMEM_BYTES = RING_BYTES + sizeof(Smem);

__device__ __forceinline__ uint8_t* ring_base() {
  extern __shared__ __align__(128) uint8_t dyn[];
  return dyn;
}
__device__ __forceinline__ Smem& sm() {
  extern __shared__ __align__(128) uint8_t dyn[];
  return *reinterpret_cast<Smem*>(dyn + RING_BYTES);
}

// ------------------------------------------------------------- item plans
struct GUPlan {
  int n_sh, n_items, rs;  // rs: rows per shared bf16 stage
};

__device__ __forceinline__ GUPlan gu_plan(const DecodeParams& p, int n_exp) {
  GUPlan g;
  if (p.shared_kind == MOE_SHARED_BF16) {
    int rs = STAGE / (4 * p.D);
    rs = rs > GU_ROWS ? GU_ROWS : rs;
    g.rs = rs;
    const int sh_stages = (p.I + rs - 1) / rs;
    g.n_sh = (sh_stages + SH_ITEM_STAGES - 1) / SH_ITEM_STAGES;
  } else {
    g.rs = GU_ROWS;
    g.n_sh = p.I / GU_TILE;
  }
  g.n_items = g.n_sh + n_exp * (p.I / GU_TILE);
  return g;
}

struct DNPlan {
  int rs2, sh_stages;  // shared bf16 rows per stage, shared stages per item
};

__device__ __forceinline__ DNPlan dn_plan(const DecodeParams& p) {
  DNPlan d;
  if (p.shared_kind == MOE_SHARED_BF16) {
    int rs = STAGE / (2 * p.I);
    d.rs2 = rs > DN_ROWS ? DN_ROWS : rs;
    d.sh_stages = (DN_ROWS + d.rs2 - 1) / d.rs2;
  } else {
    d.rs2 = DN_ROWS;
    d.sh_stages = 1;
  }
  return d;
}

// ------------------------------------------------------------- producer
// Waits for ring slot n to be free, publishes the header, and returns the
// slot's stage buffer, or nullptr after a timeout.
__device__ __forceinline__ uint8_t* producer_acquire(uint32_t n, const Hdr& h, uint64_t deadline, unsigned* status) {
  Smem& S = sm();
  const uint32_t slot = n % NST, use = n / NST;
  if (use > 0 && !mbar_wait_bounded(reinterpret_cast<uint64_t*>(&S.empty[slot]), (use - 1) & 1u, deadline, status))
    return nullptr;
  S.hdr[slot] = h;
  return ring_base() + (size_t)slot * STAGE;
}

__device__ __forceinline__ uint64_t* full_bar(uint32_t n) { return reinterpret_cast<uint64_t*>(&sm().full[n % NST]); }

// After a timeout: wait (bounded) until the copies already issued have landed
// so none targets shared memory after the block exits.
__device__ void producer_drain(uint32_t issued, uint64_t deadline2, unsigned* status) {
  const uint32_t first = issued > (uint32_t)NST ? issued - NST : 0u;
  for (uint32_t n = first; n < issued; ++n)
    mbar_wait_bounded(full_bar(n), (n / NST) & 1u, deadline2, status);
}

// ------------------------------------------------------------- consumers
// Thread 0 waits for stage n and shares its header; returns false on stop or timeout.
__device__ __forceinline__ bool consumer_next(uint32_t n, uint64_t deadline, unsigned* status, int tid, Hdr& out) {
  Smem& S = sm();
  if (tid == 0) {
    const uint32_t slot = n % NST;
    if (mbar_wait_bounded(full_bar(n), (n / NST) & 1u, deadline, status)) S.cur = S.hdr[slot];
    else S.cur.item = -2;
  }
  named_bar_sync(1, NCT);
  out = S.cur;
  return out.item >= 0;
}

__device__ __forceinline__ void consumer_release(uint32_t n, int tid) {
  named_bar_sync(1, NCT);
  if (tid == 0) mbar_arrive(reinterpret_cast<uint64_t*>(&sm().empty[n % NST]));
}

// Sum over units of the partial buffer for `rows` rows (16 threads per row,
// fixed order).  Calls f(row, value) on the row's first thread.
template <class F>
__device__ __forceinline__ void reduce_rows(int rows, int U, int tid, F f) {
  const float* P = sm().pbuf;
  if (tid < 256) {
    const int row = tid >> 4, g = tid & 15;
    float s = 0.f;
    if (row < rows)
      for (int u = g; u < U; u += 16) s += P[row * U + u];
#pragma unroll
    for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (g == 0 && row < rows) f(row, s);
  }
}

// Block reduction of nv per-thread values (nv <= 16) over the consumer
// threads in fixed order; the sums land in S.stash[v][col].
__device__ __forceinline__ void reduce_block_to_stash(const float* v, int nv, int col, int tid) {
  Smem& S = sm();
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = 0; i < nv; ++i) {
    float a = v[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) S.red[warp][i] = a;
  }
  named_bar_sync(1, NCT);
  if (tid < nv) {
    float a = 0.f;
    for (int w = 0; w < NCW; ++w) a += S.red[w][tid];
    S.stash[tid][col] = a;
  }
  named_bar_sync(1, NCT);
}

__device__ __forceinline__ void dot8_bf16(float& acc, const uint4& w, const uint4& x) {
  acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc); acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc); acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc); acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc); acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
}

// ================================================================ gate/up
__global__ void __launch_bounds__(NTH, 1) k_gateup_decode(DecodeParams p) {
  Smem& S = sm();
  const int tid = threadIdx.x;
  const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(reinterpret_cast<uint64_t*>(&S.full[i]), 1);
      mbar_init(reinterpret_cast<uint64_t*>(&S.empty[i]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const DecodePlan* plan = p.plan;
  const int n_exp = __ldg(&plan->n_exp);
  const GUPlan G = gu_plan(p, n_exp);
  const int rb = (p.D / QK) * Q2K_B;          // bytes per Q2_K row
  const int tiles = p.I / GU_TILE;

  if (tid >= NCT) {
    // ----------------------------------------------------------- producer
    if (tid != NCT) return;
    uint32_t n = 0;
    bool ok = true;
    for (;;) {
      const int item = (int)atomicAdd(&p.ctrl->ticket_gu, 1u);
      if (item >= G.n_items) {
        Hdr h{-1, 0, 0, 0};
        if (producer_acquire(n, h, deadline, &p.ctrl->status)) {
          mbar_arrive(full_bar(n));
          ++n;
        } else {
          ok = false;
        }
        break;
      }
      int nst;
      if (item < G.n_sh && p.shared_kind == MOE_SHARED_BF16) {
        const int first = item * SH_ITEM_STAGES * G.rs;
        const int rows = min(p.I - first, SH_ITEM_STAGES * G.rs);
        nst = (rows + G.rs - 1) / G.rs;
      } else {
        nst = GU_TILE / GU_ROWS;
      }
      for (int s = 0; s < nst && ok; ++s) {
        Hdr h{item, s, nst, 0};
        uint8_t* dst = producer_acquire(n, h, deadline, &p.ctrl->status);
        if (!dst) { ok = false; break; }
        const uint8_t *a = nullptr, *b = nullptr;
        uint32_t bytes = 0, off_b = 0;
        if (item < G.n_sh && p.shared_kind == MOE_SHARED_BF16) {
          const int r0 = (item * SH_ITEM_STAGES + s) * G.rs;
          const int rows = min(G.rs, p.I - r0);
          bytes = (uint32_t)rows * 2u * (uint32_t)p.D;
          a = p.sh1 + (size_t)r0 * 2 * p.D;
          b = p.sh3 + (size_t)r0 * 2 * p.D;
          off_b = (uint32_t)G.rs * 2u * (uint32_t)p.D;
        } else {
          const uint8_t *w1, *w3;
          int tile;
          if (item < G.n_sh) {
            w1 = p.sh1; w3 = p.sh3; tile = item;
          } else {
            const int slot = (item - G.n_sh) / tiles;
            tile = (item - G.n_sh) % tiles;
            w1 = reinterpret_cast<const uint8_t*>(plan->exp_ptr[slot][0]);
            w3 = reinterpret_cast<const uint8_t*>(plan->exp_ptr[slot][1]);
          }
          if (w1 && w3) {
            const int r0 = tile * GU_TILE + s * GU_ROWS;
            bytes = (uint32_t)GU_ROWS * (uint32_t)rb;
            a = w1 + (size_t)r0 * rb;
            b = w3 + (size_t)r0 * rb;
            off_b = bytes;
          }
        }
        mbar_arrive_expect_tx(full_bar(n), a ? 2u * bytes : 0u);
        if (a) {
          bulk_g2s(dst, a, bytes, full_bar(n));
          bulk_g2s(dst + off_b, b, bytes, full_bar(n));
        }
        ++n;
      }
      if (!ok) break;
    }
    if (!ok) producer_drain(n, globaltimer_ns() + p.timeout_ns, &p.ctrl->status);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int U = p.D / 64;  // units per Q2_K row
  uint32_t n = 0;
  Hdr h;
  while (consumer_next(n, deadline, &p.ctrl->status, tid, h)) {
    const uint8_t* stage = ring_base() + (size_t)(n % NST) * STAGE;
    const int item = h.item;
    if (item < G.n_sh && p.shared_kind == MOE_SHARED_BF16) {
      // ---- shared expert, bf16: rows r0.. of W1 (stage offset 0) and W3
      const int r0 = (item * SH_ITEM_STAGES + h.stage) * G.rs;
      const int rows = min(G.rs, p.I - r0);
      const int chunks = p.D / 8;
      const uint4* w = reinterpret_cast<const uint4*>(stage);
      const int wb = G.rs * chunks;  // W3 offset in uint4
      for (int t = 0; t < p.m; ++t) {
        float acc[2 * GU_ROWS];
#pragma unroll
        for (int r = 0; r < 2 * GU_ROWS; ++r) acc[r] = 0.f;
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
        for (int c = tid; c < chunks; c += NCT) {
          const uint4 xv = __ldg(xr + c);
#pragma unroll
          for (int r = 0; r < GU_ROWS; ++r) {
            if (r < rows) {
              dot8_bf16(acc[r], w[r * chunks + c], xv);
              dot8_bf16(acc[GU_ROWS + r], w[wb + r * chunks + c], xv);
            }
          }
        }
        // reduce the 2*rows values; g rows land in stash[0..rows), u rows in stash[8..8+rows)
        float v[2 * GU_ROWS];
#pragma unroll
        for (int r = 0; r < 2 * GU_ROWS; ++r) v[r] = acc[r];
        reduce_block_to_stash(v, 2 * GU_ROWS, t, tid);
      }
      if (tid < rows * p.m) {
        const int r = tid / p.m, t = tid % p.m;
        const float hv = swiglu_f32(S.stash[r][t], S.stash[GU_ROWS + r][t], p.swiglu_limit);
        reinterpret_cast<__nv_bfloat16*>(p.shh)[(size_t)t * p.I + r0 + r] = __float2bfloat16_rn(hv);
      }
    } else {
      // ---- Q2_K tile stage: rows 0..7 = W1 rows, 8..15 = W3 rows
      int slot = -1, tile, ntok, pair0 = 0;
      bool present = true;
      if (item < G.n_sh) {
        tile = item;
        ntok = p.m;
      } else {
        slot = (item - G.n_sh) / tiles;
        tile = (item - G.n_sh) % tiles;
        pair0 = __ldg(&plan->exp_off[slot]);
        ntok = __ldg(&plan->exp_off[slot + 1]) - pair0;
        present = __ldg(&plan->exp_ptr[slot][0]) != 0ull;
      }
      if (present) {
        const size_t xstride = unit_bytes(p.D) / 16;  // int4 per token
        for (int tt = 0; tt < ntok; ++tt) {
          const int tok = slot < 0 ? tt : __ldg(&plan->pair_tok[pair0 + tt]);
          const int4* xb = reinterpret_cast<const int4*>(p.xu) + (size_t)tok * xstride;
          XUnit xr;
          int cur = -1;
          for (int q = tid; q < 2 * GU_ROWS * U; q += NCT) {
            const int row = q / U, unit = q - row * U;
            if (unit != cur) {
              load_xunit(xr, xb + unit * 6);
              cur = unit;
            }
            S.pbuf[row * U + unit] = q2k_unit_dot(stage + (size_t)row * rb + (unit >> 2) * Q2K_B, unit & 3, xr);
          }
          named_bar_sync(1, NCT);
          reduce_rows(2 * GU_ROWS, U, tid, [&](int row, float v) {
            const int r = h.stage * GU_ROWS + (row & (GU_ROWS - 1));
            if (row < GU_ROWS) S.gacc[r][tt] = v;
            else S.uacc[r][tt] = v;
          });
          named_bar_sync(1, NCT);
        }
        if (h.stage == h.nstage - 1) {
          // SwiGLU over the 32 rows and q8_1 of h: one warp per token
          const int warp = tid >> 5, lane = tid & 31;
          for (int tt = warp; tt < ntok; tt += NCW) {
            const float hv = swiglu_f32(S.gacc[lane][tt], S.uacc[lane][tt], p.swiglu_limit);
            int* units;
            if (slot < 0) {
              units = reinterpret_cast<int*>(p.shh) + (size_t)tt * (unit_bytes(p.I) / 4);
            } else {
              units = p.hu + (size_t)(pair0 + tt) * (unit_bytes(p.I) / 4);
            }
            q8_block_warp(hv, tile, nullptr, units);
          }
        }
      }
    }
    consumer_release(n, tid);
    ++n;
  }
}

// =================================================================== down
__global__ void __launch_bounds__(NTH, 1) k_down_decode(DecodeParams p) {
  Smem& S = sm();
  const int tid = threadIdx.x;
  const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(reinterpret_cast<uint64_t*>(&S.full[i]), 1);
      mbar_init(reinterpret_cast<uint64_t*>(&S.empty[i]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const DecodePlan* plan = p.plan;
  const int n_exp = __ldg(&plan->n_exp);
  const DNPlan Dp = dn_plan(p);
  const int rb2 = (p.I / QK) * Q3K_B;  // bytes per Q3_K row
  const int n_items = p.D / DN_ROWS;
  const int nst = n_exp + Dp.sh_stages;

  if (tid >= NCT) {
    if (tid != NCT) return;
    uint32_t n = 0;
    bool ok = true;
    for (;;) {
      const int item = (int)atomicAdd(&p.ctrl->ticket_dn, 1u);
      if (item >= n_items) {
        Hdr h{-1, 0, 0, 0};
        if (producer_acquire(n, h, deadline, &p.ctrl->status)) {
          mbar_arrive(full_bar(n));
          ++n;
        } else {
          ok = false;
        }
        break;
      }
      const int d0 = item * DN_ROWS;
      for (int s = 0; s < nst && ok; ++s) {
        Hdr h{item, s, nst, 0};
        uint8_t* dst = producer_acquire(n, h, deadline, &p.ctrl->status);
        if (!dst) { ok = false; break; }
        const uint8_t* a = nullptr;
        uint32_t bytes = 0;
        if (s < n_exp) {
          const uint8_t* w2 = reinterpret_cast<const uint8_t*>(plan->exp_ptr[s][2]);
          if (w2) {
            a = w2 + (size_t)d0 * rb2;
            bytes = (uint32_t)DN_ROWS * (uint32_t)rb2;
          }
        } else if (p.shared_kind == MOE_SHARED_BF16) {
          const int r0 = d0 + (s - n_exp) * Dp.rs2;
          const int rows = min(Dp.rs2, d0 + DN_ROWS - r0);
          a = p.sh2 + (size_t)r0 * 2 * p.I;
          bytes = (uint32_t)rows * 2u * (uint32_t)p.I;
        } else {
          a = p.sh2 + (size_t)d0 * rb2;
          bytes = (uint32_t)DN_ROWS * (uint32_t)rb2;
        }
        mbar_arrive_expect_tx(full_bar(n), a ? bytes : 0u);
        if (a) bulk_g2s(dst, a, bytes, full_bar(n));
        ++n;
      }
      if (!ok) break;
    }
    if (!ok) producer_drain(n, globaltimer_ns() + p.timeout_ns, &p.ctrl->status);
    return;
  }

  const int U2 = p.I / 64;
  const size_t hstride = unit_bytes(p.I) / 16;  // int4 per h vector
  uint32_t n = 0;
  Hdr h;
  while (consumer_next(n, deadline, &p.ctrl->status, tid, h)) {
    const uint8_t* stage = ring_base() + (size_t)(n % NST) * STAGE;
    const int d0 = h.item * DN_ROWS;
    if (h.stage == 0) {
      if (tid < DN_ROWS * DECODE_MAX_M) S.acc[tid / DECODE_MAX_M][tid % DECODE_MAX_M] = 0.f;
      named_bar_sync(1, NCT);
    }
    const bool routed = h.stage < n_exp;
    if (routed || p.shared_kind == MOE_SHARED_KQUANT) {
      int pb, pe;
      bool present = true;
      if (routed) {
        pb = __ldg(&plan->exp_off[h.stage]);
        pe = __ldg(&plan->exp_off[h.stage + 1]);
        present = __ldg(&plan->exp_ptr[h.stage][2]) != 0ull;
      } else {
        pb = 0;
        pe = p.m;
      }
      for (int pi = pb; pi < pe && present; ++pi) {
        const int tok = routed ? __ldg(&plan->pair_tok[pi]) : pi;
        const float gw = routed ? __ldg(&plan->pair_w[pi]) : 1.0f;
        const int4* hb = routed ? reinterpret_cast<const int4*>(p.hu) + (size_t)pi * hstride
                                : reinterpret_cast<const int4*>(p.shh) + (size_t)pi * hstride;
        XUnit hr;
        int cur = -1;
        for (int q = tid; q < DN_ROWS * U2; q += NCT) {
          const int row = q / U2, unit = q - row * U2;
          if (unit != cur) {
            load_xunit(hr, hb + unit * 6);
            cur = unit;
          }
          S.pbuf[row * U2 + unit] = q3k_unit_dot(stage + (size_t)row * rb2 + (unit >> 2) * Q3K_B, unit & 3, hr);
        }
        named_bar_sync(1, NCT);
        reduce_rows(DN_ROWS, U2, tid, [&](int row, float v) { S.acc[row][tok] = fmaf(gw, v, S.acc[row][tok]); });
        named_bar_sync(1, NCT);
      }
    } else {
      // shared bf16 down: rows r0.. of W2 against h (bf16 [m, I])
      const int r0 = d0 + (h.stage - n_exp) * Dp.rs2;
      const int rows = min(Dp.rs2, d0 + DN_ROWS - r0);
      const int chunks = p.I / 8;
      const uint4* w = reinterpret_cast<const uint4*>(stage);
      for (int t = 0; t < p.m; ++t) {
        float acc[DN_ROWS];
#pragma unroll
        for (int r = 0; r < DN_ROWS; ++r) acc[r] = 0.f;
        const uint4* hr = reinterpret_cast<const uint4*>(p.shh) + (size_t)t * chunks;
        for (int c = tid; c < chunks; c += NCT) {
          const uint4 hv = __ldg(hr + c);
#pragma unroll
          for (int r = 0; r < DN_ROWS; ++r)
            if (r < rows) dot8_bf16(acc[r], w[r * chunks + c], hv);
        }
        reduce_block_to_stash(acc, DN_ROWS, t, tid);
      }
      if (tid < rows * p.m) {
        const int r = tid / p.m, t = tid % p.m;
        const int lr = r0 - d0 + r;
        S.acc[lr][t] += S.stash[r][t];
      }
      named_bar_sync(1, NCT);
    }
    if (h.stage == h.nstage - 1) {
      if (tid < DN_ROWS * p.m) {
        const int r = tid / p.m, t = tid % p.m;
        p.out[(size_t)t * p.D + d0 + r] = S.acc[r][t];
      }
    }
    consumer_release(n, tid);
    ++n;
  }
}

}  // namespace

int launch_decode_experts(const DecodeParams& p, int num_sms, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(k_gateup_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_down_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
    attr_done = true;
  }
  k_gateup_decode<<<num_sms, NTH, SMEM_BYTES, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  k_down_decode<<<num_sms, NTH, SMEM_BYTES, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
