// Shared device code of the moe_v41 kernels (sm_103a): PTX wrappers for
// mbarriers and 1-D bulk (TMA) copies, the workspace layout, the activation
// "unit" layout the K-quant dot products read, and the Q2_K / Q3_K unit dots.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_v41.h"

namespace moe {

// ---------------------------------------------------------------- sizes
constexpr int QK = 256;          // weights per K-quant super-block
constexpr int Q2K_B = 84;        // bytes per Q2_K super-block
constexpr int Q3K_B = 110;       // bytes per Q3_K super-block
constexpr int Q8_B = 36;         // bytes per q8_1 block of 32
constexpr int UNIT_WORDS = 24;   // words of one activation unit (see below)
constexpr int MAX_TOPK = 16;
constexpr int DECODE_MAX_M = 8;
constexpr int MAXP = DECODE_MAX_M * MAX_TOPK;  // token/expert pairs of a decode call
constexpr int MAX_N = 1024;

// ------------------------------------------------- workspace control block
struct Ctrl {
  unsigned status;        // MOE_STATUS_* bits, sticky
  unsigned route_arrive;  // last-block-done counter of the standalone router
  unsigned ticket;        // work tickets of the fused decode kernel
  unsigned q8_done;       // q8_1(x) tasks finished
  unsigned router_done;   // router tasks finished
  unsigned shdn_done;     // shared-expert down items finished (decode)
  unsigned shgu_done;     // shared-expert gate/up tasks finished
  unsigned rtgu_done;     // routed gate/up tasks finished
  unsigned exit_count;    // blocks that have left the fused kernel
  unsigned ticket_sh;     // shared-expert down items taken (decode)
  unsigned ticket_gu;     // routed gate/up items taken (decode)
  unsigned ticket_dn;     // routed down items taken (decode)
  unsigned pad[52];
};

// Routing of a decode call grouped by expert (ascending id), built in shared
// memory by each block's planner warp.
struct alignas(16) DecodePlan {
  int n_exp;                         // distinct experts picked
  int n_pairs;                       // m * topk
  int exp_id[MAXP];                  // ascending
  int exp_off[MAXP + 1];             // pair range of each distinct expert
  int pair_tok[MAXP];                // token of each pair, pairs sorted by (expert, token)
  float pair_w[MAXP];                // routing weight G of each pair
  int tok_pairs[DECODE_MAX_M][MAX_TOPK];  // each token's pairs in ascending expert id
  unsigned long long exp_ptr[MAXP][3];    // w1, w3, w2 of each distinct expert (0 = skip)
};

// Prefill tiling: weight rows per GEMM tile, columns (pairs or tokens) per
// tile, K values per pipeline stage, tokens per grouping chunk.
constexpr int PF_TM = 128;
constexpr int PF_TN = 256;     // router and bf16 shared-expert GEMMs
constexpr int PF_TN_GU = 128;  // routed gate/up GEMM (hi/lo split operands)
constexpr int PF_KC = 64;
constexpr int PF_GCH = 64;
constexpr int PF_TNQ = 128;    // routed down GEMM: pairs per tile (hi and lo parts stacked: an MMA of up to 256)

// Byte offsets of the prefill regions, relative to the prefill base.
struct PrefillLayout {
  size_t xgh, xgl, chunk, offsets, expert_ok, pair_tok, pair_w, pos_of, pos_sh, n_tiles, gu_tiles, dn_tiles, hh, hl,
      ep, hs, sp, total;
  size_t max_gu_tiles, max_dn_tiles;  // bounds on the column tiles over all experts
};

// Byte offsets of the workspace regions (all 256-B aligned).
struct WsLayout {
  size_t ctrl, plan, logits, sk, xq8, xu, hu, shh, pred, pre, total;
  PrefillLayout P;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Bytes of one activation vector of length K in unit layout.
__host__ __device__ inline size_t unit_bytes(int K) { return (size_t)(K / QK) * 4 * UNIT_WORDS * 4; }

inline PrefillLayout prefill_layout(const moe_v41_cfg& c) {
  PrefillLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  const size_t T = (size_t)c.max_tokens, P = T * c.topk, V = P + T;  // pairs, plus the K-quant shared expert's
  const size_t NE = (size_t)c.n_routed + 1;
  const size_t nch = (T + PF_GCH - 1) / PF_GCH;
  // an expert with n pairs takes ceil(n / tile width) column tiles
  L.max_gu_tiles = NE + V / PF_TN_GU + 1;
  L.max_dn_tiles = NE + V / PF_TNQ + 1;
  L.xgh = take(V * c.dim * 2);
  L.xgl = take(V * c.dim * 2);
  L.chunk = take(nch * NE * 4);
  L.offsets = take((NE + 1) * 4);
  L.expert_ok = take(NE * 4);
  L.pair_tok = take(V * 4);
  L.pair_w = take(V * 4);
  L.pos_of = take(P * 4);
  L.pos_sh = take(T * 4);
  L.n_tiles = take(2 * 4);
  L.gu_tiles = take(L.max_gu_tiles * (c.inter / PF_TM) * 16);  // per tile: (e, mt, column tile, 0)
  L.dn_tiles = take(L.max_dn_tiles * (c.dim / PF_TM) * 32);   // per tile: (e, mt, col0, ncol), W2 row-tile pointer
  L.hh = take(V * c.inter * 2);
  L.hl = take(V * c.inter * 2);
  L.ep = take(V * c.dim * 4);
  L.hs = take(T * c.inter * 2);
  L.sp = take(T * c.dim * 4);
  L.total = off;
  return L;
}

// Whether the fused decode kernel's stages hold one task's rows at these
// widths (defined with the kernel).
bool decode_fits(int D, int I);

// Whether a configuration can take the prefill kernels: always with
// MOE_PATH_PREFILL; with MOE_PATH_AUTO when some call may have more than 8
// tokens, or when the decode kernel cannot take these widths (then every call
// runs the prefill kernels).
inline bool prefill_possible(const moe_v41_cfg& c) {
  return c.path == MOE_PATH_PREFILL ||
         (c.path == MOE_PATH_AUTO && (c.max_tokens > DECODE_MAX_M || !decode_fits(c.dim, c.inter)));
}

inline WsLayout ws_layout(const moe_v41_cfg& c) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  const size_t T = (size_t)c.max_tokens;
  const size_t Td = T < DECODE_MAX_M ? T : DECODE_MAX_M;
  const size_t vecs = Td * c.topk + Td;  // routed pairs, then the shared expert's tokens
  L.ctrl = take(sizeof(Ctrl));
  L.plan = take(sizeof(DecodePlan));
  L.logits = take(T * c.n_routed * sizeof(float));
  L.sk = take(Td * c.n_routed * 2 * sizeof(float));  // (score, key) per token and expert, decode path
  L.xq8 = take(Td * (c.dim / 32) * Q8_B);
  L.xu = take(Td * unit_bytes(c.dim));
  L.hu = take(vecs * unit_bytes(c.inter));
  L.shh = take(Td * c.inter * 2);
  L.pred = take(Td * MAX_TOPK * 8);  // predicted picks of the next layer (weights, ids)
  if (prefill_possible(c)) {
    L.P = prefill_layout(c);
    L.pre = take(L.P.total);
  }
  L.total = off;
  return L;
}

// Activation "unit" layout.  A vector of K values (K a multiple of 256) in
// q8_1 blocks is stored per 256-block b and unit c (0..3) as 24 words:
//   words 4j+w (j, w < 4): int8 x4 of elements 256b + 128(c>>1) + 32j + 16(c&1) + 4w .. +3
//   word 16+j: f32 value of the fp16 d of q8_1 block 8b + 4(c>>1) + j
//   word 20+j: int sum of the 16 quants of that half block
// Unit c of a K-quant super-block holds exactly the 64 weights these 64
// activations meet (quant bytes 16c..16c+15 of Q2_K, the four sub-blocks
// 8(c>>1) + 2j + (c&1)), so one thread's dot needs one unit.

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same, letting the hardware suspend the thread for up to `ns`
// nanoseconds until the phase completes (a blocking wait, not a spin).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// 1-D bulk copy global -> shared, completing on an mbarrier.  src, dst
// 16-B aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait on an mbarrier phase.  Returns false (and sets the timeout
// status bit once) when the wait ran past the deadline.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t deadline,
                                                  unsigned* status) {
  uint32_t tries = 0;
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if ((++tries & 3u) == 0 && globaltimer_ns() > deadline) {
      atomicOr(status, (unsigned)MOE_STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// dot of four unsigned bytes of a with four signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_float(uint32_t h16) {
  return __half2float(__ushort_as_half((unsigned short)(h16 & 0xFFFFu)));
}

// Clipped SwiGLU in f32: g' = min(g, L), u' = clamp(u, -L, L) when L > 0;
// h = g' sigmoid(g') u'.
__device__ __forceinline__ float swiglu_f32(float g, float u, float L) {
  if (L > 0.f) {
    g = fminf(g, L);
    u = fminf(fmaxf(u, -L), L);
  }
  float sig = 1.0f / (1.0f + expf(-g));
  return g * sig * u;
}

// ------------------------------------------------------ K-quant unit dots
// One activation unit in registers.
struct XUnit {
  int q[16];
  float dq[4];
  int s16[4];
};

__device__ __forceinline__ void load_xunit(XUnit& x, const int4* p) {
  int4 v0 = __ldg(p + 0), v1 = __ldg(p + 1), v2 = __ldg(p + 2), v3 = __ldg(p + 3);
  int4 v4 = __ldg(p + 4), v5 = __ldg(p + 5);
  x.q[0] = v0.x; x.q[1] = v0.y; x.q[2] = v0.z; x.q[3] = v0.w;
  x.q[4] = v1.x; x.q[5] = v1.y; x.q[6] = v1.z; x.q[7] = v1.w;
  x.q[8] = v2.x; x.q[9] = v2.y; x.q[10] = v2.z; x.q[11] = v2.w;
  x.q[12] = v3.x; x.q[13] = v3.y; x.q[14] = v3.z; x.q[15] = v3.w;
  x.dq[0] = __int_as_float(v4.x); x.dq[1] = __int_as_float(v4.y);
  x.dq[2] = __int_as_float(v4.z); x.dq[3] = __int_as_float(v4.w);
  x.s16[0] = v5.x; x.s16[1] = v5.y; x.s16[2] = v5.z; x.s16[3] = v5.w;
}

// (float)v for |v| < 2^22, exactly: v added to the bit pattern of 1.5 * 2^23
// (whose binade has unit spacing), minus that value.  Two full-rate
// instructions instead of one quarter-rate conversion.
__device__ __forceinline__ float i2f_exact22(int v) { return __int_as_float(0x4B400000 + v) - 12582912.0f; }

// byte j of v, zero-extended
__device__ __forceinline__ int byte_of(uint32_t v, int j) { return (int)__byte_perm(v, 0u, 0x4440u + (uint32_t)j); }

// Unit c of a Q2_K block (84 B, 4-B aligned, in shared memory) dotted with
// the matching activation unit:
//   sum_j dq_j * ( d * sc_j * sum(q * qx) - dmin * m_j * sum(qx) )
// over the four sub-blocks j of the unit.  The 2-bit plane j is masked in
// place (values 4^j q), so its integer dot is shifted back by 2j.
__device__ __forceinline__ float q2k_unit_dot(const uint8_t* blk, int c, const XUnit& x) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
  const uint32_t q0 = w[4 + 4 * c], q1 = w[5 + 4 * c], q2 = w[6 + 4 * c], q3 = w[7 + 4 * c];
  const int h = c >> 1, half = c & 1;
  const uint32_t sa = w[2 * h], sb = w[2 * h + 1];
  const uint32_t dd = w[20];
  // the scale / min bytes of sub-blocks j = 0..3 of this unit (bytes half,
  // half + 2 of sa, then of sb), split into scale and min nibbles
  const uint32_t sm = __byte_perm(sa, sb, half ? 0x7531u : 0x6420u);
  const uint32_t sc4 = sm & 0x0F0F0F0Fu, mn4 = (sm >> 4) & 0x0F0F0F0Fu;
  float acc_d = 0.f, acc_m = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t mask = 0x03030303u << (2 * j);
    int a = dp4a_us(q0 & mask, x.q[4 * j + 0], 0);
    a = dp4a_us(q1 & mask, x.q[4 * j + 1], a);
    a = dp4a_us(q2 & mask, x.q[4 * j + 2], a);
    a = dp4a_us(q3 & mask, x.q[4 * j + 3], a);
    const int isum = a >> (2 * j);
    // |sc * isum| <= 15 * 16 * 3 * 127 and |m * s16| <= 15 * 16 * 127: exact below 2^22
    acc_d = fmaf(x.dq[j], i2f_exact22(byte_of(sc4, j) * isum), acc_d);
    acc_m = fmaf(x.dq[j], i2f_exact22(byte_of(mn4, j) * x.s16[j]), acc_m);
  }
  const float d = half_bits_to_float(dd), dmin = half_bits_to_float(dd >> 16);
  return d * acc_d - dmin * acc_m;
}

// Unit c of a Q3_K block (110 B, 2-B aligned, in shared memory) dotted with
// the matching activation unit.  q = lo + 4 hb - 4 with lo the 2-bit plane j
// and hb bit 4h + j of the hmask byte:
//   sum_j dq_j * d * (code_j - 32) * ( sum(lo*qx) + 4 sum(hb*qx) - 4 sum(qx) )
// The block's words are read from the 4-byte aligned window around it and
// realigned with one byte permute each (the window may reach 2 bytes past the
// block, still inside the stage buffer).
__device__ __forceinline__ float q3k_unit_dot(const uint8_t* blk, int c, const XUnit& x) {
  const int h = c >> 1, half = c & 1;
  const uintptr_t a = reinterpret_cast<uintptr_t>(blk);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sel = (a & 2u) ? 0x5432u : 0x3210u;  // block word i = prmt(w[i], w[i + 1], sel)
  uint32_t hmw[5], qsw[5], scw[4];
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    hmw[i] = w[4 * half + i];      // block words 4 half .. 4 half + 3: hmask bytes 16 half ..
    qsw[i] = w[8 + 4 * c + i];     // block words 8 + 4c ..: quant bytes 32 + 16c ..
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) scw[i] = w[24 + i];  // block words 24 .. 26: scales; 27: d
  uint32_t q[4], m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    q[i] = __byte_perm(qsw[i], qsw[i + 1], sel);
    m[i] = __byte_perm(hmw[i], hmw[i + 1], sel);
  }
  const uint32_t s_lo = __byte_perm(scw[0], scw[1], sel);   // scales bytes 0..3
  const uint32_t s_lo2 = __byte_perm(scw[1], scw[2], sel);  // scales bytes 4..7
  const uint32_t s_hi = __byte_perm(scw[2], scw[3], sel);   // scales bytes 8..11
  const uint32_t dbits = (a & 2u) ? (scw[3] >> 16) : (scw[3] & 0xFFFFu);
  // six-bit scale codes of sub-blocks 8h + 2j + half, j = 0..3, one per byte:
  // low four bits from bytes half, half + 2, half + 4, half + 6 of scales[0..7]
  // (nibble h), high two bits from scales[8 + 2(j & 1) + half] at bit 4h + 2(j >> 1)
  const uint32_t lo4 = (__byte_perm(s_lo, s_lo2, half ? 0x7531u : 0x6420u) >> (4 * h)) & 0x0F0F0F0Fu;
  const uint32_t hv = __byte_perm(s_hi, s_hi, half ? 0x3131u : 0x2020u) >> (4 * h);
  const uint32_t hi2 = ((hv & 0x0000FFFFu) | ((hv >> 2) & 0xFFFF0000u)) & 0x03030303u;
  const uint32_t codes = lo4 | (hi2 << 4);
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lmask = 0x03030303u << (2 * j);
    const uint32_t hmask = 0x01010101u << (4 * h + j);
    int a0 = dp4a_us(q[0] & lmask, x.q[4 * j + 0], 0);
    a0 = dp4a_us(q[1] & lmask, x.q[4 * j + 1], a0);
    a0 = dp4a_us(q[2] & lmask, x.q[4 * j + 2], a0);
    a0 = dp4a_us(q[3] & lmask, x.q[4 * j + 3], a0);
    int b = dp4a_us(m[0] & hmask, x.q[4 * j + 0], 0);
    b = dp4a_us(m[1] & hmask, x.q[4 * j + 1], b);
    b = dp4a_us(m[2] & hmask, x.q[4 * j + 2], b);
    b = dp4a_us(m[3] & hmask, x.q[4 * j + 3], b);
    const int isum = (a0 >> (2 * j)) + ((b >> (4 * h + j)) << 2) - 4 * x.s16[j];
    // |scale * isum| <= 32 * 16 * 7 * 127: exact below 2^22
    acc = fmaf(x.dq[j], i2f_exact22((byte_of(codes, j) - 32) * isum), acc);
  }
  return half_bits_to_float(dbits) * acc;
}

// q8_1 code of v: round-half-away(RN(v / d)), the f32 decision of the q8_1
// rule, mostly without a division.  y = v * RN(1/d) is within 2^-22 |y| of
// RN(v / d) (1/d and the product are each rounded once, 2^-24 relative, and
// v / d itself is within 2^-24 of its rounding); when y lies farther than
// 2^-19 max(|y|, 1) from every half-integer both round to the same integer.
// Otherwise (a few values in 10^4), or when 1/d overflowed, the quotient is
// computed exactly.
// The exact quotient rule, out of line: it is taken for a few values in 10^4.
static __device__ __noinline__ int q8_code_exact(float v, float d) { return (int)roundf(__fdiv_rn(v, d)); }

__device__ __forceinline__ int q8_code(float v, float d, float rd) {
  const float y = v * rd;
  const float a = fabsf(y);
  const float f = a - floorf(a);
  if (a < 1.0e30f && fabsf(f - 0.5f) > 0x1.0p-19f * fmaxf(a, 1.0f)) return (int)copysignf(floorf(a + 0.5f), y);
  return q8_code_exact(v, d);
}

// ------------------------------------------------------------------ q8_1 (warp)
// One warp quantises one q8_1 block of 32 values (lane i holds value i):
// d = amax/127, q = round-half-away(v/d), decisions in f32.  Writes the
// 36-byte block (if q8 != nullptr) and the block's two half units into the
// unit layout of its vector (if units != nullptr).  qb = block index within
// the vector.
__device__ __forceinline__ void q8_block_warp(float v, int qb, uint8_t* q8, int* units) {
  const int lane = threadIdx.x & 31;
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = amax == 0.0f ? 0 : q8_code(v, d, __frcp_rn(d));
  int s = q, s16;
#pragma unroll
  for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);  // sums within 16-lane halves
  s16 = s;
  const int sum = s16 + __shfl_xor_sync(0xffffffffu, s16, 16);
  // gather four bytes per word
  uint32_t b = (uint32_t)(q & 0xFF);
  uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 1);
  uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 2);
  uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 3);
  const uint32_t word = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
  const __half d16 = __float2half_rn(d);
  if (q8) {
    uint8_t* blk = q8 + (size_t)qb * Q8_B;
    if (lane == 0) {
      const __half s16h = __float2half_rn(__fmul_rn(d, (float)sum));
      const uint32_t hdr = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(s16h) << 16);
      *reinterpret_cast<uint32_t*>(blk) = hdr;
    }
    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(blk + 4 + lane) = word;
  }
  if (units) {
    const int b256 = qb >> 3, hj = qb & 7, h = hj >> 2, j = hj & 3;
    const int half = lane >> 4;
    int* u = units + ((size_t)b256 * 4 + 2 * h + half) * UNIT_WORDS;
    if ((lane & 3) == 0) u[4 * j + ((lane & 15) >> 2)] = (int)word;
    if ((lane & 15) == 0) {
      u[16 + j] = __float_as_int(__half2float(d16));
      u[20 + j] = s16;
    }
  }
}

// The same quantisation of one block by ONE thread (no shuffles, so a warp
// quantises 32 blocks at once): x32 = 32 bf16 values (16-B aligned), qb = the
// block's index within its vector.  Bit-identical to q8_block_warp: the same
// f32 operations in the same order for every value; amax and the integer sums
// do not depend on the order.
__device__ __forceinline__ void q8_block_thread(const uint16_t* x32, int qb, int* units) {
  const uint2* xp = reinterpret_cast<const uint2*>(x32);
  float amax = 0.f;
#pragma unroll 1
  for (int w = 0; w < 8; ++w) {
    const uint2 v = xp[w];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))), fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y)))));
  }
  const float d = __fdiv_rn(amax, 127.0f);
  const float rd = __frcp_rn(d);
  const int b256 = qb >> 3, hj = qb & 7, h = hj >> 2, j = hj & 3;
  int* u0 = units + ((size_t)b256 * 4 + 2 * h) * UNIT_WORDS;
  int s0 = 0, s1 = 0;
  // words 0..3 of the block go to the first half unit, 4..7 to the second
#pragma unroll 1
  for (int w = 0; w < 8; ++w) {
    const uint2 v = xp[w];
    const float f[4] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y)};
    uint32_t wd = 0;
    int sw = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int q = amax == 0.0f ? 0 : q8_code(f[b], d, rd);
      wd |= (uint32_t)(q & 0xFF) << (8 * b);
      sw += q;
    }
    if (w < 4) s0 += sw; else s1 += sw;
    u0[(w >> 2) * UNIT_WORDS + 4 * j + (w & 3)] = (int)wd;
  }
  const float dq = __half2float(__float2half_rn(d));
  int* u1 = u0 + UNIT_WORDS;
  u0[16 + j] = __float_as_int(dq);
  u1[16 + j] = __float_as_int(dq);
  u0[20 + j] = s0;
  u1[20 + j] = s1;
}

}  // namespace moe
