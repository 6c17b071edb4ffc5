// Prefill path (any m; taken by default above eight tokens): the expert
// projections as GEMMs on the 5th-generation tensor cores.
//
//   router  logits = x W_R^T (bf16 tensor-core GEMM, f32 accumulation), then
//           the selection per token
//   group   (expert, token) pairs ordered by expert id, tokens ascending
//           within an expert: the per-expert token lists of DeepSeek V4.1
//           atlas "Mixture of experts" (model.py MoE.forward), made
//           deterministic by a counting sort over token chunks
//   xg      the q8_1 activation values fp16(d) * q (the values the method's
//           integer dots stand for) as exact fp16 high + low parts, written
//           in pair order
//   gate/up per (expert, 128 rows, <= 128 pairs) tile: W1 and W3 rows
//           dequantised from Q2_K, split into high and low fp16 parts, times
//           the pairs' xg rows (three products: hi.hi + hi.lo + lo.hi, about
//           2^-22 relative); the epilogue applies the clipped SwiGLU,
//           quantises h to q8_1 and stores its exact values as fp16 high +
//           low parts.  The split is needed because q8_1(h) turns any error
//           in h near a rounding boundary into a whole quantisation step.
//   down    W2 (Q3_K) times those rows with exact products (the persistent
//           GEMM of k_prefill_kq.cu) -> E per pair
//   shared  bf16 shared expert: two bf16 GEMMs, h rounded to bf16 between them;
//           a K-quant shared expert is one more expert taken by every token
//   combine out = sum over the token's experts in ascending id of G_i E_i,
//           then the shared expert's output added last
//
// GEMM block (128 weight rows x up to 128 or 256 columns): a TMA thread loads
// the B rows (and bf16 A rows) of each K chunk into 128-byte-swizzled K-major
// stage tiles; for Q2_K A, sixteen producer warps dequantise staged raw
// blocks into the A tiles (four threads per weight row, one 16-value
// sub-block each, through per-sub-block lookup tables); one thread issues
// tcgen05.mma (M = 128, N = tile width, K = 16) into a tensor-memory
// accumulator and commits each stage back; the producer warps then read the
// accumulator for the epilogue.  Products accumulate in f32; bf16 operands
// (router, bf16 shared expert) are the caller's values, exact.
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int TM = PF_TM;
constexpr int KC = PF_KC;

enum : int { A_BF16 = 0, A_Q2K = 1 };
enum : int { E_F32 = 0, E_SWIGLU_Q8 = 1, E_SWIGLU_BF16 = 2 };

__device__ __forceinline__ uint32_t f2h(float v) { return (uint32_t)__half_as_ushort(__float2half_rn(v)); }

// ------------------------------------------------------------------ prep
// The q8_1 values of x, fp16(d) * q (exact in f32), as fp16 high and low
// parts, written to the row of every (expert, token) pair of the token (and
// of the K-quant shared expert's pair), so the gate/up GEMM reads its B
// operand as contiguous rows.  Four threads per block of 32 (the q8_1 rule:
// d = amax / 127, q = round-half-away(v / d), d stored as fp16), eight values
// each, so that a warp's 16-byte stores cover 512 contiguous bytes.
__global__ void k_xg(const uint16_t* __restrict__ x, int m, int D, int k, const int* __restrict__ pos_of,
                     const int* __restrict__ pos_sh, uint16_t* __restrict__ xgh, uint16_t* __restrict__ xgl) {
  const int nq = D / 32;
  const long nb = (long)m * nq * 4;  // quarter blocks; D / 8 per token, so a group of four never spans tokens
  for (long g = blockIdx.x * (long)blockDim.x + threadIdx.x; g - (threadIdx.x & 31) < nb;
       g += (long)gridDim.x * blockDim.x) {
    const bool live = g < nb;
    const long gq = live ? g : nb - 1;  // lanes past the end repeat the last quarter and store nothing
    const int t = (int)(gq / (nq * 4));
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + gq);
    const uint32_t raw[4] = {v.x, v.y, v.z, v.w};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(raw[i])), fabsf(bf16hi(raw[i]))));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float rd = __frcp_rn(d);
    const float dq = __half2float(__float2half_rn(d));
    uint32_t oh[4], ol[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q0 = amax == 0.0f ? 0 : q8_code(bf16lo(raw[i]), d, rd);
      const int q1 = amax == 0.0f ? 0 : q8_code(bf16hi(raw[i]), d, rd);
      const float v0 = dq * (float)q0, v1 = dq * (float)q1;
      const __half2 hh = __floats2half2_rn(v0, v1);
      const float2 back = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v0 - back.x, v1 - back.y);
      oh[i] = *reinterpret_cast<const uint32_t*>(&hh);
      ol[i] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    if (!live) continue;
    const long off = gq - (long)t * nq * 4;  // 16-byte chunk of the token's row
    for (int i = 0; i <= k; ++i) {
      const int pos = i < k ? __ldg(pos_of + (size_t)t * k + i) : (pos_sh ? __ldg(pos_sh + t) : -1);
      if (pos < 0) continue;
      reinterpret_cast<uint4*>(xgh + (size_t)pos * D)[off] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      reinterpret_cast<uint4*>(xgl + (size_t)pos * D)[off] = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    }
  }
}

// ----------------------------------------------------------------- group
// Pairs are (token t, slot i) at index p = t k + i.  The pseudo-expert N is a
// K-quant shared expert (every token, weight 1) when there is one.

// per chunk of PF_GCH tokens: how many of its pairs pick each expert
__global__ void k_group_hist(const int* __restrict__ idx, int m, int k, int N, int shq, int* __restrict__ chunk) {
  extern __shared__ int hist[];
  const int NE = N + 1;
  const int t0 = blockIdx.x * PF_GCH, t1 = min(m, t0 + PF_GCH);
  for (int e = threadIdx.x; e < NE; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (int p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
    const int e = __ldg(idx + p);
    if ((unsigned)e < (unsigned)N) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < NE; e += blockDim.x)
    chunk[(size_t)blockIdx.x * NE + e] = e == N ? (shq ? t1 - t0 : 0) : hist[e];
}

// exclusive scan over a 1024-thread block; returns the exclusive prefix of v
// and writes the block total to *total
__device__ __forceinline__ int block_scan_1024(int v, int* s32, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s32[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = s32[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    s32[lane] = wi - w;  // exclusive prefix of the warp totals
    if (lane == 31) s32[32] = wi;
  }
  __syncthreads();
  const int r = s32[warp] + incl - v;
  *total = s32[32];
  __syncthreads();  // s32 is reused by the next scan
  return r;
}

// One block of 1024 threads, two experts per thread: expert counts and
// offsets, the chunk bases of the scatter (in place over the chunk counts),
// which picked experts are usable, and the tile lists of both expert GEMMs.
// Gate/up tiles are (expert, row tile, column tile of 128 pairs).  Down tiles
// are two int4 each: (expert, row tile, first pair, pairs) and the address
// of the tile's first W2 row (twice); an expert with n pairs takes ceil(n /
// 64) of them with balanced widths (pairs [n t / c, n (t + 1) / c) for tile
// t of c).  Row tiles are listed fastest, so that the row tiles of one
// expert's pairs run side by side and share their activation rows in L2.
// Expert N is the K-quant shared expert (its W2 is sh2).
__global__ void __launch_bounds__(1024) k_group_scan(int* __restrict__ chunk, int nch, int N,
                                                     const unsigned long long* __restrict__ eptr, int gu_mt,
                                                     int dn_mt, size_t dn_row_tile, const uint8_t* sh2,
                                                     int* __restrict__ offsets, int* __restrict__ expert_ok,
                                                     int4* __restrict__ gu_tiles, int4* __restrict__ dn_tiles,
                                                     int* __restrict__ n_tiles, unsigned* status) {
  __shared__ int s32[33];
  const int NE = N + 1;
  int cnt[2] = {0, 0}, ok[2] = {1, 1}, ng[2] = {0, 0}, nd[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = 2 * threadIdx.x + j;
    if (e < NE) {
      for (int c = 0; c < nch; ++c) cnt[j] += chunk[(size_t)c * NE + e];
      if (e < N && cnt[j] > 0) {
        for (int q = 0; q < 3; ++q) {
          const unsigned long long v = __ldg(eptr + (size_t)e * 3 + q);
          if (v == 0ull || (v & 255ull)) ok[j] = 0;
        }
        if (!ok[j]) atomicOr(status, (unsigned)MOE_STATUS_MISSING_EXPERT);
      }
      ng[j] = ok[j] ? (cnt[j] + PF_TN_GU - 1) / PF_TN_GU : 0;
      nd[j] = ok[j] ? (cnt[j] + PF_TNQ - 1) / PF_TNQ : 0;
    }
  }
  int total_pairs, total_g, total_d;
  const int off = block_scan_1024(cnt[0] + cnt[1], s32, &total_pairs);
  const int goff = block_scan_1024(ng[0] + ng[1], s32, &total_g);
  const int doff = block_scan_1024(nd[0] + nd[1], s32, &total_d);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = 2 * threadIdx.x + j;
    if (e < NE) {
      const int o = off + (j ? cnt[0] : 0);
      const int go = goff + (j ? ng[0] : 0), dof = doff + (j ? nd[0] : 0);
      offsets[e] = o;
      expert_ok[e] = ok[j];
      int run = o;
      for (int c = 0; c < nch; ++c) {
        const int v = chunk[(size_t)c * NE + e];
        chunk[(size_t)c * NE + e] = run;
        run += v;
      }
      for (int t = 0; t < ng[j]; ++t)
        for (int mt = 0; mt < gu_mt; ++mt) gu_tiles[(size_t)(go + t) * gu_mt + mt] = make_int4(e, mt, t, 0);
      if (nd[j] > 0) {
        const unsigned long long w2 = e == N ? reinterpret_cast<unsigned long long>(sh2) : __ldg(eptr + (size_t)e * 3 + 2);
        for (int t = 0; t < nd[j]; ++t) {
          const int a = (int)((long long)cnt[j] * t / nd[j]), b = (int)((long long)cnt[j] * (t + 1) / nd[j]);
          for (int mt = 0; mt < dn_mt; ++mt) {
            const unsigned long long rp = w2 + (unsigned long long)mt * dn_row_tile;
            int4* d = dn_tiles + 2 * ((size_t)(dof + t) * dn_mt + mt);
            d[0] = make_int4(e, mt, o + a, b - a);
            d[1] = make_int4((int)(uint32_t)rp, (int)(uint32_t)(rp >> 32), (int)(uint32_t)rp, (int)(uint32_t)(rp >> 32));
          }
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    offsets[NE] = total_pairs;
    n_tiles[0] = total_g * gu_mt;
    n_tiles[1] = total_d * dn_mt;
  }
}

// per chunk: each pair's position = its expert's chunk base + the number of
// earlier tokens of the chunk that picked the same expert (a token never
// picks one expert twice)
__global__ void k_group_scatter(const int* __restrict__ idx, const float* __restrict__ w, int m, int k, int N,
                                int shq, const int* __restrict__ chunk_base, int* __restrict__ pair_tok,
                                float* __restrict__ pair_w, int* __restrict__ pos_of, int* __restrict__ pos_sh) {
  __shared__ int s_idx[PF_GCH * MAX_TOPK];
  const int NE = N + 1;
  const int t0 = blockIdx.x * PF_GCH, t1 = min(m, t0 + PF_GCH);
  const int np = (t1 - t0) * k;
  const int* base = chunk_base + (size_t)blockIdx.x * NE;
  for (int q = threadIdx.x; q < np; q += blockDim.x) s_idx[q] = __ldg(idx + (size_t)t0 * k + q);
  __syncthreads();
  for (int q = threadIdx.x; q < np; q += blockDim.x) {
    const int e = s_idx[q];
    const size_t p = (size_t)t0 * k + q;
    if ((unsigned)e >= (unsigned)N) {
      pos_of[p] = -1;
      continue;
    }
    const int tl = q / k;
    int rank = 0;
    for (int q2 = 0; q2 < tl * k; ++q2) rank += s_idx[q2] == e;
    const int pos = base[e] + rank;
    pair_tok[pos] = t0 + tl;
    pair_w[pos] = __ldg(w + p);
    pos_of[p] = pos;
  }
  if (shq) {
    for (int tl = threadIdx.x; tl < t1 - t0; tl += blockDim.x) {
      const int pos = base[N] + tl;
      pair_tok[pos] = t0 + tl;
      pair_w[pos] = 1.0f;
      pos_sh[t0 + tl] = pos;
    }
  }
}

// --------------------------------------------------------------- combine
template <class V> __device__ __forceinline__ V vzero();
template <> __device__ __forceinline__ float vzero<float>() { return 0.f; }
template <> __device__ __forceinline__ float4 vzero<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ float vfma(float w, float a, float c) { return fmaf(w, a, c); }
__device__ __forceinline__ float4 vfma(float w, float4 a, float4 c) {
  return make_float4(fmaf(w, a.x, c.x), fmaf(w, a.y, c.y), fmaf(w, a.z, c.z), fmaf(w, a.w, c.w));
}
__device__ __forceinline__ float vadd(float a, float b) { return a + b; }
__device__ __forceinline__ float4 vadd(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

// out[t] = sum over t's usable pairs in ascending expert id of G * E, then
// the shared expert's output (V = float4 where out is 16-byte aligned)
template <class V, int VW = sizeof(V) / sizeof(float)>
__global__ void k_combine(const int* __restrict__ idx, const int* __restrict__ pos_of,
                          const int* __restrict__ expert_ok, const float* __restrict__ pair_w,
                          const float* __restrict__ ep, const float* __restrict__ sp, const int* __restrict__ pos_sh,
                          int k, int D, float* __restrict__ out) {
  const int t = blockIdx.x;
  __shared__ int s_pos[MAX_TOPK];
  __shared__ float s_w[MAX_TOPK];
  __shared__ int s_n;
  if (threadIdx.x == 0) {
    int e[MAX_TOPK], pos[MAX_TOPK], n = 0;
    for (int i = 0; i < k; ++i) {
      const int ei = idx[(size_t)t * k + i], pi = pos_of[(size_t)t * k + i];
      if (pi < 0 || !expert_ok[ei]) continue;
      int j = n - 1;  // insertion by expert id
      while (j >= 0 && e[j] > ei) {
        e[j + 1] = e[j];
        pos[j + 1] = pos[j];
        --j;
      }
      e[j + 1] = ei;
      pos[j + 1] = pi;
      ++n;
    }
    for (int i = 0; i < n; ++i) {
      s_pos[i] = pos[i];
      s_w[i] = pair_w[pos[i]];
    }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  // VW values per access; every pair's value is loaded before the sums, so a
  // thread has all its streams in flight at once
  const int DV = D / VW;
  const V* e = reinterpret_cast<const V*>(ep);
  const V* sh = reinterpret_cast<const V*>(pos_sh ? ep + (size_t)pos_sh[t] * D : sp + (size_t)t * D);
  V* o = reinterpret_cast<V*>(out + (size_t)t * D);
  for (int c = threadIdx.x; c < DV; c += blockDim.x) {
    V v[MAX_TOPK];
#pragma unroll
    for (int i = 0; i < MAX_TOPK; ++i)
      if (i < n) v[i] = __ldcs(e + (size_t)s_pos[i] * DV + c);
    const V hv = __ldcs(sh + c);
    V acc = vzero<V>();
#pragma unroll
    for (int i = 0; i < MAX_TOPK; ++i)
      if (i < n) acc = vfma(s_w[i], v[i], acc);
    __stcs(o + c, vadd(acc, hv));
  }
}

// ------------------------------------------------------------------ GEMM
constexpr int B_BOX = 16;  // rows per B box of the expert GEMMs: a tile loads only the rows it uses

struct GemmArgs {
  CUtensorMap map_a[2];                // bf16 A matrices (box 64 x 128)
  CUtensorMap map_b[2];                // B rows (high, low parts): box 64 x B_BOX (expert jobs), 64 x TNM
                                       // (plain jobs)
  int K;                               // contraction length: a multiple of 256 (K-quant A) or 64 (bf16 A)
  int a_rows;                          // rows of A (the M extent)
  int a_row_bytes;                     // K-quant A: bytes per row
  const uint8_t* a0;                   // K-quant A of a plain job, or of the pseudo-expert
  const uint8_t* a1;
  const unsigned long long* eptr;      // expert jobs: the [N][3] pointer table
  int pj0, pj1;                        // pointer-table columns of the job's matrices
  int pseudo;                          // expert whose matrices are a0 / a1 (-1: none)
  int cols;                            // plain jobs: number of columns
  const int4* tiles;                   // expert jobs: (e, mt, nt) per block
  const int* n_tiles;
  const int* offsets;                  // expert jobs: column range of each expert
  int mt_count;                        // plain jobs: M tiles
  float* out_f32;                      // E_F32: out[col * ld + row]
  uint16_t* out_h;                     // E_SWIGLU_*: h[col * ld + row] (E_SWIGLU_Q8: its high fp16 part)
  uint16_t* out_h2;                    // E_SWIGLU_Q8: the low fp16 part
  int out_ld;
  float swiglu_limit;
  unsigned* status;
  unsigned long long timeout_ns;
};

constexpr uint32_t A_TILE = TM * 128;  // bytes of one A tile (128 rows x 64 values)

// Raw Q2_K staging.  A UNIT is the stretch of every tile row's blocks that
// a group of consecutive K chunks reads: half a super-block (2 chunks: its
// 32 quant bytes, 8 scale bytes and d/dmin = 11 words).  Shared memory holds
// it row-major with an odd pitch (11 words): the copies of one row's
// consecutive words coalesce, and one word of 32 consecutive rows falls in 32
// banks.
template <int AK>
struct RawGeo {
  static constexpr int words() { return 11; }
  static constexpr int PITCH = 11;
  static constexpr uint32_t BYTES = AK == A_BF16 ? 0u : (uint32_t)(TM * PITCH * 4);  // one matrix, one buffer
};

template <int NSA, int NSB, int RAWN>
struct GemmCtl {
  unsigned long long full_a[NSA], empty_a[NSA], full_b[NSB], empty_b[NSB], acc;
  unsigned long long raw_full[RAWN], raw_free[RAWN];
  uint32_t tmem;
};

// Memory plan of one GEMM variant.  A ring of NSA A stages (NMAT A tiles
// each, times two when split into high and low fp16 parts): in tensor memory
// for K-quant A (written by the dequantising threads, lane = row), in shared
// memory for bf16 A (loaded by TMA together with B, in the A stage of the B
// stage's index).  In shared memory: a ring of NSB B stages (one B tile of
// TNM rows, two when split), RAWN raw buffers per matrix for K-quant A, the
// control block and the gathered B row indices.
template <int AK, int NMAT, bool SPLIT, int TNM, int NSA, int NSB, int RAWN>
struct Plan {
  static constexpr int NPART = SPLIT ? 2 : 1;
  static constexpr uint32_t B_TILE = TNM * 128;
  static constexpr uint32_t A_STAGE = NMAT * NPART * A_TILE;
  static constexpr uint32_t B_STAGE = NPART * B_TILE;
  static constexpr bool ATMEM = AK != A_BF16;  // K-quant A lives in tensor memory
  static constexpr uint32_t B_RING = ATMEM ? 0u : NSA * A_STAGE;
  // tensor-memory columns: accumulators [0, 256), K-quant A stages from 256
  static constexpr uint32_t TA_COLS = NMAT * NPART * 32;  // columns of one A stage (64 K values per tile)
  static_assert(!ATMEM || 256 + NSA * TA_COLS <= 512, "A stages exceed tensor memory");
  static constexpr uint32_t RAW_OFF = B_RING + NSB * B_STAGE;
  static constexpr uint32_t RAW = RAWN * NMAT * RawGeo<AK>::BYTES;
  static constexpr uint32_t CTL = RAW_OFF + RAW;
  static constexpr uint32_t ROWS = CTL + ((sizeof(GemmCtl<NSA, NSB, RAWN>) + 15) & ~15);
  static constexpr size_t SMEM = 1024 + (size_t)ROWS + TNM * 4;
  static __device__ __forceinline__ uint32_t a_off(int sa, int mat, int part) {
    return sa * A_STAGE + (mat * NPART + part) * A_TILE;
  }
  static __device__ __forceinline__ uint32_t b_off(int sb, int part) { return B_RING + sb * B_STAGE + part * B_TILE; }
  static __device__ __forceinline__ uint32_t raw_off(int mat, int buf) {
    return RAW_OFF + (buf * NMAT + mat) * RawGeo<AK>::BYTES;
  }
};


__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// arrive (without a pending-count increment) on the mbarrier once every
// cp.async this thread has issued so far has landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Lookup tables of one Q2_K sub-block: w(q) = d sc q - dmin mn for q = 0..3
// as fp16 high parts (hi01 = w0 | w1 << 16, hi23 = w2 | w3 << 16) and, when
// split, the fp16 residuals w(q) - hi(q).
template <bool SPLIT>
__device__ __forceinline__ void q2k_tables(float d, float dmin, uint32_t scbyte, uint32_t& hi01, uint32_t& hi23,
                                           uint32_t& lo01, uint32_t& lo23) {
  const float A = d * (float)(scbyte & 15u), B = dmin * (float)(scbyte >> 4);
  const float w0 = -B, w1 = A - B, w2 = fmaf(2.0f, A, -B), w3 = fmaf(3.0f, A, -B);
  const __half2 ha = __floats2half2_rn(w0, w1), hb = __floats2half2_rn(w2, w3);
  hi01 = h2bits(ha);
  hi23 = h2bits(hb);
  if constexpr (SPLIT) {
    const float2 fa = __half22float2(ha), fb = __half22float2(hb);
    lo01 = h2bits(__floats2half2_rn(w0 - fa.x, w1 - fa.y));
    lo23 = h2bits(__floats2half2_rn(w2 - fb.x, w3 - fb.y));
  }
}

// PRMT selectors of table entries: for the 2-bit codes q0..q3 in bytes 0..3
// of qq, byte b of the result is (2qb + 1) << 4 | 2qb, so its low half selects
// bytes (2q0, 2q0+1, 2q1, 2q1+1) of the 8-byte table and its high half the
// same for q2, q3 (no byte carries into the next: 3 * 0x22 + 0x10 < 0x100).
__device__ __forceinline__ uint32_t pair_sels(uint32_t qq) { return qq * 0x22u + 0x10101010u; }

// q8_1 of one 32-value block of h held one value per lane: the exact value
// fp16(d) * q of this lane's element (11 x 7 significant bits) as fp16 high
// and low parts whose sum is exact
__device__ __forceinline__ void q8_hilo_warp(float v, uint16_t& hi, uint16_t& lo) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = amax == 0.0f ? 0 : q8_code(v, d, __frcp_rn(d));
  const float x = __half2float(__float2half_rn(d)) * (float)q;
  const __half h = __float2half_rn(x);
  hi = __half_as_ushort(h);
  lo = __half_as_ushort(__float2half_rn(x - __half2float(h)));
}

// One tile: D[128 rows, TN columns] (per matrix) = A . B^T over K.
//   warps 0 .. NPW-1       K-quant A: dequantise staged raw blocks into the
//                          A ring; then the epilogue (all variants)
//   next NLW warps         K-quant A: copy the raw blocks of each unit into
//                          the raw ring (asynchronous copies; these warps never
//                          fence, so no copy in flight delays a stage hand-over)
//   next warp              lane 0: TMA loads of B (and of bf16 A) per stage
//   last warp              lane 0: tcgen05.mma issue
// SPLIT: A = A_hi + A_lo and B = B_hi + B_lo in fp16, accumulating
// A_hi B_hi + A_hi B_lo + A_lo B_hi (the A_lo B_lo term is below 2^-22
// relative).
template <int AK>
constexpr int loader_warps() { return AK == A_BF16 ? 0 : 4; }

template <int AK, int NMAT, bool SPLIT, int EPI, int TNM, int NSA, int NSB, int RAWN, int NPROD>
__global__ void __launch_bounds__(NPROD + 32 * loader_warps<AK>() + 64, 1) k_gemm(const __grid_constant__ GemmArgs g) {
  using PL = Plan<AK, NMAT, SPLIT, TNM, NSA, NSB, RAWN>;
  using RG = RawGeo<AK>;
  constexpr bool KQ = AK != A_BF16;
  static_assert(KQ || NSA == NSB, "bf16 A shares the B stage index");
  static_assert(!KQ || NPROD == 4 * TM, "the K-quant producers take one 16-value sub-block each");
  constexpr int NPW = NPROD / 32;       // producer warps
  constexpr int NLW = loader_warps<AK>();  // raw loader warps
  extern __shared__ __align__(1024) uint8_t raw_smem[];
  uint8_t* sm = raw_smem + ((1024u - (smem_u32(raw_smem) & 1023u)) & 1023u);
  GemmCtl<NSA, NSB, RAWN>& C = *reinterpret_cast<GemmCtl<NSA, NSB, RAWN>*>(sm + PL::CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int W_LOAD = NPW, W_TMA = NPW + NLW, W_MMA = NPW + NLW + 1;
  auto B = [](unsigned long long& b) { return reinterpret_cast<uint64_t*>(&b); };

  // ---- the tile of this block (block-uniform)
  int mt, col0, ncol;
  const uint8_t *A0 = nullptr, *A1 = nullptr;
  if (g.tiles) {
    if ((int)blockIdx.x >= __ldg(g.n_tiles)) return;
    const int4 t = __ldg(g.tiles + blockIdx.x);
    const int e = t.x;
    mt = t.y;
    const int lo = __ldg(g.offsets + e), hi = __ldg(g.offsets + e + 1);
    col0 = lo + t.z * TNM;
    ncol = min(TNM, hi - col0);
    if (e == g.pseudo) {
      A0 = g.a0;
      A1 = g.a1;
    } else if (KQ) {
      A0 = reinterpret_cast<const uint8_t*>(__ldg(g.eptr + (size_t)e * 3 + g.pj0));
      if (NMAT == 2) A1 = reinterpret_cast<const uint8_t*>(__ldg(g.eptr + (size_t)e * 3 + g.pj1));
    }
  } else {
    mt = (int)blockIdx.x % g.mt_count;
    col0 = ((int)blockIdx.x / g.mt_count) * TNM;
    ncol = min(TNM, g.cols - col0);
    A0 = g.a0;
    A1 = g.a1;
  }
  if (ncol <= 0) return;
  const int TN = (ncol + 15) & ~15;  // MMA width: a multiple of 16, <= TNM
  // Split K-quant tiles whose four accumulators fit the 256 accumulator
  // columns stack B_lo right after B_hi in the B stage: A_hi * [B_hi; B_lo]
  // is then one MMA of width 2 TN (columns [0, TN) hi * hi, [TN, 2 TN)
  // hi * lo), followed by A_lo * B_hi (width TN) onto columns [0, TN); the
  // epilogue adds the two halves.  Two MMA instructions per matrix and K step
  // instead of three.
  const bool stack = SPLIT && PL::ATMEM && NMAT * 2 * TN <= 256;
  const int mcols = stack ? 2 * TN : TN;  // accumulator columns of one matrix
  uint32_t ncols_tmem = 32;
  while (ncols_tmem < (uint32_t)(NMAT * TN)) ncols_tmem <<= 1;
  if (PL::ATMEM) ncols_tmem = 512;
  const int row0 = mt * TM;
  const int nk = g.K / KC;
  const uint64_t deadline = globaltimer_ns() + g.timeout_ns;

  if (tid == 0) {
    for (int s = 0; s < NSA; ++s) {
      mbar_init(B(C.full_a[s]), AK == A_Q2K ? NPROD / 2 : NPROD);  // Q2_K: half the producers fill a chunk
      mbar_init(B(C.empty_a[s]), 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(B(C.full_b[s]), 1);
      mbar_init(B(C.empty_b[s]), 1);
    }
    mbar_init(B(C.acc), 1);
    if constexpr (KQ) {
      for (int b = 0; b < RAWN; ++b) {
        mbar_init(B(C.raw_full[b]), NLW * 32);
        mbar_init(B(C.raw_free[b]), NPROD);
      }
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&C.tmem, ncols_tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;

  if (warp < NPW) {
    // ------------------------------------------------------ producers
    const int r = tid & (TM - 1), qd = tid >> 7;  // A row; sub-block u = qd & 1 of plane half jj = qd >> 1
    const int jj = qd >> 1, u = qd & 1;
    bool ok = true;
    if constexpr (KQ) {
      const bool row_ok = row0 + r < g.a_rows;
      const uint8_t* Am[2] = {A0, A1};
      const uint32_t raw_base = smem_u32(sm);
      const int nunits = nk / 2;  // two K chunks per unit (half a Q2_K block)
      // this thread's 8 TMEM columns of A stage sa, matrix m, part pt: the
      // 16 K values 32 jj + 16 u .. + 15 of its row (lane = row)
      const uint32_t ta_lane = tmem + 256u + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(16 * jj + 8 * u);
      auto ta_addr = [&](int sa, int m, int pt) -> uint32_t {
        return ta_lane + (uint32_t)(sa * PL::TA_COLS + (m * PL::NPART + pt) * 32);
      };
      // Q2_K: producer half qd >> 1 fills chunk qd >> 1 of every unit, both
      // plane halves jb of its sub-block position u (one tensor-memory wait
      // and one hand-over per unit instead of two): its columns 16 jb + 8 u
      const uint32_t ta_lane_u = tmem + 256u + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(8 * u);
      auto ta_addr_q2 = [&](int sa, int m, int pt, int jb) -> uint32_t {
        return ta_lane_u + (uint32_t)(16 * jb + sa * PL::TA_COLS + (m * PL::NPART + pt) * 32);
      };
      // one K chunk: wait for the A stage, store this thread's piece, hand over
      auto chunk = [&](int kc, auto&& fillA) -> bool {
        const int sa = kc % NSA;
        if (kc >= NSA && !mbar_wait_bounded(B(C.empty_a[sa]), (uint32_t)((kc / NSA - 1) & 1), deadline, g.status))
          return false;
        tc_fence_after();
        if (row_ok) {
          fillA(sa);
        } else {
          const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int pt = 0; pt < PL::NPART; ++pt) {
              if constexpr (AK == A_Q2K) {
                tmem_st8(ta_addr_q2(sa, m, pt, 0), z);
                tmem_st8(ta_addr_q2(sa, m, pt, 1), z);
              } else {
                tmem_st8(ta_addr(sa, m, pt), z);
              }
            }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(B(C.full_a[sa]));
        return true;
      };
      for (int v = 0; v < nunits && ok; ++v) {
        const int buf = v % RAWN;
        if (!mbar_wait_bounded(B(C.raw_full[buf]), (uint32_t)((v / RAWN) & 1), deadline, g.status)) {
          ok = false;
          break;
        }
        const uint32_t* rw[2];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) rw[m] = reinterpret_cast<const uint32_t*>(sm + PL::raw_off(m, buf)) + r * RG::PITCH;
        if constexpr (AK == A_Q2K) {
          // half h of super-block v / 2: chunks 2v, 2v + 1 (parts 2h, 2h + 1)
          uint32_t qs[NMAT][4], sc[NMAT][2], dd[NMAT];
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
#pragma unroll
            for (int i = 0; i < 4; ++i) qs[m][i] = rw[m][(4 * u + i)];
            sc[m][0] = rw[m][8];
            sc[m][1] = rw[m][9];
            dd[m] = rw[m][10];
          }
          {
            const int cp = jj;  // this thread's chunk of the unit (the producer half)
            ok = chunk(2 * v + cp, [&](int sa) {
#pragma unroll
              for (int m = 0; m < NMAT; ++m) {
                const float d = half_bits_to_float(dd[m]), dmin = half_bits_to_float(dd[m] >> 16);
#pragma unroll
                for (int jb = 0; jb < 2; ++jb) {
                  const int j = 2 * cp + jb;  // 2-bit plane
                  const int sbi = 2 * j + u;  // sub-block 8h + sbi: scale byte sbi of the half
                  const uint32_t byte = (sc[m][sbi >> 2] >> (8 * (sbi & 3))) & 0xFFu;
                  uint32_t th0, th1, tl0 = 0, tl1 = 0;
                  q2k_tables<SPLIT>(d, dmin, byte, th0, th1, tl0, tl1);
                  uint32_t oh[8], ol[8];  // values l = 16u .. 16u + 15 in pairs: qs words 0..3 of the sub-block
#pragma unroll
                  for (int f = 0; f < 4; ++f) {
                    const uint32_t qq = (qs[m][f] >> (2 * j)) & 0x03030303u;
                    const uint32_t s0 = pair_sels(qq), s1 = s0 >> 16;
                    oh[2 * f] = prmt(th0, th1, s0);
                    oh[2 * f + 1] = prmt(th0, th1, s1);
                    if (SPLIT) {
                      ol[2 * f] = prmt(tl0, tl1, s0);
                      ol[2 * f + 1] = prmt(tl0, tl1, s1);
                    }
                  }
                  tmem_st8(ta_addr_q2(sa, m, 0, jb), oh);
                  if (SPLIT) tmem_st8(ta_addr_q2(sa, m, SPLIT ? 1 : 0, jb), ol);
                }
              }
            });
          }
        }
        // raw buffer `buf` is free once every producer has read it
        mbar_arrive(B(C.raw_free[buf]));
      }
    }
    // ------------------------------------------------------- epilogue
    // The MMA thread always commits the accumulator barrier (after its last
    // issued MMA), so a second bounded wait after a timeout still ends with
    // no MMA in flight before the tensor memory is read or freed.
    if (lane == 0 && !mbar_wait_bounded(B(C.acc), 0u, deadline, g.status))
      mbar_wait_bounded(B(C.acc), 0u, globaltimer_ns() + g.timeout_ns, g.status);
    __syncwarp();
    tc_fence_after();
    constexpr int CG = NPROD / 128;         // warps per TMEM lane group
    const int lg = warp & 3, cg = warp >> 2;
    const int rw = row0 + lg * 32 + lane;   // the output row of this lane
    const uint32_t tl = tmem + ((uint32_t)(lg * 32) << 16);
    for (int c0 = 16 * cg; c0 < TN; c0 += 16 * CG) {
      float v0[16], v1[16];
      tmem_ld16(tl + (uint32_t)c0, v0);
      if (NMAT == 2) tmem_ld16(tl + (uint32_t)(mcols + c0), v1);
      if (stack) {
        float w[16];
        tmem_ld16(tl + (uint32_t)(TN + c0), w);
#pragma unroll
        for (int j = 0; j < 16; ++j) v0[j] += w[j];
        if (NMAT == 2) {
          tmem_ld16(tl + (uint32_t)(mcols + TN + c0), w);
#pragma unroll
          for (int j = 0; j < 16; ++j) v1[j] += w[j];
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = c0 + j;
        if (col >= ncol) break;  // warp-uniform
        if constexpr (EPI == E_F32) {
          if (rw < g.a_rows) g.out_f32[(size_t)(col0 + col) * g.out_ld + rw] = v0[j];
        } else {
          const float hv = swiglu_f32(v0[j], v1[j], g.swiglu_limit);
          if constexpr (EPI == E_SWIGLU_Q8) {
            uint16_t hi, lo;
            q8_hilo_warp(hv, hi, lo);  // the warp's 32 rows: one q8_1 block
            g.out_h[(size_t)(col0 + col) * g.out_ld + rw] = hi;
            g.out_h2[(size_t)(col0 + col) * g.out_ld + rw] = lo;
          } else {
            g.out_h[(size_t)(col0 + col) * g.out_ld + rw] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
          }
        }
      }
    }
  } else if (KQ && warp >= W_LOAD && warp < W_LOAD + NLW) {
    // ---------------------------------------------------- raw loaders
    if constexpr (KQ) {
      // Word i of a buffer (row i / words, word i % words) goes to loader
      // thread i % NLT, so each thread copies the same (row, word) pairs of
      // every unit: their source offsets from the unit's first row are worked
      // out once, and a copy costs an add, a compare and the cp.async.
      constexpr int NLT = NLW * 32;
      constexpr int WORDS = RG::words();
      static_assert(TM * WORDS % NLT == 0, "loader threads tile the buffer");
      const int t = tid - W_LOAD * 32;
      const uint8_t* Am[2] = {A0, A1};
      const uint32_t raw_base = smem_u32(sm);
      const int nunits = nk / 2;
      const int lim = max(0, min(TM, g.a_rows - row0)) * WORDS;  // words of rows that exist
      const size_t rb = g.a_row_bytes;
      if constexpr (AK == A_Q2K) {
        // buffer word w of a row: qs words 4 + 8h .. 4 + 8h + 7 of the
        // super-block (w < 8), scale words 2h, 2h + 1 (w = 8, 9), d/dmin (w = 10)
        constexpr int NJ = TM * WORDS / NLT;
        uint32_t o0[NJ], o1[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int i = t + NLT * j, rr = i / WORDS, w = i - rr * WORDS;
          const int b0 = w < 8 ? 4 + w : (w < 10 ? w - 8 : 20), dh = w < 8 ? 8 : (w < 10 ? 2 : 0);
          o0[j] = (uint32_t)(rr * rb) + 4u * (uint32_t)b0;
          o1[j] = o0[j] + 4u * (uint32_t)dh;
        }
        for (int v = 0; v < nunits; ++v) {
          const int buf = v % RAWN;
          if (v >= RAWN && !mbar_wait_bounded(B(C.raw_free[buf]), (uint32_t)((v / RAWN - 1) & 1), deadline, g.status))
            break;
          const bool hi = v & 1;
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const uint8_t* u = Am[m] + (size_t)row0 * rb + (size_t)(v >> 1) * Q2K_B;
            const uint32_t dst = raw_base + PL::raw_off(m, buf) + 4u * (uint32_t)t;
#pragma unroll
            for (int j = 0; j < NJ; ++j)
              if (t + NLT * j < lim) cp_async4(dst + 4u * (uint32_t)(NLT * j), u + (hi ? o1[j] : o0[j]));
          }
          cp_async_arrive(B(C.raw_full[buf]));  // once this thread's copies have landed
        }
      }
      // copies still in flight land before the block can exit
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp == W_TMA && lane == 0) {
    // ------------------------------------------------------- TMA issuer
    const bool boxed = g.tiles != nullptr;  // expert jobs: B_BOX-row boxes up to TN rows
    const uint32_t bbytes = (uint32_t)(boxed ? TN : TNM) * 128u;
    const uint32_t bytes = (KQ ? 0u : NMAT * A_TILE) + PL::NPART * bbytes;
    for (int kc = 0; kc < nk; ++kc) {
      const int sb = kc % NSB;
      if (kc >= NSB && !mbar_wait_bounded(B(C.empty_b[sb]), (uint32_t)((kc / NSB - 1) & 1), deadline, g.status)) break;
      uint64_t* fb = B(C.full_b[sb]);
      mbar_arrive_expect_tx(fb, bytes);
      if constexpr (!KQ) {
#pragma unroll
        for (int mat = 0; mat < NMAT; ++mat)
          tma_load_2d(smem_u32(sm + PL::a_off(sb, mat, 0)), &g.map_a[mat], kc * KC, row0, fb);
      }
#pragma unroll
      for (int pt = 0; pt < PL::NPART; ++pt) {
        const uint32_t dst = stack && pt == 1 ? smem_u32(sm + PL::b_off(sb, 0)) + (uint32_t)TN * 128u
                                              : smem_u32(sm + PL::b_off(sb, pt));
        if (boxed) {
          for (int i = 0; i < TN; i += B_BOX) tma_load_2d(dst + (uint32_t)i * 128u, &g.map_b[pt], kc * KC, col0 + i, fb);
        } else {
          tma_load_2d(dst, &g.map_b[pt], kc * KC, col0, fb);
        }
      }
    }
  } else if (warp == W_MMA && lane == 0) {
    // ----------------------------------------------------- MMA issuer
    const uint32_t idesc = umma_idesc(TN, AK == A_BF16);
    const uint32_t idesc2 = umma_idesc(2 * TN, AK == A_BF16);  // stacked: only when 2 TN <= 128
    for (int kc = 0; kc < nk; ++kc) {
      const int sb = kc % NSB, sa = KQ ? kc % NSA : sb;
      if (!mbar_wait_bounded(B(C.full_b[sb]), (uint32_t)((kc / NSB) & 1), deadline, g.status)) break;
      if (KQ && !mbar_wait_bounded(B(C.full_a[sa]), (uint32_t)((kc / NSA) & 1), deadline, g.status)) break;
      tc_fence_after();
      const uint32_t base = smem_u32(sm);
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        const uint32_t td = tmem + (uint32_t)(mat * mcols);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bh = umma_desc(base + PL::b_off(sb, 0) + 32u * k);
          if constexpr (PL::ATMEM) {
            // A in tensor memory: 8 columns (16 K values) per MMA
            const uint32_t ta = tmem + 256u + (uint32_t)(sa * PL::TA_COLS + (mat * PL::NPART) * 32 + 8 * k);
            if (stack) {
              umma_f16_ta(td, ta, bh, idesc2, (kc | k) ? 1u : 0u);  // A_hi * [B_hi; B_lo]
              umma_f16_ta(td, ta + 32u, bh, idesc, 1u);            // A_lo * B_hi
              continue;
            }
            umma_f16_ta(td, ta, bh, idesc, (kc | k) ? 1u : 0u);
            if (SPLIT) {
              umma_f16_ta(td, ta, umma_desc(base + PL::b_off(sb, SPLIT ? 1 : 0) + 32u * k), idesc, 1u);
              umma_f16_ta(td, ta + 32u, bh, idesc, 1u);
            }
          } else {
            const uint64_t ah = umma_desc(base + PL::a_off(sa, mat, 0) + 32u * k);
            umma_f16(td, ah, bh, idesc, (kc | k) ? 1u : 0u);
            if (SPLIT) {
              umma_f16(td, ah, umma_desc(base + PL::b_off(sb, SPLIT ? 1 : 0) + 32u * k), idesc, 1u);
              umma_f16(td, umma_desc(base + PL::a_off(sa, mat, SPLIT ? 1 : 0) + 32u * k), bh, idesc, 1u);
            }
          }
        }
      }
      umma_commit(B(C.empty_b[sb]));
      if (KQ) umma_commit(B(C.empty_a[sa]));
    }
    umma_commit(B(C.acc));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols_tmem);
  }
}

template <int AK, int NMAT, bool SPLIT, int EPI, int TNM, int NSA, int NSB, int RAWN, int NPROD>
int launch_gemm(const GemmArgs& g, unsigned grid, cudaStream_t s) {
  constexpr size_t smem = Plan<AK, NMAT, SPLIT, TNM, NSA, NSB, RAWN>::SMEM;
  static_assert(smem <= 232448, "GEMM stages exceed the shared memory of a block");
  auto kern = k_gemm<AK, NMAT, SPLIT, EPI, TNM, NSA, NSB, RAWN, NPROD>;
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_dev = dev;
  }
  if (grid == 0) return MOE_OK;
  kern<<<grid, NPROD + 32 * loader_warps<AK>() + 64, smem, s>>>(g);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

constexpr int NP_KQ = 512;   // K-quant GEMMs: 16 dequantising warps
constexpr int NP_BF = 128;   // bf16 GEMMs: 4 epilogue warps

int route_steps(const PrefillParams& p, cudaStream_t s) {
  GemmArgs g{};
  if (!make_map_b16(&g.map_a[0], p.router_w, p.D, p.N, TM) || !make_map_b16(&g.map_b[0], p.x, p.D, p.m, PF_TN))
    return MOE_ERR_CUDA;
  g.K = p.D; g.a_rows = p.N; g.pseudo = -1; g.cols = p.m; g.mt_count = (p.N + TM - 1) / TM;
  g.out_f32 = p.logits; g.out_ld = p.N; g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
  const unsigned grid = (unsigned)(g.mt_count * ((p.m + PF_TN - 1) / PF_TN));
  int rc = launch_gemm<A_BF16, 1, false, E_F32, PF_TN, 4, 4, 1, NP_BF>(g, grid, s);
  if (rc) return rc;
  SelectParams sp{};
  sp.logits = p.logits; sp.bias = p.bias; sp.bias_vl = p.bias_vl; sp.image_mask = p.image_mask;
  sp.m = p.m; sp.N = p.N; sp.k = p.k; sp.norm = p.norm; sp.score_func = p.score_func;
  sp.gate_temp = p.gate_temp; sp.route_scale = p.route_scale; sp.topk_w = p.topk_w; sp.topk_idx = p.topk_idx;
  sp.ctrl = p.ctrl;
  return launch_select(sp, s);
}

}  // namespace

bool make_map_b16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || rows == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_prefill_route(const PrefillParams& p, cudaStream_t s) { return route_steps(p, s); }

int launch_prefill(const PrefillParams& p, cudaStream_t s) {
  const PrefillLayout& L = p.L;
  uint8_t* pw = p.pw;
  const int m = p.m, D = p.D, I = p.I, N = p.N, k = p.k;
  const int shq = p.shared_kind == MOE_SHARED_KQUANT;
  const int NE = N + 1;
  const int nch = (m + PF_GCH - 1) / PF_GCH;
  const int V = m * k + (shq ? m : 0);  // pair rows (the K-quant shared expert's tokens included)
  int rc;
  uint16_t* xgh = reinterpret_cast<uint16_t*>(pw + L.xgh);
  uint16_t* xgl = reinterpret_cast<uint16_t*>(pw + L.xgl);
  int* chunk = reinterpret_cast<int*>(pw + L.chunk);
  int* offsets = reinterpret_cast<int*>(pw + L.offsets);
  int* expert_ok = reinterpret_cast<int*>(pw + L.expert_ok);
  int* pair_tok = reinterpret_cast<int*>(pw + L.pair_tok);
  float* pair_w = reinterpret_cast<float*>(pw + L.pair_w);
  int* pos_of = reinterpret_cast<int*>(pw + L.pos_of);
  int* pos_sh = reinterpret_cast<int*>(pw + L.pos_sh);
  int* n_tiles = reinterpret_cast<int*>(pw + L.n_tiles);
  int4* gu_tiles = reinterpret_cast<int4*>(pw + L.gu_tiles);
  int4* dn_tiles = reinterpret_cast<int4*>(pw + L.dn_tiles);
  uint16_t* hh = reinterpret_cast<uint16_t*>(pw + L.hh);
  uint16_t* hl = reinterpret_cast<uint16_t*>(pw + L.hl);
  float* ep = reinterpret_cast<float*>(pw + L.ep);
  uint16_t* hs = reinterpret_cast<uint16_t*>(pw + L.hs);
  float* sp = reinterpret_cast<float*>(pw + L.sp);

  // 1-2. router logits and selection
  if ((rc = route_steps(p, s))) return rc;
  // 3. grouping
  k_group_hist<<<nch, 256, NE * sizeof(int), s>>>(p.topk_idx, m, k, N, shq, chunk);
  k_group_scan<<<1, 1024, 0, s>>>(chunk, nch, N, p.expert_ptrs, I / TM, D / TM, (size_t)TM * (I / QK) * Q3K_B,
                                  p.sh2, offsets, expert_ok, gu_tiles, dn_tiles, n_tiles, &p.ctrl->status);
  k_group_scatter<<<nch, 256, 0, s>>>(p.topk_idx, p.topk_w, m, k, N, shq, chunk, pair_tok, pair_w, pos_of, pos_sh);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 4. the q8_1 values of x as fp16 high and low parts, in pair order
  {
    const long nb = (long)m * (D / 32) * 4;
    long blocks = (nb + 255) / 256;
    if (blocks > 152L * 8) blocks = 152L * 8;
    k_xg<<<(unsigned)blocks, 256, 0, s>>>(p.x, m, D, k, pos_of, shq ? pos_sh : nullptr, xgh, xgl);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  // 5. gate/up of the routed experts (and of a K-quant shared expert) -> q8_1(h) as fp16 hi + lo
  {
    GemmArgs g{};
    if (!make_map_b16(&g.map_b[0], xgh, D, V, B_BOX) || !make_map_b16(&g.map_b[1], xgl, D, V, B_BOX))
      return MOE_ERR_CUDA;
    g.K = D; g.a_rows = I; g.a_row_bytes = (D / QK) * Q2K_B; g.eptr = p.expert_ptrs; g.pj0 = 0; g.pj1 = 1;
    g.pseudo = shq ? N : -1; g.a0 = p.sh1; g.a1 = p.sh3;
    g.tiles = gu_tiles; g.n_tiles = n_tiles; g.offsets = offsets; g.out_h = hh; g.out_h2 = hl; g.out_ld = I;
    g.swiglu_limit = p.swiglu_limit; g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
    const unsigned grid = (unsigned)L.max_gu_tiles * (unsigned)(I / TM);
    if ((rc = launch_gemm<A_Q2K, 2, true, E_SWIGLU_Q8, PF_TN_GU, 2, 3, 3, NP_KQ>(g, grid, s))) return rc;
  }
  // 6. down -> E per pair (exact products, k_prefill_kq.cu)
  {
    KqLaunch q{};
    q.bh = hh; q.bl = hl; q.b_rows = V; q.tiles = dn_tiles; q.n_tiles = n_tiles + 1;
    q.K = I; q.a_row_bytes = (I / QK) * Q3K_B; q.out_ld = D; q.out_e = ep;
    q.status = &p.ctrl->status; q.timeout_ns = p.timeout_ns;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    q.grid = (unsigned)sms;
    if ((rc = launch_kq_gemm(q, s))) return rc;
  }
  // 7. the bf16 shared expert
  if (!shq) {
    const unsigned ntok = (unsigned)((m + PF_TN - 1) / PF_TN);
    GemmArgs g{};
    if (!make_map_b16(&g.map_a[0], p.sh1, D, I, TM) || !make_map_b16(&g.map_a[1], p.sh3, D, I, TM) ||
        !make_map_b16(&g.map_b[0], p.x, D, m, PF_TN))
      return MOE_ERR_CUDA;
    g.K = D; g.a_rows = I; g.pseudo = -1; g.cols = m;
    g.mt_count = I / TM; g.out_h = hs; g.out_ld = I; g.swiglu_limit = p.swiglu_limit;
    g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
    if ((rc = launch_gemm<A_BF16, 2, false, E_SWIGLU_BF16, PF_TN, 3, 3, 1, NP_BF>(g, (unsigned)g.mt_count * ntok,
                                                                                      s)))
      return rc;
    GemmArgs d{};
    if (!make_map_b16(&d.map_a[0], p.sh2, I, D, TM) || !make_map_b16(&d.map_b[0], hs, I, m, PF_TN)) return MOE_ERR_CUDA;
    d.K = I; d.a_rows = D; d.pseudo = -1; d.cols = m;
    d.mt_count = D / TM; d.out_f32 = sp; d.out_ld = D; d.status = &p.ctrl->status; d.timeout_ns = p.timeout_ns;
    if ((rc = launch_gemm<A_BF16, 1, false, E_F32, PF_TN, 4, 4, 1, NP_BF>(d, (unsigned)d.mt_count * ntok, s)))
      return rc;
  }
  // 8. ordered combine
  if ((reinterpret_cast<uintptr_t>(p.out) & 15u) == 0)
    k_combine<float4><<<m, 256, 0, s>>>(p.topk_idx, pos_of, expert_ok, pair_w, ep, sp, shq ? pos_sh : nullptr, k, D,
                                        p.out);
  else
    k_combine<float><<<m, 256, 0, s>>>(p.topk_idx, pos_of, expert_ok, pair_w, ep, sp, shq ? pos_sh : nullptr, k, D,
                                       p.out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// kernel launches of one prefill call
int prefill_launches(int shared_kind) { return shared_kind == MOE_SHARED_KQUANT ? 9 : 11; }

}  // namespace moe
