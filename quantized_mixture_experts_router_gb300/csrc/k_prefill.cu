// Prefill path (any m; taken by default above eight tokens): the expert
// projections as GEMMs on the 5th-generation tensor cores.
//
//   x16     the q8_1 activation values fp16(d) * q (the values the method's
//           integer dots stand for) as a high and a low fp16 part, exact
//   router  logits = x W_R^T (bf16 tensor-core GEMM, f32 accumulation), then
//           the selection per token
//   group   (expert, token) pairs ordered by expert id, tokens ascending
//           within an expert: the per-expert token lists of DeepSeek V4.1
//           atlas "Mixture of experts" (model.py MoE.forward), made
//           deterministic by a counting sort over token chunks
//   gate/up per (expert, 128 rows, <= 128 pairs) tile: W1 and W3 rows
//           dequantised from Q2_K, split into high and low fp16 parts, times
//           the pairs' x16 rows (three products: hi.hi + hi.lo + lo.hi, about
//           2^-22 relative); the epilogue applies the clipped SwiGLU,
//           quantises h to q8_1 and stores fp16 of its values.  The split is
//           needed because q8_1(h) turns any error in h near a rounding
//           boundary into a whole quantisation step.
//   down    W2 rows dequantised from Q3_K to fp16 times those h rows (one
//           product; its rounding enters the output linearly) -> E per pair
//   shared  bf16 shared expert: two bf16 GEMMs, h rounded to bf16 between them;
//           a K-quant shared expert is one more expert taken by every token
//   combine out = sum over the token's experts in ascending id of G_i E_i,
//           then the shared expert's output added last
//
// GEMM block (128 weight rows x up to 128 or 256 columns): eight producer
// warps fill a ring of 128-byte-swizzled K-major tiles (dequantising K-quant
// blocks on the way, two threads per weight row), one thread issues
// tcgen05.mma (M = 128, N = tile width, K = 16) into a tensor-memory
// accumulator and commits each stage back to the producers, and the same
// eight warps then read the accumulator for the epilogue.  Products
// accumulate in f32; bf16 operands (router, bf16 shared expert) are the
// caller's values, exact.
#include "internal.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int TM = PF_TM;
constexpr int KC = PF_KC;
constexpr int NPROD = 256;   // producer / epilogue threads (8 warps); one more warp issues the MMAs
constexpr int GTHREADS = NPROD + 32;

enum : int { A_BF16 = 0, A_Q2K = 1, A_Q3K = 2 };
enum : int { E_F32 = 0, E_SWIGLU_Q8 = 1, E_SWIGLU_BF16 = 2 };

__device__ __forceinline__ uint32_t f2h(float v) { return (uint32_t)__half_as_ushort(__float2half_rn(v)); }

// ------------------------------------------------------------------ prep
// The q8_1 values of x, fp16(d) * q (exact in f32), as fp16 high and low
// parts; one thread per block of 32 (the q8_1 rule: d = amax / 127,
// q = round-half-away(v / d), d stored as fp16).
__global__ void k_x16(const uint16_t* __restrict__ x, int m, int D, uint16_t* __restrict__ x16h,
                      uint16_t* __restrict__ x16l) {
  const long nb = (long)m * (D / 32);
  for (long g = blockIdx.x * (long)blockDim.x + threadIdx.x; g < nb; g += (long)gridDim.x * blockDim.x) {
    const uint4* xp = reinterpret_cast<const uint4*>(x + g * 32);
    uint32_t raw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(xp + i);
      raw[4 * i + 0] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(raw[i])), fabsf(bf16hi(raw[i]))));
    const float d = __fdiv_rn(amax, 127.0f);
    const float rd = __frcp_rn(d);
    const float dq = __half2float(__float2half_rn(d));
    uint32_t oh[16], ol[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q0 = amax == 0.0f ? 0 : q8_code(bf16lo(raw[i]), d, rd);
      const int q1 = amax == 0.0f ? 0 : q8_code(bf16hi(raw[i]), d, rd);
      const float v0 = dq * (float)q0, v1 = dq * (float)q1;
      const __half2 hh = __floats2half2_rn(v0, v1);
      const float2 back = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v0 - back.x, v1 - back.y);
      oh[i] = *reinterpret_cast<const uint32_t*>(&hh);
      ol[i] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    uint4* ph = reinterpret_cast<uint4*>(x16h + g * 32);
    uint4* pl = reinterpret_cast<uint4*>(x16l + g * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ph[i] = make_uint4(oh[4 * i], oh[4 * i + 1], oh[4 * i + 2], oh[4 * i + 3]);
      pl[i] = make_uint4(ol[4 * i], ol[4 * i + 1], ol[4 * i + 2], ol[4 * i + 3]);
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
__global__ void __launch_bounds__(1024) k_group_scan(int* __restrict__ chunk, int nch, int N,
                                                     const unsigned long long* __restrict__ eptr, int gu_mt,
                                                     int dn_mt, int* __restrict__ offsets, int* __restrict__ expert_ok,
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
      nd[j] = ok[j] ? (cnt[j] + PF_TN - 1) / PF_TN : 0;
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
      for (int t = 0; t < nd[j]; ++t)
        for (int mt = 0; mt < dn_mt; ++mt) dn_tiles[(size_t)(dof + t) * dn_mt + mt] = make_int4(e, mt, t, 0);
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
// out[t] = sum over t's usable pairs in ascending expert id of G * E, then
// the shared expert's output
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
  const float* sh = pos_sh ? ep + (size_t)pos_sh[t] * D : sp + (size_t)t * D;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < n; ++i) acc = fmaf(s_w[i], ep[(size_t)s_pos[i] * D + d], acc);
    out[(size_t)t * D + d] = acc + sh[d];
  }
}

// ------------------------------------------------------------------ GEMM
struct GemmArgs {
  int K;                               // contraction length, a multiple of 64
  int a_rows;                          // rows of A (the M extent)
  int a_row_bytes;                     // bytes per A row
  const uint8_t* a0;                   // A matrices of a plain job, or of the pseudo-expert
  const uint8_t* a1;
  const unsigned long long* eptr;      // expert jobs: the [N][3] pointer table
  int pj0, pj1;                        // pointer-table columns of the job's matrices
  int pseudo;                          // expert whose matrices are a0 / a1 (-1: none)
  const uint16_t* b;                   // B rows of K values (the high parts when split)
  const uint16_t* b_lo;                // split B: the low parts
  const int* b_rows;                   // B row of each column, or null: the column itself
  int cols;                            // plain jobs: number of columns
  const int4* tiles;                   // expert jobs: (e, mt, nt) per block
  const int* n_tiles;
  const int* offsets;                  // expert jobs: column range of each expert
  int mt_count;                        // plain jobs: M tiles
  float* out_f32;                      // E_F32: out[col * ld + row]
  uint16_t* out_h;                     // E_SWIGLU_*: h[col * ld + row]
  int out_ld;
  float swiglu_limit;
  unsigned* status;
  unsigned long long timeout_ns;
};

constexpr uint32_t A_TILE = TM * 128;  // bytes of one A tile (128 rows x 64 values)

template <int NS>
struct GemmCtl {
  unsigned long long full[NS], empty[NS], acc;
  uint32_t tmem;
};

// Shared-memory plan of one GEMM variant: per stage NMAT A tiles (times two
// when split into high and low fp16 parts), then one B tile (two when split)
// of TNM rows.
template <int NMAT, bool SPLIT, int TNM, int NS>
struct Plan {
  static constexpr int NPART = SPLIT ? 2 : 1;
  static constexpr uint32_t B_TILE = TNM * 128;
  static constexpr uint32_t STAGE = NMAT * NPART * A_TILE + NPART * B_TILE;
  static constexpr size_t SMEM = 1024 + (size_t)NS * STAGE + sizeof(GemmCtl<NS>);
  static __device__ __forceinline__ uint32_t a_off(int mat, int part) { return (mat * NPART + part) * A_TILE; }
  static __device__ __forceinline__ uint32_t b_off(int part) { return NMAT * NPART * A_TILE + part * B_TILE; }
};

// 32-bit word at a 2-byte aligned address p, from the two aligned words
// around it (reads the 8 bytes [p & ~3, (p & ~3) + 8))
__device__ __forceinline__ uint32_t ldg_u32_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  return __funnelshift_r(__ldg(base), __ldg(base + 1), (uint32_t)(a & 3u) * 8u);
}

// the same from two 16-bit loads (reads exactly [p, p + 4))
__device__ __forceinline__ uint32_t ldg_u32_a2_exact(const uint8_t* p) {
  const unsigned short* h = reinterpret_cast<const unsigned short*>(p);
  return (uint32_t)__ldg(h) | ((uint32_t)__ldg(h + 1) << 16);
}

// eight f32 values as fp16 into a 16-byte tile chunk; when split, the
// residual v - fp16(v) as fp16 into the same chunk of the low tile
template <bool SPLIT>
__device__ __forceinline__ void emit8(const float* v, uint8_t* hi, uint8_t* lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2 hh = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
    h[e] = *reinterpret_cast<const uint32_t*>(&hh);
    if constexpr (SPLIT) {
      const float2 back = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v[2 * e] - back.x, v[2 * e + 1] - back.y);
      l[e] = *reinterpret_cast<const uint32_t*>(&ll);
    }
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  if constexpr (SPLIT) *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Half hf (K values 32 hf .. 32 hf + 31) of chunk kc of one A row into row r
// of the swizzled tile(s): 16-byte chunks 4 hf .. 4 hf + 3.
template <int AK, bool SPLIT>
__device__ __forceinline__ void produce_a(const uint8_t* row, int kc, int hf, uint8_t* hi, uint8_t* lo, int r) {
  if constexpr (AK == A_BF16) {
    const uint4* src = reinterpret_cast<const uint4*>(row + (size_t)kc * 128) + 4 * hf;
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(hi + swz(r, 4 * hf + c)) = __ldg(src + c);
  } else if constexpr (AK == A_Q2K) {
    // GGUF Q2_K super-block: scales[16] (low nibble scale, high nibble min),
    // qs[64] (2-bit planes), fp16 d, dmin.  Element 128h + 32j + l (l < 32)
    // is bits 2j of qs[32h + l], in sub-block 8h + 2j + (l >= 16):
    // d * sc * q - dmin * mn.  Chunk kc is quarter (kc & 3) of super-block
    // kc / 4: half h = (kc & 3) / 2, planes j0 = 2 (kc & 1) and j0 + 1; this
    // thread's half of it is plane j = j0 + hf.
    const uint8_t* blk = row + (size_t)(kc >> 2) * Q2K_B;
    const int part = kc & 3, h = part >> 1, j0 = 2 * (part & 1), j = j0 + hf;
    const uint32_t* bw = reinterpret_cast<const uint32_t*>(blk);
    uint32_t qs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[i] = __ldg(bw + 4 + 8 * h + i);
    const uint32_t sc = __ldg(bw + 2 * h + (j0 >> 1));  // scale bytes of sub-blocks 8h + 2j0 .. + 3
    const uint32_t dd = __ldg(bw + 20);
    const float d = half_bits_to_float(dd), dmin = half_bits_to_float(dd >> 16);
    float am[2], bm[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // sub-blocks 8h + 2j + u
      const uint32_t byte = (sc >> (8 * (2 * hf + u))) & 0xFFu;
      am[u] = d * (float)(byte & 15u);
      bm[u] = dmin * (float)(byte >> 4);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // l = 8c .. 8c + 7
      const int u = c >> 1;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int l = 8 * c + e;
        const float q = (float)((qs[l >> 2] >> (8 * (l & 3) + 2 * j)) & 3u);
        v[e] = fmaf(am[u], q, -bm[u]);
      }
      emit8<SPLIT>(v, hi + swz(r, 4 * hf + c), lo + swz(r, 4 * hf + c));
    }
  } else {
    // GGUF Q3_K super-block (110 bytes, 2-byte aligned): hmask[32], qs[64],
    // scales[12] (sixteen 6-bit codes: low nibbles in bytes 0-7, high bit
    // pairs in bytes 8-11), fp16 d.  Element 128h + 32j + l is
    // (bits 2j of qs[32h + l]) + 4 * (bit 4h + j of hmask[l]) - 4, times
    // d * (code - 32) of sub-block 8h + 2j + (l >= 16).
    const uint8_t* blk = row + (size_t)(kc >> 2) * Q3K_B;
    const int part = kc & 3, h = part >> 1, j = 2 * (part & 1) + hf;
    uint32_t qs[8], hm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qs[i] = ldg_u32_a2(blk + 32 + 32 * h + 4 * i);
      hm[i] = ldg_u32_a2(blk + 4 * i);
    }
    const uint32_t s_lo = ldg_u32_a2(blk + 96 + 4 * (j >> 1));  // low-nibble bytes 2j, 2j + 1
    const uint32_t s_hi = ldg_u32_a2_exact(blk + 104);           // the block's last bytes: no read past it
    const float d = half_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(blk + 108)));
    float am[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int sb = 2 * j + u;  // sub-block index mod 8
      const uint32_t lo4 = (s_lo >> (8 * (sb & 3) + 4 * h)) & 15u;
      const uint32_t hi2 = (s_hi >> (8 * (sb & 3) + 2 * (2 * h + (j >> 1)))) & 3u;
      am[u] = d * (float)((int)(lo4 | (hi2 << 4)) - 32);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int u = c >> 1;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int l = 8 * c + e;
        const uint32_t q = (qs[l >> 2] >> (8 * (l & 3) + 2 * j)) & 3u;
        const uint32_t hb = (hm[l >> 2] >> (8 * (l & 3) + 4 * h + j)) & 1u;
        v[e] = am[u] * (float)((int)(q | (hb << 2)) - 4);
      }
      emit8<SPLIT>(v, hi + swz(r, 4 * hf + c), lo + swz(r, 4 * hf + c));
    }
  }
}

// q8_1 of one 32-value block of h held one value per lane: fp16 bits of
// fp16(d) * q for this lane's value
__device__ __forceinline__ uint16_t q8_h16_warp(float v) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = amax == 0.0f ? 0 : q8_code(v, d, __frcp_rn(d));
  const float dq = __half2float(__float2half_rn(d));
  return (uint16_t)f2h(dq * (float)q);
}

// One tile: D[128 rows, TN columns] (per matrix) = A . B^T over K.
// SPLIT: A = A_hi + A_lo and B = B_hi + B_lo in fp16, accumulating
// A_hi B_hi + A_hi B_lo + A_lo B_hi (the A_lo B_lo term is below 2^-22
// relative).
template <int AK, int NMAT, bool SPLIT, int EPI, int TNM, int NS>
__global__ void __launch_bounds__(GTHREADS, 1) k_gemm(const __grid_constant__ GemmArgs g) {
  using PL = Plan<NMAT, SPLIT, TNM, NS>;
  extern __shared__ __align__(1024) uint8_t raw_smem[];
  uint8_t* sm = raw_smem + ((1024u - (smem_u32(raw_smem) & 1023u)) & 1023u);
  GemmCtl<NS>& C = *reinterpret_cast<GemmCtl<NS>*>(sm + NS * PL::STAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the tile of this block (block-uniform)
  int mt, col0, ncol;
  const uint8_t *A0, *A1 = nullptr;
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
    } else {
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
  uint32_t ncols_tmem = 32;
  while (ncols_tmem < (uint32_t)(NMAT * TN)) ncols_tmem <<= 1;
  const int row0 = mt * TM;
  const int nk = g.K / KC;
  const uint64_t deadline = globaltimer_ns() + g.timeout_ns;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(reinterpret_cast<uint64_t*>(&C.full[s]), NPROD);
      mbar_init(reinterpret_cast<uint64_t*>(&C.empty[s]), 1);
    }
    mbar_init(reinterpret_cast<uint64_t*>(&C.acc), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&C.tmem, ncols_tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;

  if (warp < NPROD / 32) {
    // ------------------------------------------------------ producers
    const int r = tid & (TM - 1), hf = tid >> 7;  // A row, and which half of its 64 K values
    const bool row_ok = row0 + r < g.a_rows;
    const uint8_t* arow0 = A0 + (size_t)(row0 + r) * g.a_row_bytes;
    const uint8_t* arow1 = NMAT == 2 ? A1 + (size_t)(row0 + r) * g.a_row_bytes : nullptr;
    for (int kc = 0; kc < nk; ++kc) {
      const int s = kc % NS;
      if (kc >= NS && !mbar_wait_bounded(reinterpret_cast<uint64_t*>(&C.empty[s]), (uint32_t)((kc / NS - 1) & 1),
                                         deadline, g.status))
        break;
      uint8_t* st = sm + (size_t)s * PL::STAGE;
      if (row_ok) {
        produce_a<AK, SPLIT>(arow0, kc, hf, st + PL::a_off(0, 0), st + PL::a_off(0, SPLIT ? 1 : 0), r);
        if (NMAT == 2)
          produce_a<AK, SPLIT>(arow1, kc, hf, st + PL::a_off(1, 0), st + PL::a_off(1, SPLIT ? 1 : 0), r);
      } else {
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
          for (int pt = 0; pt < PL::NPART; ++pt)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(st + PL::a_off(m, pt) + swz(r, 4 * hf + c)) = make_uint4(0, 0, 0, 0);
      }
      for (int q = tid; q < TN * 8; q += NPROD) {
        const int col = q >> 3, c = q & 7;
        uint4 v = make_uint4(0, 0, 0, 0), vl = make_uint4(0, 0, 0, 0);
        if (col < ncol) {
          const int brow = g.b_rows ? __ldg(g.b_rows + col0 + col) : col0 + col;
          const size_t off = (size_t)brow * g.K + (size_t)kc * KC;
          v = __ldg(reinterpret_cast<const uint4*>(g.b + off) + c);
          if (SPLIT) vl = __ldg(reinterpret_cast<const uint4*>(g.b_lo + off) + c);
        }
        *reinterpret_cast<uint4*>(st + PL::b_off(0) + swz(col, c)) = v;
        if (SPLIT) *reinterpret_cast<uint4*>(st + PL::b_off(1) + swz(col, c)) = vl;
      }
      fence_async_smem();
      mbar_arrive(reinterpret_cast<uint64_t*>(&C.full[s]));
    }
    // ------------------------------------------------------- epilogue
    // The MMA thread always commits the accumulator barrier (after its last
    // issued MMA), so a second bounded wait after a timeout still ends with
    // no MMA in flight before the tensor memory is read or freed.
    if (lane == 0 && !mbar_wait_bounded(reinterpret_cast<uint64_t*>(&C.acc), 0u, deadline, g.status))
      mbar_wait_bounded(reinterpret_cast<uint64_t*>(&C.acc), 0u, globaltimer_ns() + g.timeout_ns, g.status);
    __syncwarp();
    tc_fence_after();
    const int lg = warp & 3;                // TMEM lanes 32 lg .. 32 lg + 31 = tile rows
    const int rw = row0 + lg * 32 + lane;   // the output row of this lane
    const uint32_t tl = tmem + ((uint32_t)(lg * 32) << 16);
    for (int c0 = 16 * hf; c0 < TN; c0 += 32) {  // the two warps of a lane group alternate 16-column chunks
      float v0[16], v1[16];
      tmem_ld16(tl + (uint32_t)c0, v0);
      if (NMAT == 2) tmem_ld16(tl + (uint32_t)(TN + c0), v1);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int col = c0 + j;
        if (col >= ncol) break;  // warp-uniform
        if constexpr (EPI == E_F32) {
          if (rw < g.a_rows) g.out_f32[(size_t)(col0 + col) * g.out_ld + rw] = v0[j];
        } else {
          const float hv = swiglu_f32(v0[j], v1[j], g.swiglu_limit);
          if constexpr (EPI == E_SWIGLU_Q8) {
            g.out_h[(size_t)(col0 + col) * g.out_ld + rw] = q8_h16_warp(hv);  // the warp's 32 rows: one q8_1 block
          } else {
            g.out_h[(size_t)(col0 + col) * g.out_ld + rw] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
          }
        }
      }
    }
  } else if (lane == 0) {
    // ----------------------------------------------------- MMA issuer
    const uint32_t idesc = umma_idesc(TN, AK == A_BF16);
    for (int kc = 0; kc < nk; ++kc) {
      const int s = kc % NS;
      if (!mbar_wait_bounded(reinterpret_cast<uint64_t*>(&C.full[s]), (uint32_t)((kc / NS) & 1), deadline, g.status))
        break;
      tc_fence_after();
      const uint32_t st = smem_u32(sm + (size_t)s * PL::STAGE);
#pragma unroll
      for (int mat = 0; mat < NMAT; ++mat) {
        const uint32_t td = tmem + (uint32_t)(mat * TN);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ah = umma_desc(st + PL::a_off(mat, 0) + 32u * k);
          const uint64_t bh = umma_desc(st + PL::b_off(0) + 32u * k);
          umma_f16(td, ah, bh, idesc, (kc | k) ? 1u : 0u);
          if (SPLIT) {
            umma_f16(td, ah, umma_desc(st + PL::b_off(SPLIT ? 1 : 0) + 32u * k), idesc, 1u);
            umma_f16(td, umma_desc(st + PL::a_off(mat, SPLIT ? 1 : 0) + 32u * k), bh, idesc, 1u);
          }
        }
      }
      umma_commit(reinterpret_cast<uint64_t*>(&C.empty[s]));
    }
    umma_commit(reinterpret_cast<uint64_t*>(&C.acc));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols_tmem);
  }
}

template <int AK, int NMAT, bool SPLIT, int EPI, int TNM, int NS>
int launch_gemm(const GemmArgs& g, unsigned grid, cudaStream_t s) {
  constexpr size_t smem = Plan<NMAT, SPLIT, TNM, NS>::SMEM;
  static_assert(smem <= 232448, "GEMM stages exceed the shared memory of a block");
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(k_gemm<AK, NMAT, SPLIT, EPI, TNM, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_dev = dev;
  }
  if (grid == 0) return MOE_OK;
  k_gemm<AK, NMAT, SPLIT, EPI, TNM, NS><<<grid, GTHREADS, smem, s>>>(g);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int route_steps(const PrefillParams& p, cudaStream_t s) {
  GemmArgs g{};
  g.K = p.D; g.a_rows = p.N; g.a_row_bytes = 2 * p.D; g.a0 = reinterpret_cast<const uint8_t*>(p.router_w);
  g.pseudo = -1; g.b = p.x; g.cols = p.m; g.mt_count = (p.N + TM - 1) / TM;
  g.out_f32 = p.logits; g.out_ld = p.N; g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
  const unsigned grid = (unsigned)(g.mt_count * ((p.m + PF_TN - 1) / PF_TN));
  int rc = launch_gemm<A_BF16, 1, false, E_F32, PF_TN, 4>(g, grid, s);
  if (rc) return rc;
  SelectParams sp{};
  sp.logits = p.logits; sp.bias = p.bias; sp.m = p.m; sp.N = p.N; sp.k = p.k; sp.norm = p.norm;
  sp.gate_temp = p.gate_temp; sp.route_scale = p.route_scale; sp.topk_w = p.topk_w; sp.topk_idx = p.topk_idx;
  sp.ctrl = p.ctrl;
  return launch_select(sp, s);
}

}  // namespace

int launch_prefill_route(const PrefillParams& p, cudaStream_t s) { return route_steps(p, s); }

int launch_prefill(const PrefillParams& p, cudaStream_t s) {
  const PrefillLayout& L = p.L;
  uint8_t* pw = p.pw;
  const int m = p.m, D = p.D, I = p.I, N = p.N, k = p.k;
  const int shq = p.shared_kind == MOE_SHARED_KQUANT;
  const int NE = N + 1;
  const int nch = (m + PF_GCH - 1) / PF_GCH;
  int rc;
  uint16_t* x16h = reinterpret_cast<uint16_t*>(pw + L.x16h);
  uint16_t* x16l = reinterpret_cast<uint16_t*>(pw + L.x16l);
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
  uint16_t* h16 = reinterpret_cast<uint16_t*>(pw + L.h16);
  float* ep = reinterpret_cast<float*>(pw + L.ep);
  uint16_t* hs = reinterpret_cast<uint16_t*>(pw + L.hs);
  float* sp = reinterpret_cast<float*>(pw + L.sp);

  // 1. fp16 of q8_1(x)
  {
    const long nb = (long)m * (D / 32);
    long blocks = (nb + 255) / 256;
    if (blocks > 152L * 8) blocks = 152L * 8;
    k_x16<<<(unsigned)blocks, 256, 0, s>>>(p.x, m, D, x16h, x16l);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  // 2-3. router logits and selection
  if ((rc = route_steps(p, s))) return rc;
  // 4. grouping
  k_group_hist<<<nch, 256, NE * sizeof(int), s>>>(p.topk_idx, m, k, N, shq, chunk);
  k_group_scan<<<1, 1024, 0, s>>>(chunk, nch, N, p.expert_ptrs, I / TM, D / TM, offsets, expert_ok, gu_tiles, dn_tiles,
                                  n_tiles, &p.ctrl->status);
  k_group_scatter<<<nch, 256, 0, s>>>(p.topk_idx, p.topk_w, m, k, N, shq, chunk, pair_tok, pair_w, pos_of, pos_sh);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 5. gate/up of the routed experts (and of a K-quant shared expert) -> fp16 of q8_1(h)
  {
    GemmArgs g{};
    g.K = D; g.a_rows = I; g.a_row_bytes = (D / QK) * Q2K_B; g.eptr = p.expert_ptrs; g.pj0 = 0; g.pj1 = 1;
    g.pseudo = shq ? N : -1; g.a0 = p.sh1; g.a1 = p.sh3; g.b = x16h; g.b_lo = x16l; g.b_rows = pair_tok;
    g.tiles = gu_tiles; g.n_tiles = n_tiles; g.offsets = offsets; g.out_h = h16; g.out_ld = I;
    g.swiglu_limit = p.swiglu_limit; g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
    const unsigned grid = (unsigned)L.max_gu_tiles * (unsigned)(I / TM);
    if ((rc = launch_gemm<A_Q2K, 2, true, E_SWIGLU_Q8, PF_TN_GU, 2>(g, grid, s))) return rc;
  }
  // 6. down -> E per pair
  {
    GemmArgs g{};
    g.K = I; g.a_rows = D; g.a_row_bytes = (I / QK) * Q3K_B; g.eptr = p.expert_ptrs; g.pj0 = 2; g.pj1 = 2;
    g.pseudo = shq ? N : -1; g.a0 = p.sh2; g.b = h16;
    g.tiles = dn_tiles; g.n_tiles = n_tiles + 1; g.offsets = offsets; g.out_f32 = ep; g.out_ld = D;
    g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
    const unsigned grid = (unsigned)L.max_dn_tiles * (unsigned)(D / TM);
    if ((rc = launch_gemm<A_Q3K, 1, false, E_F32, PF_TN, 4>(g, grid, s))) return rc;
  }
  // 7. the bf16 shared expert
  if (!shq) {
    const unsigned ntok = (unsigned)((m + PF_TN - 1) / PF_TN);
    GemmArgs g{};
    g.K = D; g.a_rows = I; g.a_row_bytes = 2 * D; g.a0 = p.sh1; g.a1 = p.sh3; g.pseudo = -1; g.b = p.x; g.cols = m;
    g.mt_count = I / TM; g.out_h = hs; g.out_ld = I; g.swiglu_limit = p.swiglu_limit;
    g.status = &p.ctrl->status; g.timeout_ns = p.timeout_ns;
    if ((rc = launch_gemm<A_BF16, 2, false, E_SWIGLU_BF16, PF_TN, 3>(g, (unsigned)g.mt_count * ntok, s))) return rc;
    GemmArgs d{};
    d.K = I; d.a_rows = D; d.a_row_bytes = 2 * I; d.a0 = p.sh2; d.pseudo = -1; d.b = hs; d.cols = m;
    d.mt_count = D / TM; d.out_f32 = sp; d.out_ld = D; d.status = &p.ctrl->status; d.timeout_ns = p.timeout_ns;
    if ((rc = launch_gemm<A_BF16, 1, false, E_F32, PF_TN, 4>(d, (unsigned)d.mt_count * ntok, s))) return rc;
  }
  // 8. ordered combine
  k_combine<<<m, 256, 0, s>>>(p.topk_idx, pos_of, expert_ok, pair_w, ep, sp, shq ? pos_sh : nullptr, k, D, p.out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// kernel launches of one prefill call
int prefill_launches(int shared_kind) { return shared_kind == MOE_SHARED_KQUANT ? 9 : 11; }

}  // namespace moe
