// Prefill path, the down projection: E = W2 q8_1(h) per (expert, token) pair
// (Q3_K weights), as a persistent tcgen05 kernel over (expert, 128 rows of
// W2, <= 128 pairs) tiles with exact products.
//
//   A  the weights' integer part (code - 32) * q, q in -4..3, exact in fp16,
//      written by the dequantising warps into a 128-byte-swizzled K-major
//      shared-memory tile per 64-value chunk; the per-super-block factor d
//      (fp16) is left out of A.
//   B  the q8_1 values of h, fp16(d_h) * q_h (18 significant bits), as the two
//      fp16 parts hi + lo whose sum is exact (written so by the gate/up
//      epilogue); the tile's n pairs' hi rows and then their lo rows form one
//      B tile of 2n rows, so one MMA of width 2n forms A*hi and A*lo.
// Each super-block (256 K values) accumulates into a fresh tensor-memory
// accumulator, two of them alternating (2 x 256 columns: all of tensor
// memory); the epilogue warps drain each, add the hi and lo halves and scale
// by the super-block's d into f32 running sums in registers while the MMAs of
// the next super-block proceed.  The only rounding is the f32 accumulation,
// so an error that every clipped element of a row of h shares (they all hold
// the block maximum) cannot add up coherently along the row.  An expert with
// up to 128 pairs dequantises each W2 row tile once.
//
// Method: DeepSeek V4.1 atlas "Mixture of experts" (Routed expert step:
// E = W2 h); metrale moe_v41 module docs (Q3_K down projection on q8_1(h)).
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int TM = PF_TM;          // weight rows per tile
constexpr int TNQ = PF_TNQ;        // pairs per tile
constexpr int BBOX = 16;           // rows per B box: a tile loads only the rows of its pairs
constexpr uint32_t B_STAGE = 2 * TNQ * 128;  // B tile: n hi rows, then n lo rows, of 64 fp16 (128-byte swizzle)
constexpr uint32_t A_STAGE = TM * 128;       // A tile: 128 rows of 64 fp16 (128-byte swizzle)
constexpr int NSB = 3;             // B ring stages
constexpr int NA = 4;              // A ring stages
constexpr int NEW = 8;             // epilogue warps (0-7): pairs 0-63 (warps 0-3) and 64-127 (warps 4-7)
constexpr int NDW = 8;             // dequantising warps (8-15)
constexpr int W_TMA = NEW + NDW;   // TMA issuer
constexpr int W_MMA = W_TMA + 1;   // MMA issuer
constexpr int NTHR = (W_MMA + 1) * 32;
// Raw-block staging of the dequantising warps, two buffers per warp of 32
// rows: one super-block's 4-byte aligned window (28 words, pitch 29 words).
constexpr int Q3_PITCH = 29;
constexpr uint32_t STG_WARP = 2u * 32 * Q3_PITCH * 4;
constexpr uint32_t STG_BYTES = NDW * STG_WARP;

struct KqArgs {
  CUtensorMap map_bh, map_bl;           // B hi / lo parts: rows = pair positions, box {64 values, 16 rows}
  const int4* tiles;                    // two int4 per tile: (expert, row tile, first pair, pairs), row pointer
  const int* n_tiles;
  int K;                                // contraction length I (a multiple of 256)
  int a_row_bytes;                      // bytes per W2 row
  int out_ld;                           // E row length D
  float* out_e;                         // E f32 [pair][D]
  unsigned* status;
  unsigned long long timeout_ns;
};

struct KqCtl {
  unsigned long long b_full[NSB], b_empty[NSB];
  unsigned long long a_full[NA], a_empty[NA];
  unsigned long long acc_full[2], acc_empty[2];
  unsigned long long done;
  uint32_t tmem;
  uint32_t abort;
};

constexpr uint32_t SMEM_BYTES = 1024 + NSB * B_STAGE + NA * A_STAGE + STG_BYTES + ((sizeof(KqCtl) + 15) & ~15u);
static_assert(SMEM_BYTES <= 232448, "stages exceed the shared memory of a block");

__device__ __forceinline__ uint64_t* bp(unsigned long long& b) { return reinterpret_cast<uint64_t*>(&b); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait of one thread; on a timeout the block's abort flag is set and
// every later wait of the block returns false at once.
__device__ __forceinline__ bool kwait(KqCtl& C, unsigned long long& bar, uint32_t parity, uint64_t deadline,
                                      unsigned* status) {
  if (*reinterpret_cast<volatile uint32_t*>(&C.abort)) return false;
  if (mbar_wait_bounded(bp(bar), parity, deadline, status)) return true;
  *reinterpret_cast<volatile uint32_t*>(&C.abort) = 1u;
  return false;
}

// The same for a whole warp (lane 0 waits, the result is shared).
__device__ __forceinline__ bool kwait_warp(KqCtl& C, unsigned long long& bar, uint32_t parity, uint64_t deadline,
                                           unsigned* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = kwait(C, bar, parity, deadline, status);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One arrival per warp: every lane's tensor-memory accesses are complete
// (the warp-collective wait before this) and fenced, then lane 0 arrives.
__device__ __forceinline__ void warp_arrive(unsigned long long& b) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bp(b));
}

struct Tile {
  int e, mt, col0, ncol, tnp;
  const uint8_t* rows;  // the tile's first W2 row
};

__device__ __forceinline__ Tile tile_of(const KqArgs& g, int t) {
  const int4 v = __ldg(g.tiles + 2 * t);
  const int4 p = __ldg(g.tiles + 2 * t + 1);
  Tile T;
  T.e = v.x;
  T.mt = v.y;
  T.col0 = v.z;
  T.ncol = v.w;
  T.tnp = (v.w + 15) & ~15;
  T.rows = reinterpret_cast<const uint8_t*>(((unsigned long long)(uint32_t)p.y << 32) | (uint32_t)p.x);
  return T;
}

// ------------------------------------------------------------ MMA issuer
// Super-block s of a tile: its 4 value chunks (4 K steps each) into
// accumulator s % 2, which the epilogue has emptied.
__device__ void run_mma(const KqArgs& g, KqCtl& C, uint32_t tmem, uint32_t smem_base, int ntiles,
                        uint64_t deadline) {
  const int nsb = g.K / QK;
  const uint64_t bdesc0 = umma_desc(smem_base);  // stage st adds st * B_STAGE / 16 to the address field
  const uint64_t adesc0 = umma_desc(smem_base + NSB * B_STAGE);
  uint32_t gb = 0, ga = 0, gacc[2] = {0, 0};
  // a wait that is already satisfied costs one try; the bounded loop only runs when it is not
  auto wait = [&](unsigned long long& b, uint32_t par) -> bool {
    return mbar_try_wait(bp(b), par) || kwait(C, b, par, deadline, g.status);
  };
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = tile_of(g, t);
    const uint32_t idesc = umma_idesc(2 * T.tnp, false);
    for (int s = 0; s < nsb; ++s) {
      const int acc = s & 1;
      if (gacc[acc] > 0 && !wait(C.acc_empty[acc], (gacc[acc] - 1) & 1u)) goto out;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(256 * acc);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const uint32_t bu = gb + (uint32_t)c, st = bu % NSB;
        if (!wait(C.b_full[st], (bu / NSB) & 1u)) goto out;
        const uint32_t au = ga++, as = au % NA;
        if (!wait(C.a_full[as], (au / NA) & 1u)) goto out;
        tc_fence_after();
        const uint64_t bd = bdesc0 + (uint64_t)(st * (B_STAGE >> 4));
        const uint64_t ad = adesc0 + (uint64_t)(as * (A_STAGE >> 4));
        umma_f16(d, ad, bd, idesc, c ? 1u : 0u);
        umma_f16(d, ad + 2u, bd + 2u, idesc, 1u);
        umma_f16(d, ad + 4u, bd + 4u, idesc, 1u);
        umma_f16(d, ad + 6u, bd + 6u, idesc, 1u);
        umma_commit(bp(C.a_empty[as]));
        umma_commit(bp(C.b_empty[st]));
      }
      umma_commit(bp(C.acc_full[acc]));
      ++gacc[acc];
      gb += 4;
    }
  }
out:
  umma_commit(bp(C.done));  // after every MMA this thread issued
}

// ------------------------------------------------------------ TMA issuer
__device__ void run_tma(const KqArgs& g, KqCtl& C, uint32_t smem_base, int ntiles, uint64_t deadline) {
  const int nsb = g.K / QK;
  uint32_t gb = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = tile_of(g, t);
    for (int s = 0; s < nsb; ++s) {
      for (int c = 0; c < 4; ++c) {
        const uint32_t bu = gb++, st = bu % NSB;
        if (bu >= NSB && !kwait(C, C.b_empty[st], (bu / NSB - 1) & 1u, deadline, g.status)) goto out;
        const uint32_t dst = smem_base + st * B_STAGE;
        mbar_arrive_expect_tx(bp(C.b_full[st]), 2u * (uint32_t)T.tnp * 128u);
        for (int r = 0; r < T.tnp; r += BBOX) {
          tma_load_2d(dst + (uint32_t)r * 128u, &g.map_bh, QK * s + 64 * c, T.col0 + r, bp(C.b_full[st]));
          tma_load_2d(dst + (uint32_t)(T.tnp + r) * 128u, &g.map_bl, QK * s + 64 * c, T.col0 + r, bp(C.b_full[st]));
        }
      }
    }
  }
out:
  // copies still in flight land before the block can exit (the MMA issuer
  // consumed every stage unless the call timed out)
  {
    const uint64_t d2 = globaltimer_ns() + g.timeout_ns;
    const uint32_t first = gb > (uint32_t)NSB ? gb - NSB : 0u;
    for (uint32_t bu = first; bu < gb; ++bu) mbar_wait_bounded(bp(C.b_full[bu % NSB]), (bu / NSB) & 1u, d2, g.status);
  }
}

// --------------------------------------------------------- dequantisers
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_wait0() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The dequantising warps walk one stream of (tile, raw unit) items; a warp
// stages the unit of its 32 rows with coalesced asynchronous copies (lane i
// copies piece i of each row in turn) one item ahead of the one it writes.
struct UnitCursor {
  int t, u;  // tile index, unit within the tile
};

// Down: thread = (weight row, half of each super-block): warps 8-11 write
// value chunks 0 and 1 of every super-block, warps 12-15 chunks 2 and 3.  Unit
// = one super-block: the 4-byte aligned 28-word window around the row's
// 110-byte Q3_K block (2-byte aligned), realigned with one byte permute per
// word.  A value is (code - 32) * q with q = lo + 4 hb - 4 (exact in fp16).
__device__ void run_dequant_q3k(const KqArgs& g, KqCtl& C, uint32_t a_smem, uint32_t* stg, int ntiles,
                                uint64_t deadline) {
  const int w = (threadIdx.x >> 5) - NEW;  // 0..7
  const int lane = threadIdx.x & 31;
  const int hf = w >> 2, quarter = w & 3;
  const int row = quarter * 32 + lane;  // this thread's row of the tile
  const int nsb = g.K / QK;
  const uint32_t stg_s = smem_u32(stg);
  const __half2 m1028 = u2h(0xE404E404u);  // -1028 in both halves
  uint32_t ga = 0;  // chunk c of the n-th super-block walked is use 4 n + c of the ring
  int tcache = -1;  // the tile whose row pointer is cached
  const uint8_t* rcache = nullptr;
  auto rows_of = [&](int t) -> const uint8_t* {
    if (t != tcache) {
      tcache = t;
      rcache = tile_of(g, t).rows;
    }
    return rcache;
  };
  auto issue = [&](UnitCursor it, int buf) {
    if (it.t < ntiles) {
      const uint8_t* A = rows_of(it.t) + (size_t)(quarter * 32) * g.a_row_bytes + Q3K_B * it.u;
      const uint32_t dst = stg_s + (uint32_t)(buf * 32 * Q3_PITCH * 4) + 4u * lane;
      if (lane < 28) {
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const uintptr_t a = reinterpret_cast<uintptr_t>(A + (size_t)rr * g.a_row_bytes) & ~uintptr_t(3);
          cp_async4(dst + (uint32_t)(rr * Q3_PITCH * 4), reinterpret_cast<const void*>(a + 4 * lane));
        }
      }
    }
    cp_commit();
  };
  auto next = [&](UnitCursor it) -> UnitCursor {
    if (++it.u == nsb) {
      it.u = 0;
      it.t += gridDim.x;
    }
    return it;
  };
  UnitCursor cur{(int)blockIdx.x, 0};
  const uint8_t* cur_rows = cur.t < ntiles ? rows_of(cur.t) : nullptr;
  issue(cur, 0);
  int buf = 0;
  while (cur.t < ntiles) {
    const UnitCursor nx = next(cur);
    issue(nx, buf ^ 1);
    // this thread's row: its alignment within the staged window (the row
    // pointer of the current tile was cached when its first unit was issued)
    const uintptr_t a = reinterpret_cast<uintptr_t>(cur_rows + (size_t)(quarter * 32 + lane) * g.a_row_bytes +
                                                    (size_t)cur.u * Q3K_B);
    const uint32_t sel = (a & 2u) ? 0x5432u : 0x3210u;
    cp_wait1();
    __syncwarp();
    const uint32_t* win = stg + buf * 32 * Q3_PITCH + lane * Q3_PITCH;
    // block words: hmask 0..7, qs 8..23 (this half: 8 + 8 hf ..), scales 24..26
    uint32_t hm[8], qs[8], sw[3];
    {
      uint32_t prev = win[0];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t nw = win[i + 1];
        hm[i] = prmt(prev, nw, sel);
        prev = nw;
      }
      prev = win[8 + 8 * hf];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t nw = win[9 + 8 * hf + i];
        qs[i] = prmt(prev, nw, sel);
        prev = nw;
      }
      prev = win[24];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const uint32_t nw = win[25 + i];
        sw[i] = prmt(prev, nw, sel);
        prev = nw;
      }
    }
    __syncwarp();  // every lane is done with `buf` before it is refilled
    bool ok = true;
#pragma unroll
    for (int cc = 0; cc < 2 && ok; ++cc) {
      const int c = 2 * hf + cc;
      const uint32_t au = ga + (uint32_t)c, as = au % NA;
      if (au >= NA && !kwait_warp(C, C.a_empty[as], (au / NA - 1) & 1u, deadline, g.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int h = hf;  // value chunk c covers block half c >> 1
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        const int j = 2 * cc + jb;  // 2-bit plane
#pragma unroll
        for (int l16 = 0; l16 < 2; ++l16) {
          // sub-block b = 8 h + i (i = 2 j + l16): low four code bits from
          // scales[i] (h = 0) or the high nibble of scales[i] (h = 1), high
          // two bits from scales[8 + i % 4] at bit 2 (b / 4) = 2 (2 h + i / 4)
          const int i = 2 * j + l16;
          const uint32_t lo4 = (sw[i >> 2] >> (8 * (i & 3) + 4 * h)) & 15u;
          const uint32_t hi2 = (sw[2] >> (8 * (i & 3) + 2 * (2 * h + (i >> 2)))) & 3u;
          const __half2 ds = __float2half2_rn((float)((int)(lo4 | (hi2 << 4)) - 32));
          uint32_t o[8];
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            const uint32_t lo2 = (qs[4 * l16 + wd] >> (2 * j)) & 0x03030303u;
            const uint32_t hb = (hm[4 * l16 + wd] >> (4 * h + j)) & 0x01010101u;
            const uint32_t q = lo2 | (hb << 2);  // lo + 4 hb, per byte: 0..7
            // fp16 1024 + q per value, minus 1028 (exact: q - 4), times (code - 32) (exact)
            o[2 * wd] = h2u(__hmul2(__hadd2(u2h(prmt(q, 0x64646464u, 0x4140u)), m1028), ds));
            o[2 * wd + 1] = h2u(__hmul2(__hadd2(u2h(prmt(q, 0x64646464u, 0x4342u)), m1028), ds));
          }
          // the 16 values are K 32 jb + 16 l16 .. + 15 of the chunk: two 16-byte pieces
          const uint32_t base = a_smem + as * A_STAGE;
          sts128(base + swz(row, 4 * jb + 2 * l16), o[0], o[1], o[2], o[3]);
          sts128(base + swz(row, 4 * jb + 2 * l16 + 1), o[4], o[5], o[6], o[7]);
        }
      }
      fence_async_smem();  // the tensor cores read A through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bp(C.a_full[as]));
    }
    if (!ok) break;
    ga += 4;
    if (nx.t != cur.t && nx.t < ntiles) cur_rows = rows_of(nx.t);
    cur = nx;
    buf ^= 1;
  }
  cp_wait0();  // no copy may still be landing when the block exits
}

// ------------------------------------------------------------- epilogue
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Drain of one accumulator for np of the warp group's pairs (np a multiple of
// 16, at most 64): R[p] += c * (hi[p] + lo[p]), hi at column hi0 + p and lo
// at column lo0 + p of the warp's lanes.
__device__ __forceinline__ void drain(uint32_t hi0, uint32_t lo0, int np, float c, float (&R)[64]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (16 * q < np) {  // warp-uniform
      uint32_t hi[16], lo[16];
      tmem_ld16_nw(hi0 + (uint32_t)(16 * q), hi);
      tmem_ld16_nw(lo0 + (uint32_t)(16 * q), lo);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) R[16 * q + j] = fmaf(c, __uint_as_float(hi[j]) + __uint_as_float(lo[j]), R[16 * q + j]);
    }
  }
}

// Warps 0-3 keep the running sums of pairs 0-63 of the tile, warps 4-7 those
// of pairs 64-127, each for its quarter of the rows; both groups drain every
// super-block's accumulator (the hi parts at columns 0..n-1, the lo parts at
// n..2n-1) and then write their pairs of E.
__device__ void run_epilogue_dn(const KqArgs& g, KqCtl& C, uint32_t tmem, int ntiles, uint64_t deadline) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = w >> 2, quarter = w & 3, r = quarter * 32 + lane;
  const int nsb = g.K / QK;
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  uint32_t gacc[2] = {0, 0};
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = tile_of(g, t);
    const int row = T.mt * TM + r;
    const uint8_t* rowp = T.rows + (size_t)r * g.a_row_bytes;
    const int p0 = 64 * grp;
    const int np = min(64, T.tnp - p0);  // this group's columns (<= 0: none)
    float R[64];
#pragma unroll
    for (int p = 0; p < 64; ++p) R[p] = 0.f;
    bool ok = true;
    for (int s = 0; s < nsb; ++s) {
      const int acc = s & 1;
      const uint8_t* dp = rowp + (size_t)s * Q3K_B + 108;
      const float c = half_bits_to_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(dp)));
      if (ok && kwait_warp(C, C.acc_full[acc], gacc[acc] & 1u, deadline, g.status)) {
        tc_fence_after();
        const uint32_t a = lane_base + (uint32_t)(256 * acc);
        drain(a + (uint32_t)p0, a + (uint32_t)(T.tnp + p0), np, c, R);
        warp_arrive(C.acc_empty[acc]);
      } else {
        ok = false;
      }
      ++gacc[acc];
    }
    if (ok) {
#pragma unroll
      for (int p = 0; p < 64; ++p)
        if (p < np && p0 + p < T.ncol) g.out_e[(size_t)(T.col0 + p0 + p) * g.out_ld + row] = R[p];
    }
  }
}

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(NTHR, 1) k_down_gemm(const __grid_constant__ KqArgs g) {
  extern __shared__ __align__(1024) uint8_t raw_smem[];
  uint8_t* sm = raw_smem + ((1024u - (smem_u32(raw_smem) & 1023u)) & 1023u);
  uint32_t* stg = reinterpret_cast<uint32_t*>(sm + NSB * B_STAGE + NA * A_STAGE);
  KqCtl& C = *reinterpret_cast<KqCtl*>(sm + NSB * B_STAGE + NA * A_STAGE + STG_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = __ldg(g.n_tiles);
  if ((int)blockIdx.x >= ntiles) return;
  const uint64_t deadline = globaltimer_ns() + g.timeout_ns;
  if (tid == 0) {
    for (int i = 0; i < NSB; ++i) {
      mbar_init(bp(C.b_full[i]), 1);
      mbar_init(bp(C.b_empty[i]), 1);
    }
    for (int i = 0; i < NA; ++i) {
      mbar_init(bp(C.a_full[i]), 4);  // one arrival per dequantising warp of the stage
      mbar_init(bp(C.a_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bp(C.acc_full[i]), 1);
      mbar_init(bp(C.acc_empty[i]), NEW);  // one arrival per epilogue warp
    }
    mbar_init(bp(C.done), 1);
    C.abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&C.tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;
  const uint32_t smem_base = smem_u32(sm);

  if (warp < NEW) {
    run_epilogue_dn(g, C, tmem, ntiles, deadline);
  } else if (warp < NEW + NDW) {
    run_dequant_q3k(g, C, smem_base + NSB * B_STAGE, stg + (size_t)(warp - NEW) * (STG_WARP / 4), ntiles, deadline);
  } else if (warp == W_TMA) {
    if (lane == 0) run_tma(g, C, smem_base, ntiles, deadline);
  } else {
    if (lane == 0) run_mma(g, C, tmem, smem_base, ntiles, deadline);
  }
  __syncwarp();
  // no MMA may still be writing tensor memory when it is freed: the issuer's
  // final commit follows its last MMA (bounded wait, a fresh deadline)
  if (warp == 0 && lane == 0) mbar_wait_bounded(bp(C.done), 0u, globaltimer_ns() + g.timeout_ns, g.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// ---------------------------------------------------------------- host
int launch_kq_gemm(const KqLaunch& L, cudaStream_t s) {
  KqArgs g{};
  if (!make_map_b16(&g.map_bh, L.bh, (uint64_t)L.K, (uint64_t)L.b_rows, BBOX) ||
      !make_map_b16(&g.map_bl, L.bl, (uint64_t)L.K, (uint64_t)L.b_rows, BBOX))
    return MOE_ERR_CUDA;
  g.tiles = L.tiles; g.n_tiles = L.n_tiles; g.K = L.K; g.a_row_bytes = L.a_row_bytes; g.out_ld = L.out_ld;
  g.out_e = L.out_e; g.status = L.status; g.timeout_ns = L.timeout_ns;
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(k_down_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_dev = dev;
  }
  k_down_gemm<<<L.grid, NTHR, SMEM_BYTES, s>>>(g);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
