// Tensor-core issue-rate microbenchmark (measurement support, not part of the
// MoE library): one thread per block issues back-to-back tcgen05.mma
// (cta_group::1, M = 128, K = one instruction's depth) into one tensor-memory
// accumulator, with operands read from 128-byte-swizzled shared-memory tiles
// or A from tensor memory; the block waits for the last MMA through
// tcgen05.commit on an mbarrier (bounded wait).  The host times the launch
// with CUDA events; blocks = one per SM.  Operand values are zero: the rate
// does not depend on them.
//
// kinds: 0 f16 x f16 -> f32, 1 bf16 x bf16 -> f32, 3 e4m3 x e4m3 -> f32
// (kind::f8f6f4).  There is no int8 kind: ptxas rejects tcgen05.mma
// .kind::i8 for sm_103a ("not supported on .target 'sm_103a'"), while it
// accepts it for sm_100a.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor: D format (bits 4-5), A / B formats (7-9, 10-12),
// N >> 3 (17-22), M >> 4 (24-28); K-major operands
__device__ __forceinline__ uint32_t idesc(int kind, int n, int m) {
  const uint32_t dfmt = 1u;                   // f32 accumulator
  const uint32_t ab = kind == 1 ? 1u : 0u;    // bf16 = 1; f16 and e4m3 = 0
  return (dfmt << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

template <int KIND, bool ATMEM>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint32_t ta, uint64_t b, uint32_t id, uint32_t acc) {
  if constexpr (KIND <= 1) {
    if constexpr (ATMEM)
      asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                   " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d), "r"(ta), "l"(b),
                   "r"(id), "r"(acc) : "memory");
    else
      asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                   " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d), "l"(a), "l"(b),
                   "r"(id), "r"(acc) : "memory");
  } else {
    if constexpr (ATMEM)
      asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                   " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d), "r"(ta), "l"(b),
                   "r"(id), "r"(acc) : "memory");
    else
      asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                   " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d), "l"(a), "l"(b),
                   "r"(id), "r"(acc) : "memory");
  }
}

// alignment slack, A tile 128 x 128 B, B tile 256 x 128 B; the request is
// sized so that two blocks never share an SM (each allocates all 512
// tensor-memory columns)
constexpr int SMEM_USED = 1024 + 128 * 128 + 256 * 128;
constexpr int SMEM = 120 * 1024;
static_assert(SMEM >= SMEM_USED, "operand tiles exceed the request");

template <int KIND, bool ATMEM>
__global__ void __launch_bounds__(128, 1) k_mma_rate(int n, int m, int nacc, int iters, unsigned long long* clk,
                                                     unsigned* err) {
  extern __shared__ __align__(1024) uint8_t raw[];
  uint8_t* sm = raw + ((1024u - (su32(raw) & 1023u)) & 1023u);
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  for (int i = tid; i < (128 * 128 + 256 * 128) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&s_tmem)) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  if (tid == 0) {
    const uint32_t id = idesc(KIND, n, m);
    const uint32_t a0 = su32(sm), b0 = su32(sm + 128 * 128);
    // everything an MMA needs is computed before the loop: the loop body is
    // four MMA issues (K steps 0..3, accumulators cycled), so the issuing
    // thread's own instructions do not set the rate
    uint64_t ad[4], bd[4];
    uint32_t dd[4], ta[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ad[k] = sdesc(a0 + 32u * k);
      bd[k] = sdesc(b0 + 32u * k);
      ta[k] = tmem + 256u + 8u * k;
      dd[k] = tmem + (uint32_t)((k % nacc) * n);
    }
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int i = 0; i < iters; i += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) mma<KIND, ATMEM>(dd[k], ad[k], ta[k], bd[k], id, 1u);
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&bar))
                 : "memory");
    uint32_t ok = 0;
    for (uint32_t spin = 0; spin < (1u << 26) && !ok; ++spin)
      asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
                   " selp.u32 %0, 1, 0, p;\n}\n" : "=r"(ok) : "r"(su32(&bar)) : "memory");
    if (!ok) atomicAdd(err, 1u);
    clk[blockIdx.x] = clock64() - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid < 32) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

template <int KIND, bool ATMEM>
int run(int n, int m, int nacc, int iters, int blocks, float* ms, unsigned long long* clk_host) {
  auto kern = k_mma_rate<KIND, ATMEM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess) return 1;
  unsigned long long* clk = nullptr;
  unsigned* err = nullptr;
  if (cudaMalloc(&clk, sizeof(unsigned long long) * blocks) != cudaSuccess) return 2;
  if (cudaMalloc(&err, sizeof(unsigned)) != cudaSuccess) return 2;
  cudaMemset(err, 0, sizeof(unsigned));
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  kern<<<blocks, 128, SMEM>>>(n, m, nacc, 64, clk, err);  // warm-up
  cudaEventRecord(e0);
  kern<<<blocks, 128, SMEM>>>(n, m, nacc, iters, clk, err);
  cudaEventRecord(e1);
  int rc = cudaEventSynchronize(e1) == cudaSuccess ? 0 : 3;
  cudaEventElapsedTime(ms, e0, e1);
  unsigned herr = 0;
  cudaMemcpy(&herr, err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaMemcpy(clk_host, clk, sizeof(unsigned long long) * blocks, cudaMemcpyDeviceToHost);
  if (herr) rc = 4;
  if (cudaGetLastError() != cudaSuccess) rc = 5;
  cudaFree(clk);
  cudaFree(err);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return rc;
}

}  // namespace

// kind 0, 1 or 3 as above; n the MMA width (16..256, a multiple of 16); m the
// MMA height (64 or 128); nacc accumulators of n columns cycled through
// (1, 2 or 4; nacc * n <= 256 with A in tensor memory, which starts at
// column 256; <= 512 otherwise); a_tmem: A read from tensor memory; iters MMAs per block;
// blocks launched (one per SM).
// Writes the elapsed milliseconds and each block's issue-to-completion clock
// cycles.  Returns 0 on success.
extern "C" __attribute__((visibility("default"))) int mma_rate_run(int kind, int n, int m, int nacc, int a_tmem,
                                                                  int iters, int blocks, float* ms,
                                                                  unsigned long long* clk_per_block) {
  if (n < 16 || n > 256 || n % 16 || iters < 1 || blocks < 1) return -1;
  if ((m != 64 && m != 128) || (nacc != 1 && nacc != 2 && nacc != 4) || nacc * n > (a_tmem ? 256 : 512)) return -1;
  if (iters % 4) return -1;
  if (m == 64 && n % 8) return -1;
  switch (kind * 2 + (a_tmem ? 1 : 0)) {
    case 0: return run<0, false>(n, m, nacc, iters, blocks, ms, clk_per_block);
    case 1: return run<0, true>(n, m, nacc, iters, blocks, ms, clk_per_block);
    case 2: return run<1, false>(n, m, nacc, iters, blocks, ms, clk_per_block);
    case 3: return run<1, true>(n, m, nacc, iters, blocks, ms, clk_per_block);
    case 6: return run<3, false>(n, m, nacc, iters, blocks, ms, clk_per_block);
    case 7: return run<3, true>(n, m, nacc, iters, blocks, ms, clk_per_block);
    default: return -1;
  }
}
