// GPU twin of the seeded synthetic-input generator (synth_core.h), used to
// fill large device-resident inputs (all routed experts of a 40-layer stack
// are ~200 GB) without staging them through host memory.  Same element
// definitions as synth.c; K-quant blocks and uniform draws are bit-identical
// to the host fill, normal draws agree up to the platform log/cos note in
// synth_core.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

namespace {

__global__ void k_fill_q2k(uint8_t* out, uint64_t nblocks, uint64_t block0, uint64_t key,
                           double dlo, double dhi) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < nblocks;
       i += (uint64_t)gridDim.x * blockDim.x) {
    uint8_t b[84];
    syn_q2k_block(b, key, block0 + i, dlo, dhi);
    uint8_t* dst = out + i * 84ULL;   // 4-byte aligned (84 = 4 * 21)
    for (int k = 0; k < 84; k += 4)
      *reinterpret_cast<uint32_t*>(dst + k) =
          (uint32_t)b[k] | ((uint32_t)b[k + 1] << 8) | ((uint32_t)b[k + 2] << 16) | ((uint32_t)b[k + 3] << 24);
  }
}

__global__ void k_fill_q3k(uint8_t* out, uint64_t nblocks, uint64_t block0, uint64_t key,
                           double dlo, double dhi) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < nblocks;
       i += (uint64_t)gridDim.x * blockDim.x) {
    uint8_t b[110];
    syn_q3k_block(b, key, block0 + i, dlo, dhi);
    uint8_t* dst = out + i * 110ULL;  // 2-byte aligned (110 = 2 * 55)
    for (int k = 0; k < 110; k += 2)
      *reinterpret_cast<uint16_t*>(dst + k) = (uint16_t)((uint32_t)b[k] | ((uint32_t)b[k + 1] << 8));
  }
}

__global__ void k_fill_normal_bf16(uint16_t* out, uint64_t n, uint64_t cols, uint64_t key, double std_,
                                   const double* row_scale) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    double s = std_;
    if (row_scale) s = __dmul_rn(s, row_scale[i / cols]);
    out[i] = syn_f64_to_bf16(__dmul_rn(syn_normal(key, i), s));
  }
}

__global__ void k_fill_uniform_f32(float* out, uint64_t n, uint64_t key, double lo, double hi) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = __double2float_rn(syn_affine(lo, hi, syn_unit(syn_draw(key, i))));
}

// Every routed expert of one layer in one launch: expert e's slot starts at
// base + e * slot; w1 / w3 (Q2_K) at o1 / o3, w2 (Q3_K) at o2; stream keys
// (seed, layer, tensor, e) exactly as the host fill uses them.
__global__ void k_fill_experts(uint8_t* base, uint32_t n_experts, uint64_t slot, uint64_t o1, uint64_t o3,
                               uint64_t o2, uint64_t nb1, uint64_t nb2, uint64_t seed, uint32_t layer) {
  const uint64_t per = 2 * nb1 + nb2;
  const uint64_t total = per * n_experts;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t e = (uint32_t)(i / per);
    uint64_t r = i % per;
    uint8_t* slotp = base + e * slot;
    if (r < 2 * nb1) {
      const bool up = r >= nb1;
      const uint64_t blk = up ? r - nb1 : r;
      const uint64_t key = syn_key(seed, layer, up ? SYN_T_W3 : SYN_T_W1, e);
      uint8_t b[84];
      syn_q2k_block(b, key, blk, 1e-3, 4e-3);
      uint8_t* dst = slotp + (up ? o3 : o1) + blk * 84ULL;
      for (int k = 0; k < 84; k += 4)
        *reinterpret_cast<uint32_t*>(dst + k) =
            (uint32_t)b[k] | ((uint32_t)b[k + 1] << 8) | ((uint32_t)b[k + 2] << 16) | ((uint32_t)b[k + 3] << 24);
    } else {
      const uint64_t blk = r - 2 * nb1;
      const uint64_t key = syn_key(seed, layer, SYN_T_W2, e);
      uint8_t b[110];
      syn_q3k_block(b, key, blk, 5e-4, 2e-3);
      uint8_t* dst = slotp + o2 + blk * 110ULL;
      for (int k = 0; k < 110; k += 2)
        *reinterpret_cast<uint16_t*>(dst + k) = (uint16_t)((uint32_t)b[k] | ((uint32_t)b[k + 1] << 8));
    }
  }
}

unsigned grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ULL * 32ULL) g = 152ULL * 32ULL;
  return g ? (unsigned)g : 1u;
}

}  // namespace

extern "C" {

int syn_gpu_fill_q2k(void* out, uint64_t nblocks, uint64_t block0, uint64_t key, double dlo, double dhi,
                     void* stream) {
  if (!nblocks) return 0;
  k_fill_q2k<<<grid_for(nblocks), 256, 0, (cudaStream_t)stream>>>((uint8_t*)out, nblocks, block0, key, dlo, dhi);
  return (int)cudaGetLastError();
}

int syn_gpu_fill_q3k(void* out, uint64_t nblocks, uint64_t block0, uint64_t key, double dlo, double dhi,
                     void* stream) {
  if (!nblocks) return 0;
  k_fill_q3k<<<grid_for(nblocks), 256, 0, (cudaStream_t)stream>>>((uint8_t*)out, nblocks, block0, key, dlo, dhi);
  return (int)cudaGetLastError();
}

int syn_gpu_fill_normal_bf16(void* out, uint64_t n, uint64_t cols, uint64_t key, double std_,
                             const double* row_scale_dev, void* stream) {
  if (!n) return 0;
  k_fill_normal_bf16<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)out, n, cols ? cols : 1, key,
                                                                    std_, row_scale_dev);
  return (int)cudaGetLastError();
}

int syn_gpu_fill_uniform_f32(float* out, uint64_t n, uint64_t key, double lo, double hi, void* stream) {
  if (!n) return 0;
  k_fill_uniform_f32<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, key, lo, hi);
  return (int)cudaGetLastError();
}

int syn_gpu_fill_experts(void* base, uint32_t n_experts, uint64_t slot, uint64_t o1, uint64_t o3, uint64_t o2,
                         uint64_t nb1, uint64_t nb2, uint64_t seed, uint32_t layer, void* stream) {
  const uint64_t total = (2 * nb1 + nb2) * n_experts;
  if (!total) return 0;
  k_fill_experts<<<grid_for(total), 256, 0, (cudaStream_t)stream>>>((uint8_t*)base, n_experts, slot, o1, o3, o2,
                                                                     nb1, nb2, seed, layer);
  return (int)cudaGetLastError();
}

}  // extern "C"
