// moe_v41_forward_noalloc: the decode-path forward with its scratch memory in
// a fixed array that the library itself holds on each GPU, for callers that
// cannot allocate device memory (see include/moe_v41.h).  It launches the same
// fused decode kernel as moe_v41_forward; only where the scratch lives differs.
#include "internal.h"

using namespace moe;

namespace {

// The scratch.  Every GPU that loads the library holds these bytes until the
// process exits.  Kernels receive its device address, which host code looks
// up on every call with cudaGetSymbolAddress (no allocation; it stays correct
// if the device's context is torn down and the module reloaded at another
// address); host code never dereferences the symbol itself.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_V41_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch on the current device.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  *out = p;
  return MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int moe_v41_forward_noalloc(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w,
                                       const float* bias, const uint64_t* expert_ptrs, int shared_kind,
                                       const void* sh_w1, const void* sh_w3, const void* sh_w2, float* out,
                                       float* topk_w, int32_t* topk_idx, float* logits_out, uint32_t* status_out,
                                       void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  const moe_v41_cfg& c = *cfg;
  // the decode kernels only: at most eight tokens, never the prefill path
  if (c.max_tokens > DECODE_MAX_M || c.path == MOE_PATH_PREFILL) return MOE_ERR_ARG;
  if (m < 1 || m > c.max_tokens) return MOE_ERR_ARG;
  if (!x || !router_w || !bias || !expert_ptrs || !sh_w1 || !sh_w3 || !sh_w2 || !out || !topk_w || !topk_idx)
    return MOE_ERR_ARG;
  if (shared_kind != MOE_SHARED_BF16 && shared_kind != MOE_SHARED_KQUANT) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(expert_ptrs, 8)) return MOE_ERR_ALIGN;
  if (!aligned(sh_w1, 256) || !aligned(sh_w3, 256) || !aligned(sh_w2, 256)) return MOE_ERR_ALIGN;
  if (!decode_fits(c.dim, c.inter)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(c);
  if (L.total > (size_t)MOE_V41_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;  // beyond the fixed scratch

  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = static_cast<uint8_t*>(base);
  // The array keeps whatever the previous call left: clear the control block
  // (status word and counters) this call starts from.
  if (cudaMemsetAsync(w + L.ctrl, 0, sizeof(Ctrl), s) != cudaSuccess) return MOE_ERR_CUDA;

  DecodeParams dp{};
  dp.m = m; dp.D = c.dim; dp.I = c.inter; dp.N = c.n_routed; dp.k = c.topk;
  dp.norm = c.norm_topk_prob != 0; dp.score_func = c.score_func;
  dp.gate_temp = c.gate_temp; dp.route_scale = c.route_scale; dp.swiglu_limit = c.swiglu_limit;
  dp.shared_kind = shared_kind;
  dp.x = static_cast<const uint16_t*>(x);
  dp.router_w = static_cast<const uint16_t*>(router_w);
  dp.bias = bias;
  dp.expert_ptrs = reinterpret_cast<const unsigned long long*>(expert_ptrs);
  dp.sh1 = static_cast<const uint8_t*>(sh_w1);
  dp.sh3 = static_cast<const uint8_t*>(sh_w3);
  dp.sh2 = static_cast<const uint8_t*>(sh_w2);
  dp.logits = logits_out ? logits_out : reinterpret_cast<float*>(w + L.logits);
  dp.topk_w = topk_w; dp.topk_idx = topk_idx;
  dp.sk = reinterpret_cast<float2*>(w + L.sk);
  dp.xu = reinterpret_cast<int*>(w + L.xu);
  dp.hu = reinterpret_cast<int*>(w + L.hu);
  dp.shh = w + L.shh;
  dp.shvec0 = c.max_tokens * c.topk;
  dp.out = out;
  dp.ctrl = reinterpret_cast<Ctrl*>(w + L.ctrl);
  dp.timeout_ns = (uint64_t)(c.wait_timeout_us ? c.wait_timeout_us : 2000000u) * 1000ull;
  if ((rc = launch_decode_layer(dp, sms, s))) return rc;
  if (status_out &&
      cudaMemcpyAsync(status_out, w + L.ctrl, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
