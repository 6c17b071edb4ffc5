// The C-ABI of moe_v41 (declared in include/moe_v41.h): argument checks on
// the host, the workspace layout, and the kernel launches.  Nothing here
// allocates device memory; every buffer is the caller's.
#include "internal.h"

using namespace moe;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_ws(const moe_v41_cfg* c, void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGN;
  if (ws_bytes < ws_layout(*c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

uint64_t timeout_ns(const moe_v41_cfg* c) {
  return (uint64_t)(c->wait_timeout_us ? c->wait_timeout_us : 2000000u) * 1000ull;
}

bool use_decode(const moe_v41_cfg* c, int m) {
  if (c->path == MOE_PATH_DECODE) return true;
  if (c->path == MOE_PATH_PREFILL) return false;
  return m <= DECODE_MAX_M && decode_fits(c->dim, c->inter);
}

RouteParams route_params(const moe_v41_cfg* c, const void* x, int m, const void* router_w, const float* bias,
                         const float* bias_vl, const uint8_t* image_mask, float* logits, float* topk_w,
                         int32_t* topk_idx, uint8_t* ws, const WsLayout& L) {
  RouteParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.router_w = static_cast<const uint16_t*>(router_w);
  p.bias = bias; p.bias_vl = bias_vl; p.image_mask = image_mask;
  p.m = m; p.D = c->dim; p.N = c->n_routed; p.k = c->topk; p.norm = c->norm_topk_prob != 0;
  p.score_func = c->score_func;
  p.gate_temp = c->gate_temp; p.route_scale = c->route_scale;
  p.logits = logits ? logits : reinterpret_cast<float*>(ws + L.logits);
  p.topk_w = topk_w; p.topk_idx = topk_idx;
  p.xq8 = ws + L.xq8;
  p.xu = reinterpret_cast<int*>(ws + L.xu);
  p.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  return p;
}

PrefillParams prefill_params(const moe_v41_cfg* c, const void* x, int m, const void* router_w, const float* bias,
                             const float* bias_vl, const uint8_t* image_mask, const uint64_t* expert_ptrs,
                             int shared_kind, const void* sh1, const void* sh3, const void* sh2, float* out,
                             float* topk_w, int32_t* topk_idx, float* logits, uint8_t* ws, const WsLayout& L) {
  PrefillParams p{};
  p.m = m; p.D = c->dim; p.I = c->inter; p.N = c->n_routed; p.k = c->topk; p.norm = c->norm_topk_prob != 0;
  p.score_func = c->score_func;
  p.bias_vl = bias_vl; p.image_mask = image_mask;
  p.gate_temp = c->gate_temp; p.route_scale = c->route_scale; p.swiglu_limit = c->swiglu_limit;
  p.shared_kind = shared_kind;
  p.x = static_cast<const uint16_t*>(x);
  p.router_w = static_cast<const uint16_t*>(router_w);
  p.bias = bias;
  p.expert_ptrs = reinterpret_cast<const unsigned long long*>(expert_ptrs);
  p.sh1 = static_cast<const uint8_t*>(sh1);
  p.sh3 = static_cast<const uint8_t*>(sh3);
  p.sh2 = static_cast<const uint8_t*>(sh2);
  p.logits = logits ? logits : reinterpret_cast<float*>(ws + L.logits);
  p.topk_w = topk_w; p.topk_idx = topk_idx; p.out = out;
  p.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  p.pw = ws + L.pre;
  p.L = L.P;
  p.timeout_ns = timeout_ns(c);
  return p;
}

}  // namespace

int moe::route_topk(const moe_v41_cfg* cfg, int k, const void* x, int m, const void* router_w, const float* bias,
                    int32_t** idx_out, void* ws, size_t ws_bytes, cudaStream_t s) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!x || !router_w || !bias || !idx_out || m < 1 || m > cfg->max_tokens || m > DECODE_MAX_M) return MOE_ERR_ARG;
  if (k < 1 || k > MAX_TOPK || k > cfg->n_routed) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16)) return MOE_ERR_ALIGN;
  if ((rc = check_ws(cfg, ws, ws_bytes))) return rc;
  const WsLayout L = ws_layout(*cfg);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* idx = reinterpret_cast<int32_t*>(w + L.pred);
  float* wt = reinterpret_cast<float*>(idx + (size_t)m * k);
  *idx_out = idx;
  if (use_decode(cfg, m)) {
    RouteParams p = route_params(cfg, x, m, router_w, bias, nullptr, nullptr, nullptr, wt, idx, w, L);
    p.k = k;
    return launch_route_decode(p, s);
  }
  PrefillParams p = prefill_params(cfg, x, m, router_w, bias, nullptr, nullptr, nullptr, MOE_SHARED_BF16, nullptr,
                                   nullptr, nullptr, nullptr, wt, idx, nullptr, w, L);
  p.k = k;
  return launch_prefill_route(p, s);
}

extern "C" {

size_t moe_v41_workspace_bytes(const moe_v41_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

int moe_v41_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGN;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_v41_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, void* q8_out, void* stream) {
  if (!x || !q8_out || rows < 1 || cols < 32 || cols % 32) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(q8_out, 16)) return MOE_ERR_ALIGN;
  return launch_quantize_q8_1(x, x_is_f32, rows, cols, q8_out, (cudaStream_t)stream);
}

int moe_v41_select_from_logits(const moe_v41_cfg* cfg, const float* logits, int m, const float* bias,
                               float* topk_w, int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream) {
  return moe_v41_select_from_logits_vl(cfg, logits, m, bias, nullptr, nullptr, topk_w, topk_idx, ws, ws_bytes,
                                       stream);
}

int moe_v41_select_from_logits_vl(const moe_v41_cfg* cfg, const float* logits, int m, const float* bias,
                                  const float* bias_vl, const uint8_t* image_mask, float* topk_w,
                                  int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!logits || !bias || !topk_w || !topk_idx || m < 1 || m > cfg->max_tokens) return MOE_ERR_ARG;
  if ((rc = check_ws(cfg, ws, ws_bytes))) return rc;
  const WsLayout L = ws_layout(*cfg);
  SelectParams p{};
  p.logits = logits; p.bias = bias; p.bias_vl = bias_vl; p.image_mask = image_mask;
  p.m = m; p.N = cfg->n_routed; p.k = cfg->topk; p.score_func = cfg->score_func;
  p.norm = cfg->norm_topk_prob != 0; p.gate_temp = cfg->gate_temp; p.route_scale = cfg->route_scale;
  p.topk_w = topk_w; p.topk_idx = topk_idx;
  p.ctrl = reinterpret_cast<Ctrl*>(static_cast<uint8_t*>(ws) + L.ctrl);
  return launch_select(p, (cudaStream_t)stream);
}

int moe_v41_route(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                  float* logits_out, float* topk_w, int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream) {
  return moe_v41_route_vl(cfg, x, m, router_w, bias, nullptr, nullptr, logits_out, topk_w, topk_idx, ws, ws_bytes,
                          stream);
}

int moe_v41_route_vl(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                     const float* bias_vl, const uint8_t* image_mask, float* logits_out, float* topk_w,
                     int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!x || !router_w || !bias || !topk_w || !topk_idx || m < 1 || m > cfg->max_tokens) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16)) return MOE_ERR_ALIGN;
  if ((rc = check_ws(cfg, ws, ws_bytes))) return rc;
  const WsLayout L = ws_layout(*cfg);
  uint8_t* w = static_cast<uint8_t*>(ws);
  // the router kernel of the forward that would take these tokens (same logits)
  if (m <= DECODE_MAX_M && use_decode(cfg, m)) {
    RouteParams p = route_params(cfg, x, m, router_w, bias, bias_vl, image_mask, logits_out, topk_w, topk_idx, w, L);
    return launch_route_decode(p, (cudaStream_t)stream);
  }
  PrefillParams p = prefill_params(cfg, x, m, router_w, bias, bias_vl, image_mask, nullptr, MOE_SHARED_BF16, nullptr,
                                   nullptr, nullptr, nullptr, topk_w, topk_idx, logits_out, w, L);
  return launch_prefill_route(p, (cudaStream_t)stream);
}

int moe_v41_forward(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                    const uint64_t* expert_ptrs, int shared_kind, const void* sh_w1, const void* sh_w3,
                    const void* sh_w2, float* out, float* topk_w, int32_t* topk_idx, float* logits_out, void* ws,
                    size_t ws_bytes, void* stream) {
  return moe_v41_forward_vl(cfg, x, m, router_w, bias, nullptr, nullptr, expert_ptrs, shared_kind, sh_w1, sh_w3,
                            sh_w2, out, topk_w, topk_idx, logits_out, ws, ws_bytes, stream);
}

int moe_v41_forward_vl(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                       const float* bias_vl, const uint8_t* image_mask, const uint64_t* expert_ptrs, int shared_kind,
                       const void* sh_w1, const void* sh_w3, const void* sh_w2, float* out, float* topk_w,
                       int32_t* topk_idx, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!x || !router_w || !bias || !expert_ptrs || !sh_w1 || !sh_w3 || !sh_w2 || !out || !topk_w || !topk_idx)
    return MOE_ERR_ARG;
  if (m < 1 || m > cfg->max_tokens) return MOE_ERR_ARG;
  if (shared_kind != MOE_SHARED_BF16 && shared_kind != MOE_SHARED_KQUANT) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(expert_ptrs, 8)) return MOE_ERR_ALIGN;
  if (!aligned(sh_w1, 256) || !aligned(sh_w3, 256) || !aligned(sh_w2, 256)) return MOE_ERR_ALIGN;
  if ((rc = check_ws(cfg, ws, ws_bytes))) return rc;
  const WsLayout L = ws_layout(*cfg);
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaStream_t s = (cudaStream_t)stream;
  if (!use_decode(cfg, m)) {
    if (!prefill_possible(*cfg)) return MOE_ERR_ARG;
    PrefillParams p = prefill_params(cfg, x, m, router_w, bias, bias_vl, image_mask, expert_ptrs, shared_kind, sh_w1,
                                     sh_w3, sh_w2, out, topk_w, topk_idx, logits_out, w, L);
    return launch_prefill(p, s);
  }
  if (m > DECODE_MAX_M) return MOE_ERR_ARG;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;

  if (!decode_fits(cfg->dim, cfg->inter)) return MOE_ERR_ARG;
  DecodeParams dp{};
  dp.m = m; dp.D = cfg->dim; dp.I = cfg->inter; dp.N = cfg->n_routed; dp.k = cfg->topk;
  dp.norm = cfg->norm_topk_prob != 0; dp.score_func = cfg->score_func;
  dp.gate_temp = cfg->gate_temp; dp.route_scale = cfg->route_scale; dp.swiglu_limit = cfg->swiglu_limit;
  dp.shared_kind = shared_kind;
  dp.x = static_cast<const uint16_t*>(x);
  dp.router_w = static_cast<const uint16_t*>(router_w);
  dp.bias = bias; dp.bias_vl = bias_vl; dp.image_mask = image_mask;
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
  const int Td = cfg->max_tokens < DECODE_MAX_M ? cfg->max_tokens : DECODE_MAX_M;
  dp.shvec0 = Td * cfg->topk;
  dp.out = out;
  dp.ctrl = reinterpret_cast<Ctrl*>(w + L.ctrl);
  dp.timeout_ns = timeout_ns(cfg);
  return launch_decode_layer(dp, sms, s);
}

int moe_v41_kernel_launches(const moe_v41_cfg* cfg, int m, int shared_kind) {
  if (check_cfg(cfg) != MOE_OK || m < 1 || m > cfg->max_tokens) return -1;
  if (shared_kind != MOE_SHARED_BF16 && shared_kind != MOE_SHARED_KQUANT) return -1;
  if (use_decode(cfg, m)) return m <= DECODE_MAX_M && decode_fits(cfg->dim, cfg->inter) ? 1 : -1;
  return prefill_possible(*cfg) ? prefill_launches(shared_kind) : -1;
}

int moe_v41_read_status(void* ws, void* stream, uint32_t* status, int clear) {
  if (!ws || !status) return MOE_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, ws, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  if (clear) {
    if (cudaMemsetAsync(ws, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

const char* moe_v41_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_ALIGN: return "misaligned pointer";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA launch failure";
    default: return "unknown moe_v41 error";
  }
}

}  // extern "C"
