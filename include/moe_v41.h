/* moe_v41 — one DeepSeek-V4.1 MoE FFN layer forward on still-quantized experts,
 * hand-written for GB300 (sm_103a).
 *
 * The method (docs.metrale.ai, module metrale_model_arch::moe_v41 and its
 * moe_v41.rs source page; open-model-atlas "DeepSeek V4.1 · Mixture of
 * experts", the Router / Routed expert / Shared expert steps):
 *   z = x W_R^T (f32 accumulation)        s = sqrt(softplus(z / gate_temp))
 *   T = top-k of s + bias (stable, ties to the lower id)
 *   G_i = route_scale * s_i / (sum_T s + 1e-20)   (plain s_i when !norm or k == 1)
 *   per picked expert: g = W1 q8_1(x), u = W3 q8_1(x)  (Q2_K blocks)
 *                      h = min(g,L) sigmoid(min(g,L)) clip(u,-L,L)
 *                      E = W2 q8_1(h)                   (Q3_K blocks)
 *   out = sum_{i in T, ascending id} G_i E_i  +  S(x)   (shared expert last)
 *
 * Conventions for every call:
 *  - All pointers are caller-owned DEVICE memory unless stated otherwise.  The
 *    library allocates nothing and keeps no state between calls.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    is asynchronous on it; only moe_v41_read_status synchronises.
 *  - The return value reports argument and launch errors found on the host
 *    (MOE_ERR_*).  Conditions only the GPU can see (a NaN routing key, a picked
 *    expert with a NULL or misaligned slot pointer, an in-kernel wait that ran
 *    out) set bits of a status word inside the workspace (MOE_STATUS_*), read
 *    with moe_v41_read_status.
 *  - A workspace serves one call at a time.  It must be prepared once with
 *    moe_v41_workspace_init; every call leaves it ready for the next one.
 */
#ifndef MOE_V41_H
#define MOE_V41_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Layer configuration; mirrors the metrale MoeV41Cfg struct (moe_v41.rs source)
 * plus two execution fields and the DeepSeek Gate's score function. */
typedef struct {
  int32_t dim;              /* D, model width: multiple of 256, <= 7680 */
  int32_t inter;            /* I, expert hidden width: multiple of 256, <= 7680 */
  int32_t n_routed;         /* N, routed experts: 1..1024 */
  int32_t topk;             /* k, experts per token: 1..min(N, 16) */
  float gate_temp;          /* > 0; the logit is divided by it before the score function */
  int32_t norm_topk_prob;   /* non-zero: renormalise the k weights (when k > 1) */
  float route_scale;        /* weights are multiplied by it */
  float swiglu_limit;       /* L; <= 0 disables both clamps */
  int32_t max_tokens;       /* largest m the workspace is sized for: 1..65536 */
  int32_t path;             /* MOE_PATH_*: which kernel family runs */
  uint32_t wait_timeout_us; /* bound of every in-kernel wait; 0 = 2,000,000 */
  int32_t score_func;       /* MOE_SCORE_*; 0 = sqrt(softplus), the moe_v41 default */
} moe_v41_cfg;

/* Score functions of the DeepSeek V4.1 Gate (atlas page "Mixture of experts",
 * model.py Gate.forward), on t = f32(logit / gate_temp).  Each score is the
 * f64 evaluation of the formula rounded once to f32:
 *   MOE_SCORE_SQRTSOFTPLUS  sqrt(softplus(t)), softplus(t) = t above 20
 *   MOE_SCORE_SIGMOID       1 / (1 + exp(-t))
 *   MOE_SCORE_SOFTMAX       exp(t - max t) / sum over the experts of the same */
enum { MOE_SCORE_SQRTSOFTPLUS = 0, MOE_SCORE_SIGMOID = 1, MOE_SCORE_SOFTMAX = 2 };

enum {
  MOE_PATH_AUTO = 0,    /* decode kernels for m <= 8 when dim <= 5120 and inter <= 3328 (the widths one
                           decode stage holds), prefill kernels otherwise */
  MOE_PATH_DECODE = 1,  /* decode kernels for any m <= 8 (error above, or at wider shapes) */
  MOE_PATH_PREFILL = 2  /* prefill kernels for any m */
};

enum {
  MOE_SHARED_BF16 = 0,   /* shared w1/w3 bf16 [inter, dim] row-major, w2 bf16 [dim, inter] */
  MOE_SHARED_KQUANT = 1  /* shared w1/w3 Q2_K [inter][dim/256], w2 Q3_K [dim][inter/256] */
};

/* host-returned codes */
enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,        /* a size, count or configuration value out of range, or a NULL pointer */
  MOE_ERR_ALIGN = 2,      /* a pointer that must be aligned is not */
  MOE_ERR_WORKSPACE = 3,  /* workspace NULL, too small, or sized for fewer tokens */
  MOE_ERR_CUDA = 4        /* a CUDA launch or attribute call failed */
};

/* device status bits (moe_v41_read_status) */
enum {
  MOE_STATUS_NAN_KEY = 1u,          /* a routing key was NaN; it ranked below every number */
  MOE_STATUS_MISSING_EXPERT = 2u,   /* a picked expert's slot pointer was NULL or not 256-B aligned;
                                       its contribution was left out */
  MOE_STATUS_TIMEOUT = 4u           /* an in-kernel wait exceeded wait_timeout_us; outputs are invalid */
};

/* Bytes of workspace a configuration needs (for up to cfg->max_tokens tokens;
 * it includes the prefill kernels' buffers when cfg->path is MOE_PATH_PREFILL,
 * or MOE_PATH_AUTO with max_tokens > 8).  Returns 0 for an invalid
 * configuration. */
MOE_API size_t moe_v41_workspace_bytes(const moe_v41_cfg* cfg);

/* Prepare a workspace for first use: clears its control block and status word
 * (asynchronous on stream).  ws must be 256-B aligned. */
MOE_API int moe_v41_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* q8_1 quantisation of `rows` activation rows of `cols` values (cols a multiple
 * of 32): x is bf16 (x_is_f32 == 0) or f32, row-major [rows, cols].  Writes
 * rows * cols/32 blocks of 36 bytes to q8_out: fp16 d, fp16 s = d * sum(q),
 * int8 q[32]; d = amax/127, q = round-half-away(x/d), all decisions in f32
 * (the q8_1 activation format named in the moe_v41 module docs).  x and
 * q8_out 16-B aligned. */
MOE_API int moe_v41_quantize_q8_1(const void* x, int x_is_f32, int rows, int cols, void* q8_out, void* stream);

/* The routing step alone from given f32 logits [m, n_routed] (metrale
 * moe_v41.rs, fn route_from_logits; DeepSeek model.py Gate.forward): scores,
 * biased stable top-k, weights.  bias f32 [n_routed].  Writes topk_w f32
 * [m, topk] and topk_idx int32 [m, topk], each token's picks in descending
 * key order.  1 <= m <= cfg->max_tokens. */
MOE_API int moe_v41_select_from_logits(const moe_v41_cfg* cfg, const float* logits, int m, const float* bias,
                               float* topk_w, int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream);

/* The same with the image-token bias of the DeepSeek Gate (model.py
 * Gate.forward, torch.where(image_mask, bias_vl, bias)): token t picks with
 * bias_vl when image_mask[t] is non-zero.  bias_vl f32 [n_routed] and
 * image_mask uint8 [m] are DEVICE arrays; either NULL means no image token.
 * The weights stay the raw scores for every token.  The _vl forms of route
 * and forward below take the same two arguments after bias. */
MOE_API int moe_v41_select_from_logits_vl(const moe_v41_cfg* cfg, const float* logits, int m, const float* bias,
                                          const float* bias_vl, const uint8_t* image_mask, float* topk_w,
                                          int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream);

/* Router logits and routing for m tokens (the metrale route call, with the
 * selection on the device): x bf16 [m, dim], router_w bf16 [n_routed, dim]
 * (16-B aligned), bias f32 [n_routed].  logits_out (may be NULL) receives the
 * f32 logits [m, n_routed].  The router kernel is the one the forward of the
 * same tokens runs, with the same accumulation order, so the logits and the
 * picks equal the forward's bit for bit. */
MOE_API int moe_v41_route(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                  float* logits_out, float* topk_w, int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream);
MOE_API int moe_v41_route_vl(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                             const float* bias_vl, const uint8_t* image_mask, float* logits_out, float* topk_w,
                             int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream);

/* One MoE layer forward for m tokens (the metrale MoeV41::forward call, all
 * experts resident).  Up to eight tokens run the decode kernels (one
 * persistent launch of integer-dot GEMVs); above that, at widths the decode
 * kernel does not take, or with MOE_PATH_PREFILL, the prefill kernels (tokens grouped by expert, tensor-core
 * GEMMs on dequantised tiles; router logits then carry the tensor cores' f32
 * accumulation order).  The decode launch allows programmatic stream
 * serialisation: its blocks may set up while the previous launch on the
 * stream finishes, and read or write no global memory before it has
 * completed, so stream order holds as for any launch.
 *   x           bf16 [m, dim], 16-B aligned
 *   router_w    bf16 [n_routed, dim], 16-B aligned
 *   bias        f32 [n_routed]
 *   expert_ptrs DEVICE array of n_routed * 3 uint64 device addresses
 *               {w1, w3, w2} per expert: w1, w3 Q2_K [inter rows][dim/256
 *               blocks of 84 B]; w2 Q3_K [dim rows][inter/256 blocks of 110 B];
 *               raw GGUF block order, each 256-B aligned; 0 = not resident
 *               (picking it sets MOE_STATUS_MISSING_EXPERT)
 *   shared_kind MOE_SHARED_BF16 or MOE_SHARED_KQUANT; sh_w1, sh_w3, sh_w2 as
 *               described there, each 256-B aligned
 *   out         f32 [m, dim], overwritten (never accumulated into)
 *   topk_w      f32 [m, topk], topk_idx int32 [m, topk]: the routing
 *   logits_out  f32 [m, n_routed] or NULL
 *   ws          workspace of moe_v41_workspace_bytes(cfg) bytes, 256-B aligned */
MOE_API int moe_v41_forward(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                    const uint64_t* expert_ptrs, int shared_kind, const void* sh_w1, const void* sh_w3,
                    const void* sh_w2, float* out, float* topk_w, int32_t* topk_idx, float* logits_out, void* ws,
                    size_t ws_bytes, void* stream);
MOE_API int moe_v41_forward_vl(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w, const float* bias,
                               const float* bias_vl, const uint8_t* image_mask, const uint64_t* expert_ptrs,
                               int shared_kind, const void* sh_w1, const void* sh_w3, const void* sh_w2, float* out,
                               float* topk_w, int32_t* topk_idx, float* logits_out, void* ws, size_t ws_bytes,
                               void* stream);

/* Bytes of the fixed scratch array behind moe_v41_forward_noalloc (512 KiB).
 * Each GPU that loads this library holds it until the process exits. */
#define MOE_V41_NOALLOC_SCRATCH_BYTES (512u << 10)

/* moe_v41_forward for up to eight tokens (the decode kernels) WITHOUT a
 * caller workspace: the scratch lives in a fixed 512 KiB array owned by the
 * library on each device.  The pages describe no such call; it exists for
 * callers that have no way to obtain device memory at call time: a plugin
 * running inside a host engine that owns every byte of the GPU's memory
 * through its own pool and hands plugins no allocator, or a latency-critical
 * loop that must not call cudaMalloc (which can synchronise the device).
 *   Arguments are those of moe_v41_forward minus ws/ws_bytes, plus
 *   status_out: a DEVICE uint32_t (may be NULL) that receives this call's
 *   MOE_STATUS_* bits, written asynchronously on `stream`.
 *   Limits: cfg->max_tokens <= 8 and 1 <= m <= cfg->max_tokens; the
 *   workspace moe_v41_workspace_bytes(cfg) would need must fit in
 *   MOE_V41_NOALLOC_SCRATCH_BYTES, else MOE_ERR_WORKSPACE (the DeepSeek-V4.1
 *   shape, dim 5120 / inter 2304 / 384 experts / top-6 at 8 tokens, needs
 *   381,952 bytes).  Nothing is allocated: no cudaMalloc, cudaFree or
 *   allocating library call.
 *   Set-up: every call looks the array's device address up on the current
 *   device (cudaGetSymbolAddress, which allocates nothing).  The first call
 *   on a device may load the library's device code there: make that first
 *   call before any stream capture.  Each call first clears the control
 *   words and counters it starts from.  All calls share the one array, so
 *   calls whose work overlaps on the GPU (different streams, or different
 *   host threads) race: serialise
 *   them, e.g. by issuing them on one stream. */
MOE_API int moe_v41_forward_noalloc(const moe_v41_cfg* cfg, const void* x, int m, const void* router_w,
                                    const float* bias, const uint64_t* expert_ptrs, int shared_kind,
                                    const void* sh_w1, const void* sh_w3, const void* sh_w2, float* out,
                                    float* topk_w, int32_t* topk_idx, float* logits_out, uint32_t* status_out,
                                    void* stream);

/* Kernel launches one moe_v41_forward call with these arguments makes (for
 * launch accounting and graph capture sizing); -1 for invalid arguments. */
MOE_API int moe_v41_kernel_launches(const moe_v41_cfg* cfg, int m, int shared_kind);

/* Synchronise `stream`, then copy the workspace status word (MOE_STATUS_* bits
 * accumulated since the last clear) to *status (host memory); clear == non-zero
 * resets it to 0. */
MOE_API int moe_v41_read_status(void* ws, void* stream, uint32_t* status, int clear);

/* Static text for a MOE_ERR_* code. */
MOE_API const char* moe_v41_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif
