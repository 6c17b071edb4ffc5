/* moe_v41 expert cache — routed experts streamed from a host-resident arena
 * into a least-recently-used set of HBM slots, and the next layer's experts
 * predicted and fetched ahead.
 *
 * The method (docs.metrale.ai, module metrale_model_arch::moe_v41: the
 * routed experts are streamed, still quantized; per token the router picks
 * topk experts and the ExpertLru gathers their raw slices into its
 * device-visible slots, reading misses from the ExpertSource; the
 * deepseek_v41 layer page: the arena is page-locked host memory with
 * METRALE_DS41_ARENA_DEVICE=0; moe_v41.rs source: the slot table marks a
 * non-resident expert with -1, and METRALE_DS41_PREFETCH_K, read once,
 * sets how many of the next layer's experts, predicted by the next layer's
 * router on this layer's single-token input, start loading while this layer
 * computes; struct MoeV41 stage_m1 / compute_m1: the host span between the
 * router and the expert compute selects, fetches the cache and refreshes the
 * pointer table, and the compute then reads only the table).
 *
 * The arena holds every expert of every covered layer in one slot layout
 * ([n_layers][n_routed] slots of slot_bytes, the gate / up / down blocks at
 * off_w1 / off_w3 / off_w2, each 256-B aligned); the HBM slots use the same
 * layout.  The cache keeps, for every covered layer, the [n_routed][3] slot
 * pointer table that moe_v41_forward reads: the HBM addresses of a resident
 * expert's three matrices, or NULL (not resident: a forward that picks it
 * sets MOE_STATUS_MISSING_EXPERT and leaves it out).
 *
 * Ownership: the arena (host), the slots and the tables (device) are the
 * caller's; the cache object holds only host-side bookkeeping and CUDA
 * events, created by moe_v41_cache_create and released by
 * moe_v41_cache_destroy.  It is not thread-safe: one host thread drives it.
 *
 * Streams: misses are copied (one cudaMemcpyAsync per expert from the arena,
 * which should be page-locked so the copies are asynchronous) and the tables
 * updated on a copy stream.  Work on other streams is ordered against them by
 * two calls: moe_v41_cache_wait before work that reads a layer's table, and
 * moe_v41_cache_reads after work that reads experts, so a slot is never
 * overwritten while enqueued work may still read it.
 *
 * Errors: a call that returns MOE_ERR_ARG changed nothing.  After
 * MOE_ERR_CUDA the host bookkeeping may no longer match the device tables:
 * drain the streams and destroy the cache.
 *
 * Simulation mode: with slots and tables both NULL the cache makes no CUDA
 * call at all; moe_v41_cache_fetch then only runs the replacement policy and
 * counts (hits, misses, evictions, bytes), e.g. to size the slot count from a
 * routing trace.
 */
#ifndef MOE_V41_CACHE_H
#define MOE_V41_CACHE_H

#include "moe_v41.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_v41_cache moe_v41_cache; /* opaque */

typedef struct {
  int32_t n_layers;    /* layers the arena covers: 1..4096 */
  int32_t n_routed;    /* experts per layer: 1..1024 */
  int32_t n_slots;     /* HBM slots: 1..65536 */
  uint64_t slot_bytes; /* bytes of one expert slot: a multiple of 256 */
  uint64_t off_w1, off_w3, off_w2; /* offsets of the gate, up and down blocks in a slot: multiples of 256 */
  const void* arena;   /* HOST [n_layers][n_routed] slots (page-locked for asynchronous copies), or NULL in simulation mode */
  void* slots;         /* DEVICE [n_slots] slots, 256-B aligned, or NULL (simulation mode) */
  uint64_t* tables;    /* DEVICE [n_layers][n_routed][3] slot pointer tables, 8-B aligned, or NULL (simulation mode) */
} moe_v41_cache_cfg;

typedef struct {
  uint64_t hits;            /* demanded experts found resident */
  uint64_t misses;          /* demanded experts copied in */
  uint64_t evictions;       /* resident experts dropped to make room */
  uint64_t bytes_copied;    /* arena -> slot bytes, demand and prefetch */
  uint64_t prefetched;      /* experts copied in by a prefetch */
  uint64_t prefetch_hits;   /* demanded experts that a prefetch had brought in */
} moe_v41_cache_stats;

/* Creates the cache with every table entry NULL (a memset of the tables on
 * `stream`; none in simulation mode).  Errors: MOE_ERR_ARG (sizes, offsets,
 * or exactly one of slots / tables NULL, or arena NULL with slots given),
 * MOE_ERR_ALIGN, MOE_ERR_CUDA. */
MOE_API int moe_v41_cache_create(const moe_v41_cache_cfg* cfg, void* stream, moe_v41_cache** out);

/* Releases the host state.  The caller must have drained the streams the
 * cache used. */
MOE_API int moe_v41_cache_destroy(moe_v41_cache* cache);

/* Makes experts[0..n) of `layer` (host array; repeats allowed) resident.
 * Resident ones become the most recently used; each miss takes the least
 * recently used slot that this call does not need (its old expert's table
 * entry becomes NULL), is copied in on `copy_stream`, and gets its table
 * entry.  prefetch != 0 marks the copies as a prefetch (the experts need not
 * be used soon; counted apart).  The distinct count must not exceed n_slots.
 * Free slots are taken in ascending order first.  Asynchronous: the table
 * update completes on copy_stream (every fetch of a cache must use the same
 * copy stream); order a reader with moe_v41_cache_wait.  Errors: MOE_ERR_ARG,
 * MOE_ERR_CUDA. */
MOE_API int moe_v41_cache_fetch(moe_v41_cache* cache, int layer, const int32_t* experts, int n, int prefetch,
                                void* copy_stream);

/* Makes `stream` wait for every table update of `layer` issued so far. */
MOE_API int moe_v41_cache_wait(moe_v41_cache* cache, int layer, void* stream);

/* Records that the work enqueued on `stream` so far reads experts[0..n) of
 * `layer` (host array), or, with experts NULL, every expert of the layer
 * resident now: a later fetch does not overwrite those slots before that
 * work completes. */
MOE_API int moe_v41_cache_reads(moe_v41_cache* cache, int layer, const int32_t* experts, int n, void* stream);

/* The slot holding (layer, expert), or -1. */
MOE_API int moe_v41_cache_slot_of(const moe_v41_cache* cache, int layer, int expert);

/* Counters since creation. */
MOE_API int moe_v41_cache_get_stats(const moe_v41_cache* cache, moe_v41_cache_stats* out);

/* One layer forward with the routed experts streamed through the cache (the
 * metrale single-token step: router, host selection span, cache fetch,
 * pointer-table compute).  In order:
 *  1. when next_router_w is given, prefetch_k > 0, m == 1 and layer + 1 <
 *     n_layers: the next layer's router and selection on this x (topk =
 *     prefetch_k, the next layer's bias; score function as cfg) -- the
 *     prediction;
 *  2. moe_v41_route on this layer (same logits and picks as the forward's
 *     own: the two router kernels share one accumulation order);
 *  3. the picks (and predictions) are copied to host_picks (HOST, m*topk +
 *     prefetch_k int32, page-locked for speed) and `stream` is synchronised;
 *  4. moe_v41_cache_fetch of the picks on copy_stream, `stream` waits for it;
 *  5. moe_v41_forward with this layer's cache table on `stream`, then
 *     moe_v41_cache_reads of the picks;
 *  6. moe_v41_cache_fetch of the predictions (prefetch) on copy_stream,
 *     overlapping the forward.
 * Arguments as moe_v41_forward; cfg->path must not be MOE_PATH_PREFILL when
 * m <= 8 is to use the decode kernels (any path works).  The slot count must
 * hold min(m*topk, n_routed) + prefetch_k experts.  Returns after enqueuing step 5 and 6;
 * synchronises `stream` once (step 3). */
MOE_API int moe_v41_forward_streamed(const moe_v41_cfg* cfg, moe_v41_cache* cache, int layer, const void* x, int m,
                                     const void* router_w, const float* bias, const void* next_router_w,
                                     const float* next_bias, int prefetch_k, int shared_kind, const void* sh_w1,
                                     const void* sh_w3, const void* sh_w2, float* out, float* topk_w,
                                     int32_t* topk_idx, void* ws, size_t ws_bytes, int32_t* host_picks,
                                     void* stream, void* copy_stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_V41_CACHE_H */
