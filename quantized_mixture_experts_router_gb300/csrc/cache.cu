// The expert cache of include/moe_v41_cache.h: routed experts of a
// host-resident arena held in a least-recently-used set of HBM slots, the
// per-layer slot pointer tables the forward reads, and the streamed forward
// that routes, fetches and predicts the next layer's experts.
//
// Method: docs.metrale.ai moe_v41 module docs (the ExpertLru gathers the
// picked experts' raw slices into device-visible slots, misses read from the
// ExpertSource); the deepseek_v41 layer page (a page-locked host arena,
// METRALE_DS41_ARENA_DEVICE=0); moe_v41.rs source (slot table with -1 for a
// non-resident expert; METRALE_DS41_PREFETCH_K, the next layer's router on
// this layer's single-token input); struct MoeV41 stage_m1 / compute_m1.
//
// Host bookkeeping only lives here; the device work is cudaMemcpyAsync of
// whole expert slots, one small kernel that rewrites table entries, and the
// library's own route / forward launches.
#include <algorithm>
#include <new>
#include <vector>

#include "internal.h"
#include "../../include/moe_v41_cache.h"

namespace moe {
namespace {

constexpr int TS_MAX = 64;   // table entries one k_table_set launch writes
constexpr int RING = 256;    // reader events in flight before the host waits

struct TableSet {
  int n;
  uint32_t index[TS_MAX];                // layer * n_routed + expert
  unsigned long long ptr[TS_MAX][3];     // gate, up, down block addresses (0 = not resident)
};

__global__ void k_table_set(unsigned long long* tables, TableSet s) {
  const int i = threadIdx.x;
  if (i < s.n) {
    unsigned long long* e = tables + (size_t)s.index[i] * 3;
    e[0] = s.ptr[i][0];
    e[1] = s.ptr[i][1];
    e[2] = s.ptr[i][2];
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

struct moe_v41_cache {
  moe_v41_cache_cfg c{};
  bool sim = false;
  std::vector<int32_t> slot_of;      // key (layer * n_routed + expert) -> slot, or -1
  std::vector<int64_t> key_of;       // slot -> key, or -1 (free)
  std::vector<int32_t> prv, nxt;     // recency list over the slots: head = most recently used
  int32_t head = -1, tail = -1;
  std::vector<uint8_t> pre;          // slot brought in by a prefetch, not demanded since
  std::vector<uint64_t> last_read;   // slot -> reader sequence number (0: none)
  std::vector<uint32_t> mark;        // slot -> stamp of the fetch that needs it
  uint32_t stamp = 0;
  uint64_t seq = 0;                  // reader sequence numbers handed out
  cudaEvent_t ring[RING] = {};
  std::vector<cudaEvent_t> table_ev; // per layer: after its latest table update
  std::vector<uint8_t> table_rec;
  moe_v41_cache_stats st{};

  void unlink(int32_t s) {
    if (prv[s] >= 0) nxt[prv[s]] = nxt[s]; else head = nxt[s];
    if (nxt[s] >= 0) prv[nxt[s]] = prv[s]; else tail = prv[s];
    prv[s] = nxt[s] = -1;
  }
  void push_head(int32_t s) {
    prv[s] = -1;
    nxt[s] = head;
    if (head >= 0) prv[head] = s;
    head = s;
    if (tail < 0) tail = s;
  }
  void touch(int32_t s) {
    if (head == s) return;
    unlink(s);
    push_head(s);
  }
  unsigned long long addr(int32_t s, uint64_t off) const {
    return (unsigned long long)(reinterpret_cast<uintptr_t>(c.slots) + (uint64_t)s * c.slot_bytes + off);
  }
};

namespace {

int release(moe_v41_cache* k) {
  if (!k) return MOE_ERR_ARG;
  if (!k->sim) {
    for (cudaEvent_t& e : k->ring)
      if (e) cudaEventDestroy(e);
    for (cudaEvent_t& e : k->table_ev)
      if (e) cudaEventDestroy(e);
  }
  delete k;
  return MOE_OK;
}

// Table entries of one fetch, written by as few k_table_set launches as needed.
int write_tables(moe_v41_cache* k, const std::vector<std::pair<int64_t, int32_t>>& sets, cudaStream_t s) {
  TableSet ts{};
  for (size_t i = 0; i < sets.size(); ++i) {
    const int j = ts.n++;
    ts.index[j] = (uint32_t)sets[i].first;
    const int32_t slot = sets[i].second;
    ts.ptr[j][0] = slot < 0 ? 0ull : k->addr(slot, k->c.off_w1);
    ts.ptr[j][1] = slot < 0 ? 0ull : k->addr(slot, k->c.off_w3);
    ts.ptr[j][2] = slot < 0 ? 0ull : k->addr(slot, k->c.off_w2);
    if (ts.n == TS_MAX || i + 1 == sets.size()) {
      k_table_set<<<1, TS_MAX, 0, s>>>(reinterpret_cast<unsigned long long*>(k->c.tables), ts);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
      ts.n = 0;
    }
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_v41_cache_create(const moe_v41_cache_cfg* cfg, void* stream, moe_v41_cache** out) {
  if (!cfg || !out) return MOE_ERR_ARG;
  *out = nullptr;
  const moe_v41_cache_cfg& c = *cfg;
  if (c.n_layers < 1 || c.n_layers > 4096 || c.n_routed < 1 || c.n_routed > MAX_N || c.n_slots < 1 ||
      c.n_slots > 65536)
    return MOE_ERR_ARG;
  if (c.slot_bytes == 0 || c.slot_bytes % 256 || c.off_w1 % 256 || c.off_w3 % 256 || c.off_w2 % 256 ||
      c.off_w1 >= c.slot_bytes || c.off_w3 >= c.slot_bytes || c.off_w2 >= c.slot_bytes)
    return MOE_ERR_ARG;
  const bool sim = !c.slots && !c.tables;
  if (!sim && (!c.slots || !c.tables || !c.arena)) return MOE_ERR_ARG;
  if (!sim && (!aligned(c.slots, 256) || !aligned(c.tables, 8))) return MOE_ERR_ALIGN;

  moe_v41_cache* k = new (std::nothrow) moe_v41_cache();
  if (!k) return MOE_ERR_ARG;
  k->c = c;
  k->sim = sim;
  const size_t keys = (size_t)c.n_layers * c.n_routed;
  k->slot_of.assign(keys, -1);
  k->key_of.assign(c.n_slots, -1);
  k->prv.assign(c.n_slots, -1);
  k->nxt.assign(c.n_slots, -1);
  k->pre.assign(c.n_slots, 0);
  k->last_read.assign(c.n_slots, 0);
  k->mark.assign(c.n_slots, 0);
  for (int32_t s = 0; s < c.n_slots; ++s) k->push_head(s);  // the tail (taken first) is slot 0
  k->table_ev.assign(c.n_layers, nullptr);
  k->table_rec.assign(c.n_layers, 0);
  if (!sim) {
    bool ok = true;
    for (cudaEvent_t& e : k->ring) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    for (cudaEvent_t& e : k->table_ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    cudaStream_t s = (cudaStream_t)stream;
    ok = ok && cudaMemsetAsync(c.tables, 0, keys * 3 * sizeof(uint64_t), s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) {
      release(k);
      return MOE_ERR_CUDA;
    }
  }
  *out = k;
  return MOE_OK;
}

int moe_v41_cache_destroy(moe_v41_cache* cache) { return release(cache); }

int moe_v41_cache_fetch(moe_v41_cache* k, int layer, const int32_t* experts, int n, int prefetch, void* copy_stream) {
  if (!k || layer < 0 || layer >= k->c.n_layers || n < 0 || (n > 0 && !experts)) return MOE_ERR_ARG;
  const int N = k->c.n_routed;
  std::vector<int32_t> ids(experts, experts + n);
  for (int32_t e : ids)
    if (e < 0 || e >= N) return MOE_ERR_ARG;
  std::sort(ids.begin(), ids.end());
  ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
  if ((int)ids.size() > k->c.n_slots) return MOE_ERR_ARG;

  const uint32_t stamp = ++k->stamp;
  const int64_t base = (int64_t)layer * N;
  // resident ones: most recently used now, and off limits to this call's evictions
  for (int32_t e : ids) {
    const int32_t s = k->slot_of[base + e];
    if (s < 0) continue;
    k->mark[s] = stamp;
    k->touch(s);
    if (!prefetch) {
      ++k->st.hits;
      if (k->pre[s]) {
        ++k->st.prefetch_hits;
        k->pre[s] = 0;
      }
    }
  }
  // misses: the least recently used slot this call does not need
  std::vector<std::pair<int32_t, int64_t>> fills;       // (slot, key)
  std::vector<std::pair<int64_t, int32_t>> sets;        // (key, slot or -1)
  std::vector<uint64_t> waits;                          // reader sequence numbers to wait for
  std::vector<int32_t> layers_touched{layer};
  for (int32_t e : ids) {
    const int64_t key = base + e;
    if (k->slot_of[key] >= 0) continue;
    int32_t s = k->tail;
    while (s >= 0 && k->mark[s] == stamp) s = k->prv[s];
    if (s < 0) return MOE_ERR_ARG;  // cannot happen: ids.size() <= n_slots
    const int64_t old = k->key_of[s];
    if (old >= 0) {
      k->slot_of[old] = -1;
      ++k->st.evictions;
      sets.emplace_back(old, -1);
      layers_touched.push_back((int32_t)(old / N));
      if (k->last_read[s]) waits.push_back(k->last_read[s]);
    }
    k->key_of[s] = key;
    k->slot_of[key] = s;
    k->mark[s] = stamp;
    k->pre[s] = prefetch ? 1 : 0;
    k->last_read[s] = 0;
    k->touch(s);
    if (prefetch) ++k->st.prefetched; else ++k->st.misses;
    k->st.bytes_copied += k->c.slot_bytes;
    fills.emplace_back(s, key);
    sets.emplace_back(key, s);
  }
  if (k->sim || fills.empty()) return MOE_OK;

  cudaStream_t cs = (cudaStream_t)copy_stream;
  // readers of the slots about to be overwritten finish first (a ring event is
  // only re-recorded after it completed, so a newer record is a later point)
  std::sort(waits.begin(), waits.end());
  waits.erase(std::unique(waits.begin(), waits.end()), waits.end());
  for (uint64_t r : waits)
    if (cudaStreamWaitEvent(cs, k->ring[r % RING], 0) != cudaSuccess) return MOE_ERR_CUDA;
  const uint8_t* arena = static_cast<const uint8_t*>(k->c.arena);
  uint8_t* slots = static_cast<uint8_t*>(k->c.slots);
  for (const auto& f : fills)
    if (cudaMemcpyAsync(slots + (size_t)f.first * k->c.slot_bytes, arena + (size_t)f.second * k->c.slot_bytes,
                        k->c.slot_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return MOE_ERR_CUDA;
  int rc = write_tables(k, sets, cs);
  if (rc) return rc;
  std::sort(layers_touched.begin(), layers_touched.end());
  layers_touched.erase(std::unique(layers_touched.begin(), layers_touched.end()), layers_touched.end());
  for (int32_t l : layers_touched) {
    if (cudaEventRecord(k->table_ev[l], cs) != cudaSuccess) return MOE_ERR_CUDA;
    k->table_rec[l] = 1;
  }
  return MOE_OK;
}

int moe_v41_cache_wait(moe_v41_cache* k, int layer, void* stream) {
  if (!k || layer < 0 || layer >= k->c.n_layers) return MOE_ERR_ARG;
  if (k->sim || !k->table_rec[layer]) return MOE_OK;
  return cudaStreamWaitEvent((cudaStream_t)stream, k->table_ev[layer], 0) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_v41_cache_reads(moe_v41_cache* k, int layer, const int32_t* experts, int n, void* stream) {
  if (!k || layer < 0 || layer >= k->c.n_layers || n < 0) return MOE_ERR_ARG;
  const int N = k->c.n_routed;
  const uint64_t q = ++k->seq;
  if (!k->sim) {
    cudaEvent_t& e = k->ring[q % RING];
    // the ring entry's previous reader must be done before the event is reused
    if (q > (uint64_t)RING && cudaEventSynchronize(e) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventRecord(e, (cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  const int64_t base = (int64_t)layer * N;
  if (experts) {
    for (int i = 0; i < n; ++i) {
      if (experts[i] < 0 || experts[i] >= N) return MOE_ERR_ARG;
      const int32_t s = k->slot_of[base + experts[i]];
      if (s >= 0) k->last_read[s] = q;
    }
  } else {
    for (int e = 0; e < N; ++e) {
      const int32_t s = k->slot_of[base + e];
      if (s >= 0) k->last_read[s] = q;
    }
  }
  return MOE_OK;
}

int moe_v41_cache_slot_of(const moe_v41_cache* k, int layer, int expert) {
  if (!k || layer < 0 || layer >= k->c.n_layers || expert < 0 || expert >= k->c.n_routed) return -1;
  return k->slot_of[(size_t)layer * k->c.n_routed + expert];
}

int moe_v41_cache_get_stats(const moe_v41_cache* k, moe_v41_cache_stats* out) {
  if (!k || !out) return MOE_ERR_ARG;
  *out = k->st;
  return MOE_OK;
}

int moe_v41_forward_streamed(const moe_v41_cfg* cfg, moe_v41_cache* k, int layer, const void* x, int m,
                             const void* router_w, const float* bias, const void* next_router_w,
                             const float* next_bias, int prefetch_k, int shared_kind, const void* sh_w1,
                             const void* sh_w3, const void* sh_w2, float* out, float* topk_w, int32_t* topk_idx,
                             void* ws, size_t ws_bytes, int32_t* host_picks, void* stream, void* copy_stream) {
  if (!cfg || !k || k->sim || !host_picks || layer < 0 || layer >= k->c.n_layers) return MOE_ERR_ARG;
  if (cfg->n_routed != k->c.n_routed || m < 1 || m > cfg->max_tokens || prefetch_k < 0 || prefetch_k > MAX_TOPK ||
      prefetch_k > cfg->n_routed)
    return MOE_ERR_ARG;
  const int P = (next_router_w && next_bias && prefetch_k > 0 && m == 1 && layer + 1 < k->c.n_layers) ? prefetch_k : 0;
  const int picks = m * cfg->topk;
  if (std::min(picks, cfg->n_routed) + P > k->c.n_slots) return MOE_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int rc;
  // 1. the prediction: the next layer's router and selection on this input
  int32_t* pred_idx = nullptr;
  if (P && (rc = route_topk(cfg, P, x, m, next_router_w, next_bias, &pred_idx, ws, ws_bytes, s))) return rc;
  // 2. this layer's routing (the same picks the forward makes)
  if ((rc = moe_v41_route(cfg, x, m, router_w, bias, nullptr, topk_w, topk_idx, ws, ws_bytes, stream))) return rc;
  // 3. the host span: picks and predictions to the host
  if (cudaMemcpyAsync(host_picks, topk_idx, (size_t)picks * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (P && cudaMemcpyAsync(host_picks + picks, pred_idx, (size_t)P * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  // 4. the picks resident, the forward's stream after the table update
  if ((rc = moe_v41_cache_fetch(k, layer, host_picks, picks, 0, copy_stream))) return rc;
  if ((rc = moe_v41_cache_wait(k, layer, stream))) return rc;
  // 5. the layer on the cache's table
  const uint64_t* table = k->c.tables + (size_t)layer * k->c.n_routed * 3;
  if ((rc = moe_v41_forward(cfg, x, m, router_w, bias, table, shared_kind, sh_w1, sh_w3, sh_w2, out, topk_w,
                            topk_idx, nullptr, ws, ws_bytes, stream)))
    return rc;
  if ((rc = moe_v41_cache_reads(k, layer, host_picks, picks, stream))) return rc;
  // 6. the predicted experts of the next layer, behind this layer's compute
  if (P && (rc = moe_v41_cache_fetch(k, layer + 1, host_picks + picks, P, 1, copy_stream))) return rc;
  return MOE_OK;
}

}  // extern "C"
