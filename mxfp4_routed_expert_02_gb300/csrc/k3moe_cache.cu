// k3moe_cache.cu -- host-side expert cache (slot states, LRU victims, pinned hits) and its
// C ABI: create, destroy, lookup (host only), statistics.  The streamed layer step that
// uses it is in k3moe_api.cu.  Policy: README of FareedKhan-dev/kimi-k3-in-c, section 12
// "An LRU cache for the experts"; README of Maknee/Kimi-K3.cpp, "The consumer-memory
// idea", items 3-5.
#include <algorithm>
#include <new>

#include "k3moe_cache.h"

namespace k3 {

namespace {

// The page's victim choice: skip slots in flight; an empty slot is taken at once; skip
// pinned slots; otherwise the least recently used.  -1 when every slot is pinned or in
// flight.
int pick_victim(const k3moe_expert_cache *c) {
  int best = -1;
  uint64_t oldest = ~0ull;
  for (int s = 0; s < c->n_slots; s++) {
    if (c->key_of[s] == kSlotInflight) continue;
    if (c->key_of[s] == kSlotEmpty) return s;
    if (c->pinned[s]) continue;
    if (c->used_at[s] < oldest) {
      oldest = c->used_at[s];
      best = s;
    }
  }
  return best;
}

}  // namespace

k3moe_status cache_reserve(k3moe_expert_cache *c, int layer, const int32_t *experts, int n,
                           int32_t *slots, int32_t *load) {
  const int64_t E = c->n_experts;
  // first, without changing anything: do the call's distinct misses fit in the slots that
  // its hits leave (between calls no slot is pinned or in flight)?
  {
    std::vector<int64_t> keys;
    keys.reserve(n);
    for (int j = 0; j < n; j++)
      if (experts[j] >= 0 && experts[j] < E) keys.push_back((int64_t)layer * E + experts[j]);
    std::sort(keys.begin(), keys.end());
    keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
    if ((int)keys.size() > c->n_slots) {  // hits keep their slots; misses need the rest
      for (int j = 0; j < n; j++) {
        slots[j] = -1;
        load[j] = 0;
      }
      return K3MOE_ERR_CACHE_FULL;
    }
  }
  c->clock++;
  // phase 1a: pin every selected hit before any victim is chosen
  for (int j = 0; j < n; j++) {
    slots[j] = -1;
    load[j] = 0;
    const int32_t e = experts[j];
    if (e < 0 || e >= E) continue;
    const int64_t key = (int64_t)layer * E + e;
    const int32_t s = c->slot_of[key];
    if (s >= 0 && c->key_of[s] == key) {
      if (!c->pinned[s]) c->hits++;
      c->pinned[s] = 1;
      c->used_at[s] = c->clock;
      slots[j] = s;
    }
  }
  // phase 1b: reserve a slot for every miss, serially
  for (int j = 0; j < n; j++) {
    const int32_t e = experts[j];
    if (e < 0 || e >= E || slots[j] >= 0) continue;
    const int64_t key = (int64_t)layer * E + e;
    const int32_t r = c->slot_of[key];
    if (r >= 0 && c->key_of[r] == kSlotInflight && c->pinned[r]) {  // reserved above
      slots[j] = r;
      continue;
    }
    const int s = pick_victim(c);  // never -1: the count above left room for every miss
    const int64_t old = c->key_of[s];
    if (old >= 0) c->slot_of[old] = -1;  // evicted
    c->key_of[s] = kSlotInflight;
    c->pinned[s] = 1;
    c->used_at[s] = c->clock;
    c->slot_of[key] = s;
    slots[j] = s;
    load[j] = 1;
    c->misses++;
  }
  return K3MOE_OK;
}

void cache_publish(k3moe_expert_cache *c, int layer, const int32_t *experts, int n,
                   const int32_t *slots, const int32_t *load, const int32_t *ok) {
  const int64_t E = c->n_experts;
  for (int j = 0; j < n; j++) {
    if (!load[j]) continue;
    const int64_t key = (int64_t)layer * E + experts[j];
    if (ok[j]) {
      c->key_of[slots[j]] = key;
      c->bytes_loaded += c->record_bytes;
    } else {
      c->key_of[slots[j]] = kSlotEmpty;
      c->slot_of[key] = -1;
    }
  }
  for (int s = 0; s < c->n_slots; s++) c->pinned[s] = 0;
}

}  // namespace k3

extern "C" {

k3moe_status k3moe_cache_create(int32_t n_layers, const uint8_t *const *host_experts,
                                int32_t n_experts, int64_t record_bytes, int64_t host_stride,
                                uint8_t *slots, int32_t n_slots, int64_t slot_stride,
                                k3moe_expert_cache **out) {
  if (!out) return K3MOE_ERR_ARG;
  *out = nullptr;
  if (n_layers < 1 || n_experts < 1 || n_experts > 4096 || n_slots < 1 || record_bytes < 1 ||
      !host_experts || !slots)
    return K3MOE_ERR_ARG;
  if ((long long)n_layers * n_experts > (1ll << 24)) return K3MOE_ERR_ARG;
  if (host_stride < record_bytes || slot_stride < record_bytes || slot_stride % 16)
    return K3MOE_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(slots) & 15) return K3MOE_ERR_ALIGN;
  for (int l = 0; l < n_layers; l++)
    if (!host_experts[l]) return K3MOE_ERR_ARG;
  k3moe_expert_cache *c = new (std::nothrow) k3moe_expert_cache();
  if (!c) return K3MOE_ERR_ARG;
  c->n_layers = n_layers;
  c->n_experts = n_experts;
  c->n_slots = n_slots;
  c->record_bytes = record_bytes;
  c->host_stride = host_stride;
  c->slot_stride = slot_stride;
  c->host.assign(host_experts, host_experts + n_layers);
  c->slots = slots;
  c->key_of.assign(n_slots, k3::kSlotEmpty);
  c->used_at.assign(n_slots, 0);
  c->pinned.assign(n_slots, 0);
  c->slot_of.assign((size_t)n_layers * n_experts, -1);
  *out = c;
  return K3MOE_OK;
}

k3moe_status k3moe_cache_destroy(k3moe_expert_cache *cache) {
  delete cache;
  return K3MOE_OK;
}

k3moe_status k3moe_cache_lookup(k3moe_expert_cache *c, int32_t layer, const int32_t *experts,
                                int32_t n, int32_t *slots, int32_t *load) {
  if (!c || !experts || !slots || !load || n < 0) return K3MOE_ERR_ARG;
  if (layer < 0 || layer >= c->n_layers) return K3MOE_ERR_ARG;
  std::lock_guard<std::mutex> lk(c->mu);
  const k3moe_status s = k3::cache_reserve(c, layer, experts, n, slots, load);
  if (s != K3MOE_OK) return s;
  std::vector<int32_t> ok(load, load + n);  // the caller reads what it was told to load
  k3::cache_publish(c, layer, experts, n, slots, load, ok.data());
  return K3MOE_OK;
}

k3moe_status k3moe_cache_stats(k3moe_expert_cache *c, int64_t *hits, int64_t *misses,
                               int64_t *bytes_loaded) {
  if (!c) return K3MOE_ERR_ARG;
  std::lock_guard<std::mutex> lk(c->mu);
  if (hits) *hits = c->hits;
  if (misses) *misses = c->misses;
  if (bytes_loaded) *bytes_loaded = c->bytes_loaded;
  return K3MOE_OK;
}

}  // extern "C"
