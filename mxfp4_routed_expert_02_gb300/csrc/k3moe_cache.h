// k3moe_cache.h -- the host-side expert cache behind k3moe_layer_streamed (internal).
//
// The policy is the pages' (README of FareedKhan-dev/kimi-k3-in-c, section 12 "An LRU
// cache for the experts": slot states, victim choice, reserve / read / publish; README of
// Maknee/Kimi-K3.cpp, "The consumer-memory idea", items 3-5: fixed slots of one expert
// each, every selected hit pinned before any victim is chosen, all misses of a step read
// as one batch).  Here a slot is a record-sized piece of the caller's device memory and a
// read is a host-to-device copy from the caller's host copy of the layer's experts.
#pragma once
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "k3moe.h"

struct k3moe_expert_cache {
  int32_t n_layers = 0, n_experts = 0, n_slots = 0;
  int64_t record_bytes = 0, host_stride = 0, slot_stride = 0;
  std::vector<const uint8_t *> host;  // per layer: expert e at host[l] + e * host_stride
  uint8_t *slots = nullptr;           // device: slot s at slots + s * slot_stride
  std::vector<int64_t> key_of;        // per slot: layer * E + expert, or kEmpty / kInflight
  std::vector<uint64_t> used_at;      // per slot: clock of its last use
  std::vector<uint8_t> pinned;        // per slot: selected by the call in progress
  std::vector<int32_t> slot_of;       // per (layer, expert): its slot, or -1
  uint64_t clock = 0;
  int64_t hits = 0, misses = 0, bytes_loaded = 0;
  std::mutex mu;
  // host scratch of one call (routes in, slots out)
  std::vector<int32_t> route_host, slot_host, load_host;
  // pinned copy of a pass's slot indices, read by a copy on the call's stream; the next
  // pass rewrites it only after its own route read-back has synchronised that stream
  int32_t *slot_pin = nullptr;
  size_t slot_pin_n = 0;
  ~k3moe_expert_cache() {
    if (slot_pin) cudaFreeHost(slot_pin);
  }
};

namespace k3 {

constexpr int64_t kSlotEmpty = -1;
constexpr int64_t kSlotInflight = -2;

// Phases 1 and 2 of one call under the cache's lock: every expert of experts[0..n) that is
// resident is pinned and marked used (a hit); then every other expert, in the order given,
// reserves a victim slot (an empty one first, else the least recently used slot that is
// neither pinned nor in flight), which goes in flight.  An expert listed twice takes the
// slot of its first mention.  slots[j] = the slot of expert j; load[j] = 1 when the expert
// must be read into it.  Experts outside [0, n_experts) get slot -1 and are not loaded.
// K3MOE_ERR_CACHE_FULL (nothing reserved, nothing pinned) when the call's distinct experts
// do not fit in the slots.
k3moe_status cache_reserve(k3moe_expert_cache *c, int layer, const int32_t *experts, int n,
                           int32_t *slots, int32_t *load);
// Phase 3: publish the slots that were read (ok[j] != 0 for a load that was issued), return
// the ones that were not to the empty state, and unpin everything the call pinned.
void cache_publish(k3moe_expert_cache *c, int layer, const int32_t *experts, int n,
                   const int32_t *slots, const int32_t *load, const int32_t *ok);

}  // namespace k3
