// expert_cache.cu -- the decode-time expert cache's replacement policy
// (host only): least recently used over C device slots, as specified in
// include/moe.h.  The forward pass over cached slots is moe_forward_cached
// (moe_api.cu); the expert GEMMs read expert e from slot slot_of[e].
#include <cstring>

#include "internal.h"

namespace {

// The state's two maps agree and every index is in range.
bool consistent(const moe_expert_cache *c) {
  if (c->E < 1 || c->E > MOE_CACHE_MAX_E || c->C < 1 || c->C > c->E) return false;
  for (int e = 0; e < c->E; ++e) {
    const int s = c->slot_of[e];
    if (s < -1 || s >= c->C) return false;
    if (s >= 0 && c->expert_in[s] != e) return false;
  }
  for (int s = 0; s < c->C; ++s) {
    const int e = c->expert_in[s];
    if (e < -1 || e >= c->E) return false;
    if (e >= 0 && c->slot_of[e] != s) return false;
  }
  return true;
}

}  // namespace

extern "C" {

int moe_expert_cache_init(moe_expert_cache *cache, int E, int C) {
  if (!cache || E < 1 || E > MOE_CACHE_MAX_E || C < 1 || C > E) return MOE_ERR_INVALID_ARG;
  std::memset(cache, 0, sizeof(*cache));
  cache->E = E;
  cache->C = C;
  for (int i = 0; i < MOE_CACHE_MAX_E; ++i) {
    cache->slot_of[i] = -1;
    cache->expert_in[i] = -1;
    cache->last_use[i] = -1;
  }
  return MOE_OK;
}

int moe_expert_cache_plan(moe_expert_cache *cache, const int *needed, int *load_expert, int *load_slot,
                          int *n_loads) {
  if (!cache || !needed || !load_expert || !load_slot || !n_loads) return MOE_ERR_INVALID_ARG;
  if (!consistent(cache)) return MOE_ERR_INVALID_ARG;
  const int E = cache->E, C = cache->C;
  int n_needed = 0;
  for (int e = 0; e < E; ++e) n_needed += needed[e] != 0;
  if (n_needed > C) return MOE_ERR_UNSUPPORTED;
  int n = 0;
  for (int e = 0; e < E; ++e) {
    if (!needed[e]) continue;
    if (cache->slot_of[e] >= 0) {
      ++cache->hits;
      continue;
    }
    ++cache->misses;
    int s = -1;
    for (int i = 0; i < C && s < 0; ++i)
      if (cache->expert_in[i] < 0) s = i;  // the lowest empty slot
    if (s < 0) {
      // the least recently used resident expert outside the needed set
      // (one exists: at most n_needed - 1 <= C - 1 slots hold needed experts)
      for (int i = 0; i < C; ++i) {
        if (needed[cache->expert_in[i]]) continue;
        if (s < 0 || cache->last_use[i] < cache->last_use[s]) s = i;
      }
      cache->slot_of[cache->expert_in[s]] = -1;
    }
    cache->expert_in[s] = e;
    cache->slot_of[e] = s;
    load_expert[n] = e;
    load_slot[n] = s;
    ++n;
  }
  for (int e = 0; e < E; ++e)
    if (needed[e]) cache->last_use[cache->slot_of[e]] = cache->step;
  ++cache->step;
  *n_loads = n;
  return MOE_OK;
}

}  // extern "C"
