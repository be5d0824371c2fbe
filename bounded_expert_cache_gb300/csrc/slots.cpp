// Host-side slot manager of the bounded expert cache (one per layer).
//
// "MawForge" §IV-C: per-layer slot tensors; a miss materialises the expert
// block into an available slot and updates route-to-slot metadata.
// "Paging the Experts" §3.2: entries are pinned while their layer is
// evaluated; §4.1/§5.1: LRU versus seeded random eviction; §4.2: materialised
// bytes = demand misses x payload. "Nanite for Experts" §5.4: page-table
// entries carry generations so a stale slot is never read.
//
// Step semantics: resident experts of the union are touched in ascending id,
// then missing experts are admitted in ascending id; every access takes the
// next tick. A miss takes the lowest free slot, else the LRU victim (oldest
// tick) or, for the random policy, cand[next() mod n] where cand lists the
// resident experts outside the current union by slot index and next() is
// SplitMix64. Hits count assignments minus missing experts.
//
// When the union exceeds the slot count (LRU only) fills evict experts of
// the same step; such a fill is assigned to the compute wave after the one
// of the expert it evicts, so a slot is overwritten only after the compute
// that reads it.
//
// Prefetch ("Paging the Experts" §3.3): before a step, a predicted expert
// that is absent is loaded like a miss with nothing pinned (one tick, the
// lowest free slot, else the policy's victim over every slot); a resident
// one is touched like a hit (resident refresh) or only recorded
// (preserve-resident). The next step counts the load useful if its union
// holds the expert, else wasted; speculative bytes are counted apart from
// the demand misses' (§4.2).
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

namespace {

constexpr uint64_t kGoldenGamma = 0x9E3779B97F4A7C15ull;

}  // namespace

extern "C" uint64_t moe_splitmix64_next(uint64_t* state) {
  uint64_t z = (*state += kGoldenGamma);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct moe_slots {
  int32_t E = 0, S = 0, policy = 0, layer = 0;
  int64_t payload = 0;
  uint64_t rng = 0;
  uint64_t tick = 0;
  std::vector<int32_t> pt, owner;
  std::vector<uint32_t> gen;
  std::vector<uint64_t> last;
  std::vector<int32_t> f_expert, f_slot, f_victim, f_wave;
  std::vector<int32_t> wave_of;   // per expert, for the current step
  std::vector<uint8_t> in_step;   // per expert, member of the current union
  int32_t pending = -1;           // expert of the last speculative load, until its step
  moe_stats_t stats{};
};

namespace moe {

moe_slots* slots_new(int32_t E, int32_t S, int32_t policy, uint64_t seed, int32_t layer,
                     int64_t payload) {
  auto* s = new moe_slots();
  s->E = E;
  s->S = S;
  s->policy = policy;
  s->layer = layer;
  s->payload = payload;
  s->rng = seed ^ (static_cast<uint64_t>(layer) * kGoldenGamma);
  s->pt.assign(E, -1);
  s->owner.assign(S, -1);
  s->gen.assign(S, 0);
  s->last.assign(S, 0);
  s->wave_of.assign(E, 0);
  s->in_step.assign(E, 0);
  return s;
}

static int32_t lowest_free(const moe_slots* s) {
  for (int32_t i = 0; i < s->S; ++i)
    if (s->owner[i] < 0) return i;
  return -1;
}

// Slot of the policy's victim when no slot is free: LRU the oldest access;
// random cand[next() mod n] over the slots whose expert is not in the
// current union (in_step), listed by slot index.
static int32_t victim_slot(moe_slots* s, std::vector<int32_t>& cand) {
  if (s->policy == MOE_LRU) {
    int32_t slot = 0;
    for (int32_t i = 1; i < s->S; ++i)
      if (s->last[i] < s->last[slot]) slot = i;
    return slot;
  }
  cand.clear();
  for (int32_t i = 0; i < s->S; ++i)
    if (!s->in_step[s->owner[i]]) cand.push_back(i);
  uint64_t r = moe_splitmix64_next(&s->rng);
  return cand[r % cand.size()];
}

moe_status_t slots_step(moe_slots* s, const int32_t* uniq, int32_t n_uniq, const int32_t* counts,
                        moe_miss_list_t* out, std::string* err) {
  if (n_uniq < 0 || n_uniq > s->E || (n_uniq > 0 && !uniq) || !counts) {
    *err = "slots_step: bad union";
    return MOE_ERR_ARG;
  }
  std::vector<int32_t> U(uniq, uniq + n_uniq);
  std::sort(U.begin(), U.end());
  for (int32_t i = 0; i < n_uniq; ++i) {
    if (U[i] < 0 || U[i] >= s->E || (i > 0 && U[i] == U[i - 1])) {
      *err = "slots_step: union holds an invalid or repeated expert";
      return MOE_ERR_ARG;
    }
  }
  // The random policy never evicts an expert of the current step: check the
  // capacity first so a failing step leaves the state unchanged.
  int32_t n_miss = 0;
  for (int32_t e : U) n_miss += s->pt[e] < 0;
  if (s->policy == MOE_RANDOM) {
    int32_t free_slots = 0, resident_in_u = 0;
    for (int32_t i = 0; i < s->S; ++i) free_slots += s->owner[i] < 0;
    for (int32_t e : U) resident_in_u += s->pt[e] >= 0;
    int32_t candidates = (s->S - free_slots) - resident_in_u;
    if (n_miss > free_slots + candidates) {
      *err = "slots_step: random policy has no unpinned victim (union larger than the slots)";
      return MOE_ERR_CAPACITY;
    }
  }
  if (s->pending >= 0) {  // the last speculative load meets its step
    const bool used = std::binary_search(U.begin(), U.end(), s->pending);
    (used ? s->stats.prefetch_useful : s->stats.prefetch_wasted)++;
    s->pending = -1;
  }
  for (int32_t e : U) {
    s->in_step[e] = 1;
    s->wave_of[e] = 0;
  }
  s->f_expert.clear();
  s->f_slot.clear();
  s->f_victim.clear();
  s->f_wave.clear();
  for (int32_t e : U) {
    if (s->pt[e] >= 0) s->last[s->pt[e]] = ++s->tick;
  }
  // the misses are fixed before any fill: a resident expert of the union
  // that a fill evicts (|U| > S) was still a hit of this step
  std::vector<int32_t> M;
  for (int32_t e : U)
    if (s->pt[e] < 0) M.push_back(e);
  int32_t n_waves = 1;
  std::vector<int32_t> cand;
  for (int32_t e : M) {
    ++s->tick;
    int32_t slot = lowest_free(s), victim = -1;
    if (slot < 0) {
      slot = victim_slot(s, cand);
      victim = s->owner[slot];
      s->pt[victim] = -1;
      s->owner[slot] = -1;
      s->stats.evictions++;
    }
    int32_t wave = (victim >= 0 && s->in_step[victim]) ? s->wave_of[victim] + 1 : 0;
    s->wave_of[e] = wave;
    if (wave + 1 > n_waves) n_waves = wave + 1;
    s->owner[slot] = e;
    s->pt[e] = slot;
    s->gen[slot]++;
    s->last[slot] = s->tick;
    s->f_expert.push_back(e);
    s->f_slot.push_back(slot);
    s->f_victim.push_back(victim);
    s->f_wave.push_back(wave);
  }
  int64_t assignments = 0;
  for (int32_t e : U) {
    assignments += counts[e];
    s->in_step[e] = 0;
  }
  int32_t hits = static_cast<int32_t>(assignments) - n_miss;
  s->stats.steps++;
  s->stats.hits += hits;
  s->stats.misses += n_miss;
  s->stats.materialized_bytes += static_cast<int64_t>(n_miss) * s->payload;
  out->n = n_miss;
  out->expert = s->f_expert.data();
  out->slot = s->f_slot.data();
  out->victim = s->f_victim.data();
  out->wave = s->f_wave.data();
  out->n_waves = n_waves;
  out->hits = hits;
  out->misses = n_miss;
  out->layer = s->layer;
  return MOE_OK;
}

moe_status_t slots_prefetch(moe_slots* s, int32_t e, int32_t mode, int32_t* action, moe_miss_list_t* fill,
                            std::string* err) {
  if (e < 0 || e >= s->E || (mode != MOE_PREFETCH_REFRESH && mode != MOE_PREFETCH_PRESERVE)) {
    *err = "prefetch: bad expert or mode";
    return MOE_ERR_ARG;
  }
  s->f_expert.clear();
  s->f_slot.clear();
  s->f_victim.clear();
  s->f_wave.clear();
  *fill = moe_miss_list_t{};
  fill->layer = s->layer;
  fill->n_waves = 1;
  const int32_t at = s->pt[e];
  if (at >= 0) {
    if (mode == MOE_PREFETCH_REFRESH) {
      s->last[at] = ++s->tick;
      s->stats.prefetch_refreshes++;
      *action = MOE_PREFETCH_REFRESHED;
    } else {
      s->stats.prefetch_probes++;
      *action = MOE_PREFETCH_PROBED;
    }
    return MOE_OK;
  }
  ++s->tick;
  std::vector<int32_t> cand;
  int32_t slot = lowest_free(s), victim = -1;
  if (slot < 0) {  // nothing is pinned outside a step
    slot = victim_slot(s, cand);
    victim = s->owner[slot];
    s->pt[victim] = -1;
    s->owner[slot] = -1;
    s->stats.evictions++;
  }
  s->owner[slot] = e;
  s->pt[e] = slot;
  s->gen[slot]++;
  s->last[slot] = s->tick;
  s->pending = e;
  s->stats.prefetch_loads++;
  s->stats.prefetch_bytes += s->payload;
  s->f_expert.push_back(e);
  s->f_slot.push_back(slot);
  s->f_victim.push_back(victim);
  s->f_wave.push_back(0);
  fill->n = 1;
  fill->expert = s->f_expert.data();
  fill->slot = s->f_slot.data();
  fill->victim = s->f_victim.data();
  fill->wave = s->f_wave.data();
  *action = MOE_PREFETCH_LOADED;
  return MOE_OK;
}

moe_status_t slots_preload(moe_slots* s, const int32_t* experts, int32_t n, std::vector<int32_t>* filled,
                           std::vector<int32_t>* filled_slots, std::string* err) {
  std::vector<int32_t> v(experts, experts + n);
  std::sort(v.begin(), v.end());
  for (int32_t e : v) {
    if (e < 0 || e >= s->E) {
      *err = "preload: expert id out of range";
      return MOE_ERR_ARG;
    }
  }
  for (int32_t e : v) {
    if (s->pt[e] >= 0) continue;
    int32_t slot = lowest_free(s);
    if (slot < 0) {
      *err = "preload: more experts than free slots";
      return MOE_ERR_CAPACITY;
    }
    ++s->tick;
    s->owner[slot] = e;
    s->pt[e] = slot;
    s->gen[slot]++;
    s->last[slot] = s->tick;
    if (filled) filled->push_back(e);
    if (filled_slots) filled_slots->push_back(slot);
  }
  return MOE_OK;
}

moe_status_t slots_evict(moe_slots* s, int32_t e, std::string* err) {
  if (e < 0 || e >= s->E) {
    *err = "evict: expert id out of range";
    return MOE_ERR_ARG;
  }
  int32_t slot = s->pt[e];
  if (slot < 0) return MOE_OK;
  s->pt[e] = -1;
  s->owner[slot] = -1;
  s->stats.evictions++;
  return MOE_OK;
}

const int32_t* slots_pt(const moe_slots* s) { return s->pt.data(); }
const int32_t* slots_owner(const moe_slots* s) { return s->owner.data(); }
const uint64_t* slots_last(const moe_slots* s) { return s->last.data(); }
uint64_t slots_tick(const moe_slots* s) { return s->tick; }
uint64_t slots_rng(const moe_slots* s) { return s->rng; }
const uint32_t* slots_gen(const moe_slots* s) { return s->gen.data(); }
moe_stats_t slots_stats(const moe_slots* s) { return s->stats; }

}  // namespace moe

// ------------------------------------------------------------ C ABI
namespace {
thread_local std::string g_slots_err;
}

extern "C" moe_status_t moe_slots_create(int32_t n_experts, int32_t n_slots, int32_t policy,
                                         uint64_t seed, int32_t layer, int64_t payload_bytes,
                                         moe_slots_t** out) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  if (n_experts <= 0 || n_slots <= 0 || n_slots > n_experts ||
      (policy != MOE_LRU && policy != MOE_RANDOM) || layer < 0 || payload_bytes < 0)
    return MOE_ERR_ARG;
  *out = moe::slots_new(n_experts, n_slots, policy, seed, layer, payload_bytes);
  return MOE_OK;
}

extern "C" void moe_slots_destroy(moe_slots_t* s) { delete s; }

extern "C" moe_status_t moe_slots_step(moe_slots_t* s, const int32_t* uniq, int32_t n_uniq,
                                       const int32_t* counts, moe_miss_list_t* out) {
  if (!s || !out) return MOE_ERR_ARG;
  return moe::slots_step(s, uniq, n_uniq, counts, out, &g_slots_err);
}

extern "C" moe_status_t moe_slots_prefetch(moe_slots_t* s, int32_t expert, int32_t mode, int32_t* action,
                                           moe_miss_list_t* fill) {
  if (!s || !action || !fill) return MOE_ERR_ARG;
  return moe::slots_prefetch(s, expert, mode, action, fill, &g_slots_err);
}

extern "C" moe_status_t moe_slots_preload(moe_slots_t* s, const int32_t* experts, int32_t n) {
  if (!s || (n > 0 && !experts) || n < 0) return MOE_ERR_ARG;
  return moe::slots_preload(s, experts, n, nullptr, nullptr, &g_slots_err);
}

extern "C" moe_status_t moe_slots_evict(moe_slots_t* s, int32_t expert) {
  if (!s) return MOE_ERR_ARG;
  return moe::slots_evict(s, expert, &g_slots_err);
}

extern "C" moe_status_t moe_slots_read(const moe_slots_t* s, int32_t* pt, uint32_t* gen) {
  if (!s) return MOE_ERR_ARG;
  if (pt) std::memcpy(pt, s->pt.data(), sizeof(int32_t) * s->E);
  if (gen) std::memcpy(gen, s->gen.data(), sizeof(uint32_t) * s->S);
  return MOE_OK;
}

extern "C" moe_status_t moe_slots_stats(const moe_slots_t* s, moe_stats_t* out) {
  if (!s || !out) return MOE_ERR_ARG;
  *out = s->stats;
  return MOE_OK;
}
