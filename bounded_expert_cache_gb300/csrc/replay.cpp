// Offline replays of one layer's step sequence under other cache policies,
// for policy comparisons on fixed route traces.
//
// "Paging the Experts" §2: farthest-next-use is an offline paging reference
// (it needs future routing); §5.1 compares policies on fixed route replays.
// "Nanite for Experts" §5.6 and §7.4: a learned, static working set of 16 (or
// 20) experts per layer instead of rolling replacement.
//
// A step is one layer evaluation; its whole union is pinned. Farthest next
// use touches resident experts, then admits the missing ones in ascending
// id: the lowest free slot, else the slot of the resident expert outside the
// union whose next step of use is the farthest (never again is farthest;
// ties to the lower slot). The static working set keeps the W experts with
// the most assignments over the first calib steps (ties to the lower id),
// resident before the first step and never evicted; every other expert of
// a step is a miss that is materialised for the step and not admitted. LRU
// and seeded random run through the slot manager itself.
#include <algorithm>
#include <limits>
#include <string>
#include <vector>

#include "internal.h"

namespace {

moe_status_t replay_farthest(int32_t E, int32_t S, int32_t n, const int32_t* off, const int32_t* ex,
                             const int32_t* cnt, moe_stats_t* out) {
  // for every expert, the steps that use it, in order
  std::vector<std::vector<int32_t>> uses(E);
  for (int32_t t = 0; t < n; ++t)
    for (int32_t i = off[t]; i < off[t + 1]; ++i) uses[ex[i]].push_back(t);
  std::vector<size_t> cur(E, 0);  // index of the first use at or after the current step
  std::vector<int32_t> owner(S, -1), where(E, -1);
  std::vector<char> in_step(E, 0);
  const int64_t kNever = std::numeric_limits<int64_t>::max();
  for (int32_t t = 0; t < n; ++t) {
    std::vector<int32_t> U(ex + off[t], ex + off[t + 1]);
    std::sort(U.begin(), U.end());
    if (static_cast<int32_t>(U.size()) > S) return MOE_ERR_CAPACITY;
    for (int32_t e : U) {
      in_step[e] = 1;
      while (cur[e] < uses[e].size() && uses[e][cur[e]] <= t) ++cur[e];  // now: first use after t
    }
    int64_t assignments = 0;
    for (int32_t i = off[t]; i < off[t + 1]; ++i) assignments += cnt[i];
    int32_t nmiss = 0;
    for (int32_t e : U) {
      if (where[e] >= 0) continue;
      ++nmiss;
      int32_t slot = -1;
      for (int32_t s = 0; s < S && slot < 0; ++s)
        if (owner[s] < 0) slot = s;
      if (slot < 0) {
        int64_t far = -1;
        for (int32_t s = 0; s < S; ++s) {
          const int32_t o = owner[s];
          if (in_step[o]) continue;
          // next use of o after step t
          size_t c = cur[o];
          while (c < uses[o].size() && uses[o][c] <= t) ++c;
          const int64_t nu = c < uses[o].size() ? uses[o][c] : kNever;
          if (nu > far) {
            far = nu;
            slot = s;
          }
        }
        where[owner[slot]] = -1;
        out->evictions++;
      }
      owner[slot] = e;
      where[e] = slot;
    }
    for (int32_t e : U) in_step[e] = 0;
    out->misses += nmiss;
    out->hits += assignments - nmiss;
  }
  return MOE_OK;
}

moe_status_t replay_static(int32_t E, int32_t S, int32_t n, const int32_t* off, const int32_t* ex,
                           const int32_t* cnt, int32_t width, int32_t calib, moe_stats_t* out) {
  if (width > S || width > E) return MOE_ERR_CAPACITY;
  std::vector<int64_t> total(E, 0);
  for (int32_t t = 0; t < std::min(calib, n); ++t)
    for (int32_t i = off[t]; i < off[t + 1]; ++i) total[ex[i]] += cnt[i];
  std::vector<int32_t> order(E);
  for (int32_t e = 0; e < E; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return total[a] > total[b]; });
  std::vector<char> keep(E, 0);
  for (int32_t i = 0; i < width; ++i) keep[order[i]] = 1;
  for (int32_t t = 0; t < n; ++t) {
    int64_t assignments = 0, nmiss = 0;
    for (int32_t i = off[t]; i < off[t + 1]; ++i) {
      assignments += cnt[i];
      nmiss += keep[ex[i]] ? 0 : 1;
    }
    out->misses += nmiss;
    out->hits += assignments - nmiss;
  }
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_replay(int32_t policy, int32_t n_experts, int32_t n_slots, uint64_t seed,
                                   int32_t layer, int64_t payload_bytes, int32_t width, int32_t calib,
                                   int32_t n_steps, const int32_t* offsets, const int32_t* experts,
                                   const int32_t* counts, moe_stats_t* out) {
  if (!out || n_experts < 1 || n_slots < 1 || n_slots > n_experts || n_steps < 0 || payload_bytes < 0 || width < 0 || calib < 0 ||
      (n_steps > 0 && (!offsets || !experts || !counts)))
    return MOE_ERR_ARG;
  if (offsets && offsets[0] != 0) return MOE_ERR_ARG;
  for (int32_t t = 0; t < n_steps; ++t) {
    if (offsets[t + 1] < offsets[t]) return MOE_ERR_ARG;
    std::vector<int32_t> U(experts + offsets[t], experts + offsets[t + 1]);
    std::sort(U.begin(), U.end());
    for (size_t i = 0; i < U.size(); ++i)
      if (U[i] < 0 || U[i] >= n_experts || (i > 0 && U[i] == U[i - 1])) return MOE_ERR_ARG;
    for (int32_t i = offsets[t]; i < offsets[t + 1]; ++i)
      if (counts[i] < 0) return MOE_ERR_ARG;
  }
  *out = moe_stats_t{};
  moe_status_t st = MOE_OK;
  if (policy == MOE_LRU || policy == MOE_RANDOM) {
    moe_slots* s = moe::slots_new(n_experts, n_slots, policy, seed, layer, payload_bytes);
    std::vector<int32_t> cnt(n_experts, 0);
    std::string err;
    for (int32_t t = 0; t < n_steps && st == MOE_OK; ++t) {
      for (int32_t i = offsets[t]; i < offsets[t + 1]; ++i) cnt[experts[i]] = counts[i];
      moe_miss_list_t ml{};
      st = moe::slots_step(s, experts + offsets[t], offsets[t + 1] - offsets[t], cnt.data(), &ml, &err);
      for (int32_t i = offsets[t]; i < offsets[t + 1]; ++i) cnt[experts[i]] = 0;
    }
    if (st == MOE_OK) *out = moe::slots_stats(s);
    moe_slots_destroy(s);
  } else if (policy == MOE_FARTHEST_NEXT_USE) {
    st = replay_farthest(n_experts, n_slots, n_steps, offsets, experts, counts, out);
  } else if (policy == MOE_STATIC_SET) {
    st = replay_static(n_experts, n_slots, n_steps, offsets, experts, counts, width, calib, out);
  } else {
    return MOE_ERR_ARG;
  }
  if (st != MOE_OK) return st;
  out->steps = n_steps;
  if (policy != MOE_LRU && policy != MOE_RANDOM) out->materialized_bytes = out->misses * payload_bytes;
  return MOE_OK;
}
