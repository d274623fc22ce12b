// kv_plan.cu - query-aware anchor-KV cache plan (host code). "Motor de inferência Quail
// atinge 1 bilhão de tokens por minuto por GPU", section "Como funciona", first bullet: the
// engine knows the whole query plan in advance, so it can evict without regret; "Quail, il
// motore di inferenza che supera il miliardo di token al minuto su una H100", the KV
// regret paragraph (tokens prefilled again because their KV had been discarded).
//
// Given the plan's sequence of anchor accesses, each anchor's KV size in tokens and the
// token capacity for anchor KV, it decides which accesses hit, what is evicted, and counts
// compulsory and regret prefill tokens. Policies: LRU (a general server's choice) and
// furthest next use (the incoming anchor is a candidate too: if its next access is the
// furthest it is bypassed). Residents are kept in an ordered set, O(n log n) in all.
#include <cstdint>
#include <limits>
#include <set>
#include <tuple>
#include <vector>

#include "quail.h"

namespace {

constexpr int64_t kNever = std::numeric_limits<int64_t>::max();

}  // namespace

extern "C" quail_status quail_kv_plan(int32_t num_anchors, const int64_t* anchor_tokens,
                                      int64_t num_accesses, const int32_t* access_anchor,
                                      int64_t capacity_tokens, int32_t policy, uint8_t* hit,
                                      quail_kv_plan_stats* stats) {
  if (num_anchors < 0 || num_accesses < 0 || capacity_tokens < 0 || stats == nullptr)
    return QUAIL_ERR_INVALID_ARG;
  if (policy != QUAIL_KV_LRU && policy != QUAIL_KV_FURTHEST_NEXT_USE) return QUAIL_ERR_INVALID_ARG;
  if (num_anchors > 0 && anchor_tokens == nullptr) return QUAIL_ERR_INVALID_ARG;
  if (num_accesses > 0 && access_anchor == nullptr) return QUAIL_ERR_INVALID_ARG;
  for (int32_t a = 0; a < num_anchors; ++a)
    if (anchor_tokens[a] < 0) return QUAIL_ERR_INVALID_ARG;
  for (int64_t i = 0; i < num_accesses; ++i)
    if (access_anchor[i] < 0 || access_anchor[i] >= num_anchors) return QUAIL_ERR_INVALID_ARG;

  // next access of the same anchor after access i (kNever if none)
  std::vector<int64_t> next_use(static_cast<size_t>(num_accesses));
  {
    std::vector<int64_t> seen(static_cast<size_t>(num_anchors), kNever);
    for (int64_t i = num_accesses - 1; i >= 0; --i) {
      next_use[i] = seen[access_anchor[i]];
      seen[access_anchor[i]] = i;
    }
  }
  // per anchor: resident?, ever prefilled?, its key in the resident set
  std::vector<uint8_t> resident(static_cast<size_t>(num_anchors), 0);
  std::vector<uint8_t> seen(static_cast<size_t>(num_anchors), 0);
  std::vector<int64_t> key(static_cast<size_t>(num_anchors), 0);  // last or next access
  // LRU: (last access, anchor), smallest first. Furthest next use: (next access, size,
  // anchor), largest first - the same order as the tie rule (larger size, larger id).
  std::set<std::pair<int64_t, int32_t>> lru;
  std::set<std::tuple<int64_t, int64_t, int32_t>> far;
  int64_t used = 0;
  quail_kv_plan_stats st{};
  for (int64_t i = 0; i < num_accesses; ++i) {
    const int32_t a = access_anchor[i];
    const int64_t sz = anchor_tokens[a];
    if (resident[a]) {
      ++st.hits;
      if (hit) hit[i] = 1;
      if (policy == QUAIL_KV_LRU) {
        lru.erase({key[a], a});
        key[a] = i;
        lru.insert({key[a], a});
      } else {
        far.erase({key[a], sz, a});
        key[a] = next_use[i];
        far.insert({key[a], sz, a});
      }
      continue;
    }
    ++st.misses;
    if (hit) hit[i] = 0;
    if (seen[a]) {
      st.regret_tokens += sz;
    } else {
      st.compulsory_tokens += sz;
      seen[a] = 1;
    }
    if (sz > capacity_tokens) continue;  // streamed: never resident
    if (policy == QUAIL_KV_LRU) {
      while (used + sz > capacity_tokens) {
        const auto victim = *lru.begin();
        lru.erase(lru.begin());
        resident[victim.second] = 0;
        used -= anchor_tokens[victim.second];
      }
      key[a] = i;
      lru.insert({key[a], a});
    } else {
      // walk the residents from the furthest next use down; the incoming anchor is
      // bypassed (and nothing evicted) as soon as it is the furthest of what remains
      const std::tuple<int64_t, int64_t, int32_t> incoming{next_use[i], sz, a};
      int64_t free_tokens = capacity_tokens - used;
      auto it = far.rbegin();
      int64_t n_victims = 0;
      bool bypass = false;
      while (free_tokens < sz) {
        if (it == far.rend() || incoming > *it) {
          bypass = true;
          break;
        }
        free_tokens += std::get<1>(*it);
        ++n_victims;
        ++it;
      }
      if (bypass) continue;
      for (int64_t v = 0; v < n_victims; ++v) {
        const auto top = std::prev(far.end());
        resident[std::get<2>(*top)] = 0;
        used -= std::get<1>(*top);
        far.erase(top);
      }
      key[a] = next_use[i];
      far.insert({key[a], sz, a});
    }
    resident[a] = 1;
    used += sz;
    if (used > st.peak_resident_tokens) st.peak_resident_tokens = used;
  }
  *stats = st;
  return QUAIL_OK;
}
