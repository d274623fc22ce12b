// shard.cu - sharding one join batch over ranks by anchor (host code). "Motor de
// inferência Quail atinge 1 bilhão de tokens por minuto por GPU", section "Como funciona",
// cascade-attention bullet: a suffix attends only to its own anchor and to itself, so an
// anchor with its suffixes is an independent unit; ranks then need no data exchange.
//
// Work of anchor a = its visible (query, key) pairs, sum over its suffixes s of
// l_s L_a + l_s (l_s + 1) / 2 (exact in int64: both terms are below T_S * 2^31). Longest
// processing time first (Graham, 1969): anchors by decreasing work (ties: lower index),
// each to the rank with the least work so far (ties: lower rank), kept in a min-heap.
// O(A log A + A log R).
#include <algorithm>
#include <cstdint>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "quail.h"

extern "C" quail_status quail_shard_anchors(int32_t num_anchors, const int32_t* anchor_offsets,
                                            const int32_t* anchor_suffix_ptr,
                                            const int32_t* suffix_offsets, int32_t num_ranks,
                                            int32_t* rank_of_anchor, int64_t* rank_pairs) {
  if (num_anchors < 0 || num_ranks < 1) return QUAIL_ERR_INVALID_ARG;
  if (anchor_offsets == nullptr || anchor_suffix_ptr == nullptr || suffix_offsets == nullptr)
    return QUAIL_ERR_INVALID_ARG;
  if (num_anchors > 0 && rank_of_anchor == nullptr) return QUAIL_ERR_INVALID_ARG;
  if (anchor_suffix_ptr[0] != 0) return QUAIL_ERR_INVALID_ARG;
  for (int32_t a = 0; a < num_anchors; ++a)
    if (anchor_offsets[a + 1] < anchor_offsets[a] ||
        anchor_suffix_ptr[a + 1] < anchor_suffix_ptr[a])
      return QUAIL_ERR_INVALID_ARG;
  const int32_t S = anchor_suffix_ptr[num_anchors];
  for (int32_t s = 0; s < S; ++s)
    if (suffix_offsets[s + 1] < suffix_offsets[s]) return QUAIL_ERR_INVALID_ARG;

  std::vector<int64_t> work(static_cast<size_t>(num_anchors), 0);
  for (int32_t a = 0; a < num_anchors; ++a) {
    const int64_t la = static_cast<int64_t>(anchor_offsets[a + 1]) - anchor_offsets[a];
    int64_t w = 0;
    for (int32_t s = anchor_suffix_ptr[a]; s < anchor_suffix_ptr[a + 1]; ++s) {
      const int64_t ls = static_cast<int64_t>(suffix_offsets[s + 1]) - suffix_offsets[s];
      w += ls * la + ls * (ls + 1) / 2;
    }
    work[a] = w;
  }
  std::vector<int32_t> order(static_cast<size_t>(num_anchors));
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    return work[x] != work[y] ? work[x] > work[y] : x < y;
  });
  // (load, rank), smallest first: the least-loaded rank, the lower rank on ties
  using Slot = std::pair<int64_t, int32_t>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int32_t r = 0; r < num_ranks; ++r) heap.push({0, r});
  std::vector<int64_t> load(static_cast<size_t>(num_ranks), 0);
  for (const int32_t a : order) {
    Slot top = heap.top();
    heap.pop();
    rank_of_anchor[a] = top.second;
    top.first += work[a];
    load[top.second] = top.first;
    heap.push(top);
  }
  if (rank_pairs != nullptr)
    for (int32_t r = 0; r < num_ranks; ++r) rank_pairs[r] = load[r];
  return QUAIL_OK;
}

// One rank's sub-batch: its anchors in their original order, each with all its suffixes.
// Offsets are rebased prefix sums of the kept lengths; rows are indices into the full
// batch's tensors (anchor rows of k_anc / v_anc; suffix rows of q_suf / k_suf / v_suf and of
// out / lse). Two passes: sizes, then (if the arrays are given) the arrays.
extern "C" quail_status quail_shard_batch(
    int32_t num_anchors, const int32_t* anchor_offsets, const int32_t* anchor_suffix_ptr,
    const int32_t* suffix_offsets, const int32_t* rank_of_anchor, int32_t rank,
    quail_shard_sizes* sizes, int32_t* sub_anchor_offsets, int32_t* sub_anchor_suffix_ptr,
    int32_t* sub_suffix_offsets, int32_t* anchors, int64_t* anchor_rows, int64_t* suffix_rows) {
  if (num_anchors < 0 || rank < 0 || sizes == nullptr) return QUAIL_ERR_INVALID_ARG;
  if (anchor_offsets == nullptr || anchor_suffix_ptr == nullptr || suffix_offsets == nullptr ||
      (num_anchors > 0 && rank_of_anchor == nullptr))
    return QUAIL_ERR_INVALID_ARG;
  if (anchor_suffix_ptr[0] != 0) return QUAIL_ERR_INVALID_ARG;
  const bool any_out = sub_anchor_offsets || sub_anchor_suffix_ptr || sub_suffix_offsets ||
                       anchors || anchor_rows || suffix_rows;
  const bool all_out = sub_anchor_offsets && sub_anchor_suffix_ptr && sub_suffix_offsets &&
                       anchors && anchor_rows && suffix_rows;
  if (any_out && !all_out) return QUAIL_ERR_INVALID_ARG;
  // sizes (and the same checks as quail_shard_anchors)
  int64_t n_anchor = 0, n_suffix = 0, t_anchor = 0, t_suffix = 0;
  for (int32_t a = 0; a < num_anchors; ++a) {
    if (anchor_offsets[a + 1] < anchor_offsets[a] ||
        anchor_suffix_ptr[a + 1] < anchor_suffix_ptr[a])
      return QUAIL_ERR_INVALID_ARG;
    for (int32_t s = anchor_suffix_ptr[a]; s < anchor_suffix_ptr[a + 1]; ++s)
      if (suffix_offsets[s + 1] < suffix_offsets[s]) return QUAIL_ERR_INVALID_ARG;
    if (rank_of_anchor[a] != rank) continue;
    ++n_anchor;
    n_suffix += anchor_suffix_ptr[a + 1] - anchor_suffix_ptr[a];
    t_anchor += static_cast<int64_t>(anchor_offsets[a + 1]) - anchor_offsets[a];
    t_suffix += static_cast<int64_t>(suffix_offsets[anchor_suffix_ptr[a + 1]]) -
                suffix_offsets[anchor_suffix_ptr[a]];
  }
  if (t_anchor > INT32_MAX || t_suffix > INT32_MAX) return QUAIL_ERR_UNSUPPORTED;
  sizes->num_anchors = static_cast<int32_t>(n_anchor);
  sizes->num_suffixes = static_cast<int32_t>(n_suffix);
  sizes->anchor_tokens = t_anchor;
  sizes->suffix_tokens = t_suffix;
  if (!all_out) return QUAIL_OK;
  // arrays
  int32_t ia = 0, is = 0;
  int64_t ra = 0, rs = 0;
  sub_anchor_offsets[0] = 0;
  sub_anchor_suffix_ptr[0] = 0;
  sub_suffix_offsets[0] = 0;
  for (int32_t a = 0; a < num_anchors; ++a) {
    if (rank_of_anchor[a] != rank) continue;
    anchors[ia] = a;
    for (int32_t r = anchor_offsets[a]; r < anchor_offsets[a + 1]; ++r) anchor_rows[ra++] = r;
    sub_anchor_offsets[ia + 1] = static_cast<int32_t>(ra);
    for (int32_t s = anchor_suffix_ptr[a]; s < anchor_suffix_ptr[a + 1]; ++s) {
      for (int32_t r = suffix_offsets[s]; r < suffix_offsets[s + 1]; ++r) suffix_rows[rs++] = r;
      sub_suffix_offsets[++is] = static_cast<int32_t>(rs);
    }
    sub_anchor_suffix_ptr[ia + 1] = is;
    ++ia;
  }
  return QUAIL_OK;
}
