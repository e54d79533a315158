// Host plan of the softmax-attention layer over a packed pass.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "The Workload"
// (branches attend to their view and never to each other) and section
// "Kernels" (the branches of a pass share one launch, short ones packed).
//
// Query tiles: each view is cut into 128-row tiles from its first row; a
// branch longer than 128 rows likewise (after its parent view's rows as a
// prefix); runs of consecutive short branches of the same parent are packed
// into one tile of at most 128 rows, so that the parent's keys are read once
// for all of them.  Every (tile, head) pair is one item; items are dealt to
// CTAs longest first, each to the CTA with the least work so far.
#include <algorithm>
#include <functional>
#include <queue>
#include <utility>

#include "spanla_internal.h"

namespace spanla {

namespace {

int32_t blocks_of(const SaItem& it) {
  return (it.pn + kTileRows - 1) / kTileRows + (it.r0 - it.os) / kTileRows + 1;
}

}  // namespace

SoftmaxPlan make_softmax_plan(const int32_t* view_cu, int32_t V, const int32_t* branch_cu, int32_t B,
                              const int32_t* parent, int H, int max_ctas, bool branches_only) {
  SoftmaxPlan plan;
  std::vector<SaItem> tiles;   // head 0; replicated per head below
  auto add_segment = [&](int32_t a, int32_t e, int32_t ps, int32_t pn) {
    for (int32_t r0 = a; r0 < e; r0 += kTileRows)
      tiles.push_back({r0, std::min<int32_t>(kTileRows, e - r0), 0, ps, pn, a, 0, 0});
  };
  if (!branches_only)
    for (int32_t s = 0; s < V; ++s) add_segment(view_cu[s], view_cu[s + 1], 0, 0);
  for (int32_t b = 0; b < B;) {
    const int32_t a = branch_cu[b], e = branch_cu[b + 1];
    const int32_t p = parent[b];
    const int32_t ps = view_cu[p], pn = view_cu[p + 1] - view_cu[p];
    if (e == a) {
      ++b;
      continue;
    }
    if (e - a > kTileRows) {
      add_segment(a, e, ps, pn);
      ++b;
      continue;
    }
    // Pack b and the following short branches of the same parent.
    int32_t c = b;
    std::vector<uint8_t> starts;
    while (c < B && parent[c] == p && branch_cu[c + 1] - branch_cu[c] <= kTileRows &&
           branch_cu[c + 1] - a <= kTileRows) {
      if (branch_cu[c + 1] > branch_cu[c]) starts.push_back(static_cast<uint8_t>(branch_cu[c] - a));
      ++c;
    }
    SaItem it{a, branch_cu[c] - a, 0, ps, pn, a, 0, 0};
    if (starts.size() > 1) {
      it.seg0 = static_cast<int32_t>(plan.bounds.size());
      it.nseg = static_cast<int32_t>(starts.size());
      plan.bounds.insert(plan.bounds.end(), starts.begin(), starts.end());
    }
    tiles.push_back(it);
    b = c;
  }
  if (tiles.empty()) return plan;

  // Items longest first; each goes to the least loaded CTA.
  std::vector<std::pair<int32_t, int32_t>> order;   // (blocks, tile index)
  order.reserve(tiles.size());
  for (size_t t = 0; t < tiles.size(); ++t) order.push_back({blocks_of(tiles[t]), static_cast<int32_t>(t)});
  std::stable_sort(order.begin(), order.end(),
                   [](const auto& x, const auto& y) { return x.first > y.first; });
  const int64_t n_items = static_cast<int64_t>(tiles.size()) * H;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_ctas, n_items)));
  using Load = std::pair<int64_t, int>;   // (blocks so far, cta)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0, c});
  std::vector<std::vector<SaItem>> per_cta(grid);
  for (const auto& o : order) {
    for (int h = 0; h < H; ++h) {
      Load l = heap.top();
      heap.pop();
      SaItem it = tiles[o.second];
      it.head = h;
      per_cta[l.second].push_back(it);
      l.first += o.first;
      plan.key_blocks += o.first;
      heap.push(l);
    }
  }
  plan.grid = grid;
  plan.cta_begin.assign(grid + 1, 0);
  plan.items.reserve(n_items);
  for (int c = 0; c < grid; ++c) {
    plan.cta_begin[c] = static_cast<int32_t>(plan.items.size());
    plan.items.insert(plan.items.end(), per_cta[c].begin(), per_cta[c].end());
  }
  plan.cta_begin[grid] = static_cast<int32_t>(plan.items.size());
  return plan;
}

}  // namespace spanla
