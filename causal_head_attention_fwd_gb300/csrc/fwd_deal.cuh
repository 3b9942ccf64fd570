// Deal of the persistent kernels' work items over their CTAs.
//
// A work item is two 128-row query tiles of one (b, h); item idx starts at
// query row 2*BM*(n_pairs-1-idx/BH) of head idx%BH, so low indices are the
// long causal rows. Causal items differ in length (2 to 2*ceil(T/256) key
// steps), so the host deals them longest first, each to the CTA with the least
// work so far (greedy longest-processing-time), and passes every CTA's list in
// the launch parameters. Without a table (too many items, or equal items when
// non-causal) CTA c takes items c, 2G-1-c, 2G+c, ... in rounds of G CTAs.
// The backward deals its causal items (one key tile of one head each) the
// same way.
#pragma once
#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "common.cuh"

namespace attn {

constexpr int DEAL_MAX_ITEMS = 2048, DEAL_MAX_CTAS = 160;

struct WorkDeal {
  int use;                                 // 0: snake order
  uint16_t off[DEAL_MAX_CTAS + 1];         // CTA c's items: item[off[c] .. off[c+1])
  uint16_t item[DEAL_MAX_ITEMS];
};

// Item k of this CTA.
__device__ __forceinline__ int deal_item(const WorkDeal& s, int k) {
  const int G = gridDim.x, c = blockIdx.x;
  if (s.use) return s.item[s.off[c] + k];
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Number of items of this CTA.
__device__ __forceinline__ int deal_count(const WorkDeal& s, int n_items) {
  if (s.use) return s.off[blockIdx.x + 1] - s.off[blockIdx.x];
  int n = 0;
  while (deal_item(s, n) < n_items) ++n;
  return n;
}

// Key-tile steps of causal item idx: those of its longer query tile.
inline int causal_item_steps(int idx, int n_pairs, int BH, int T) {
  const int q0 = (n_pairs - 1 - idx / BH) * 2 * BM;
  int n = 0;
  for (int i = 0; i < 2; ++i) {
    const int qs = q0 + i * BM;
    if (qs < T) n = std::max(n, qs / BN + 1);
  }
  return n;
}

// Greedy longest-processing-time deal of n_items items over `grid` CTAs:
// items in index order (the callers number them longest first), each to the
// CTA with the least work so far; cost(idx) is an item's work in key-tile
// steps, `overhead` its start-up in the same unit.
template <typename Cost>
inline void build_lpt_deal(WorkDeal& s, int n_items, int grid, float overhead, Cost cost) {
  s.use = 0;
  if (n_items > DEAL_MAX_ITEMS || grid < 1 || grid > DEAL_MAX_CTAS) return;
  using Load = std::pair<float, int>;      // (work so far, CTA): least work, then lowest CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0.f, c});
  std::vector<std::vector<int>> per(grid);
  for (int idx = 0; idx < n_items; ++idx) {
    const Load l = heap.top();
    heap.pop();
    per[l.second].push_back(idx);
    heap.push({l.first + (float)cost(idx) + overhead, l.second});
  }
  int n = 0;
  for (int c = 0; c < grid; ++c) {
    s.off[c] = (uint16_t)n;
    for (int idx : per[c]) s.item[n++] = (uint16_t)idx;
  }
  s.off[grid] = (uint16_t)n;
  s.use = 1;
}

// The forward's causal items: an item weighs its key steps plus 1.7 for its
// start-up (measured: ~4k cycles from an item's last P to the next item's
// first scores, against ~2.4k per key step).
inline void build_causal_deal(WorkDeal& s, int n_pairs, int BH, int T, int grid) {
  build_lpt_deal(s, n_pairs * BH, grid, 1.7f,
                 [&](int idx) { return causal_item_steps(idx, n_pairs, BH, T); });
}

// The deal a launch uses: the causal table (built once per shape, then
// reused) or the snake order.
inline WorkDeal launch_deal(bool causal, int n_pairs, int BH, int T, int grid) {
  WorkDeal d;
  d.use = 0;
  if (!causal) return d;
  static std::mutex mu;
  static WorkDeal cached;
  static long long key0[4] = {-1, -1, -1, -1};
  const long long key[4] = {n_pairs, BH, T, grid};
  std::lock_guard<std::mutex> lk(mu);
  if (!std::equal(key, key + 4, key0)) {
    build_causal_deal(cached, n_pairs, BH, T, grid);
    std::copy(key, key + 4, key0);
  }
  return cached;
}

// The backward's causal deal: item idx = key tile idx / BH of head idx % BH
// walks the query tiles from that key tile on, n_kv - idx / BH steps (key tile
// 0 first); an item weighs its steps plus 0.5 for its start-up (the first
// step's K/V wait and the previous item's dK/dV hand-over). Built once per
// shape; the snake order when the items are equal (no mask) or too many.
inline WorkDeal launch_deal_bwd(bool causal, int n_kv, int BH, int grid) {
  WorkDeal d;
  d.use = 0;
  if (!causal) return d;
  static std::mutex mu;
  static WorkDeal cached;
  static long long key0[3] = {-1, -1, -1};
  const long long key[3] = {n_kv, BH, grid};
  std::lock_guard<std::mutex> lk(mu);
  if (!std::equal(key, key + 3, key0)) {
    build_lpt_deal(cached, n_kv * BH, grid, 0.5f, [&](int idx) { return n_kv - idx / BH; });
    std::copy(key, key + 3, key0);
  }
  return cached;
}

}  // namespace attn
