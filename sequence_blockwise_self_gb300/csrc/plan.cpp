// plan.cpp -- ring visiting order and launch order (see plan.h).
#include "plan.h"

#include <algorithm>
#include <numeric>

namespace ra {

namespace {

int n_tiles(int L) { return (L + kTileRows - 1) / kTileRows; }

// Group an ordered list of tile indices into maximal runs of consecutive
// indices and append them as (begin, end) pairs.
void append_ranges(const std::vector<int>& tiles, std::vector<int32_t>& out) {
  size_t i = 0;
  while (i < tiles.size()) {
    size_t j = i + 1;
    while (j < tiles.size() && tiles[j] == tiles[j - 1] + 1) ++j;
    out.push_back(tiles[i]);
    out.push_back(tiles[j - 1] + 1);
    i = j;
  }
}

void finish(Plan& p) {
  p.order.resize(p.n_blocks);
  std::iota(p.order.begin(), p.order.end(), 0);
  // Longest-processing-time first: the hardware hands CTAs to SMs in launch
  // order, so heavy items go first and light ones fill the tail.
  std::stable_sort(p.order.begin(), p.order.end(),
                   [&](int a, int b) { return p.work[a] > p.work[b]; });
}

}  // namespace

Plan build_fwd_plan(int L, int N, bool causal) {
  Plan p;
  const int nt = n_tiles(L);
  p.n_blocks = (L + kQBlockRows - 1) / kQBlockRows;
  p.offsets.push_back(0);
  std::vector<int> tiles;
  for (int u = 0; u < p.n_blocks; ++u) {
    const int q_first = u * kQBlockRows;
    const int q_last = std::min(q_first + kQBlockRows, L) - 1;
    const int r = owner_rank(L, N, causal, q_first);
    const int last_kv = causal ? q_last / kTileRows : nt - 1;
    tiles.clear();
    for (int t = 0; t <= last_kv; ++t) tiles.push_back(t);
    auto step = [&](int t) {
      const int src = owner_rank(L, N, causal, t * kTileRows);
      return ((r - src) % N + N) % N;
    };
    std::stable_sort(tiles.begin(), tiles.end(), [&](int a, int b) {
      const int sa = step(a), sb = step(b);
      return sa != sb ? sa < sb : a < b;
    });
    append_ranges(tiles, p.ranges);
    p.offsets.push_back(static_cast<int32_t>(p.ranges.size() / 2));
    const int q_tiles = (q_last - q_first) / kTileRows + 1;
    p.work.push_back(static_cast<int64_t>(tiles.size()) * q_tiles);
  }
  finish(p);
  return p;
}

Plan build_bwd_plan(int L, int N, bool causal) {
  Plan p;
  const int nt = n_tiles(L);
  p.n_blocks = nt;
  p.offsets.push_back(0);
  std::vector<int> tiles;
  for (int t = 0; t < nt; ++t) {
    const int rk = owner_rank(L, N, causal, t * kTileRows);
    tiles.clear();
    for (int q = causal ? t : 0; q < nt; ++q) tiles.push_back(q);
    auto step = [&](int q) {
      const int dst = owner_rank(L, N, causal, q * kTileRows);
      return ((dst - rk) % N + N) % N;
    };
    std::stable_sort(tiles.begin(), tiles.end(), [&](int a, int b) {
      const int sa = step(a), sb = step(b);
      return sa != sb ? sa < sb : a < b;
    });
    append_ranges(tiles, p.ranges);
    p.offsets.push_back(static_cast<int32_t>(p.ranges.size() / 2));
    p.work.push_back(static_cast<int64_t>(tiles.size()));
  }
  finish(p);
  return p;
}

Plan build_step_plan(int L, int N, bool causal, int sched, int step, int rank_lo, int rank_hi) {
  Plan p;
  const int C = L / N;
  const int nt = C / kTileRows;                       // tiles per chunk
  const int nb = (C + kQBlockRows - 1) / kQBlockRows;  // 256-row blocks per chunk
  p.n_blocks = (rank_hi - rank_lo) * nb;
  p.offsets.push_back(0);
  std::vector<int> tiles;
  for (int w = rank_lo; w < rank_hi; ++w) {
    int r, src;
    const bool busy = schedule_pair(N, sched, step, w, &r, &src);
    for (int u = 0; u < nb; ++u) {
      tiles.clear();
      int q_tiles = 0;
      for (int qt = 2 * u; qt < 2 * u + 2 && qt < nt; ++qt) ++q_tiles;
      for (int kt = 0; kt < nt && busy; ++kt) {
        bool seen = !causal;
        for (int qt = 2 * u; qt < 2 * u + 2 && qt < nt && !seen; ++qt)
          seen = chunk_pos(L, N, true, sched, src, kt * kTileRows) <=
                 chunk_pos(L, N, true, sched, r, qt * kTileRows + kTileRows - 1);
        if (seen) tiles.push_back(kt);
      }
      append_ranges(tiles, p.ranges);
      p.offsets.push_back(static_cast<int32_t>(p.ranges.size() / 2));
      p.work.push_back(static_cast<int64_t>(tiles.size()) * q_tiles);
    }
  }
  finish(p);
  return p;
}

Plan build_bwd_step_plan(int L, int N, bool causal, int sched, int step, int rank_lo, int rank_hi) {
  Plan p;
  const int C = L / N;
  const int nt = C / kTileRows;
  p.n_blocks = (rank_hi - rank_lo) * nt;
  p.offsets.push_back(0);
  std::vector<int> tiles;
  for (int w = rank_lo; w < rank_hi; ++w) {
    int r, src;
    const bool busy = schedule_pair(N, sched, step, w, &r, &src);
    for (int kt = 0; kt < nt; ++kt) {
      tiles.clear();
      const int kmin = chunk_pos(L, N, causal, sched, src, kt * kTileRows);
      for (int qt = 0; qt < nt && busy; ++qt)
        if (!causal || kmin <= chunk_pos(L, N, causal, sched, r, qt * kTileRows + kTileRows - 1)) tiles.push_back(qt);
      append_ranges(tiles, p.ranges);
      p.offsets.push_back(static_cast<int32_t>(p.ranges.size() / 2));
      p.work.push_back(static_cast<int64_t>(tiles.size()));
    }
  }
  finish(p);
  return p;
}

}  // namespace ra
