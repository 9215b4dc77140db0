// Host-side ring scheduler: shard layouts, the ring schedule, the expected
// per-(rank, step) work, and the derived ring traffic and imbalance.
//
// Layouts: contiguous (rank k owns [kS/c, (k+1)S/c), "06 - Sequence / Context
// Parallelism", section 1), zig-zag (2c chunks, rank k owns chunks k and
// 2c-1-k, plate "Splitting the Sequence") and striped (rank k owns positions
// k mod c, the tutorial's section 5).  Schedule: at step t rank i holds
// the block of rank (i - t) mod c (tutorial section 4).  Work: the tutorial's
// exercise B and the plate's "1.94 times the average" compare per-rank causal
// work; here it is counted per 128x128 tile pair from each tile's smallest
// and largest position (a tile pair is hidden entirely when its smallest key
// position exceeds its largest query position, and visible entirely when its
// largest key position is at most its smallest query position), and per
// visible (query, key) pair by a merge of the two sorted position lists.

#include <algorithm>
#include <cstdint>
#include <vector>

#include "ra_internal.h"

namespace ra {

void shard_positions(int S, int c, int layout, int32_t* pos) {
  const int n = S / c;
  for (int r = 0; r < c; ++r) {
    for (int i = 0; i < n; ++i) {
      int nat;
      if (layout == RA_ZIGZAG) {
        const int ch = n / 2;
        nat = i < ch ? r * ch + i : (2 * c - 1 - r) * ch + (i - ch);
      } else if (layout == RA_STRIPED) {
        nat = r + c * i;
      } else {
        nat = r * n + i;
      }
      pos[static_cast<long long>(r) * n + i] = nat;
    }
  }
}

namespace {

struct TileRange {
  int mn, mx;
};

std::vector<TileRange> tile_ranges(const int32_t* pos, int n) {
  std::vector<TileRange> out;
  for (int a = 0; a < n; a += kTile) {
    const int e = std::min(n, a + kTile);
    TileRange t{pos[a], pos[a]};
    for (int i = a; i < e; ++i) {
      t.mn = std::min(t.mn, pos[i]);
      t.mx = std::max(t.mx, pos[i]);
    }
    out.push_back(t);
  }
  return out;
}

// Visible pairs between two position lists: for each query, the keys at or
// before it (both lists sorted first).
uint64_t visible_pairs(std::vector<int32_t> q, std::vector<int32_t> k, bool causal) {
  if (!causal) return static_cast<uint64_t>(q.size()) * k.size();
  std::sort(q.begin(), q.end());
  std::sort(k.begin(), k.end());
  uint64_t total = 0;
  size_t j = 0;
  for (int32_t qp : q) {
    while (j < k.size() && k[j] <= qp) ++j;
    total += j;
  }
  return total;
}

}  // namespace

void expected_work(int S, int c, int layout, int causal, ra_work* out) {
  const int n = S / c;
  std::vector<int32_t> pos(static_cast<size_t>(S));
  shard_positions(S, c, layout, pos.data());
  std::vector<std::vector<TileRange>> tiles(c);
  for (int r = 0; r < c; ++r) tiles[r] = tile_ranges(pos.data() + static_cast<long long>(r) * n, n);
  for (int i = 0; i < c; ++i) {
    const std::vector<int32_t> qi(pos.begin() + static_cast<long long>(i) * n,
                                  pos.begin() + static_cast<long long>(i + 1) * n);
    for (int t = 0; t < c; ++t) {
      const int j = ((i - t) % c + c) % c;
      ra_work w{0, 0, 0, 0};
      const std::vector<int32_t> kj(pos.begin() + static_cast<long long>(j) * n,
                                    pos.begin() + static_cast<long long>(j + 1) * n);
      w.pairs = visible_pairs(qi, kj, causal != 0);
      for (const TileRange& qt : tiles[i]) {
        for (const TileRange& kt : tiles[j]) {
          if (!causal || kt.mx <= qt.mn) ++w.tiles_full;
          else if (kt.mn > qt.mx) ++w.tiles_skipped;
          else ++w.tiles_partial;
        }
      }
      out[static_cast<long long>(i) * c + t] = w;
    }
  }
}

}  // namespace ra
