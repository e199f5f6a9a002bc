// Host-side check of the grouped FFN's tile order (tile_order.cuh): for
// random segment layouts, every (segment, n-block, m-block) tile appears at
// exactly one merged position, each stream keeps its own (segment, n-block,
// m-block) order, and after u positions exactly floor(u * Lh / L) hot tiles
// have been placed.  The incremental MergedWalk, started at every CTA index
// below the grid size G, visits the same tiles as merged() at u0, u0 + G, ...
// Built with nvcc as a host program; needs no GPU.  Exit code 0 = all cases
// pass.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "tile_order.cuh"

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32() {
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 7;
  rng_state ^= rng_state << 17;
  return (uint32_t)(rng_state >> 11);
}

static int check(const std::vector<int> &mt, int NB, bool interleave) {
  const int S = (int)mt.size();
  std::vector<int32_t> pre_h(S + 1, 0), pre_c(S + 1, 0);
  for (int s = 0; s < S; ++s) {
    const bool hot = interleave && mt[s] >= 2;
    pre_h[s + 1] = pre_h[s] + (hot ? mt[s] : 0);
    pre_c[s + 1] = pre_c[s] + (hot ? 0 : mt[s]);
  }
  const int64_t Mh = pre_h[S], Mc = pre_c[S];
  const int64_t total = (Mh + Mc) * NB, Lh = Mh * NB;
  std::vector<int64_t> pos;  // position of tile (s, n, m), -1 = not seen
  std::vector<int64_t> base(S + 1, 0);
  for (int s = 0; s < S; ++s) base[s + 1] = base[s] + (int64_t)mt[s] * NB;
  pos.assign(base[S], -1);
  if (base[S] != total) return 1;
  int64_t hot_seen = 0, cold_seen = 0, last_hot = -1, last_cold = -1;
  for (int64_t u = 0; u < total; ++u) {
    int s = -1, n = -1, m = -1;
    tile_order::merged(u, pre_h.data(), pre_c.data(), S, NB, Mh, Mc, s, n, m);
    if (s < 0 || s >= S || n < 0 || n >= NB || m < 0 || m >= mt[s]) {
      std::printf("u=%lld -> out of range (%d, %d, %d)\n", (long long)u, s, n, m);
      return 1;
    }
    const int64_t id = base[s] + (int64_t)n * mt[s] + m;
    if (pos[id] >= 0) {
      std::printf("tile (%d, %d, %d) at %lld and %lld\n", s, n, m, (long long)pos[id], (long long)u);
      return 1;
    }
    pos[id] = u;
    const bool hot = interleave && mt[s] >= 2;
    // streams keep their own order: tile ids rise within each stream
    int64_t &last = hot ? last_hot : last_cold;
    if (id <= last) {
      std::printf("stream order broken at u=%lld\n", (long long)u);
      return 1;
    }
    last = id;
    (hot ? hot_seen : cold_seen) += 1;
    if (total > 0 && hot_seen != (u + 1) * Lh / total) {
      std::printf("mix broken at u=%lld: %lld hot placed\n", (long long)u, (long long)hot_seen);
      return 1;
    }
  }
  // the walk of each CTA u0 < G matches merged() position by position
  for (int64_t G : {(int64_t)1, (int64_t)3, (int64_t)152, (int64_t)1000}) {
    for (int64_t u0 = 0; u0 < G && u0 < total; ++u0) {
      tile_order::MergedWalk w;
      w.start(u0, G, Mh, Mc, NB);
      for (int64_t u = u0; u < total; u += G, w.advance()) {
        int s0, n0, m0, s1, n1, m1;
        tile_order::merged(u, pre_h.data(), pre_c.data(), S, NB, Mh, Mc, s0, n0, m0);
        w.tile(pre_h.data(), pre_c.data(), S, NB, s1, n1, m1);
        if (w.u != u || s0 != s1 || n0 != n1 || m0 != m1) {
          std::printf("walk G=%lld u0=%lld differs at u=%lld: (%d,%d,%d) vs (%d,%d,%d)\n",
                      (long long)G, (long long)u0, (long long)u, s1, n1, m1, s0, n0, m0);
          return 1;
        }
      }
    }
  }
  for (int s = 0; s < S; ++s)
    for (int n = 0; n < NB; ++n)
      for (int m = 0; m < mt[s]; ++m) {
        const int64_t id = base[s] + (int64_t)n * mt[s] + m;
        if (pos[id] < 0) {
          std::printf("tile (%d, %d, %d) never placed\n", s, n, m);
          return 1;
        }
        if (!interleave && id > 0 && pos[id] != id) {  // plain order without interleave
          std::printf("plain order broken at tile %lld\n", (long long)id);
          return 1;
        }
      }
  return 0;
}

int main() {
  int cases = 0;
  // hand-made layouts: no hot segment, only hot segments, empty segments, one segment
  const std::vector<std::vector<int>> fixed = {
      {1, 1, 1, 0, 1}, {2, 3, 14}, {0, 0, 5, 0}, {1}, {9}, {0, 1, 0, 2, 0, 1, 0, 3, 0}};
  for (const auto &mt : fixed)
    for (int NB : {1, 2, 16, 32})
      for (int il = 0; il < 2; ++il) {
        ++cases;
        if (check(mt, NB, il != 0)) return 1;
      }
  // random layouts shaped like routed loads: a few hot experts, many one-block ones
  for (int it = 0; it < 3000; ++it) {
    const int S = 1 + (int)(next_u32() % 300);
    std::vector<int> mt(S);
    for (int s = 0; s < S; ++s) {
      const uint32_t r = next_u32() % 100;
      mt[s] = r < 10 ? 0 : (r < 70 ? 1 : 2 + (int)(next_u32() % (r < 95 ? 4 : 20)));
    }
    const int NB = 1 + (int)(next_u32() % 64);
    ++cases;
    if (check(mt, NB, (it & 3) != 0)) return 1;
  }
  std::printf("tile order ok: %d cases\n", cases);
  return 0;
}
