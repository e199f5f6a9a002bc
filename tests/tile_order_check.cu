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

// Every CTA's two-phase walk (CtaWalk): each phase-0 position once, by CTA
// u mod G; each phase-1 position once, by the CTA Ph1Plan names; a CTA's
// phase-0 tiles before its phase-1 tiles, positions rising within a phase;
// the tile at each position is merged()'s; and with the first leg not cut
// short, CTAs that reach phase 1 early take delta more phase-1 tiles (+-1).
static int check_walks(const std::vector<int> &mt, int NB0, int NB1, int G, int delta) {
  const int S = (int)mt.size();
  std::vector<int32_t> pre_h(S + 1, 0), pre_c(S + 1, 0);
  for (int s = 0; s < S; ++s) {
    const bool hot = mt[s] >= 2;
    pre_h[s + 1] = pre_h[s] + (hot ? mt[s] : 0);
    pre_c[s + 1] = pre_c[s] + (hot ? 0 : mt[s]);
  }
  const int64_t Mh = pre_h[S], Mc = pre_c[S];
  const int64_t T0 = (Mh + Mc) * NB0, T1 = (Mh + Mc) * NB1;
  std::vector<int> seen0(T0, -1), seen1(T1, -1);
  std::vector<int64_t> n1(G, 0);
  tile_order::Ph1Plan plan;
  plan.init(T0, T1, G, delta);
  for (int c = 0; c < G; ++c) {
    tile_order::CtaWalk w;
    w.start(c, G, Mh, Mc, NB0, NB1, delta);
    int last_ph = 0;
    int64_t last = -1;
    for (int guard = 0; w.valid(); w.next()) {
      if (++guard > T0 + T1 + 2) {
        std::printf("walk of CTA %d does not end\n", c);
        return 1;
      }
      const int64_t u = w.pos();
      if (w.ph < last_ph || (w.ph == last_ph && u <= last)) {
        std::printf("CTA %d: order broken at phase %d position %lld\n", c, w.ph, (long long)u);
        return 1;
      }
      if (w.ph != last_ph) last = -1;
      last_ph = w.ph;
      last = u;
      const int NB = w.ph ? NB1 : NB0;
      int s0, n0, m0, s1, nn1, m1;
      tile_order::merged(u, pre_h.data(), pre_c.data(), S, NB, Mh, Mc, s0, n0, m0);
      w.tile(pre_h.data(), pre_c.data(), S, s1, nn1, m1);
      if (s0 != s1 || n0 != nn1 || m0 != m1) {
        std::printf("CTA %d phase %d position %lld: tile differs from merged()\n", c, w.ph,
                    (long long)u);
        return 1;
      }
      if (w.ph == 0) {
        if (u < 0 || u >= T0 || seen0[u] >= 0 || u % G != c) {
          std::printf("phase-0 position %lld: bad owner %d\n", (long long)u, c);
          return 1;
        }
        seen0[u] = c;
      } else {
        const int owner = u < plan.PA ? plan.r0 + (int)(u % (G - plan.r0))
                                      : (int)((u - plan.PA) % G);
        if (u < 0 || u >= T1 || seen1[u] >= 0 || owner != c) {
          std::printf("phase-1 position %lld: bad owner %d (plan says %d)\n", (long long)u, c,
                      owner);
          return 1;
        }
        seen1[u] = c;
        ++n1[c];
      }
    }
  }
  for (int64_t u = 0; u < T0; ++u)
    if (seen0[u] < 0) {
      std::printf("phase-0 position %lld never taken\n", (long long)u);
      return 1;
    }
  for (int64_t u = 0; u < T1; ++u)
    if (seen1[u] < 0) {
      std::printf("phase-1 position %lld never taken\n", (long long)u);
      return 1;
    }
  if (plan.r0 > 0 && plan.PA == (int64_t)delta * (G - plan.r0) && T1 >= plan.PA + G) {
    int64_t lo_late = 1 << 30, hi_late = -1, lo_early = 1 << 30, hi_early = -1;
    for (int c = 0; c < G; ++c) {
      int64_t &lo = c < plan.r0 ? lo_late : lo_early, &hi = c < plan.r0 ? hi_late : hi_early;
      if (n1[c] < lo) lo = n1[c];
      if (n1[c] > hi) hi = n1[c];
    }
    if (lo_early - hi_late < delta - 1 || hi_early - lo_late > delta + 1) {
      std::printf("phase-1 shares: late CTAs %lld..%lld, early %lld..%lld, delta %d\n",
                  (long long)lo_late, (long long)hi_late, (long long)lo_early,
                  (long long)hi_early, delta);
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
  // the two-phase walks of every CTA, over grids and shifts
  for (int it = 0; it < 1500; ++it) {
    const int S = 1 + (int)(next_u32() % 200);
    std::vector<int> mt(S);
    for (int s = 0; s < S; ++s) {
      const uint32_t r = next_u32() % 100;
      mt[s] = r < 10 ? 0 : (r < 70 ? 1 : 2 + (int)(next_u32() % (r < 95 ? 4 : 20)));
    }
    const int NB0 = 1 + (int)(next_u32() % 32), NB1 = 1 + (int)(next_u32() % 64);
    const int grids[] = {1, 2, 7, 152, 160};
    const int G = grids[next_u32() % 5];
    const int delta = (int)(next_u32() % 6);
    ++cases;
    if (check_walks(mt, NB0, NB1, G, delta)) {
      std::printf("  (S=%d NB0=%d NB1=%d G=%d delta=%d)\n", S, NB0, NB1, G, delta);
      return 1;
    }
  }
  for (const auto &mt : fixed)
    for (int G : {1, 3, 152})
      for (int delta : {0, 4}) {
        ++cases;
        if (check_walks(mt, 16, 32, G, delta)) return 1;
      }
  std::printf("tile order ok: %d cases\n", cases);
  return 0;
}
