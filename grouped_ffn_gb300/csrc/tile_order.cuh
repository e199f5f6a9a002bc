// Order in which the grouped FFN's persistent CTAs take the tiles of one
// GEMM phase.  Host and device code: the kernel decodes its tiles with it,
// and a host-side check (tests/tile_order_check.cu) proves it is a
// bijection.
//
// A phase has NB n-blocks per segment and two tile streams:
//   hot  segments with two or more 128-row m-blocks; their weight tiles are
//        re-read from L2 by every m-block and so lean on the tensor cores;
//   cold one-block segments, which stream fresh weights from HBM.
// pre_h[s] / pre_c[s] (S + 1 entries each) are the exclusive prefix sums of
// the hot / cold m-block counts (a segment counts in one of them, or in
// neither if empty); Mh = pre_h[S], Mc = pre_c[S].  Each stream is ordered
// (segment, n-block, m-block), so a segment's A rows and a weight tile's
// m-blocks stay close in time.
//
// The two streams of Lh = Mh * NB and Lc = Mc * NB tiles are merged in
// proportion to their lengths (Bresenham): position u holds a hot tile when
// floor((u + 1) * Lh / L) > floor(u * Lh / L), with L = Lh + Lc, so that every
// wave of CTAs mixes both kinds of work and neither the tensor pipe nor HBM
// idles for a whole wave.
//
// A persistent CTA visits positions u0, u0 + G, u0 + 2G, ... (G = grid size).
// MergedWalk steps through them with additions only: the division of
// merged() happens once per phase, not once per tile, which keeps the
// bookkeeping between two tiles off the k-block pipeline's critical path.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define TILE_ORDER_HD __host__ __device__ __forceinline__
#else
#define TILE_ORDER_HD inline
#endif

namespace tile_order {

// Tile t of a stream ordered (segment, n-block, m-block), where segment s
// owns tiles [prefix[s] * NB, prefix[s + 1] * NB).  A segment holds fewer
// than 2^32 tiles (under 2^24 m-blocks of 128 rows times NB <= 256), so the
// split into (n-block, m-block) is a 32-bit division.
TILE_ORDER_HD void in_stream(int64_t t, const int32_t *prefix, int S, int NB, int &s, int &n_blk,
                             int &m_blk) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)prefix[mid] * NB <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  s = lo;
  const uint32_t local = (uint32_t)(t - (int64_t)prefix[s] * NB);
  const uint32_t mt = (uint32_t)(prefix[s + 1] - prefix[s]);
  n_blk = (int)(local / mt);
  m_blk = (int)(local - (uint32_t)n_blk * mt);
}

// Merged position u in [0, (Mh + Mc) * NB) -> (segment, n-block, m-block).
TILE_ORDER_HD void merged(int64_t u, const int32_t *pre_h, const int32_t *pre_c, int S, int NB,
                          int64_t Mh, int64_t Mc, int &s, int &n_blk, int &m_blk) {
  const int64_t Lh = Mh * NB, L = (Mh + Mc) * NB;
  const int64_t hb = u * Lh / L;  // hot tiles before position u
  if ((u + 1) * Lh / L > hb)
    in_stream(hb, pre_h, S, NB, s, n_blk, m_blk);
  else
    in_stream(u - hb, pre_c, S, NB, s, n_blk, m_blk);
}

// The positions u0, u0 + G, u0 + 2G, ... of merged(), in order.  The walk
// carries q = floor(u * Lh / L) (hot tiles before u) and r = u * Lh - q * L,
// 0 <= r < L.  Position u is hot when floor((u + 1) * Lh / L) > q, which is
// r + Lh >= L; its index is q in the hot stream, u - q in the cold one.
struct MergedWalk {
  int64_t u, q, r, Lh, L, dq, dr, G;

  TILE_ORDER_HD void start(int64_t u0, int64_t step, int64_t Mh, int64_t Mc, int NB) {
    u = u0;
    G = step;
    Lh = Mh * NB;
    L = (Mh + Mc) * NB;
    if (L > 0) {
      q = u0 * Lh / L;
      r = u0 * Lh - q * L;
      dq = step * Lh / L;
      dr = step * Lh - dq * L;
    } else {
      q = r = dq = dr = 0;
    }
  }
  TILE_ORDER_HD void advance() {
    u += G;
    q += dq;
    r += dr;  // both below L, so one correction restores 0 <= r < L
    if (r >= L) {
      r -= L;
      ++q;
    }
  }
  TILE_ORDER_HD bool hot() const { return r + Lh >= L; }
  // The tile at the current position; the same as merged(u, ...).
  TILE_ORDER_HD void tile(const int32_t *pre_h, const int32_t *pre_c, int S, int NB, int &s,
                          int &n_blk, int &m_blk) const {
    if (hot())
      in_stream(q, pre_h, S, NB, s, n_blk, m_blk);
    else
      in_stream(u - q, pre_c, S, NB, s, n_blk, m_blk);
  }
};

}  // namespace tile_order
