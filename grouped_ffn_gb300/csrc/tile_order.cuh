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

// Which merged positions of the down-projection phase (phase 1) CTA c of G
// takes.  Phase 0 hands position u to CTA u mod G, so with T0 = q*G + r0
// tiles the first r0 CTAs take one tile more (about K0/K1 phase-1 tiles'
// worth of work, K the GEMMs' depths) and reach phase 1 late.  The first
// PA = min(delta * (G - r0), T1) phase-1 positions therefore go round-robin
// to the G - r0 CTAs that arrive early (delta each), and the rest to all G
// CTAs in turn:
//   v <  PA:  CTA r0 + (v mod (G - r0))
//   v >= PA:  CTA (v - PA) mod G
// With r0 = 0 or delta = 0 this is plain round-robin.  A CTA's positions
// rise, and every position has exactly one CTA.
struct Ph1Plan {
  int64_t T1, PA;
  int G, r0;

  TILE_ORDER_HD void init(int64_t T0, int64_t T1_, int G_, int delta) {
    T1 = T1_;
    G = G_;
    r0 = (int)(T0 % G_);
    const int64_t pa = (r0 > 0 && delta > 0) ? (int64_t)delta * (G_ - r0) : 0;
    PA = pa < T1_ ? pa : T1_;
  }
  // First position of CTA c and its step (first leg: v < PA).
  TILE_ORDER_HD bool first_leg(int c, int64_t &v0, int64_t &step) const {
    if (c < r0 || PA == 0 || c - r0 >= PA) return false;
    v0 = c - r0;
    step = G - r0;
    return true;
  }
  TILE_ORDER_HD void second_leg(int c, int64_t &v0, int64_t &step) const {
    v0 = PA + c;
    step = G;
  }
};

// The tiles of CTA c of G over both phases, in its order: phase-0
// positions c, c + G, ... below T0 = (Mh + Mc) * NB0, then its phase-1
// positions by Ph1Plan (T1 = (Mh + Mc) * NB1).  Additions per step; a
// division when a leg starts.
struct CtaWalk {
  MergedWalk w;
  Ph1Plan plan;
  int64_t T0, Mh, Mc, step, leg_end;
  int NB0, NB1, c, G, ph, leg;
  bool done;

  TILE_ORDER_HD void start(int c_, int G_, int64_t Mh_, int64_t Mc_, int NB0_, int NB1_,
                           int delta) {
    c = c_;
    G = G_;
    Mh = Mh_;
    Mc = Mc_;
    NB0 = NB0_;
    NB1 = NB1_;
    T0 = (Mh + Mc) * NB0;
    plan.init(T0, (Mh + Mc) * NB1, G, delta);
    done = false;
    if (c < T0) {
      ph = 0;
      step = G;
      leg_end = T0;
      w.start(c, G, Mh, Mc, NB0);
    } else {
      enter_ph1();
    }
  }
  TILE_ORDER_HD void enter_ph1() {
    ph = 1;
    int64_t v0;
    if (plan.first_leg(c, v0, step)) {
      leg = 0;
      leg_end = plan.PA;
    } else {
      leg = 1;
      plan.second_leg(c, v0, step);
      leg_end = plan.T1;
    }
    if (v0 >= leg_end) {
      done = true;
      return;
    }
    w.start(v0, step, Mh, Mc, NB1);
  }
  TILE_ORDER_HD void next() {
    if (w.u + step < leg_end) {
      w.advance();
      return;
    }
    if (ph == 0) {
      enter_ph1();
    } else if (leg == 0) {
      leg = 1;
      int64_t v0;
      plan.second_leg(c, v0, step);
      leg_end = plan.T1;
      if (v0 >= leg_end)
        done = true;
      else
        w.start(v0, step, Mh, Mc, NB1);
    } else {
      done = true;
    }
  }
  TILE_ORDER_HD bool valid() const { return !done; }
  // Position within the current phase.
  TILE_ORDER_HD int64_t pos() const { return w.u; }
  TILE_ORDER_HD void tile(const int32_t *pre_h, const int32_t *pre_c, int S, int &s, int &n_blk,
                          int &m_blk) const {
    w.tile(pre_h, pre_c, S, ph ? NB1 : NB0, s, n_blk, m_blk);
  }
};

}  // namespace tile_order
