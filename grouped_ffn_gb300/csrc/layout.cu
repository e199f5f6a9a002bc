// Dispatch layout: slot choice, histogram, stable prefix-scan permutation
// into contiguous per-slot segments, and per-rank counts.
// "14. Serving Mixture-of-Experts Models", "Follow one token through an MoE
// layer", steps 1-2: a permutation built from a histogram over the expert
// ids, so that the kernels that follow see contiguous per-expert segments,
// each sent to the rank that owns the expert.  Replica preference: "The
// network topology is visible in every MoE layer" (a copy on the same node
// first, otherwise spread).
//
// One pass over the assignments, single launch plus a tiny finalize:
//  * CTAs take 1024-assignment tiles in launch order from an atomic ticket
//    (smaller tiles measured faster: more CTAs, two rounds per warp).
//  * Each warp ranks its 256 assignments stably with __match_any_sync and a
//    per-warp shared-memory histogram; a per-slot scan over the 16 warps
//    gives the tile's own histogram and each warp's offset.
//  * Tiles chain their per-slot histograms with a decoupled look-back
//    (one 32-bit word per (tile, slot): 2-bit flag + 30-bit count), so each
//    assignment's rank within its slot is known after one read of the
//    input.  Every spin is bounded by a %globaltimer deadline.
//  * The CTA of the last tile turns the totals into seg_counts,
//    seg_offsets (exclusive scan) and rank_counts; the finalize kernel adds
//    seg_offsets to every partial rank and writes the inverse permutation.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerWarp = 64;
constexpr int kRounds = kPerWarp / 32;
constexpr int kTileA = kWarps * kPerWarp;  // 1024 assignments per tile
constexpr int kMaxSlots = 1024;
constexpr int kMaxRanks = 1024;
constexpr int kMaxExperts = 4096;

constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kFlagErr = 3u << 30;
constexpr uint32_t kValMask = (1u << 30) - 1;

struct LayoutArgs {
  const int32_t *topk_ids;
  int64_t A;
  int32_t k, E, S, R, rpn;
  const int32_t *slot_expert, *slot_rank, *rep_offsets, *rep_slots, *token_src_rank;
  int32_t *slot, *seg_counts, *seg_offsets, *dest_row, *src_assign, *rank_counts;
  uint32_t *tile_flags;  // [n_tiles][K]
  int32_t *ticket;
  int32_t *status;
  int32_t n_tiles;
  int32_t K;                // keys counted by the scan (S in slot modes)
  const int32_t *slot_in;   // kModeSlots: the chosen slot of each assignment
  const int32_t *rkey;      // kModeKeys: [E] replicated-expert index or -1
  int32_t *key_totals;      // kModeKeys: [K] assignments per key
  // One tile only (and a contiguous layout): the scan CTA also does the
  // finalize's work, with no look-back flags written and no second launch.
  int32_t fused_finalize;
};

// What the scan counts and ranks: the slot given by the fixed replica rule,
// a slot chosen beforehand (routed layout), or the (replicated expert,
// source rank) key of replica routing.
enum ScanMode { kModeRule = 0, kModeSlots = 1, kModeKeys = 2 };

// Placement tables cached in shared memory by every layout CTA.
struct PlacementCache {
  const int32_t *rep_offsets;  // [E+1]
  const int32_t *rep_slots;    // [S]
  const int32_t *slot_expert;  // [S]
  const int32_t *slot_rank;    // [S]
};

// Slot serving assignment a (expert e), or -1 after reporting an error.
__device__ int choose_slot(const LayoutArgs &p, const PlacementCache &c, int64_t a, int e) {
  if (e < 0 || e >= p.E) {
    moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, (int32_t)a, moe::K_LAYOUT_SCAN);
    return -1;
  }
  const int64_t t = a / p.k;
  const int lo = c.rep_offsets[e], hi = c.rep_offsets[e + 1];
  const int n = hi - lo;
  int s = -1;
  if (lo < 0 || hi > p.S || n < 1) {
    s = -1;
  } else if (n == 1) {
    s = c.rep_slots[lo];
  } else {
    const int src = p.token_src_rank ? p.token_src_rank[t] : (int)(t % p.R);
    const int node = src / p.rpn;
    for (int i = lo; i < hi; ++i) {
      const int cs = c.rep_slots[i];
      if (cs >= 0 && cs < p.S && c.slot_rank[cs] / p.rpn == node) {
        s = cs;
        break;
      }
    }
    if (s < 0) s = c.rep_slots[lo + (int)(t % n)];
  }
  if (s < 0 || s >= p.S || c.slot_expert[s] != e) {
    moe::report_error(p.status, MOE_ERR_PLACEMENT, e, moe::K_LAYOUT_SCAN);
    return -1;
  }
  return s;
}

// Dynamic shared memory of layout_scan_kernel, in 32-bit words.
inline size_t layout_smem_words(int S, int R, int E, int K) {
  return (size_t)(kWarps + 2) * K + R + (E + 1) + 3 * (size_t)S + E;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) layout_scan_kernel(LayoutArgs p) {
  extern __shared__ int32_t smem[];
  const int K = p.K;
  int32_t *whist = smem;                       // [kWarps][K]: counts, then warp offsets
  int32_t *tile_prefix = smem + kWarps * K;    // [K]
  int32_t *tile_agg = tile_prefix + K;         // [K]
  int32_t *rload = tile_agg + K;               // [R], last tile only
  int32_t *c_rep_offsets = rload + p.R;        // [E+1]
  int32_t *c_rep_slots = c_rep_offsets + p.E + 1;  // [S]
  int32_t *c_slot_expert = c_rep_slots + p.S;      // [S]
  int32_t *c_slot_rank = c_slot_expert + p.S;      // [S]
  int32_t *c_rkey = c_slot_rank + p.S;             // [E], kModeKeys
  __shared__ int32_t s_tile;

  moe::pdl_wait();
  moe::pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) s_tile = atomicAdd(p.ticket, 1);
  for (int i = tid; i < kWarps * K; i += kThreads) whist[i] = 0;
  for (int i = tid; i <= p.E; i += kThreads) c_rep_offsets[i] = p.rep_offsets[i];
  for (int i = tid; i < p.S; i += kThreads) {
    c_rep_slots[i] = p.rep_slots[i];
    c_slot_expert[i] = p.slot_expert[i];
    c_slot_rank[i] = p.slot_rank[i];
  }
  if (MODE == kModeKeys)
    for (int i = tid; i < p.E; i += kThreads) c_rkey[i] = p.rkey[i];
  __syncthreads();
  const int tile = s_tile;
  const PlacementCache cache{c_rep_offsets, c_rep_slots, c_slot_expert, c_slot_rank};

  // ---- keys of this warp's 256 assignments (all loads issued together)
  const int64_t base = (int64_t)tile * kTileA + (int64_t)warp * kPerWarp;
  int ids[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t a = base + r * 32 + lane;
    ids[r] = (a < p.A) ? __ldg(p.topk_ids + a) : 0;
  }
  int my_slot[kRounds], my_rank[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t a = base + r * 32 + lane;
    int s = -1;
    if (a < p.A) {
      const int e = ids[r];
      if (MODE == kModeRule) {
        s = choose_slot(p, cache, a, e);
      } else if (MODE == kModeSlots) {
        s = __ldg(p.slot_in + a);
        if (e < 0 || e >= p.E) {
          moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, (int32_t)a, moe::K_LAYOUT_SCAN);
          s = -1;
        } else if (s < 0 || s >= p.S || cache.slot_expert[s] != e) {
          moe::report_error(p.status, MOE_ERR_PLACEMENT, (int32_t)a, moe::K_LAYOUT_SCAN);
          s = -1;
        }
      } else {  // kModeKeys: only experts with several replicas are keyed
        if (e < 0 || e >= p.E) {
          moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, (int32_t)a, moe::K_LAYOUT_SCAN);
        } else if (c_rkey[e] >= 0) {
          const int64_t t = a / p.k;
          const int src = p.token_src_rank ? p.token_src_rank[t] : (int)(t % p.R);
          if (src < 0 || src >= p.R)
            moe::report_error(p.status, MOE_ERR_PLACEMENT, (int32_t)a, moe::K_LAYOUT_SCAN);
          else
            s = c_rkey[e] * p.R + src;
        }
      }
    }
    my_slot[r] = s;
  }

  // ---- stable rank of each assignment inside its warp's 256-run
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int s = my_slot[r];
    const uint32_t peers = __match_any_sync(0xffffffffu, s);
    const int leader = __ffs(peers) - 1;
    const int before = (s >= 0) ? whist[warp * K + s] : 0;
    __syncwarp();
    if (s >= 0 && lane == leader) whist[warp * K + s] = before + __popc(peers);
    __syncwarp();
    my_rank[r] = before + __popc(peers & ((1u << lane) - 1u));
  }
  __syncthreads();

  // ---- per key: warp offsets, tile aggregate, decoupled look-back
  for (int s = tid; s < K; s += kThreads) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = whist[w * K + s];
      whist[w * K + s] = run;
      run += c;
    }
    tile_agg[s] = run;
    uint32_t *my_flag = p.tile_flags + (size_t)tile * K + s;
    int prefix = 0;
    bool ok = true;
    if (p.fused_finalize) {
      // the only tile: no other CTA reads a flag
    } else if (tile == 0) {
      moe::st_relaxed_u32(my_flag, kFlagInc | (uint32_t)run);
    } else {
      moe::st_relaxed_u32(my_flag, kFlagAgg | (uint32_t)run);
      const uint64_t t0 = moe::global_timer_ns();
      for (int j = tile - 1; j >= 0;) {
        const uint32_t f = moe::ld_relaxed_u32(p.tile_flags + (size_t)j * K + s);
        const uint32_t flag = f & ~kValMask;
        if (flag == 0) {
          if (moe::global_timer_ns() - t0 > moe::kWaitLimitNs) {
            moe::report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, tile, moe::K_LAYOUT_SCAN);
            ok = false;
            break;
          }
          __nanosleep(32);
          continue;
        }
        if (flag == kFlagErr) {
          ok = false;
          break;
        }
        prefix += (int)(f & kValMask);
        if (flag == kFlagInc) break;
        --j;
      }
      moe::st_relaxed_u32(my_flag, ok ? (kFlagInc | (uint32_t)(prefix + run)) : kFlagErr);
    }
    tile_prefix[s] = prefix;
  }
  __syncthreads();
  if (MODE != kModeKeys && p.fused_finalize && warp == 0) {
    // the only tile's per-slot totals are final: their exclusive scan is
    // the segment offsets, which take the place of the (zero) tile prefix
    const int per = (K + 31) / 32;
    const int lo = lane * per, hi = min(K, lo + per);
    int sum = 0;
    for (int s = lo; s < hi; ++s) sum += tile_agg[s];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - sum;
    for (int s = lo; s < hi; ++s) {
      tile_prefix[s] = run;
      run += tile_agg[s];
    }
  }
  __syncthreads();

  // ---- ranks: partial (seg_offsets added by the finalize kernel), or final
  // with the inverse permutation when this CTA finalizes too
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t a = base + r * 32 + lane;
    if (a < p.A) {
      const int s = my_slot[r];
      if (MODE == kModeRule) p.slot[a] = s;
      int d = (s >= 0) ? tile_prefix[s] + whist[warp * K + s] + my_rank[r] : -1;
      if (MODE != kModeKeys && p.fused_finalize && d >= 0) {
        if (d >= p.A) {
          moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, (int32_t)a, moe::K_LAYOUT_SCAN);
          d = -1;
        } else {
          p.src_assign[d] = (int32_t)a;
        }
      }
      p.dest_row[a] = d;
    }
  }

  // ---- the last tile knows the totals
  if (tile != p.n_tiles - 1) return;
  if (MODE == kModeKeys) {
    for (int s = tid; s < K; s += kThreads) p.key_totals[s] = tile_prefix[s] + tile_agg[s];
    return;
  }
  int32_t *tot = whist;  // reuse: [S] totals
  __syncthreads();
  for (int s = tid; s < p.S; s += kThreads) {
    tot[s] = p.fused_finalize ? tile_agg[s] : tile_prefix[s] + tile_agg[s];
    p.seg_counts[s] = tot[s];
  }
  for (int r = tid; r < p.R; r += kThreads) rload[r] = 0;
  __syncthreads();
  for (int s = tid; s < p.S; s += kThreads) {
    const int r = p.slot_rank[s], e = p.slot_expert[s];
    bool bad = r < 0 || r >= p.R || e < 0 || e >= p.E;
    if (s > 0) {
      const int pr = p.slot_rank[s - 1], pe = p.slot_expert[s - 1];
      bad = bad || pr > r || (pr == r && pe >= e);
    }
    if (bad)
      moe::report_error(p.status, MOE_ERR_PLACEMENT, s, moe::K_LAYOUT_SCAN);
    else
      atomicAdd(&rload[r], tot[s]);
  }
  // exclusive scan of the totals by warp 0: lane L owns a contiguous chunk
  // (the fixed-capacity layout has no offsets and passes none)
  if (warp == 0 && p.seg_offsets != nullptr) {
    const int per = (p.S + 31) / 32;
    const int lo = lane * per, hi = min(p.S, lo + per);
    int sum = 0;
    for (int s = lo; s < hi; ++s) sum += tot[s];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - sum;
    for (int s = lo; s < hi; ++s) {
      p.seg_offsets[s] = run;
      run += tot[s];
    }
    if (lane == 31) p.seg_offsets[p.S] = incl;
  }
  __syncthreads();
  for (int r = tid; r < p.R; r += kThreads) p.rank_counts[r] = rload[r];
  // the finalize kernel would clear the ticket for the next call
  if (p.fused_finalize && tid == 0) *p.ticket = 0;
}

// Adds seg_offsets to the partial ranks and writes the inverse permutation;
// then clears the scan's ticket and look-back flags, so the next call on
// this workspace finds them zero without a separate memset.
__global__ void layout_finalize_kernel(LayoutArgs p) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n_flags = (int64_t)p.n_tiles * p.K;
  for (int64_t i = i0; i < n_flags; i += stride) p.tile_flags[i] = 0u;
  if (i0 == 0) *p.ticket = 0;
  for (int64_t a = i0; a < p.A; a += stride) {
    const int s = p.slot[a];
    if (s < 0 || p.dest_row[a] < 0) continue;
    const int d = p.dest_row[a] + p.seg_offsets[s];
    if (d < 0 || d >= p.A) {
      moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, (int32_t)a, moe::K_LAYOUT_FINALIZE);
      p.dest_row[a] = -1;
      continue;
    }
    p.dest_row[a] = d;
    p.src_assign[d] = (int32_t)a;
  }
}

// Fixed-capacity ("masked") layout: slot s owns rows [s*cap, (s+1)*cap).
// "14. Serving Mixture-of-Experts Models", "Capacity, padding, and the drop
// decision" (a fixed per-expert capacity; what overflows is dropped and its
// output is zero); "Mixture-of-Experts Inference", "Communication pressure"
// (decode pads tokens into fixed-size masked layouts so that one captured
// graph can be replayed).  The scan left each assignment's stable rank
// within its slot in dest_row; the first `cap` of a slot keep a row, later
// ones get -1.  Also marks unused rows in src_assign, clips the per-slot and
// per-rank counts to what runs, counts the drops, and clears the scan's
// ticket and flags.  Block 0 does the per-slot work.
__global__ void layout_finalize_masked_kernel(LayoutArgs p, int32_t cap, int32_t *masked_m,
                                              int32_t *n_dropped) {
  __shared__ int32_t rload[kMaxRanks];
  __shared__ int32_t dropped;
  moe::pdl_wait();
  moe::pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n_flags = (int64_t)p.n_tiles * p.K;
  for (int64_t i = i0; i < n_flags; i += stride) p.tile_flags[i] = 0u;
  if (i0 == 0) *p.ticket = 0;
  for (int64_t a = i0; a < p.A; a += stride) {
    const int s = p.slot[a];
    const int pos = p.dest_row[a];
    if (s < 0 || s >= p.S || pos < 0 || pos >= cap) {
      p.dest_row[a] = -1;
      continue;
    }
    const int d = s * cap + pos;
    p.dest_row[a] = d;
    p.src_assign[d] = (int32_t)a;
  }
  const int64_t rows = (int64_t)p.S * cap;
  for (int64_t i = i0; i < rows; i += stride) {
    const int s = (int)(i / cap);
    if ((int)(i - (int64_t)s * cap) >= min(p.seg_counts[s], cap)) p.src_assign[i] = -1;
  }
  if (blockIdx.x != 0) return;
  for (int r = threadIdx.x; r < p.R; r += blockDim.x) rload[r] = 0;
  if (threadIdx.x == 0) dropped = 0;
  __syncthreads();
  int my_drop = 0;
  for (int s = threadIdx.x; s < p.S; s += blockDim.x) {
    const int c = p.seg_counts[s];
    const int m = min(c, cap);
    masked_m[s] = m;
    my_drop += c - m;
    const int r = p.slot_rank[s];
    if (r >= 0 && r < p.R) atomicAdd(&rload[r], m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) my_drop += __shfl_xor_sync(0xffffffffu, my_drop, off);
  if ((threadIdx.x & 31) == 0 && my_drop) atomicAdd(&dropped, my_drop);
  __syncthreads();
  for (int r = threadIdx.x; r < p.R; r += blockDim.x) p.rank_counts[r] = rload[r];
  if (threadIdx.x == 0) *n_dropped = dropped;
}

inline int64_t n_tiles_for(int64_t A) { return A > 0 ? (A + kTileA - 1) / kTileA : 0; }

// ---------------------------------------------------------------- replica routing
// "Zepp", Section 4.1 (Eq. 1) and Section 5 "Routing": per expert with
// several replicas, a greedy water-filling decides how many of each source
// rank's assignments each replica serves, preferring the source's own GPU,
// then its node, then remote nodes, within integer load bounds around the
// even split; a source's assignments then take those destinations in
// ascending order.
constexpr int kMaxRep = 16;      // replicas of one expert
constexpr int kMaxKeys = 1024;   // (replicated experts) x ranks

struct RouteArgs {
  int32_t E, S, R, rpn, Kx;  // Kx = S - E bounds the number of replicated experts
  int32_t c_num, c_den;
  const int32_t *rep_offsets, *rep_slots, *slot_rank;
  int32_t *rkey;         // [E] replicated-expert index or -1
  int32_t *repl_expert;  // [Kx]
  int32_t *n_repl;       // [1]
  const int32_t *key_totals;  // [Kx * R] demand d[c][i]
  int32_t *left;         // [Kx * R] scratch
  int32_t *M;            // [Kx * R * kMaxRep] assignments of source i served by replica p
  int32_t *inter_node;   // [1] output
  int32_t *status;
};

// Index the experts that have several replicas (one warp).
__global__ void route_prep_kernel(RouteArgs r) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  int base = 0;
  for (int e0 = 0; e0 < r.E; e0 += 32) {
    const int e = e0 + lane;
    int n = 0;
    if (e < r.E) n = r.rep_offsets[e + 1] - r.rep_offsets[e];
    bool rep = n >= 2;
    if (rep && n > kMaxRep) {
      moe::report_error(r.status, MOE_ERR_PLACEMENT, e, moe::K_LAYOUT_SCAN);
      rep = false;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, rep);
    const int idx = base + __popc(m & ((1u << lane) - 1u));
    if (rep && idx >= r.Kx) {
      moe::report_error(r.status, MOE_ERR_PLACEMENT, e, moe::K_LAYOUT_SCAN);
      rep = false;
    }
    if (e < r.E) r.rkey[e] = rep ? idx : -1;
    if (rep) r.repl_expert[idx] = e;
    base += __popc(m);
  }
  if (lane == 0) {
    *r.n_repl = min(base, r.Kx);
    *r.inter_node = 0;
  }
}

// One thread per replicated expert: the water-filling of its demand.
__global__ void route_waterfill_kernel(RouteArgs r) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= *r.n_repl) return;
  const int e = r.repl_expert[c];
  const int off = r.rep_offsets[e];
  const int n = r.rep_offsets[e + 1] - off;
  int rank_of[kMaxRep];
  int lo[kMaxRep], hi[kMaxRep], load[kMaxRep];
  const int32_t *d = r.key_totals + (size_t)c * r.R;
  int32_t *left = r.left + (size_t)c * r.R;
  int32_t *M = r.M + (size_t)c * r.R * kMaxRep;
  int64_t D = 0;
  for (int i = 0; i < r.R; ++i) {
    left[i] = d[i];
    D += d[i];
    for (int q = 0; q < kMaxRep; ++q) M[i * kMaxRep + q] = 0;
  }
  const int base = (int)(D / n), rem = (int)(D % n);
  const int slack = (int)(((int64_t)r.c_num * D) / ((int64_t)r.c_den * n));
  for (int q = 0; q < kMaxRep; ++q) {
    if (q < n) {
      rank_of[q] = r.slot_rank[r.rep_slots[off + q]];
      const int qq = base + (q < rem ? 1 : 0);
      lo[q] = max(0, qq - slack);
      hi[q] = qq + slack;
      load[q] = 0;
    }
  }
  int64_t U = D;
  auto deficit_total = [&]() {
    int64_t t = 0;
    for (int q = 0; q < n; ++q) t += max(0, lo[q] - load[q]);
    return t;
  };
  auto give = [&](int i, int q, int64_t x) {
    if (x <= 0) return;
    left[i] -= (int)x;
    load[q] += (int)x;
    U -= x;
    M[i * kMaxRep + q] += (int)x;
  };
  // passes 1-3: own GPU, own node, remote; each capped by capacity and by
  // the demand the other replicas' lower bounds still need
  for (int pass = 0; pass < 3; ++pass) {
    for (int i = 0; i < r.R; ++i) {
      for (int q = 0; q < n && left[i] > 0; ++q) {
        const int rq = rank_of[q];
        const bool same_node = rq / r.rpn == i / r.rpn;
        const bool in_pass = pass == 0 ? rq == i : (pass == 1 ? (rq != i && same_node) : !same_node);
        if (!in_pass) continue;
        const int64_t others = deficit_total() - max(0, lo[q] - load[q]);
        const int64_t allow = min((int64_t)(hi[q] - load[q]), U - others);
        give(i, q, min((int64_t)left[i], max((int64_t)0, allow)));
      }
    }
  }
  // pass 4: what the reserve rule held back, deficits first
  for (int i = 0; i < r.R; ++i) {
    for (int q = 0; q < n && left[i] > 0; ++q)
      if (lo[q] > load[q]) give(i, q, min(left[i], lo[q] - load[q]));
    for (int q = 0; q < n && left[i] > 0; ++q) give(i, q, min(left[i], hi[q] - load[q]));
  }
  if (U != 0) moe::report_error(r.status, MOE_ERR_PLACEMENT, e, moe::K_LAYOUT_SCAN);
}

// Per assignment: the replica its rank within (expert, source) falls into,
// walking the source's locality order; counts inter-node assignments and
// clears the scan's ticket and flags for the next call.
__global__ void route_assign_kernel(RouteArgs r, LayoutArgs p, int32_t *slot) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n_flags = (int64_t)p.n_tiles * p.K;
  int inter = 0;
  for (int64_t a = i0; a < p.A; a += stride) {
    const int e = p.topk_ids[a];
    if (e < 0 || e >= p.E) {
      slot[a] = -1;
      continue;
    }
    const int64_t t = a / p.k;
    const int src = p.token_src_rank ? p.token_src_rank[t] : (int)(t % p.R);
    const int off = r.rep_offsets[e];
    const int n = r.rep_offsets[e + 1] - off;
    int s = -1;
    if (n == 1) {
      s = r.rep_slots[off];
    } else if (r.rkey[e] >= 0 && src >= 0 && src < p.R) {
      const int rank = slot[a];  // rank within (expert, source), from the scan
      const int32_t *M = r.M + ((size_t)r.rkey[e] * p.R + src) * kMaxRep;
      int cum = 0;
      for (int pass = 0; pass < 3 && s < 0; ++pass) {
        for (int q = 0; q < n; ++q) {
          const int rq = r.slot_rank[r.rep_slots[off + q]];
          const bool same_node = rq / p.rpn == src / p.rpn;
          const bool in_pass =
              pass == 0 ? rq == src : (pass == 1 ? (rq != src && same_node) : !same_node);
          if (!in_pass) continue;
          cum += M[q];
          if (rank >= 0 && rank < cum) {
            s = r.rep_slots[off + q];
            break;
          }
        }
      }
    }
    if (s < 0) {
      moe::report_error(p.status, MOE_ERR_PLACEMENT, (int32_t)a, moe::K_LAYOUT_FINALIZE);
    } else if (r.slot_rank[s] / p.rpn != src / p.rpn) {
      ++inter;
    }
    slot[a] = s;
  }
  for (int64_t i = i0; i < n_flags; i += stride) p.tile_flags[i] = 0u;
  if (i0 == 0) *p.ticket = 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) inter += __shfl_xor_sync(0xffffffffu, inter, off);
  if ((threadIdx.x & 31) == 0 && inter) atomicAdd(r.inter_node, inter);
}

// "Zepp", Section 5 "Routing": starting from a feasible routing, a greedy
// refinement consolidates each token's remote expert requests onto fewer
// nodes within the same load bounds.  Each source rank's counts per copy
// stay as given, so every copy's load, the bounds and the number of
// inter-node assignments are unchanged; a request of a replicated expert
// that was sent to a remote copy may move to another remote copy of its
// expert whose count for this rank is not used up.  One CTA per source
// rank: its tokens in ascending order; each token covers its open requests
// node by node -- a node it already sends to first, then the node that
// covers most of them, ties to the lower node id -- and a request takes the
// lowest-rank copy on that node with count left.  The rank keeps the result
// only if its (token, remote node) pairs do not rise.
constexpr int kRefineThreads = 256;

struct RefineArgs {
  const int32_t *topk_ids;
  const int32_t *token_src_rank;  // [T] or null: token t lives on rank t mod R
  int64_t T;
  int32_t k, E, S, R, rpn, n_nodes;
  const int32_t *rep_offsets, *rep_slots, *slot_rank;
  int32_t *slot;      // [A] in: the routing to refine; out: refined
  int32_t *cand;      // [A] scratch: the refined slot of every open request
  int32_t *messages;  // [2] (token, remote node) pairs before / after (accumulated)
  int32_t *status;
};

// Shared memory (int32 words) of route_refine_kernel.
inline size_t refine_smem_words(int E, int S, int kmax) {
  return 2 * (size_t)E + 1 + 5 * (size_t)S + kRefineThreads + 16 +
         2 * (size_t)kRefineThreads * kmax;
}

// The placement and count tables a CTA keeps in shared memory.
struct RefineTables {
  const int32_t *rep_off;    // [E+1] clamped to [0, S]
  const int32_t *rep_sl;     // [S] slot per copy, -1 if invalid
  const int32_t *slot_node;  // [S] node of each slot, -1 if invalid
  int32_t *left;             // [S] this rank's count left per remote copy
  int n_i;                   // the rank's node
};

// One token's greedy cover, by one thread, against counts that no other
// token of the same round changes (see route_refine_kernel).  e/s0/m0: the
// token's k <= KMAX requests (expert, input slot, remote node or -1); open:
// requests that may move.  Returns the refined slot of each request in
// cur_s and the token's remote-node count before and after.  Every loop over
// requests runs to the compile-time KMAX, so the per-request values stay in
// registers.
template <int KMAX>
__device__ __forceinline__ void refine_token_lane(const RefineTables &tb, int k, const int (&e)[KMAX],
                                                  const int (&s0)[KMAX], const int (&m0)[KMAX],
                                                  uint32_t open, int (&cur_s)[KMAX], int &before,
                                                  int &after, bool &failed) {
  // distinct remote nodes: the token's before, and those of the requests
  // that do not move
  int usedn[KMAX];
  int nu = 0;
  before = 0;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    cur_s[j] = s0[j];
    usedn[j] = -1;
    if (j >= k || m0[j] < 0) continue;
    bool seen = false;
#pragma unroll
    for (int q = 0; q < j; ++q) seen |= q < k && m0[q] == m0[j];
    before += seen ? 0 : 1;
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j >= k || m0[j] < 0 || ((open >> j) & 1u)) continue;
    bool seen = false;
#pragma unroll
    for (int q = 0; q < KMAX; ++q) seen |= usedn[q] == m0[j];
    if (!seen) {
#pragma unroll
      for (int q = 0; q < KMAX; ++q)
        if (q == nu) usedn[q] = m0[j];
      ++nu;
    }
  }
  // a copy this token already took once counts one less for its later
  // requests (only a token that repeats an expert id takes a copy twice)
  int took_s[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) took_s[j] = -1;
  auto avail = [&](int s2) {
    int c = tb.left[s2];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) c -= took_s[q] == s2 ? 1 : 0;
    return c > 0;
  };
  auto cand_node = [&](int s2) {  // remote node of a copy with count left, else -1
    if (s2 < 0) return -1;
    const int m2 = tb.slot_node[s2];
    return (m2 >= 0 && m2 != tb.n_i && avail(s2)) ? m2 : -1;
  };
  // whether request q has a copy with count left on node m2
  auto has_on = [&](int eq, int m2) {
    for (int c = tb.rep_off[eq]; c < tb.rep_off[eq + 1]; ++c)
      if (cand_node(tb.rep_sl[c]) == m2) return true;
    return false;
  };
  failed = false;
  for (int iter = 0; iter < KMAX && open; ++iter) {
    uint32_t best_key = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (!((open >> j) & 1u)) continue;
      const int lo = tb.rep_off[e[j]], hi = tb.rep_off[e[j] + 1];
      for (int c = lo; c < hi; ++c) {
        const int m2 = cand_node(tb.rep_sl[c]);
        if (m2 < 0) continue;
        bool dup = false;
        for (int c2 = lo; c2 < c && !dup; ++c2) dup = cand_node(tb.rep_sl[c2]) == m2;
        if (dup) continue;
        int cover = 0;  // open requests with a copy on m2
#pragma unroll
        for (int q = 0; q < KMAX; ++q)
          if ((open >> q) & 1u) cover += (q == j || has_on(e[q], m2)) ? 1 : 0;
        bool in_used = false;
#pragma unroll
        for (int q = 0; q < KMAX; ++q) in_used |= usedn[q] == m2;
        const uint32_t key =
            (in_used ? 0u : 1u) << 16 | (uint32_t)(32 - cover) << 10 | (uint32_t)m2;
        best_key = min(best_key, key);
      }
    }
    if (best_key == 0xffffffffu) {  // no copy left: inconsistent input
      failed = true;
      break;
    }
    const int best = (int)(best_key & 1023u);
    uint32_t took = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (!((open >> j) & 1u)) continue;
      for (int c = tb.rep_off[e[j]]; c < tb.rep_off[e[j] + 1]; ++c) {
        const int s2 = tb.rep_sl[c];
        if (cand_node(s2) != best) continue;
        took_s[j] = s2;
        cur_s[j] = s2;
        took |= 1u << j;
        break;
      }
    }
#pragma unroll
    for (int q = 0; q < KMAX; ++q)
      if (q == nu) usedn[q] = best;
    ++nu;
    open &= ~took;
  }
  after = 0;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const int mj = j >= k ? -1 : (cur_s[j] == s0[j] ? m0[j] : tb.slot_node[cur_s[j]]);
    if (mj < 0) continue;
    bool seen = false;
#pragma unroll
    for (int q = 0; q < j; ++q) {
      const int mq = q >= k ? -1 : (cur_s[q] == s0[q] ? m0[q] : tb.slot_node[cur_s[q]]);
      seen |= mq == mj;
    }
    after += seen ? 0 : 1;
  }
}

// refine_token_lane for at most 32 nodes and a token without repeated
// expert ids: node sets are bit masks, and nmask[e] holds the remote nodes on
// which expert e has a copy with count left (valid for the whole round).
template <int KMAX>
__device__ __forceinline__ void refine_token_lane_masks(
    const RefineTables &tb, const uint32_t *nmask, int k, const int (&e)[KMAX],
    const int (&s0)[KMAX], const int (&m0)[KMAX], uint32_t open, int (&cur_s)[KMAX],
    int &before, int &after, bool &failed) {
  uint32_t all0 = 0, used = 0, mj[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    cur_s[j] = s0[j];
    mj[j] = 0;
    if (j >= k || m0[j] < 0) continue;
    all0 |= 1u << m0[j];
    if ((open >> j) & 1u)
      mj[j] = nmask[e[j]];
    else
      used |= 1u << m0[j];
  }
  before = __popc(all0);
  failed = false;
  while (open) {
    uint32_t uni = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) uni |= ((open >> j) & 1u) ? mj[j] : 0u;
    if (uni == 0) {  // no copy left: inconsistent input
      failed = true;
      break;
    }
    uint32_t best_key = 0xffffffffu;
    for (uint32_t u = uni; u; u &= u - 1) {
      const int m = __ffs(u) - 1;
      int cover = 0;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) cover += ((open >> j) & (mj[j] >> m) & 1u) ? 1 : 0;
      const uint32_t key = (((used >> m) & 1u) ^ 1u) << 16 | (uint32_t)(32 - cover) << 10 |
                           (uint32_t)m;
      best_key = min(best_key, key);
    }
    const int best = (int)(best_key & 1023u);
    uint32_t took = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (!((open >> j) & (mj[j] >> best) & 1u)) continue;
      for (int c = tb.rep_off[e[j]]; c < tb.rep_off[e[j] + 1]; ++c) {
        const int s2 = tb.rep_sl[c];
        if (s2 >= 0 && tb.slot_node[s2] == best && tb.left[s2] > 0) {
          cur_s[j] = s2;
          took |= 1u << j;
          break;
        }
      }
    }
    used |= 1u << best;
    open &= ~took;
    if (!took) {  // a mask that disagrees with the counts: inconsistent input
      failed = true;
      break;
    }
  }
  uint32_t all1 = 0;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j >= k) continue;
    const int mj2 = cur_s[j] == s0[j] ? m0[j] : tb.slot_node[cur_s[j]];
    if (mj2 >= 0) all1 |= 1u << mj2;
  }
  after = __popc(all1);
}

// nmask[e] for every expert: remote nodes (bits) holding a copy of e whose
// count for this rank is left; experts with one copy get 0.  By `lanes`
// threads starting at `first`.
__device__ __forceinline__ void refine_node_masks(const RefineTables &tb, uint32_t *nmask, int E,
                                                  int first, int lanes) {
  for (int ex = first; ex < E; ex += lanes) {
    uint32_t mk = 0;
    const int lo = tb.rep_off[ex], hi = tb.rep_off[ex + 1];
    if (hi - lo > 1)
      for (int c = lo; c < hi; ++c) {
        const int s2 = tb.rep_sl[c];
        const int m2 = s2 >= 0 ? tb.slot_node[s2] : -1;
        if (m2 >= 0 && m2 != tb.n_i && tb.left[s2] > 0) mk |= 1u << m2;
      }
    nmask[ex] = mk;
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kRefineThreads) route_refine_kernel(RefineArgs r) {
  moe::pdl_wait();
  moe::pdl_trigger();
  extern __shared__ int32_t rs[];
  int32_t *rep_off = rs;                    // [E+1]
  int32_t *rep_sl = rep_off + (r.E + 1);    // [S]
  int32_t *slot_node = rep_sl + r.S;        // [S] node of each slot, -1 if invalid
  int32_t *left = slot_node + r.S;          // [S] this rank's count left per remote copy
  int32_t *use = left + r.S;                // [S] a round's takes per copy
  int32_t *list = use + r.S;                // [kRefineThreads] open tokens of a chunk
  uint32_t *nmask = reinterpret_cast<uint32_t *>(list + kRefineThreads + 16);  // [E]
  // [kRefineThreads * KMAX] each: the chunk's open tokens' expert ids and slots
  int32_t *stage_e = reinterpret_cast<int32_t *>(nmask + r.E);
  int32_t *stage_s = stage_e + kRefineThreads * KMAX;
  // [S] a round's takers of each copy, one bit per lane of warp 0
  uint32_t *takers = reinterpret_cast<uint32_t *>(stage_s + kRefineThreads * KMAX);
  int32_t *misc = list + kRefineThreads;    // [1] pairs, [2] saved, [4..11] per-warp counts

  const int i = blockIdx.x;  // source rank
  const int n_i = i / r.rpn;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // placement tables, clamped so that no entry indexes outside them
  for (int e = tid; e <= r.E; e += blockDim.x) rep_off[e] = min(max(r.rep_offsets[e], 0), r.S);
  for (int s = tid; s < r.S; s += blockDim.x) {
    const int v = r.rep_slots[s];
    rep_sl[s] = (v >= 0 && v < r.S) ? v : -1;
    const int rk = r.slot_rank[s];
    slot_node[s] = (rk >= 0 && rk < r.R) ? rk / r.rpn : -1;
    left[s] = use[s] = 0;
    takers[s] = 0u;
  }
  if (tid < 16) misc[tid] = 0;
  __syncthreads();
  const RefineTables tb{rep_off, rep_sl, slot_node, left, n_i};

  const bool by_mod = r.token_src_rank == nullptr;
  const int64_t n_pos = by_mod ? (r.T > i ? (r.T - 1 - i) / r.R + 1 : 0) : r.T;
  auto token_of = [&](int64_t u) { return by_mod ? i + u * r.R : u; };
  auto belongs = [&](int64_t u) { return by_mod || __ldg(r.token_src_rank + u) == i; };
  // request a of this rank: its expert, its slot's remote node (-1 if local
  // or invalid), and whether it may move
  auto classify = [&](int64_t a, int &e, int &s, int &m, bool &open) {
    e = __ldg(r.topk_ids + a);
    s = r.slot[a];
    m = (s >= 0 && s < r.S) ? slot_node[s] : -1;
    const bool remote = m >= 0 && m != n_i;
    open = remote && e >= 0 && e < r.E && rep_off[e + 1] - rep_off[e] > 1;
    if (!remote) m = -1;
  };

  // pass 1: this rank's count per remote copy, and its pairs before
  int pairs = 0;
  for (int64_t u = tid; u < n_pos; u += blockDim.x) {
    if (!belongs(u)) continue;
    const int64_t t = token_of(u);
    int nodes[32];
    int nd = 0;
    for (int j = 0; j < r.k; ++j) {
      int e, s, m;
      bool open;
      classify(t * r.k + j, e, s, m, open);
      if (open) atomicAdd(&left[s], 1);
      if (m < 0) continue;
      bool seen = false;
      for (int q = 0; q < nd; ++q) seen |= nodes[q] == m;
      if (!seen) nodes[nd++] = m;
    }
    pairs += nd;
  }
  atomicAdd(&misc[1], pairs);
  __syncthreads();
  const bool masks = r.n_nodes <= 32;
  if (masks) refine_node_masks(tb, nmask, r.E, tid, blockDim.x);
  __syncthreads();

  // pass 2: chunks of positions; warp 0 refines the chunk's open tokens in
  // order.  Batches of 32 consecutive open tokens, one per lane, decide
  // against the counts as they stand before the batch.  That is exactly the
  // one-by-one result unless a copy's count runs out inside the batch (then
  // a later token could see that copy gone): if any copy's takes reach its
  // count, the batch is redone one token at a time, the whole warp on each.
  int delta = 0;  // pairs saved (warp 0)
  for (int64_t base = 0; base < n_pos; base += blockDim.x) {
    const int64_t u = base + tid;
    bool has_open = false;
    int ce[KMAX], cs[KMAX];
    if (u < n_pos && belongs(u)) {
      const int64_t t = token_of(u);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        int m;
        bool o = false;
        ce[j] = cs[j] = -1;
        if (j < r.k) classify(t * r.k + j, ce[j], cs[j], m, o);
        has_open |= o;
      }
    }
    // compact the chunk's open tokens in ascending position: per-warp counts,
    // then each warp's offset is the sum of the lower warps' counts
    const uint32_t b = __ballot_sync(0xffffffffu, has_open);
    if (lane == 0) misc[4 + warp] = __popc(b);
    __syncthreads();
    int wbase = 0, n_open = 0;
    for (int w = 0; w < kRefineThreads / 32; ++w) {
      wbase += w < warp ? misc[4 + w] : 0;
      n_open += misc[4 + w];
    }
    if (has_open) {
      const int idx = wbase + __popc(b & ((1u << lane) - 1u));
      list[idx] = (int32_t)(u - base);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        stage_e[idx * KMAX + j] = ce[j];
        stage_s[idx * KMAX + j] = cs[j];
      }
    }
    __syncthreads();
    if (warp == 0) {
      // Rounds of up to 32 consecutive open tokens, one per lane, decided
      // against the counts as they stand before the round.  A token's
      // decision is the one-by-one result as long as every count it looked
      // at is still positive at its turn, i.e. up to and including the first
      // token whose take empties a copy; the round commits that prefix and
      // the next round starts after it.
      int q0 = 0;
      while (q0 < n_open) {
        const int n_here = min(32, n_open - q0);
        const bool mine = lane < n_here;
        int e[KMAX], s0[KMAX], m0[KMAX], cur_s[KMAX];
        uint32_t open = 0;
        int64_t t = 0;
        int before = 0, after = 0;
        bool failed = false, repeats = false;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) e[j] = s0[j] = m0[j] = -1;
        if (mine) {
          t = token_of(base + list[q0 + lane]);
#pragma unroll
          for (int j = 0; j < KMAX; ++j) {
            if (j >= r.k) continue;
            // as classify(), from the chunk's staged copies
            const int ej = stage_e[(q0 + lane) * KMAX + j], sj = stage_s[(q0 + lane) * KMAX + j];
            int mj = (sj >= 0 && sj < r.S) ? slot_node[sj] : -1;
            const bool remote = mj >= 0 && mj != n_i;
            if (remote && ej >= 0 && ej < r.E && rep_off[ej + 1] - rep_off[ej] > 1)
              open |= 1u << j;
            e[j] = ej;
            s0[j] = sj;
            m0[j] = remote ? mj : -1;
          }
          // an expert id twice among the token's requests
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
#pragma unroll
            for (int q = 0; q < j; ++q) repeats |= j < r.k && e[q] == e[j];
          if (masks && !repeats)
            refine_token_lane_masks<KMAX>(tb, nmask, r.k, e, s0, m0, open, cur_s, before, after,
                                          failed);
          else
            refine_token_lane<KMAX>(tb, r.k, e, s0, m0, open, cur_s, before, after, failed);
          if (failed)
            moe::report_error(r.status, MOE_ERR_PLACEMENT, (int32_t)t, moe::K_LAYOUT_FINALIZE);
        }
        // takes in token order: the first token that empties a copy ends the
        // prefix.  A token that names an expert twice may take one copy twice,
        // so its choice depends on the counts' values, not only on which are
        // positive: it is exact only as the round's first token, and ends
        // the prefix before itself elsewhere.
        int stop = n_here;
        bool emptied = false;
        const bool lead_repeats = __shfl_sync(0xffffffffu, repeats ? 1 : 0, 0) != 0;
        if (!lead_repeats) {
          // All lanes at once: each marks its takes in the copies' lane
          // masks; a take empties its copy when the takers up to and
          // including this lane (one take per lane: no repeated ids here)
          // reach the copy's count.  The first such lane, or the first lane
          // with repeated ids (which stops before itself), ends the prefix:
          // the same prefix as taking the lanes one by one.
          if (mine && !repeats) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
              if ((open >> j) & 1u) atomicOr(&takers[cur_s[j]], 1u << lane);
          }
          __syncwarp();
          int flag = 0;
          if (mine) {
            if (repeats) {
              flag = 2;
            } else {
              const uint32_t upto = lane == 31 ? 0xffffffffu : (2u << lane) - 1u;
#pragma unroll
              for (int j = 0; j < KMAX; ++j)
                if (((open >> j) & 1u) &&
                    __popc(takers[cur_s[j]] & upto) >= left[cur_s[j]])
                  flag = 1;
            }
          }
          const uint32_t b1 = __ballot_sync(0xffffffffu, flag == 1);
          const uint32_t b2 = __ballot_sync(0xffffffffu, flag == 2);
          const int f1 = b1 ? __ffs(b1) - 1 : 32, f2 = b2 ? __ffs(b2) - 1 : 32;
          if (f2 < f1) {
            stop = f2;
          } else if (f1 < 32) {
            stop = f1 + 1;
            emptied = true;
          }
          __syncwarp();
          if (mine && !repeats) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
              if ((open >> j) & 1u) takers[cur_s[j]] = 0u;
          }
          __syncwarp();
        }
        for (int l = 0; lead_repeats && l < n_here; ++l) {
          int flag = 0;  // 1: empties a copy (kept, then stop); 2: stop before it
          if (lane == l) {
            if (repeats && l > 0) {
              flag = 2;
            } else {
#pragma unroll
              for (int j = 0; j < KMAX; ++j)
                if (((open >> j) & 1u) && ++use[cur_s[j]] >= left[cur_s[j]]) flag = 1;
            }
          }
          flag = __shfl_sync(0xffffffffu, flag, l);
          if (flag) {
            stop = flag == 1 ? l + 1 : l;
            emptied = flag == 1;
            break;
          }
        }
        __syncwarp();
        if (mine && lane < stop) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if ((open >> j) & 1u) {
              use[cur_s[j]] = 0;
              r.cand[t * r.k + j] = cur_s[j];
            }
          delta += before - after;
        }
        __syncwarp();
        if (mine && lane < stop) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if ((open >> j) & 1u) atomicSub(&left[cur_s[j]], 1);
        }
        __syncwarp();
        // counts change availability only when a copy runs out: then the
        // node masks are rebuilt from them
        if (masks && emptied) {
          refine_node_masks(tb, nmask, r.E, lane, 32);
          __syncwarp();
        }
        q0 += stop;
      }
    }
    __syncthreads();
  }
  // each of warp 0's lanes holds the pairs saved by its tokens
  if (warp == 0) atomicAdd(&misc[2], delta);
  __syncthreads();
  const int before = misc[1], saved = misc[2];
  const bool keep = saved >= 0;
  if (keep) {  // pass 3: move the open requests to their refined copies
    for (int64_t u = tid; u < n_pos; u += blockDim.x) {
      if (!belongs(u)) continue;
      const int64_t t = token_of(u);
      for (int j = 0; j < r.k; ++j) {
        int e, s, m;
        bool open;
        const int64_t a = t * r.k + j;
        classify(a, e, s, m, open);
        if (open) r.slot[a] = r.cand[a];
      }
    }
  }
  if (tid == 0) {
    atomicAdd(r.messages, before);
    atomicAdd(r.messages + 1, keep ? before - saved : before);
  }
}



constexpr size_t kTicketOff = moe::kLayoutTicketOff;
constexpr size_t kFlagsOff = moe::kLayoutFlagsOff;

}  // namespace

extern "C" size_t moe_workspace_size(int64_t T, int32_t k, int32_t n_slots) {
  if (T < 0 || k < 1 || n_slots < 1) return 0;
  const int64_t tiles = std::max<int64_t>(n_tiles_for(T * (int64_t)k), 1);
  return kFlagsOff + (size_t)tiles * (size_t)n_slots * sizeof(uint32_t);
}

extern "C" moe_status moe_dispatch_layout(const int32_t *topk_ids, int64_t T, int32_t k,
                                          const moe_placement *pl, int32_t *slot,
                                          int32_t *seg_counts, int32_t *seg_offsets,
                                          int32_t *dest_row, int32_t *src_assign,
                                          int32_t *rank_counts, void *ws, size_t ws_bytes,
                                          void *stream) {
  if (pl == nullptr || T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  const int64_t A = T * (int64_t)k;
  if (A >= (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  if (pl->n_experts < 1 || pl->n_slots < 1 || pl->n_ranks < 1 || pl->ranks_per_node < 1)
    return MOE_ERR_INVALID_ARG;
  if (pl->n_slots > kMaxSlots || pl->n_ranks > kMaxRanks || pl->n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (!pl->slot_expert || !pl->slot_rank || !pl->rep_offsets || !pl->rep_slots || !seg_counts ||
      !seg_offsets || !rank_counts)
    return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_ids || !slot || !dest_row || !src_assign)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size(T, k, pl->n_slots);
  if (moe_status st = moe_host::check_ws(ws, ws_bytes, need)) return st;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n_tiles = std::max<int64_t>(n_tiles_for(A), 1);
  char *wsb = static_cast<char *>(ws);
  // The ticket and flags are zero on entry: moe_workspace_init clears them
  // once, and every call leaves them clear (the finalize kernel, or with a
  // single tile the scan CTA itself, which writes no flag).

  LayoutArgs p{};
  p.topk_ids = topk_ids;
  p.A = A;
  p.k = k;
  p.E = pl->n_experts;
  p.S = pl->n_slots;
  p.R = pl->n_ranks;
  p.rpn = pl->ranks_per_node;
  p.slot_expert = pl->slot_expert;
  p.slot_rank = pl->slot_rank;
  p.rep_offsets = pl->rep_offsets;
  p.rep_slots = pl->rep_slots;
  p.token_src_rank = pl->token_src_rank;
  p.slot = slot;
  p.seg_counts = seg_counts;
  p.seg_offsets = seg_offsets;
  p.dest_row = dest_row;
  p.src_assign = src_assign;
  p.rank_counts = rank_counts;
  p.tile_flags = reinterpret_cast<uint32_t *>(wsb + kFlagsOff);
  p.ticket = reinterpret_cast<int32_t *>(wsb + kTicketOff);
  p.status = moe_host::status_ptr(ws);
  p.n_tiles = (int32_t)n_tiles;

  p.K = p.S;
  const size_t smem = layout_smem_words(p.S, p.R, p.E, p.K) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(layout_scan_kernel<kModeRule>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  p.fused_finalize = n_tiles == 1 ? 1 : 0;
  if (moe_status s = moe_host::launch_pdl(layout_scan_kernel<kModeRule>, dim3((unsigned)n_tiles),
                                          dim3(kThreads), smem, st, p))
    return s;
  if (p.fused_finalize) return MOE_OK;
  int64_t blocks = (std::max<int64_t>(A, n_tiles * p.K) + 255) / 256;
  const int64_t cap = (int64_t)moe_host::sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return moe_host::launch_pdl(layout_finalize_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p);
}

extern "C" moe_status moe_dispatch_layout_masked(const int32_t *topk_ids, int64_t T, int32_t k,
                                                 const moe_placement *pl, int32_t cap,
                                                 int32_t *slot, int32_t *seg_counts,
                                                 int32_t *masked_m, int32_t *dest_row,
                                                 int32_t *src_assign, int32_t *rank_counts,
                                                 int32_t *n_dropped, void *ws, size_t ws_bytes,
                                                 void *stream) {
  if (pl == nullptr || T < 0 || k < 1 || cap < 1) return MOE_ERR_INVALID_ARG;
  const int64_t A = T * (int64_t)k;
  if (A >= (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  if (pl->n_experts < 1 || pl->n_slots < 1 || pl->n_ranks < 1 || pl->ranks_per_node < 1)
    return MOE_ERR_INVALID_ARG;
  if (pl->n_slots > kMaxSlots || pl->n_ranks > kMaxRanks || pl->n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if ((int64_t)pl->n_slots * cap >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (!pl->slot_expert || !pl->slot_rank || !pl->rep_offsets || !pl->rep_slots || !seg_counts ||
      !masked_m || !rank_counts || !n_dropped || !src_assign)
    return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_ids || !slot || !dest_row)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size(T, k, pl->n_slots);
  if (moe_status st = moe_host::check_ws(ws, ws_bytes, need)) return st;

  LayoutArgs p{};
  p.topk_ids = topk_ids;
  p.A = A;
  p.k = k;
  p.E = pl->n_experts;
  p.S = pl->n_slots;
  p.R = pl->n_ranks;
  p.rpn = pl->ranks_per_node;
  p.slot_expert = pl->slot_expert;
  p.slot_rank = pl->slot_rank;
  p.rep_offsets = pl->rep_offsets;
  p.rep_slots = pl->rep_slots;
  p.token_src_rank = pl->token_src_rank;
  p.slot = slot;
  p.seg_counts = seg_counts;
  p.seg_offsets = nullptr;  // no contiguous offsets in this layout
  p.dest_row = dest_row;
  p.src_assign = src_assign;
  p.rank_counts = rank_counts;
  char *wsb = static_cast<char *>(ws);
  p.tile_flags = reinterpret_cast<uint32_t *>(wsb + kFlagsOff);
  p.ticket = reinterpret_cast<int32_t *>(wsb + kTicketOff);
  p.status = moe_host::status_ptr(ws);
  p.n_tiles = (int32_t)std::max<int64_t>(n_tiles_for(A), 1);
  p.K = p.S;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = layout_smem_words(p.S, p.R, p.E, p.K) * sizeof(int32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(layout_scan_kernel<kModeRule>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe_status s = moe_host::launch_pdl(layout_scan_kernel<kModeRule>, dim3((unsigned)p.n_tiles),
                                          dim3(kThreads), smem, st, p))
    return s;
  const int64_t rows = (int64_t)p.S * cap;
  int64_t blocks = (std::max<int64_t>(std::max<int64_t>(A, rows), (int64_t)p.n_tiles * p.K) + 255) / 256;
  const int64_t lim = (int64_t)moe_host::sm_count() * 8;
  if (blocks > lim) blocks = lim;
  return moe_host::launch_pdl(layout_finalize_masked_kernel, dim3((unsigned)blocks), dim3(256), 0,
                              st, p, cap, masked_m, n_dropped);
}

// ---------------------------------------------------------------------------
// Dispatch layout for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// run the layout: a serving engine that has already handed every free byte
// of HBM to its weight and KV-cache pools, or a plugin hosted by another
// runtime that neither passes it a workspace nor lets it call cudaMalloc
// while that runtime is executing.  This entry point keeps the look-back
// scratch (the tile ticket and one 32-bit flag per (1024-assignment tile,
// slot)) in the fixed device array below instead of a caller workspace.
//
// The array is 1 MiB on every GPU that loads this library and stays there
// until the process exits.  Host code may not pass its name to a kernel (on
// the host it is only a stand-in symbol); the device address is looked up
// once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) uint32_t g_layout_noalloc_scratch[262144];

namespace {

constexpr size_t kNoAllocWords = sizeof(g_layout_noalloc_scratch) / sizeof(uint32_t);
constexpr size_t kNoAllocTicketWords = 64;  // ticket word, padded to 256 bytes

// Device address of the scratch array on the current device; nullptr on a
// CUDA error.  The first call on each device does the lookup.
uint32_t *noalloc_scratch() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static uint32_t *addr[kMaxDevices] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_noalloc_scratch) != cudaSuccess || p == nullptr)
      return nullptr;
    addr[dev] = static_cast<uint32_t *>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" moe_status moe_dispatch_layout_noalloc(const int32_t *topk_ids, int64_t T, int32_t k,
                                                  const moe_placement *pl, int32_t *slot,
                                                  int32_t *seg_counts, int32_t *seg_offsets,
                                                  int32_t *dest_row, int32_t *src_assign,
                                                  int32_t *rank_counts, int32_t *status,
                                                  void *stream) {
  if (pl == nullptr || T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  const int64_t A = T * (int64_t)k;
  if (A >= (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  if (pl->n_experts < 1 || pl->n_slots < 1 || pl->n_ranks < 1 || pl->ranks_per_node < 1)
    return MOE_ERR_INVALID_ARG;
  if (pl->n_slots > kMaxSlots || pl->n_ranks > kMaxRanks || pl->n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (!pl->slot_expert || !pl->slot_rank || !pl->rep_offsets || !pl->rep_slots || !seg_counts ||
      !seg_offsets || !rank_counts)
    return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_ids || !slot || !dest_row || !src_assign)) return MOE_ERR_INVALID_ARG;
  const int64_t n_tiles = std::max<int64_t>(n_tiles_for(A), 1);
  const size_t words = kNoAllocTicketWords + (size_t)n_tiles * (size_t)pl->n_slots;
  if (words > kNoAllocWords) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch

  uint32_t *scratch = noalloc_scratch();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left: clear the part used.
  if (cudaMemsetAsync(scratch, 0, words * sizeof(uint32_t), st) != cudaSuccess)
    return MOE_ERR_CUDA;

  LayoutArgs p{};
  p.topk_ids = topk_ids;
  p.A = A;
  p.k = k;
  p.E = pl->n_experts;
  p.S = pl->n_slots;
  p.R = pl->n_ranks;
  p.rpn = pl->ranks_per_node;
  p.slot_expert = pl->slot_expert;
  p.slot_rank = pl->slot_rank;
  p.rep_offsets = pl->rep_offsets;
  p.rep_slots = pl->rep_slots;
  p.token_src_rank = pl->token_src_rank;
  p.slot = slot;
  p.seg_counts = seg_counts;
  p.seg_offsets = seg_offsets;
  p.dest_row = dest_row;
  p.src_assign = src_assign;
  p.rank_counts = rank_counts;
  p.ticket = reinterpret_cast<int32_t *>(scratch);
  p.tile_flags = scratch + kNoAllocTicketWords;
  p.status = status;
  p.n_tiles = (int32_t)n_tiles;

  p.K = p.S;
  const size_t smem = layout_smem_words(p.S, p.R, p.E, p.K) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(layout_scan_kernel<kModeRule>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // one tile (this includes A == 0): the scan CTA finalizes and leaves the
  // ticket and flags clear itself
  p.fused_finalize = n_tiles == 1 ? 1 : 0;
  layout_scan_kernel<kModeRule><<<(unsigned)n_tiles, kThreads, smem, st>>>(p);
  if (moe_status s = moe_host::launch_status()) return s;
  if (!p.fused_finalize) {
    int64_t blocks = (A + 255) / 256;
    const int64_t cap = (int64_t)moe_host::sm_count() * 8;
    if (blocks > cap) blocks = cap;
    layout_finalize_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
    if (moe_status s = moe_host::launch_status()) return s;
  }
  return MOE_OK;
}

// ---------------------------------------------------------------------------
namespace {

size_t route_ws_words_after_flags(int32_t E, int32_t S, int32_t R) {
  const size_t Kx = (size_t)(S > E ? S - E : 0);
  // key totals, rkey, replicated experts, count, left, M
  return Kx * R + (size_t)E + Kx + 1 + Kx * R + Kx * R * kMaxRep;
}

moe_status fill_layout_args(LayoutArgs &p, const int32_t *topk_ids, int64_t T, int32_t k,
                            const moe_placement *pl, void *ws) {
  p = LayoutArgs{};
  p.topk_ids = topk_ids;
  p.A = T * (int64_t)k;
  p.k = k;
  p.E = pl->n_experts;
  p.S = pl->n_slots;
  p.R = pl->n_ranks;
  p.rpn = pl->ranks_per_node;
  p.slot_expert = pl->slot_expert;
  p.slot_rank = pl->slot_rank;
  p.rep_offsets = pl->rep_offsets;
  p.rep_slots = pl->rep_slots;
  p.token_src_rank = pl->token_src_rank;
  char *wsb = static_cast<char *>(ws);
  p.tile_flags = reinterpret_cast<uint32_t *>(wsb + kFlagsOff);
  p.ticket = reinterpret_cast<int32_t *>(wsb + kTicketOff);
  p.status = moe_host::status_ptr(ws);
  p.n_tiles = (int32_t)std::max<int64_t>(n_tiles_for(p.A), 1);
  return MOE_OK;
}

moe_status check_placement(const moe_placement *pl, int64_t T, int32_t k) {
  if (pl == nullptr || T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  if (T * (int64_t)k >= (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  if (pl->n_experts < 1 || pl->n_slots < 1 || pl->n_ranks < 1 || pl->ranks_per_node < 1)
    return MOE_ERR_INVALID_ARG;
  if (pl->n_slots > kMaxSlots || pl->n_ranks > kMaxRanks || pl->n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (!pl->slot_expert || !pl->slot_rank || !pl->rep_offsets || !pl->rep_slots)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Bytes of the replica routing's workspace before the refinement's scratch.
size_t route_ws_bytes(int64_t T, int32_t k, int32_t n_experts, int32_t n_slots, int32_t n_ranks) {
  const int64_t Kx = n_slots > n_experts ? n_slots - n_experts : 0;
  // flags sized for the routing keys and for the slots of a following
  // layout call on the same workspace, so neither reaches the scratch tail
  const int64_t K = std::max<int64_t>(std::max<int64_t>(Kx * n_ranks, 1), n_slots);
  const int64_t tiles = std::max<int64_t>(n_tiles_for(T * (int64_t)k), 1);
  const size_t b = kFlagsOff + (size_t)(tiles * K) * sizeof(uint32_t) +
                   route_ws_words_after_flags(n_experts, n_slots, n_ranks) * sizeof(int32_t);
  return (b + 15) & ~(size_t)15;
}

}  // namespace

extern "C" size_t moe_route_replicas_workspace_size(int64_t T, int32_t k, int32_t n_experts,
                                                    int32_t n_slots, int32_t n_ranks) {
  if (T < 0 || k < 1 || n_experts < 1 || n_slots < 1 || n_ranks < 1) return 0;
  // + the refinement's scratch: one int32 per assignment
  return route_ws_bytes(T, k, n_experts, n_slots, n_ranks) +
         (size_t)(T * (int64_t)k) * sizeof(int32_t);
}

extern "C" moe_status moe_route_refine(const int32_t *topk_ids, int64_t T, int32_t k,
                                       const moe_placement *pl, int32_t *slot, int32_t *messages,
                                       void *ws, size_t ws_bytes, void *stream) {
  if (moe_status s = check_placement(pl, T, k)) return s;
  const int64_t A = T * (int64_t)k;
  if (!messages || (A > 0 && (!topk_ids || !slot))) return MOE_ERR_INVALID_ARG;
  if (k > 32) return MOE_ERR_UNSUPPORTED;
  const size_t need = moe_route_replicas_workspace_size(T, k, pl->n_experts, pl->n_slots,
                                                        pl->n_ranks);
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, need)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(messages, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (A == 0) return MOE_OK;
  RefineArgs r{};
  r.topk_ids = topk_ids;
  r.token_src_rank = pl->token_src_rank;
  r.T = T;
  r.k = k;
  r.E = pl->n_experts;
  r.S = pl->n_slots;
  r.R = pl->n_ranks;
  r.rpn = pl->ranks_per_node;
  r.n_nodes = (pl->n_ranks + pl->ranks_per_node - 1) / pl->ranks_per_node;
  r.rep_offsets = pl->rep_offsets;
  r.rep_slots = pl->rep_slots;
  r.slot_rank = pl->slot_rank;
  r.slot = slot;
  r.cand = reinterpret_cast<int32_t *>(
      static_cast<char *>(ws) + route_ws_bytes(T, k, pl->n_experts, pl->n_slots, pl->n_ranks));
  r.messages = messages;
  r.status = moe_host::status_ptr(ws);
  // shared memory: at most 2 * 4096 + 1 + 5 * 1024 + 272 + 2 * 256 * 32 words (117 KiB)
  const int kmax = k <= 4 ? 4 : k <= 8 ? 8 : k <= 16 ? 16 : 32;
  const size_t smem = refine_smem_words(r.E, r.S, kmax) * sizeof(int32_t);
  auto kern = kmax == 4 ? route_refine_kernel<4>
              : kmax == 8 ? route_refine_kernel<8>
              : kmax == 16 ? route_refine_kernel<16> : route_refine_kernel<32>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_host::launch_pdl(kern, dim3((unsigned)r.R), dim3(kRefineThreads), smem, st, r);
}

extern "C" moe_status moe_route_replicas(const int32_t *topk_ids, int64_t T, int32_t k,
                                         const moe_placement *pl, int32_t c_num, int32_t c_den,
                                         int32_t *slot, int32_t *inter_node, void *ws,
                                         size_t ws_bytes, void *stream) {
  if (moe_status s = check_placement(pl, T, k)) return s;
  if (c_num < 0 || c_den < 1 || !inter_node) return MOE_ERR_INVALID_ARG;
  const int64_t A = T * (int64_t)k;
  if (A > 0 && (!topk_ids || !slot)) return MOE_ERR_INVALID_ARG;
  const int Kx = pl->n_slots > pl->n_experts ? pl->n_slots - pl->n_experts : 0;
  if ((int64_t)Kx * pl->n_ranks > kMaxKeys) return MOE_ERR_UNSUPPORTED;
  const size_t need = moe_route_replicas_workspace_size(T, k, pl->n_experts, pl->n_slots,
                                                        pl->n_ranks);
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, need)) return s;

  LayoutArgs p;
  fill_layout_args(p, topk_ids, T, k, pl, ws);
  p.K = std::max(Kx * pl->n_ranks, 1);
  const int64_t flag_words = (int64_t)p.n_tiles * std::max(p.K, p.S);
  int32_t *tail = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kFlagsOff +
                                              (size_t)flag_words * sizeof(uint32_t));
  RouteArgs r{};
  r.E = p.E;
  r.S = p.S;
  r.R = p.R;
  r.rpn = p.rpn;
  r.Kx = Kx;
  r.c_num = c_num;
  r.c_den = c_den;
  r.rep_offsets = pl->rep_offsets;
  r.rep_slots = pl->rep_slots;
  r.slot_rank = pl->slot_rank;
  int32_t *key_totals = tail;
  r.key_totals = key_totals;
  r.rkey = key_totals + (size_t)Kx * p.R;
  r.repl_expert = r.rkey + p.E;
  r.n_repl = r.repl_expert + Kx;
  r.left = r.n_repl + 1;
  r.M = r.left + (size_t)Kx * p.R;
  r.inter_node = inter_node;
  r.status = p.status;
  p.rkey = r.rkey;
  p.key_totals = key_totals;
  p.dest_row = slot;  // the scan leaves each assignment's rank within its key here
  p.slot = nullptr;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (moe_status s = moe_host::launch_pdl(route_prep_kernel, dim3(1), dim3(32), 0, st, r)) return s;
  if (A > 0 && Kx > 0) {
    const size_t smem = layout_smem_words(p.S, p.R, p.E, p.K) * sizeof(int32_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(layout_scan_kernel<kModeKeys>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (moe_status s = moe_host::launch_pdl(layout_scan_kernel<kModeKeys>, dim3((unsigned)p.n_tiles),
                                            dim3(kThreads), smem, st, p))
      return s;
    if (moe_status s = moe_host::launch_pdl(route_waterfill_kernel, dim3((Kx + 63) / 64), dim3(64),
                                            0, st, r))
      return s;
  }
  int64_t blocks = (std::max<int64_t>(A, (int64_t)p.n_tiles * p.K) + 255) / 256;
  const int64_t cap = (int64_t)moe_host::sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return moe_host::launch_pdl(route_assign_kernel, dim3((unsigned)blocks), dim3(256), 0, st, r, p,
                              slot);
}

extern "C" moe_status moe_dispatch_layout_routed(const int32_t *topk_ids, const int32_t *slot_in,
                                                 int64_t T, int32_t k, const moe_placement *pl,
                                                 int32_t *seg_counts, int32_t *seg_offsets,
                                                 int32_t *dest_row, int32_t *src_assign,
                                                 int32_t *rank_counts, void *ws, size_t ws_bytes,
                                                 void *stream) {
  if (moe_status s = check_placement(pl, T, k)) return s;
  const int64_t A = T * (int64_t)k;
  if (!seg_counts || !seg_offsets || !rank_counts) return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_ids || !slot_in || !dest_row || !src_assign)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size(T, k, pl->n_slots);
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, need)) return s;

  LayoutArgs p;
  fill_layout_args(p, topk_ids, T, k, pl, ws);
  p.K = p.S;
  p.slot_in = slot_in;
  p.slot = const_cast<int32_t *>(slot_in);  // read by the finalize kernel only
  p.seg_counts = seg_counts;
  p.seg_offsets = seg_offsets;
  p.dest_row = dest_row;
  p.src_assign = src_assign;
  p.rank_counts = rank_counts;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = layout_smem_words(p.S, p.R, p.E, p.K) * sizeof(int32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(layout_scan_kernel<kModeSlots>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  p.fused_finalize = p.n_tiles == 1 ? 1 : 0;
  if (moe_status s = moe_host::launch_pdl(layout_scan_kernel<kModeSlots>, dim3((unsigned)p.n_tiles),
                                          dim3(kThreads), smem, st, p))
    return s;
  if (p.fused_finalize) return MOE_OK;
  int64_t blocks = (std::max<int64_t>(A, (int64_t)p.n_tiles * p.K) + 255) / 256;
  const int64_t cap = (int64_t)moe_host::sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return moe_host::launch_pdl(layout_finalize_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p);
}
