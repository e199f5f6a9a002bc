// Router: softmax or sigmoid top-k with optional group limit, one warp per
// token.  "14. Serving Mixture-of-Experts Models", "Follow one token through
// an MoE layer": the router produces expert ids and weights for every
// token.  "Mixture-of-Experts Inference", "MoE architecture recap": grouped
// routing picks a limited number of expert groups first, then the top
// experts within them.
//
// Layout: lane L of the warp holds logits L, L+32, L+64, ... of its token
// (VPL values per lane, coalesced 128-byte loads).  Each of the k rounds is
// a per-lane scan of its unselected values followed by a 5-step butterfly
// arg-max; the order (value descending, id ascending) is exactly the one of
// the result, so no sort is needed.  Selection compares the fp32 logits as
// IEEE values (so -0 == +0 and ties go to the lower id).
//
// GB300 issues fp64 at a small fraction of the fp32 rate, so fp64 is used
// only where a floating value decides an integer, and only when needed:
// group scores (the fp64 sum of fp64 sigmoids, by definition) are first
// computed in fp32, one group per lane; the kept set is provably the fp64
// one unless the fp32 margin at the cut is within the fp32 error bound, and
// only then does the warp recompute the scores in fp64.
// Weights are fp32: the softmax exponent l_j - l_max is split error-free
// (TwoSum) into hi + lo and exp(hi + lo) = expf(hi) * (1 + lo); the k terms
// are summed with a TwoSum-compensated butterfly; one IEEE division.  The
// weights are within a few fp32 ulps of the exact values.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace {

struct RouteArgs {
  int32_t score_fn, k, n_groups, topk_groups, group_topn;
};

__device__ __forceinline__ double sigmoid64(float x) { return 1.0 / (1.0 + exp(-(double)x)); }

// Does candidate (ov, oid) beat (bv, bid)?  oid == INT_MAX marks "none".
__device__ __forceinline__ bool beats(float ov, int oid, float bv, int bid) {
  if (oid == INT_MAX) return false;
  if (bid == INT_MAX) return true;
  return ov > bv || (ov == bv && oid < bid);
}

// Arg-max over the warp of the values whose bit is set in `mask` (bit i =
// this lane's element i, id = lane + 32 i).  Returns the winner in all lanes.
template <int VPL>
__device__ __forceinline__ void warp_argmax(const float (&v)[VPL], uint32_t mask, int lane,
                                            float &bv, int &bid) {
  bv = -FLT_MAX;
  bid = INT_MAX;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if ((mask >> i) & 1u) {
      if (beats(v[i], lane + 32 * i, bv, bid)) {
        bv = v[i];
        bid = lane + 32 * i;
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    int oid = __shfl_xor_sync(0xffffffffu, bid, off);
    if (beats(ov, oid, bv, bid)) {
      bv = ov;
      bid = oid;
    }
  }
}

constexpr int kMaxGroupTopn = 8;

__device__ __forceinline__ float sigmoid32(float x) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-x)));
}

__device__ __forceinline__ float sigmoid_of(float x, float) { return sigmoid32(x); }
__device__ __forceinline__ double sigmoid_of(float x, double) { return sigmoid64(x); }

// Lane g returns group g's score: the sum, in descending order, of the
// sigmoids (in precision F) of the group's top_n largest logits.
template <int VPL, typename F>
__device__ F group_score(const float (&v)[VPL], uint32_t avail, int lane, int n_groups,
                         const int (&gid)[VPL], int top_n) {
  F mine = (F)0;
  for (int g = 0; g < n_groups; ++g) {
    uint32_t gmask = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (((avail >> i) & 1u) && gid[i] == g) gmask |= 1u << i;
    for (int r = 0; r < top_n; ++r) {
      float bv;
      int bid;
      warp_argmax<VPL>(v, gmask, lane, bv, bid);
      if (lane == g) mine = mine + sigmoid_of(bv, (F)0);
      if ((bid & 31) == lane) gmask &= ~(1u << (bid >> 5));
    }
  }
  return mine;
}

// Groups of exactly 32 experts (element i of every lane is group i) with a
// score over at most the top 2 logits: every lane computes every group's
// score at once.  Per group, a 5-step butterfly merges the lanes' (largest,
// second largest) pairs into the group's two largest logits (as a multiset,
// so equal logits count twice, as in a selection one at a time); the score
// is sigmoid(largest) + sigmoid(second), in the same order and precision as
// group_score.  Then each lane ranks the groups itself (score descending,
// id ascending, the order select_groups uses): the kept set, the last kept
// score and the best dropped one, with no further shuffles.
template <int VPL>
__device__ __forceinline__ uint32_t select_groups_g32(const float (&v)[VPL], int n_groups,
                                                      int top_n, int n_sel, float &last_kept,
                                                      float &best_dropped) {
  float a1[VPL], a2[VPL];
#pragma unroll
  for (int g = 0; g < VPL; ++g) {
    a1[g] = v[g];
    a2[g] = -FLT_MAX;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int g = 0; g < VPL; ++g) {
      if (g < n_groups) {
        const float o1 = __shfl_xor_sync(0xffffffffu, a1[g], off);
        const float o2 = __shfl_xor_sync(0xffffffffu, a2[g], off);
        const float hi = a1[g] >= o1 ? a1[g] : o1;
        const float lo = a1[g] >= o1 ? o1 : a1[g];
        const float sec = a2[g] >= o2 ? a2[g] : o2;
        a1[g] = hi;
        a2[g] = lo >= sec ? lo : sec;
      }
    }
  }
  float sc[VPL];
#pragma unroll
  for (int g = 0; g < VPL; ++g) {
    sc[g] = 0.0f;
    if (g < n_groups) {
      sc[g] = sigmoid32(a1[g]);
      if (top_n > 1) sc[g] = sc[g] + sigmoid32(a2[g]);
    }
  }
  uint32_t kept = 0;
  last_kept = 0.0f;
  best_dropped = -INFINITY;
#pragma unroll
  for (int g = 0; g < VPL; ++g) {
    if (g >= n_groups) continue;
    int rank = 0;
#pragma unroll
    for (int h = 0; h < VPL; ++h)
      if (h < n_groups && h != g && (sc[h] > sc[g] || (sc[h] == sc[g] && h < g))) ++rank;
    if (rank < n_sel) kept |= 1u << g;
    if (rank == n_sel - 1) last_kept = sc[g];
    if (rank == n_sel) best_dropped = sc[g];
  }
  return kept;
}

// Bit mask of the n_sel best groups (lane g holds group g's score; ties to
// the lower id), with the score of the last one kept and of the best one
// left out (-inf if none).
template <typename F>
__device__ __forceinline__ uint32_t select_groups(F my_score, bool valid, int lane, int n_sel,
                                                  F &last_kept, F &best_dropped) {
  bool free_ = valid;
  uint32_t kept = 0;
  last_kept = (F)0;
  best_dropped = -(F)INFINITY;
  for (int r = 0; r <= n_sel; ++r) {
    F bs = free_ ? my_score : (F)0;
    int bg = free_ ? lane : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const F os = __shfl_xor_sync(0xffffffffu, bs, off);
      const int og = __shfl_xor_sync(0xffffffffu, bg, off);
      if (og != INT_MAX && (bg == INT_MAX || os > bs || (os == bs && og < bg))) {
        bs = os;
        bg = og;
      }
    }
    if (bg == INT_MAX) break;  // no group left
    if (r == n_sel) {
      best_dropped = bs;
      break;
    }
    kept |= 1u << bg;
    last_kept = bs;
    if (lane == bg) free_ = false;
  }
  return kept;
}

// s + e == a + b exactly (round-to-nearest, no overflow).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Compensated butterfly sum; every lane ends with the same value.
__device__ __forceinline__ float warp_sum_compensated(float x) {
  float s = x, c = 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, s, off);
    const float oc = __shfl_xor_sync(0xffffffffu, c, off);
    float e;
    two_sum(s, os, s, e);
    c = __fadd_rn(__fadd_rn(c, oc), e);
  }
  return __fadd_rn(s, c);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int64_t T,
                                                    int E, RouteArgs a, int32_t *__restrict__ ids,
                                                    float *__restrict__ w) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int gsz = a.n_groups > 1 ? E / a.n_groups : E;
  int gid[VPL];  // group of this lane's element i (constant for the whole launch)
#pragma unroll
  for (int i = 0; i < VPL; ++i) gid[i] = (lane + 32 * i) / gsz;

  for (int64_t t = warp0; t < T; t += nwarps) {
    const float *row = logits + t * E;
    float v[VPL];
    uint32_t avail = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        v[i] = __ldg(row + e);
        avail |= 1u << i;
      } else {
        v[i] = 0.0f;
      }
    }

    if (a.n_groups > 1) {
      // Group score: the sum of the sigmoids of the group's group_topn
      // largest logits, taken in descending order; lane g accumulates group
      // g's.  Keep the topk_groups best groups (score descending, id
      // ascending).  The fp32 scores satisfy |s32 - s64| <= eps (expf within
      // 2 ulp, one rounding each for 1 + e, the reciprocal and every add).
      // If the last kept group beats the best dropped one by more than 2 eps
      // the fp64 selection is the same set; otherwise the warp recomputes
      // the scores in fp64 and selects again.
      const bool gvalid = lane < a.n_groups;
      float last_kept, best_dropped;
      uint32_t kept;
      if (gsz == 32 && a.group_topn <= 2) {
        kept = select_groups_g32<VPL>(v, a.n_groups, a.group_topn, a.topk_groups, last_kept,
                                      best_dropped);
      } else {
        const float my_g32 =
            group_score<VPL, float>(v, avail, lane, a.n_groups, gid, a.group_topn);
        kept = select_groups<float>(my_g32, gvalid, lane, a.topk_groups, last_kept, best_dropped);
      }
      const float n = (float)a.group_topn;
      const float eps = n * 2e-7f + (n - 1.0f) * n * 6e-8f;
      if (a.topk_groups < a.n_groups && !(last_kept - best_dropped > 4.0f * eps)) {
        const double my_g64 =
            group_score<VPL, double>(v, avail, lane, a.n_groups, gid, a.group_topn);
        double l64, b64;
        kept = select_groups<double>(my_g64, gvalid, lane, a.topk_groups, l64, b64);
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (!((kept >> gid[i]) & 1u)) avail &= ~(1u << i);
    }

    // Top-k: lane j keeps the j-th selection.
    float my_v = 0.0f;
    int my_id = 0;
    for (int j = 0; j < a.k; ++j) {
      float bv;
      int bid;
      warp_argmax<VPL>(v, avail, lane, bv, bid);
      if ((bid & 31) == lane) avail &= ~(1u << (bid >> 5));
      if (lane == j) {
        my_v = bv;
        my_id = bid;
      }
    }

    float num = 0.0f;
    if (a.score_fn == MOE_SCORE_SOFTMAX) {
      const float m = __shfl_sync(0xffffffffu, my_v, 0);  // the largest logit
      if (lane < a.k) {
        float d, dlo;
        two_sum(my_v, -m, d, dlo);
        num = __fmul_rn(expf(d), __fadd_rn(1.0f, dlo));
      }
    } else {
      if (lane < a.k) num = __frcp_rn(__fadd_rn(1.0f, expf(-my_v)));
    }
    const float den = warp_sum_compensated(num);
    if (lane < a.k) {
      ids[t * a.k + lane] = my_id;
      w[t * a.k + lane] = __fdiv_rn(num, den);
    }
  }
}

template <int VPL>
void launch_route(const float *logits, int64_t T, int E, RouteArgs a, int32_t *ids, float *w,
                  cudaStream_t st) {
  const int threads = 256;
  int64_t blocks = (T + 7) / 8;
  const int64_t cap = (int64_t)moe_host::sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  moe_host::launch_pdl(route_kernel<VPL>, dim3((unsigned)blocks), dim3(threads), 0, st, logits, T, E,
                       a, ids, w);
}

}  // namespace

extern "C" moe_status moe_route(const float *logits, int64_t T, int32_t E, const moe_route_cfg *cfg,
                                int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                                void *stream) {
  (void)ws;
  (void)ws_bytes;
  if (cfg == nullptr || T < 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (logits == nullptr || topk_ids == nullptr || topk_w == nullptr))
    return MOE_ERR_INVALID_ARG;
  RouteArgs a{cfg->score_fn, cfg->k, cfg->n_groups, cfg->topk_groups, cfg->group_topn};
  if (a.score_fn != MOE_SCORE_SOFTMAX && a.score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (a.k < 1 || a.k > E) return MOE_ERR_INVALID_ARG;
  if (a.k > 16 || E > 512) return MOE_ERR_UNSUPPORTED;
  if (a.n_groups < 1) return MOE_ERR_INVALID_ARG;
  if (a.n_groups > 1) {
    if (a.score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    if (a.n_groups > 32 || E % a.n_groups != 0) return MOE_ERR_UNSUPPORTED;
    const int gsz = E / a.n_groups;
    if (a.topk_groups < 1 || a.topk_groups > a.n_groups) return MOE_ERR_INVALID_ARG;
    if (a.group_topn < 1 || a.group_topn > gsz) return MOE_ERR_INVALID_ARG;
    if (a.group_topn > kMaxGroupTopn) return MOE_ERR_UNSUPPORTED;
    if (a.k > a.topk_groups * gsz) return MOE_ERR_INVALID_ARG;
  }
  if (T == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    launch_route<1>(logits, T, E, a, topk_ids, topk_w, st);
  else if (vpl <= 2)
    launch_route<2>(logits, T, E, a, topk_ids, topk_w, st);
  else if (vpl <= 4)
    launch_route<4>(logits, T, E, a, topk_ids, topk_w, st);
  else if (vpl <= 8)
    launch_route<8>(logits, T, E, a, topk_ids, topk_w, st);
  else
    launch_route<16>(logits, T, E, a, topk_ids, topk_w, st);
  return moe_host::launch_status();
}
