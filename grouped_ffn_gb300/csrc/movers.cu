// Row movers and the balancedness statistic.
//
// permute: "14. Serving Mixture-of-Experts Models", "Price one dispatch" --
//   every assignment carries one copy of its token's hidden row (2*H bytes).
//   One CTA per token reads the row once with 128-bit streaming loads and
//   writes it to its k destination rows.
// combine: same chapter, "Follow one token", step 4 -- the inverse
//   permutation followed by the router-weighted sum; plus the shared
//   expert's output ("Mixture-of-Experts Inference", "MoE architecture
//   recap").  One CTA per token gathers the k expert rows 16 bytes at a time
//   and accumulates in fp32 with fmaf in j order, starting from the shared
//   output (or 0), then rounds once to bf16.
// balance: "The slowest expert sets the pace" -- avg/max per-rank load.
#include <cuda_bf16.h>

#include "common.cuh"

namespace {

constexpr int kMoverThreads = 128;
// The permute loads up to 8 x 16 bytes a thread before storing: a 16 KiB
// row (hidden 8192) in one pass of its 128 threads (measured 3-4% faster
// than 4 on the group-limited and replica layers, the same on prefill).
constexpr int kPermUnroll = 8;

// EXTRA: token t is also copied to row extra_row0 + t (the rows a shared
// expert runs on inside the same grouped FFN launch).
template <bool DROP, bool EXTRA>
__global__ void __launch_bounds__(kMoverThreads) permute_kernel(
    const uint4 *__restrict__ x, int64_t T, int H8, int k, const int32_t *__restrict__ dest_row,
    uint4 *__restrict__ xp, int64_t A, int64_t extra_row0, int32_t *status) {
  moe::pdl_wait();
  moe::pdl_trigger();
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4 *src = x + t * H8;
    const int32_t *dr = dest_row + t * k;
    for (int c0 = threadIdx.x; c0 < H8; c0 += kMoverThreads * kPermUnroll) {
      uint4 v[kPermUnroll];
#pragma unroll
      for (int u = 0; u < kPermUnroll; ++u) {
        const int c = c0 + u * kMoverThreads;
        if (c < H8) v[u] = moe::ld_stream_u4(src + c);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(dr + j);
        if (r < 0 || r >= A) {  // DROP: -1 marks a dropped assignment
          if (threadIdx.x == 0 && c0 == 0 && !(DROP && r == -1))
            moe::report_error(status, MOE_ERR_DEVICE_INDEX, (int32_t)(t * k + j), moe::K_PERMUTE);
          continue;
        }
        uint4 *dst = xp + (int64_t)r * H8;
#pragma unroll
        for (int u = 0; u < kPermUnroll; ++u) {
          const int c = c0 + u * kMoverThreads;
          if (c < H8) dst[c] = v[u];
        }
      }
      if (EXTRA) {
        uint4 *dst = xp + (extra_row0 + t) * H8;
#pragma unroll
        for (int u = 0; u < kPermUnroll; ++u) {
          const int c = c0 + u * kMoverThreads;
          if (c < H8) dst[c] = v[u];
        }
      }
    }
  }
}

__device__ __forceinline__ void bf16x8_fma(const uint4 &v, float w, float (&acc)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(u[i] << 16);
    const float hi = __uint_as_float(u[i] & 0xFFFF0000u);
    acc[2 * i] = fmaf(w, lo, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, hi, acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&p);
}

template <int KMAX>
__global__ void __launch_bounds__(kMoverThreads) combine_kernel(
    const uint4 *__restrict__ yp, const int32_t *__restrict__ dest_row,
    const float *__restrict__ topk_w, int64_t T, int k, int H8, const uint4 *__restrict__ shared,
    uint4 *__restrict__ y, int64_t A, int allow_drop, int32_t *status) {
  moe::pdl_wait();
  moe::pdl_trigger();
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    int32_t r[KMAX];
    float w[KMAX];
    bool ok = true;
    uint32_t live = 0;  // terms that take part; a dropped one (-1) adds nothing
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        r[j] = __ldg(dest_row + t * k + j);
        w[j] = __ldg(topk_w + t * k + j);
        if (r[j] >= 0 && r[j] < A)
          live |= 1u << j;
        else if (!(allow_drop && r[j] == -1))
          ok = false;
      }
    }
    if (!ok) {
      if (threadIdx.x == 0) moe::report_error(status, MOE_ERR_DEVICE_INDEX, (int32_t)t, moe::K_COMBINE);
      continue;
    }
    // U column chunks per thread and step, all their row loads issued
    // before any arithmetic (more bytes in flight when k is small)
    constexpr int U = KMAX <= 4 ? 4 : (KMAX <= 8 ? 2 : 1);
    for (int c0 = threadIdx.x; c0 < H8; c0 += kMoverThreads * U) {
      uint4 v[U][KMAX];
      uint4 sv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kMoverThreads;
        if (c < H8) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if ((live >> j) & 1u) v[u][j] = moe::ld_stream_u4(yp + (int64_t)r[j] * H8 + c);
          if (shared) sv[u] = moe::ld_stream_u4(shared + t * H8 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kMoverThreads;
        if (c >= H8) continue;
        float acc[8];
        if (shared) {
          const uint32_t w4[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __uint_as_float(w4[i] << 16);
            acc[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if ((live >> j) & 1u) bf16x8_fma(v[u][j], w[j], acc);
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        y[t * H8 + c] = o;
      }
    }
  }
}

// Combine with node-local pre-reduction ("Zepp", Section 4.2, "Merge";
// Algorithm 1's PreReduce and Reduce), simulated on one GPU: the weighted
// outputs of a token's experts on one node are summed there (fp32 fmaf in
// j order) and returned as one bf16 partial; the source adds the partials
// in ascending node order onto the shared output (or 0) and rounds once.
// Also counts the step's inter-node dispatch messages before merge (remote
// assignments) and after it (distinct remote nodes per token).
template <int KMAX>
__global__ void __launch_bounds__(kMoverThreads) combine_merged_kernel(
    const uint4 *__restrict__ yp, const int32_t *__restrict__ dest_row,
    const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
    const int32_t *__restrict__ slot_rank, const int32_t *__restrict__ token_src_rank, int S,
    int R, int rpn, int64_t T, int k, int H8, const uint4 *__restrict__ shared,
    uint4 *__restrict__ y, int64_t A, int32_t *messages, int32_t *status) {
  moe::pdl_wait();
  moe::pdl_trigger();
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    int32_t r[KMAX], nd[KMAX];
    float w[KMAX];
    bool ok = true;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      nd[j] = 0x7fffffff;
      if (j < k) {
        r[j] = __ldg(dest_row + t * k + j);
        w[j] = __ldg(topk_w + t * k + j);
        const int s = __ldg(slot + t * k + j);
        if (r[j] < 0 || r[j] >= A || s < 0 || s >= S) {
          ok = false;
        } else {
          nd[j] = __ldg(slot_rank + s) / rpn;
        }
      }
    }
    if (!ok) {
      if (threadIdx.x == 0)
        moe::report_error(status, MOE_ERR_DEVICE_INDEX, (int32_t)t, moe::K_COMBINE);
      continue;
    }
    if (threadIdx.x == 0) {
      const int src = token_src_rank ? token_src_rank[t] : (int)(t % R);
      const int sn = src / rpn;
      int before = 0, after = 0;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && nd[j] != sn) {
          ++before;
          bool first = true;
          for (int i = 0; i < j; ++i)
            if (nd[i] == nd[j]) first = false;
          if (first) ++after;
        }
      }
      if (before) {
        atomicAdd(messages, before);
        atomicAdd(messages + 1, after);
      }
    }
    for (int c = threadIdx.x; c < H8; c += kMoverThreads) {
      uint4 v[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) v[j] = moe::ld_stream_u4(yp + (int64_t)r[j] * H8 + c);
      float acc[8];
      if (shared) {
        const uint4 sv = moe::ld_stream_u4(shared + t * H8 + c);
        const uint32_t u[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __uint_as_float(u[i] << 16);
          acc[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      }
      int prev = -1;
      for (;;) {  // destination nodes in ascending order
        int n = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k && nd[j] > prev && nd[j] < n) n = nd[j];
        if (n == 0x7fffffff) break;
        float part[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k && nd[j] == n) bf16x8_fma(v[j], w[j], part);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          acc[i] = __fadd_rn(acc[i], __bfloat162float(__float2bfloat16_rn(part[i])));
        prev = n;
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      y[t * H8 + c] = o;
    }
  }
}

__global__ void balance_kernel(const int32_t *__restrict__ rc, int R, double *bal, int32_t *mx,
                               int64_t *total) {
  moe::pdl_wait();
  moe::pdl_trigger();
  __shared__ long long s_tot[32];
  __shared__ int s_max[32];
  long long tsum = 0;
  int tmax = 0;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int v = rc[r];
    tsum += v;
    tmax = max(tmax, v);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_tot[warp] = tsum;
    s_max[warp] = tmax;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long T = 0;
    int M = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      T += s_tot[i];
      M = max(M, s_max[i]);
    }
    *total = T;
    *mx = M;
    *bal = (T == 0) ? 1.0 : (double)T / ((double)R * (double)M);
  }
}

// Balancedness over L layers: the sum of the layers' mean per-rank loads
// over the sum of their busiest-rank loads ("The slowest expert sets the
// pace": avg_tokens / max_tokens summed across layers).  One warp per layer
// at a time, then a block reduction; the fp64 division is the per-layer
// formula's, total / (R * sum of maxima).
__global__ void balance_layers_kernel(const int32_t *__restrict__ rc, int L, int R, double *bal,
                                      int64_t *max_sum, int64_t *total) {
  moe::pdl_wait();
  moe::pdl_trigger();
  __shared__ long long s_tot[32], s_max[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  long long tsum = 0, msum = 0;
  for (int l = warp; l < L; l += nw) {
    const int32_t *row = rc + (int64_t)l * R;
    long long ls = 0;
    int lm = 0;
    for (int r = lane; r < R; r += 32) {
      const int v = row[r];
      ls += v;
      lm = max(lm, v);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ls += __shfl_xor_sync(0xffffffffu, ls, off);
      lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, off));
    }
    tsum += ls;
    msum += lm;
  }
  if (lane == 0) {
    s_tot[warp] = tsum;
    s_max[warp] = msum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long T = 0, M = 0;
    for (int i = 0; i < nw; ++i) {
      T += s_tot[i];
      M += s_max[i];
    }
    *total = T;
    *max_sum = M;
    *bal = (T == 0) ? 1.0 : (double)T / ((double)R * (double)M);
  }
}

unsigned mover_grid(int64_t T) {
  const int64_t cap = (int64_t)moe_host::sm_count() * 32;
  return (unsigned)(T < cap ? T : cap);
}

}  // namespace

namespace {

// n_rows: rows of x_perm that assignments may land on; allow_drop: dest_row
// -1 marks a dropped assignment; extra_row0 >= 0: also copy token t to row
// extra_row0 + t.
moe_status run_permute(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                       const int32_t *dest_row, int64_t n_rows, uint16_t *x_perm, int allow_drop,
                       void *ws, size_t ws_bytes, void *stream, int64_t extra_row0 = -1) {
  if (T < 0 || H < 1 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !dest_row || (!x_perm && n_rows > 0)) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(x) || !moe_host::aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return moe_host::launch_pdl(extra_row0 >= 0 ? permute_kernel<false, true>
                              : allow_drop   ? permute_kernel<true, false>
                                             : permute_kernel<false, false>,
                              dim3(mover_grid(T)), dim3(kMoverThreads), 0, st,
                              reinterpret_cast<const uint4 *>(x), T, H / 8, k, dest_row,
                              reinterpret_cast<uint4 *>(x_perm), n_rows, extra_row0,
                              moe_host::status_ptr(ws));
}

moe_status run_combine(const uint16_t *y_perm, int64_t n_rows, const int32_t *dest_row,
                       const float *topk_w, int64_t T, int32_t k, int32_t H,
                       const uint16_t *shared, uint16_t *y, int allow_drop, void *ws,
                       size_t ws_bytes, void *stream) {
  if (T < 0 || H < 1 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || k > 16) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if ((!y_perm && n_rows > 0) || !dest_row || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(y_perm) || !moe_host::aligned16(y) ||
      (shared && !moe_host::aligned16(shared)))
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint4 *yp = reinterpret_cast<const uint4 *>(y_perm);
  const uint4 *sh = reinterpret_cast<const uint4 *>(shared);
  uint4 *yo = reinterpret_cast<uint4 *>(y);
  int32_t *status = moe_host::status_ptr(ws);
  const dim3 g(mover_grid(T)), b(kMoverThreads);
  const int H8 = H / 8;
  const int64_t A = n_rows;
  const int d = allow_drop;
  if (k <= 2)
    return moe_host::launch_pdl(combine_kernel<2>, g, b, 0, st, yp, dest_row, topk_w, T, k, H8, sh, yo, A, d, status);
  if (k <= 4)
    return moe_host::launch_pdl(combine_kernel<4>, g, b, 0, st, yp, dest_row, topk_w, T, k, H8, sh, yo, A, d, status);
  if (k <= 8)
    return moe_host::launch_pdl(combine_kernel<8>, g, b, 0, st, yp, dest_row, topk_w, T, k, H8, sh, yo, A, d, status);
  return moe_host::launch_pdl(combine_kernel<16>, g, b, 0, st, yp, dest_row, topk_w, T, k, H8, sh, yo, A, d, status);
}

}  // namespace

extern "C" moe_status moe_permute(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                                  const int32_t *dest_row, uint16_t *x_perm, void *ws,
                                  size_t ws_bytes, void *stream) {
  if (T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  return run_permute(x, T, H, k, dest_row, T * (int64_t)k, x_perm, 0, ws, ws_bytes, stream);
}

extern "C" moe_status moe_permute_shared(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                                         const int32_t *dest_row, uint16_t *x_perm, void *ws,
                                         size_t ws_bytes, void *stream) {
  if (T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  const int64_t A = T * (int64_t)k;
  return run_permute(x, T, H, k, dest_row, A, x_perm, 0, ws, ws_bytes, stream, A);
}

extern "C" moe_status moe_permute_masked(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                                         const int32_t *dest_row, int64_t n_rows,
                                         uint16_t *x_perm, void *ws, size_t ws_bytes,
                                         void *stream) {
  return run_permute(x, T, H, k, dest_row, n_rows, x_perm, 1, ws, ws_bytes, stream);
}

extern "C" moe_status moe_combine(const uint16_t *y_perm, const int32_t *dest_row,
                                  const float *topk_w, int64_t T, int32_t k, int32_t H,
                                  const uint16_t *shared, uint16_t *y, void *ws, size_t ws_bytes,
                                  void *stream) {
  if (T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  return run_combine(y_perm, T * (int64_t)k, dest_row, topk_w, T, k, H, shared, y, 0, ws,
                     ws_bytes, stream);
}

extern "C" moe_status moe_combine_masked(const uint16_t *y_perm, int64_t n_rows,
                                         const int32_t *dest_row, const float *topk_w, int64_t T,
                                         int32_t k, int32_t H, const uint16_t *shared, uint16_t *y,
                                         void *ws, size_t ws_bytes, void *stream) {
  return run_combine(y_perm, n_rows, dest_row, topk_w, T, k, H, shared, y, 1, ws, ws_bytes,
                     stream);
}

extern "C" moe_status moe_balance_stats_layers(const int32_t *rank_counts, int32_t L, int32_t R,
                                               double *balancedness, int64_t *max_sum,
                                               int64_t *total, void *stream) {
  if (L < 1 || R < 1 || !rank_counts || !balancedness || !max_sum || !total)
    return MOE_ERR_INVALID_ARG;
  return moe_host::launch_pdl(balance_layers_kernel, dim3(1), dim3(256), 0,
                              static_cast<cudaStream_t>(stream), rank_counts, L, R, balancedness,
                              max_sum, total);
}

extern "C" moe_status moe_balance_stats(const int32_t *rank_counts, int32_t R, double *balancedness,
                                        int32_t *max_count, int64_t *total, void *ws,
                                        size_t ws_bytes, void *stream) {
  (void)ws;
  (void)ws_bytes;
  if (R < 1 || !rank_counts || !balancedness || !max_count || !total) return MOE_ERR_INVALID_ARG;
  return moe_host::launch_pdl(balance_kernel, dim3(1), dim3(256), 0, static_cast<cudaStream_t>(stream),
                              rank_counts, R, balancedness, max_count, total);
}

extern "C" moe_status moe_combine_merged(const uint16_t *y_perm, const int32_t *dest_row,
                                         const float *topk_w, const int32_t *slot,
                                         const moe_placement *pl, int64_t T, int32_t k, int32_t H,
                                         const uint16_t *shared, uint16_t *y, int32_t *messages,
                                         void *ws, size_t ws_bytes, void *stream) {
  if (T < 0 || H < 1 || k < 1 || !pl || !messages) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || k > 16) return MOE_ERR_UNSUPPORTED;
  if (pl->n_slots < 1 || pl->n_ranks < 1 || pl->ranks_per_node < 1 || !pl->slot_rank)
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(messages, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) return MOE_OK;
  if (!y_perm || !dest_row || !topk_w || !slot || !y) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(y_perm) || !moe_host::aligned16(y) ||
      (shared && !moe_host::aligned16(shared)))
    return MOE_ERR_INVALID_ARG;
  const uint4 *yp = reinterpret_cast<const uint4 *>(y_perm);
  const uint4 *sh = reinterpret_cast<const uint4 *>(shared);
  uint4 *yo = reinterpret_cast<uint4 *>(y);
  const int64_t A = T * (int64_t)k;
  int32_t *status = moe_host::status_ptr(ws);
  const dim3 g(mover_grid(T)), b(kMoverThreads);
  const int H8 = H / 8;
  const int S = pl->n_slots, R = pl->n_ranks, rpn = pl->ranks_per_node;
  const int32_t *sr = pl->slot_rank, *tsr = pl->token_src_rank;
  if (k <= 2)
    return moe_host::launch_pdl(combine_merged_kernel<2>, g, b, 0, st, yp, dest_row, topk_w, slot, sr,
                                tsr, S, R, rpn, T, k, H8, sh, yo, A, messages, status);
  if (k <= 4)
    return moe_host::launch_pdl(combine_merged_kernel<4>, g, b, 0, st, yp, dest_row, topk_w, slot, sr,
                                tsr, S, R, rpn, T, k, H8, sh, yo, A, messages, status);
  if (k <= 8)
    return moe_host::launch_pdl(combine_merged_kernel<8>, g, b, 0, st, yp, dest_row, topk_w, slot, sr,
                                tsr, S, R, rpn, T, k, H8, sh, yo, A, messages, status);
  return moe_host::launch_pdl(combine_merged_kernel<16>, g, b, 0, st, yp, dest_row, topk_w, slot, sr,
                              tsr, S, R, rpn, T, k, H8, sh, yo, A, messages, status);
}
