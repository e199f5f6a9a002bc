// Grouped SwiGLU expert FFN on pairs of SMs (tcgen05.mma.cta_group::2).
//
// The arithmetic is that of grouped_ffn.cu ("14. Serving Mixture-of-Experts
// Models", "Follow one token through an MoE layer", step 3: one grouped GEMM
// over every expert's segment; SwiGLU h = silu(x Wg^T) * (x Wu^T), y = h Wd^T,
// fp32 accumulators, one bf16 rounding each), and a row's bits are the same.
// An opt-in schedule (moe_ffn_schedule.cta_pairs): measured slower than the
// single-SM kernel on the layers of this library's workloads, so not the
// default.  What changes is how the tensor cores are fed.  A stage of the single-SM
// kernel moves 48 KiB through one SM's shared memory (an A tile and a full
// 256-row weight tile) and its MMAs read 48 KiB back; on a layer whose
// weights sit in L2 that shared-memory traffic, not the MMA, sets the pace.
// Here a cluster of two CTAs on two SMs runs each tile together:
//   pair tile  256 rows of a segment (M = 256): each CTA stages its own 128
//              A rows and HALF of the weight tile; the leader CTA (cluster
//              rank 0) issues one MMA that reads both CTAs' shared memory
//              and writes each CTA's accumulator (its 128 rows x 256) in
//              its own TMEM.  32 KiB a stage per SM instead of 48.
//   small      a segment's last block of at most 128 rows (M = 128): 64 rows
//   pair tile  and half the weights per CTA, 24 KiB a stage per SM; the
//              accumulator of a CTA's 64 rows is folded into its TMEM: lanes
//              0-63 hold columns 0-127, lanes 64-127 columns 128-255.
// The weight half of a gate/up stage is [64 gate rows | 64 up rows] of the
// n-block (leader: channels 0-63, peer: 64-127), so every CTA's accumulator
// holds gate and up of the same channels side by side (columns j and 64 + j
// of each 128-column half) and SwiGLU needs no exchange between lanes.
//
// The stages live in six 32 KiB slots (a small pair tile's 24 KiB stage
// leaves 8 KiB of its slot unused).  A byte-granular ring that packed 24 KiB
// stages tighter was built first and measured slower: its bookkeeping sat on
// the producer's path at every stage.
//
// Per CTA (192 threads): warp 0 TMA producer (its own A rows and weight
// half, completion counted on the leader's full barrier); warp 1 allocates
// 512 TMEM columns with the pair (two 256-column accumulators) and, in the
// leader, one lane issues the MMAs and commits to both CTAs' barriers;
// warps 2-5 drain their CTA's accumulator (SwiGLU or plain) and store bf16
// rows.  Gate/up then down run in one cooperative launch as in the
// single-SM kernel, with per-segment readiness counters between them.
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "ffn_pair.h"
#include "tile_order.cuh"
#include "umma.cuh"

namespace {

using namespace umma;

constexpr int kBK = 64;        // K per stage: one 128-byte swizzle row
constexpr int kSlots = 6;      // ring stages of 32 KiB
constexpr int kSlotBytes = 32768;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSegs = 1024;

// kind::f16 instruction descriptor (D fp32, A and B bf16, K-major) with
// N = 256 and the pair's M (256, or 128 for a small pair tile).
constexpr uint32_t idesc_for(int m) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t kIdescBig = idesc_for(256);
constexpr uint32_t kIdescSmall = idesc_for(128);

struct __align__(8) PairBars {
  uint64_t full[kSlots];   // leader: both CTAs' bytes of a stage landed
  uint64_t empty[kSlots];  // each CTA: the stage's MMAs are done with its slot
  uint64_t tfull[2];       // each CTA: accumulator ready
  uint64_t tempty[2];      // leader: both CTAs drained the accumulator
  uint64_t drain;
};

constexpr size_t kBarsOff = (size_t)kSlots * kSlotBytes;
constexpr size_t kMiscOff = kBarsOff + sizeof(PairBars);
constexpr size_t kSegOff = kMiscOff + 64;
constexpr size_t kSmemBytes = kSegOff + (size_t)(5 * kMaxSegs + 3) * 4 + 1024;

struct PairPhase {
  int32_t K, n_blocks;
  uint16_t *out;
  int32_t out_ld;
  int32_t mode;  // 0 gate/up + SwiGLU, 1 down
};

struct PairParams {
  const int32_t *seg_offsets, *seg_expert, *masked_m;
  int32_t S, E, n_rows, cap, n_listed, extra_lo, extra_hi, extra_expert;
  int32_t interleave, ph1_shift;
  int32_t I;        // intermediate width (packed gate/up rows per expert: 2I)
  int32_t *ready;   // [S] finished phase-0 halves per segment
  int32_t *status;
  PairPhase ph[2];
};

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// A tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier that may sit in the peer CTA (cluster address), with an L2
// eviction-priority hint.
__device__ __forceinline__ void tma_load_pair(void *dst, const CUtensorMap *m, int32_t x, int32_t y,
                                              uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this offset in both CTAs of the pair once the
// leader's MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// Arrive on this CTA's mbarrier once the MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair_local(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Arrive on an mbarrier of a CTA of the cluster (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

struct PairTile {
  int ph, s, n_blk, p;
};

// Rows [r0, r0 + 256) of segment s form pair tile p: M = 256 while more than
// 128 rows remain, else the small (M = 128) form.
__device__ __forceinline__ bool pair_is_big(const int32_t *seg_off, const int32_t *seg_end, int s,
                                            int p) {
  return seg_end[s] - (seg_off[s] + 256 * p) > 128;
}

__global__ void __launch_bounds__(kThreads, 1)
    grouped_ffn_pair_kernel(const __grid_constant__ CUtensorMap tmap_a0,
                            const __grid_constant__ CUtensorMap tmap_a0s,
                            const __grid_constant__ CUtensorMap tmap_a1,
                            const __grid_constant__ CUtensorMap tmap_a1s,
                            const __grid_constant__ CUtensorMap tmap_b0,
                            const __grid_constant__ CUtensorMap tmap_b1, const PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PairBars *bars = reinterpret_cast<PairBars *>(smem + kBarsOff);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + kMiscOff + 4);
  volatile int32_t *epi_ok = reinterpret_cast<int32_t *>(smem + kMiscOff + 8);
  // Per tile, in walk order mod 8 (leader): 1 for a big pair tile.  The
  // producer writes it before arming the tile's first stage, the MMA issuer
  // reads it after that stage's full barrier.  The producer runs at most 8
  // stages, so at most 8 tiles, ahead of the MMA.
  uint8_t *tile_big = smem + kMiscOff + 16;
  int32_t *seg_off = reinterpret_cast<int32_t *>(smem + kSegOff);
  int32_t *pre_h = seg_off + (kMaxSegs + 1);
  int32_t *pre_c = pre_h + (kMaxSegs + 1);
  int32_t *seg_exp = pre_c + (kMaxSegs + 1);
  int32_t *seg_end = seg_exp + kMaxSegs;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank_in_cluster();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int32_t kid = moe::K_FFN_GATE_UP;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 8);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  moe::pdl_trigger();
  for (int s = threadIdx.x; s < p.S; s += kThreads) {
    int lo, hi, e;
    if (s >= p.n_listed) {
      lo = p.extra_lo;
      hi = p.extra_hi;
      e = p.extra_expert;
    } else if (p.masked_m != nullptr) {
      int m = p.masked_m[s];
      if (m < 0 || m > p.cap) {
        moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, s, kid);
        m = m < 0 ? 0 : p.cap;
      }
      lo = s * p.cap;
      hi = lo + m;
      e = p.seg_expert[s];
    } else {
      lo = p.seg_offsets[s];
      hi = p.seg_offsets[s + 1];
      e = p.seg_expert[s];
    }
    hi = min(hi, p.n_rows);
    seg_off[s] = lo;
    seg_end[s] = hi;
    seg_exp[s] = e;
    int pt = (hi > lo && lo >= 0) ? (hi - lo + 255) / 256 : 0;
    if (pt > 0 && (e < 0 || e >= p.E)) {
      if (leader) moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, s, kid);
      pt = 0;
    }
    const bool hot = p.interleave && pt >= 2;
    pre_h[s] = hot ? pt : 0;
    pre_c[s] = hot ? 0 : pt;
  }
  __syncthreads();
  if (warp == 0) warp_exclusive_scan(pre_h, p.S, lane);
  if (warp == 2) warp_exclusive_scan(pre_c, p.S, lane);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int NB0 = p.ph[0].n_blocks, NB1 = p.ph[1].n_blocks;
  const int64_t Mh = pre_h[p.S], Mc = pre_c[p.S];
  auto tile_at = [&](const tile_order::CtaWalk &w) {
    PairTile t;
    t.ph = w.ph;
    w.tile(pre_h, pre_c, p.S, t.s, t.n_blk, t.p);
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (warp 0)
    // The whole warp steps through the stages in lockstep; in each, lanes
    // 0-2 issue one load each (A rows, and one or two weight boxes), so the
    // three copies leave in one instruction.
    if (lane == 0) {
      prefetch_tmap(&tmap_a0);
      prefetch_tmap(&tmap_a0s);
      prefetch_tmap(&tmap_a1);
      prefetch_tmap(&tmap_a1s);
      prefetch_tmap(&tmap_b0);
      prefetch_tmap(&tmap_b1);
    }
    uint32_t q = 0, armed = 0, armed_par = 0, tile_seq = 0;
    bool ok = true;
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    const uint64_t pol_a = policy_evict_normal();
    const uint32_t full_c0 = map_shared(&bars->full[0], 0);  // the leader's barriers
    tile_order::CtaWalk w;
    w.start(cluster, n_clusters, Mh, Mc, NB0, NB1, p.ph1_shift);
    for (; w.valid() && ok; w.next()) {
      const PairTile t = tile_at(w);
      const PairPhase &P = p.ph[t.ph];
      const int nk = P.K / kBK;
      const bool big = pair_is_big(seg_off, seg_end, t.s, t.p);
      const int pt = pre_h[t.s + 1] - pre_h[t.s] + pre_c[t.s + 1] - pre_c[t.s];
      const int e = seg_exp[t.s];
      const int NB = t.ph ? NB1 : NB0;
      // packed weights: [e][n_blk][kb][half][128 rows][64 cols]
      const int row_b = (int)((int64_t)(e * NB + t.n_blk) * nk * 256);
      // this lane's copy for every stage of the tile (lane 0: A rows; lane
      // 1: the gate rows [64*rank, +64) of half 0, or the down rows
      // [128*rank, +128); lane 2: the up rows of half 1, phase 0 only)
      const CUtensorMap *map;
      int y, dst_off;
      uint64_t pol;
      bool issues;
      if (lane == 0) {
        map = t.ph ? (big ? &tmap_a1 : &tmap_a1s) : (big ? &tmap_a0 : &tmap_a0s);
        y = seg_off[t.s] + 256 * t.p + (int)rank * (big ? 128 : 64);
        dst_off = 0;
        pol = pol_a;
        issues = true;
      } else {
        // a weight tile read by one pair tile only need not stay in L2
        pol = pt >= 2 ? pol_last : pol_first;
        map = t.ph ? &tmap_b1 : &tmap_b0;
        const int a_bytes = big ? 16384 : 8192;
        if (t.ph == 0) {
          y = row_b + 64 * (int)rank + (lane == 2 ? 128 : 0);
          dst_off = a_bytes + (lane == 2 ? 8192 : 0);
          issues = lane <= 2;
        } else {
          y = row_b + 128 * (int)rank;
          dst_off = a_bytes;
          issues = lane == 1;
        }
      }
      const int x_step = lane == 0 ? kBK : 0;   // A: next 64 columns
      const int y_step = lane == 0 ? 0 : 256;   // packed weights: next k-block
      if (t.ph == 1) {
        // every phase-0 half of the segment has stored its h rows (lane 0
        // waits, then orders its later TMA reads of h after the counter)
        int got = 1;
        if (lane == 0) {
          got = wait_counter(p.ready + t.s, pt * NB0 * 2, abort_flag, p.status, kid) ? 1 : 0;
          if (got) fence_proxy_async_global();
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
      }
      const uint32_t stage_bytes = big ? 32768u : 24576u;  // this CTA's A rows + weight half
      for (int kb = 0; kb < nk; ++kb) {
        const int slot = q % kSlots;
        if (q >= (uint32_t)kSlots) {  // the MMAs of the slot's previous stage are done
          int got = 1;
          if (lane == 0)
            got = mbar_wait(&bars->empty[slot], ((q / kSlots) - 1) & 1u, abort_flag, p.status, kid)
                      ? 1
                      : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
          }
        }
        const uint32_t off = (uint32_t)slot * kSlotBytes;
        if (leader && lane == 0) {
          if (kb == 0) tile_big[tile_seq++ & 7u] = big ? 1 : 0;
          mbar_arrive_expect_tx(&bars->full[slot], 2 * stage_bytes);
          armed |= 1u << slot;
          armed_par = (armed_par & ~(1u << slot)) | (((q / kSlots) & 1u) << slot);
        }
        __syncwarp();
        if (issues)
          tma_load_pair(smem + off + dst_off, map, kb * x_step, y + kb * y_step,
                        full_c0 + 8u * (uint32_t)slot, pol);
        ++q;
      }
    }
    if (lane == 0) {
      if (leader) {
        for (int i = 0; i < kSlots; ++i)  // own and peer copies land before the CTA exits
          if ((armed >> i) & 1u) mbar_wait_drain(&bars->full[i], (armed_par >> i) & 1u);
      } else if (!ok) {
        // copies already issued land within microseconds; give them that
        // before the CTA can exit (their barrier lives in the leader)
        const uint64_t t0 = moe::global_timer_ns();
        while (moe::global_timer_ns() - t0 < 20000) {
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ------------------------------------------------ MMA issuer (leader)
      uint32_t q = 0, tile_seq = 0, acc_phase = 0;
      int acc = 0;
      bool ok = true;
      tile_order::CtaWalk w;
      w.start(cluster, n_clusters, Mh, Mc, NB0, NB1, p.ph1_shift);
      for (; w.valid() && ok; w.next()) {
        const int nk = p.ph[w.ph].K / kBK;
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort_flag, p.status, kid)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        // the tile's first stage has landed, so its size flag is visible
        if (!mbar_wait(&bars->full[q % kSlots], (q / kSlots) & 1u, abort_flag, p.status, kid)) break;
        const bool big = tile_big[tile_seq++ & 7u] != 0;
        const uint32_t a_bytes = big ? 16384u : 8192u;
        for (int kb = 0; kb < nk; ++kb) {
          if (kb > 0 &&
              !mbar_wait(&bars->full[q % kSlots], (q / kSlots) & 1u, abort_flag, p.status, kid)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (q % kSlots) * kSlotBytes);
          const uint32_t sb = sa + a_bytes;
          if (big) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_pair(d_tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), kIdescBig,
                        (kb | kk) != 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_pair(d_tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), kIdescSmall,
                        (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(&bars->empty[q % kSlots]);
          ++q;
        }
        if (!ok) break;
        umma_commit_pair(&bars->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit_pair_local(&bars->drain);  // every MMA of this thread has finished
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // -------------------------------------------------- epilogue warps 2..5
    const int qd = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t tempty_c0 = map_shared(&bars->tempty[0], 0);
    const uint32_t tempty_c1 = map_shared(&bars->tempty[1], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    tile_order::CtaWalk w;
    w.start(cluster, n_clusters, Mh, Mc, NB0, NB1, p.ph1_shift);
    for (; w.valid(); w.next()) {
      const PairTile t = tile_at(w);
      const PairPhase &P = p.ph[t.ph];
      const bool big = pair_is_big(seg_off, seg_end, t.s, t.p);
      // this thread's row of the segment and which columns it holds:
      // big: row 128*rank + 32*qd + lane, all 256 columns;
      // small: row 64*rank + 32*(qd & 1) + lane, accumulator columns
      // 0-127 holding tile columns 128*(qd >> 1) + 0..127
      const int r_in = big ? 128 * (int)rank + 32 * qd + lane : 64 * (int)rank + 32 * (qd & 1) + lane;
      const int row = seg_off[t.s] + 256 * t.p + r_in;
      const bool valid = row < seg_end[t.s];
      if (warp == 2 && lane == 0)
        epi_ok[acc] = mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, p.status, kid) ? 1 : 0;
      epilogue_bar();
      if (!epi_ok[acc]) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * 256);
      uint16_t *orow = valid ? P.out + (int64_t)row * P.out_ld : nullptr;
      if (P.mode == 0) {
        // h channels of this n-block: big, gate/up at columns (j, 64 + j)
        // and (128 + j, 192 + j) for channels j and 64 + j; small, at (j,
        // 64 + j) for channel 64 * (qd >> 1) + j
        const int halves = big ? 2 : 1;
        for (int hf = 0; hf < halves; ++hf) {
          const int ch0 = t.n_blk * 128 + (big ? 64 * hf : 64 * (qd >> 1));
#pragma unroll 1
          for (int c = 0; c < 64; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tbase + 128 * hf + c, g);
            tmem_ld32(tbase + 128 * hf + 64 + c, u);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(silu_mul(g[2 * i], u[2 * i]), silu_mul(g[2 * i + 1], u[2 * i + 1]));
            if (valid) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + ch0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
      } else {
        // y columns: big, all 256 of the n-block; small, 128 * (qd >> 1) + 0..127
        const int ncol = big ? 256 : 128;
        const int col0 = t.n_blk * 256 + (big ? 0 : 128 * (qd >> 1));
#pragma unroll 1
        for (int c = 0; c < ncol; c += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      // this warp's TMEM reads are done: one arrival on the leader's barrier
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty_c1 : tempty_c0);
      if (t.ph == 0) {
        // publish this CTA's h rows to the phase-1 TMA loads of any CTA
        fence_proxy_async_global();
        __threadfence();
        epilogue_bar();
        if (warp == 2 && lane == 0) atomicAdd(p.ready + t.s, 1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per device: the dynamic shared-memory attribute, and how many clusters of
// two run at once (cooperative launches need every CTA resident).
int max_pair_clusters() {
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    if (cudaFuncSetAttribute(grouped_ffn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * moe_host::sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_ffn_pair_kernel, &cfg) != cudaSuccess || n < 1)
      return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

namespace moe_pair {

moe_status run(const PairRun &r, cudaStream_t st) {
  if (r.n_rows == 0) return MOE_OK;
  const int max_clusters = max_pair_clusters();
  if (max_clusters < 1) return MOE_ERR_CUDA;
  CUtensorMap m_x, m_xs, m_h, m_hs, m_wgu, m_wd;
  const uint64_t gu_rows = (uint64_t)r.E * 2 * r.I * r.H / kBK;
  const uint64_t d_rows = (uint64_t)r.E * r.H * r.I / kBK;
  if (!make_map(&m_x, r.x_perm, (uint64_t)r.n_rows, (uint64_t)r.H, 128) ||
      !make_map(&m_xs, r.x_perm, (uint64_t)r.n_rows, (uint64_t)r.H, 64) ||
      !make_map(&m_h, r.h, (uint64_t)r.n_rows, (uint64_t)r.I, 128) ||
      !make_map(&m_hs, r.h, (uint64_t)r.n_rows, (uint64_t)r.I, 64) ||
      !make_map(&m_wgu, r.w_gate_up_packed, gu_rows, (uint64_t)kBK, 64) ||
      !make_map(&m_wd, r.w_down_packed, d_rows, (uint64_t)kBK, 128))
    return MOE_ERR_CUDA;

  PairParams p{};
  p.seg_offsets = r.seg_offsets;
  p.seg_expert = r.seg_expert;
  p.masked_m = r.masked_m;
  p.S = r.S;
  p.E = r.E;
  p.n_rows = (int32_t)r.n_rows;
  p.cap = r.cap;
  p.n_listed = r.n_listed;
  p.extra_lo = (int32_t)r.extra_lo;
  p.extra_hi = (int32_t)r.extra_hi;
  p.extra_expert = r.extra_expert;
  p.interleave = r.interleave;
  p.ph1_shift = r.ph1_shift;
  p.I = r.I;
  p.ready = r.ready;
  p.status = r.status;
  p.ph[0] = PairPhase{r.H, r.I / 128, r.h, r.I, 0};
  p.ph[1] = PairPhase{r.I, r.H / 256, r.y_perm, r.H, 1};

  int64_t clusters = max_clusters;
  if (r.max_pair_tiles < clusters) clusters = r.max_pair_tiles;
  if (clusters < 1) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, grouped_ffn_pair_kernel, m_x, m_xs, m_h, m_hs, m_wgu, m_wd, p) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_host::launch_status();
}

}  // namespace moe_pair
