// Grouped SwiGLU expert FFN on 5th-generation tensor cores (sm_103a).
//
// "14. Serving Mixture-of-Experts Models", "Follow one token through an MoE
// layer", step 3: one kernel processes every expert's segment as a matrix
// with its own row count.  "Mixture-of-Experts Inference", "Optimized
// kernels for MoE": grouped GEMM over a contiguous layout.  The gated MLP
// (gate, up, activation, down) is SwiGLU: h = silu(x Wg^T) * (x Wu^T),
// y = h Wd^T.
//
// One persistent, warp-specialised kernel runs both GEMMs in a single
// cooperative launch, over one tile list:
//   phase 0 (gate/up): acc[128 x 256] = X[128 x H] * [Wg; Wu]^T tile,
//                      epilogue h = bf16(silu(acc[:, :128]) * acc[:, 128:])
//   phase 1 (down):    acc[128 x 256] = h[128 x I] * Wd^T tile, epilogue bf16.
// A segment's phase-1 tiles start once all its phase-0 tiles have stored
// their h rows (a per-segment counter; bounded wait).  A tile (128 rows, or 64)
// always starts at a segment's first row plus a multiple of 128 and uses
// that segment's expert; rows past the segment's end are computed from
// whatever follows (or TMA zero fill) and are never stored.
//
// Per CTA (one per SM, 192 threads):
//   warp 0     TMA producer: A tile 128x64 and two B halves 128x64 per
//              k-block into a 4-stage ring (48 KiB per stage, 128-byte
//              swizzle), completion via mbarrier transaction counts.
//   warp 1     allocates 512 TMEM columns (two 128x256 fp32 accumulators);
//              one lane issues tcgen05.mma kind::f16 (M=128, N=256, K=16,
//              4 per k-block) and tcgen05.commit to free smem stages and to
//              hand a finished accumulator to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows),
//              SwiGLU in fp32, bf16 stores masked to the segment.
// A tile with at most 64 rows left in its segment (a small segment, or the
// last block of a longer one; rows not gathered) is an M = 64 tile instead:
// 64 A rows a stage and M = 64 MMAs, so a stage moves 40 KiB through shared
// memory, and the epilogue takes rows from lanes 0..15 of each quadrant.
// Double-buffered accumulators overlap a tile's epilogue with the next
// tile's main loop.  Tiles are ordered (segment, n-block, m-block) so that
// CTAs running side by side share B tiles (weights) and A rows in L2; a
// weight tile that only one m-block reads is loaded with an L2 evict_first
// policy, one that several m-blocks read with evict_last.
// The launch follows the permute with programmatic dependent launch (the
// set-up above overlaps its tail; griddepcontrol.wait precedes every read),
// and the per-segment counters are cleared by the last CTA to finish, so no
// memset sits in between.  All waits are bounded (%globaltimer); on expiry
// the CTA records MOE_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs,
// frees TMEM, exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "ffn_pair.h"
#include "tile_order.cuh"
#include "umma.cuh"

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBHalfBytes = 128 * kBK * 2;
constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
constexpr int kMaxSegs = 1024;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
// Workspace: one readiness counter per segment at moe::kFfnReadyOff.
constexpr size_t kReadyOff = moe::kFfnReadyOff;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
// Tiles with at most kBMSmall rows left in their segment run M = 64: half the
// A tile is loaded and read, so a stage moves 40 KiB through shared memory
// instead of 48.  Their accumulator row r sits in TMEM lane 32 (r / 16) + r % 16
// (16 rows in each warp's lane quadrant), column n in column n.
constexpr int kBMSmall = 64;
constexpr uint32_t kIdescSmall = (kIdesc & ~(0x1Fu << 24)) | ((uint32_t)(kBMSmall >> 4) << 24);

struct __align__(8) Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
};

constexpr size_t kBarsOff = (size_t)kStages * kStageBytes;
constexpr size_t kMiscOff = kBarsOff + sizeof(Bars);
constexpr size_t kSegOff = kMiscOff + 32;
constexpr size_t kGidxOff = kSegOff + (size_t)(5 * kMaxSegs + 3) * 4;  // [kBM] gathered token rows
constexpr size_t kSmemBytes = kGidxOff + kBM * 4 + 1024;

// One GEMM phase: gate/up with the SwiGLU epilogue (mode 0) or down (mode 1).
struct Phase {
  int32_t K, n_blocks;
  int32_t b_rows_per_expert;  // rows of one expert's B matrix (2I or H)
  int32_t b_nblk_stride;      // B row step per n-block (128 or 256)
  int32_t b_second_off;       // row offset of the second 128-row half (I or 128)
  uint16_t *out;
  int32_t out_ld;
  int32_t out_nblk_stride;    // output column step per n-block (128 or 256)
  int32_t mode;               // 0 gate/up + SwiGLU, 1 down
};

struct FfnParams {
  const int32_t *seg_offsets;
  const int32_t *seg_expert;
  int32_t S, E, n_rows;
  int32_t b_packed;   // B in the tile-contiguous layout (see moe_pack_expert_weights)
  int32_t n_phases;   // 2: phase 1 reads what phase 0 writes, in the same launch
  int32_t *ready;     // [S] finished phase-0 tiles per segment (zero on entry)
  uint32_t *exit_count;  // finished CTAs; the last one re-zeroes ready[0, S) and this
  int32_t interleave; // merge multi-tile and one-tile segments' tiles (tile_order.cuh)
  int32_t ph1_shift;  // phase-1 positions that go first to the CTAs with one gate/up tile fewer
  int32_t small_rows; // segments with at most this many rows run M = 64 tiles (0: none)
  // Gather mode: phase 0 reads row r of a segment from x[gather_src[r] / gather_k]
  // (token rows, gather_T of them) instead of a permuted copy.
  const int32_t *gather_src;
  int32_t gather_k, gather_T;
  // Fixed-capacity layout: segment s is rows [s*cap, s*cap + masked_m[s])
  // (seg_offsets unused) when masked_m is set.
  const int32_t *masked_m;
  int32_t cap;
  // Segments [0, n_listed) come from seg_offsets / masked_m; when S is one
  // more, segment n_listed is rows [extra_lo, extra_hi) with expert
  // extra_expert (a shared expert run in the same launch).
  int32_t n_listed;
  int32_t extra_lo, extra_hi, extra_expert;
  int32_t *status;
  Phase ph[2];
};

using namespace umma;

// --------------------------------------------------------------- the kernel
struct TileInfo {
  int ph, s, n_blk, m_blk;
};

// Phase 0 (gate/up) and phase 1 (down) each order their tiles by merging
// the hot stream (segments with two or more m-blocks, whose weight tiles are
// re-read from L2 and so lean on the tensor cores) and the cold stream
// (one-block segments, which stream fresh weights from HBM) in proportion
// to their lengths, so that every wave of CTAs mixes both kinds of work.
// A CTA takes phase-0 positions blockIdx.x, + gridDim.x, ..., then its
// phase-1 positions, shifted so that CTAs which took one more gate/up tile
// take about as many fewer down tiles (tile_order.cuh, Ph1Plan).  Each role
// walks that sequence with additions only: a division per tile on the
// producer's single thread stalled the k-block pipeline at every tile
// boundary.
struct TileWalk {
  tile_order::CtaWalk w;

  __device__ __forceinline__ void start(int64_t Mh, int64_t Mc, int NB0, int NB1, int shift) {
    w.start(blockIdx.x, gridDim.x, Mh, Mc, NB0, NB1, shift);
  }
  __device__ __forceinline__ bool valid() const { return w.valid(); }
  __device__ __forceinline__ void next() { w.next(); }
  __device__ __forceinline__ int phase() const { return w.ph; }
  __device__ __forceinline__ TileInfo info(const int32_t *pre_h, const int32_t *pre_c,
                                           int S) const {
    TileInfo ti;
    ti.ph = w.ph;
    w.tile(pre_h, pre_c, S, ti.s, ti.n_blk, ti.m_blk);
    return ti;
  }
};

// Whether m-block m_blk of segment s is an M = 64 tile: at most small_rows
// rows from its first row to the segment's end (a one-block segment of at
// most 64 rows, or the last block of a longer one), never with gathered rows.
__device__ __forceinline__ bool small_tile(const FfnParams &p, const int32_t *seg_off,
                                           const int32_t *seg_end, int s, int m_blk) {
  return p.gather_src == nullptr && seg_end[s] - (seg_off[s] + m_blk * kBM) <= p.small_rows;
}

// The k-block loop of one tile, with its instruction descriptor fixed at
// compile time (one instantiation for M = 128 tiles, one for M = 64).
// WAIT_FIRST false: the caller has waited for the first stage's full barrier.
template <uint32_t IDESC, bool WAIT_FIRST>
__device__ __forceinline__ bool mma_tile(int nk, uint32_t d_tmem, uint8_t *smem, Bars *bars,
                                         int &stage, uint32_t &phase,
                                         volatile int32_t *abort_flag, int32_t *status,
                                         int32_t kid) {
  for (int kb = 0; kb < nk; ++kb) {
    if ((WAIT_FIRST || kb > 0) && !mbar_wait(&bars->full[stage], phase, abort_flag, status, kid))
      return false;
    tc_fence_after();
    const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
    const uint32_t sb = sa + kABytes;
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)
      umma_bf16(d_tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), IDESC,
                (kb | kk) != 0 ? 1u : 0u);
    umma_commit(&bars->empty[stage]);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// tmap_a0s / tmap_a1s: the A maps with 64-row boxes, for M = 64 tiles.
__global__ void __launch_bounds__(kThreads, 1)
    grouped_ffn_kernel(const __grid_constant__ CUtensorMap tmap_a0,
                       const __grid_constant__ CUtensorMap tmap_b0,
                       const __grid_constant__ CUtensorMap tmap_a1,
                       const __grid_constant__ CUtensorMap tmap_b1,
                       const __grid_constant__ CUtensorMap tmap_a0s,
                       const __grid_constant__ CUtensorMap tmap_a1s, const FfnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + kBarsOff);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + kMiscOff + 4);
  // the epilogue's shared go/stop decision, one per accumulator buffer
  volatile int32_t *epi_ok = reinterpret_cast<int32_t *>(smem + kMiscOff + 8);
  // Per tile, in walk order mod 8 (only when the launch has M = 64 tiles,
  // which gathered rows never do): 1 for an M = 64 tile.  The producer writes
  // it before arming the tile's first stage and the MMA reads it after that
  // stage's full barrier, which orders the two.  The producer runs at most
  // kStages stages, so at most kStages tiles, ahead of the MMA: 8 entries
  // are never overwritten before they are read.
  uint8_t *tile_small = smem + kMiscOff + 16;
  // set in the CTA that finishes last (the one that clears the counters)
  volatile int32_t *last_cta = reinterpret_cast<int32_t *>(smem + kMiscOff + 24);
  int32_t *seg_off = reinterpret_cast<int32_t *>(smem + kSegOff);  // [S] first row of s
  int32_t *pre_h = seg_off + (kMaxSegs + 1);  // [S+1] m-tiles before s, multi-tile segments
  int32_t *pre_c = pre_h + (kMaxSegs + 1);    // [S+1] m-tiles before s, one-tile segments
  int32_t *seg_exp = pre_c + (kMaxSegs + 1);  // [S]
  int32_t *seg_end = seg_exp + kMaxSegs;      // [S] one past the last row of s (<= n_rows)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t kid = p.ph[0].mode == 0 ? moe::K_FFN_GATE_UP : moe::K_FFN_DOWN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 128);
    }
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // Launched behind the permute with programmatic dependent launch: the
  // set-up above overlaps its tail; nothing it writes is read before this.
  moe::pdl_wait();
  // the next kernel on the stream (the combine) may start launching now; it
  // waits (griddepcontrol.wait) until this grid has finished
  moe::pdl_trigger();
  int has_small = 0;
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
    int mt = (hi > lo && lo >= 0) ? (hi - lo + kBM - 1) / kBM : 0;
    if (mt > 0 && (e < 0 || e >= p.E)) {
      moe::report_error(p.status, MOE_ERR_DEVICE_INDEX, s, kid);
      mt = 0;
    }
    const bool hot = p.interleave && mt >= 2;
    pre_h[s] = hot ? mt : 0;
    pre_c[s] = hot ? 0 : mt;
    if (mt > 0 && small_tile(p, seg_off, seg_end, s, mt - 1)) has_small = 1;
  }
  // any M = 64 tile in this launch?  If not, every role runs the plain path.
  const bool any_small = __syncthreads_or(has_small) != 0;
  if (warp == 0) warp_exclusive_scan(pre_h, p.S, lane);
  if (warp == 2) warp_exclusive_scan(pre_c, p.S, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int NB0 = p.ph[0].n_blocks;
  const int NB1 = p.n_phases > 1 ? p.ph[1].n_blocks : 0;
  const int64_t Mh = pre_h[p.S], Mc = pre_c[p.S];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (lane 0;
    // the whole warp stages gathered row indices)
    int32_t *gidx = reinterpret_cast<int32_t *>(smem + kGidxOff);
    if (lane == 0) {
      prefetch_tmap(&tmap_a0);
      prefetch_tmap(&tmap_b0);
      if (p.small_rows > 0) prefetch_tmap(&tmap_a0s);
      if (p.n_phases > 1) {
        prefetch_tmap(&tmap_a1);
        prefetch_tmap(&tmap_b1);
        if (p.small_rows > 0) prefetch_tmap(&tmap_a1s);
      }
    }
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0, tile_seq = 0;
    bool ok = true;
    // Everything one tile's loads need, prepared by lane 0 from its TileInfo.
    struct Loads {
      int ph, s, nk, need, row_a, row_b0, row_b1, b_x_step, b_y_step;
      bool small;  // an M = 64 tile: 64 A rows a stage
      uint64_t wpol;
    };
    auto prepare = [&](const TileInfo &ti) {
      Loads L;
      const Phase &P = p.ph[ti.ph];
      const int NB = ti.ph ? NB1 : NB0;
      const int mt = pre_h[ti.s + 1] - pre_h[ti.s] + pre_c[ti.s + 1] - pre_c[ti.s];
      L.ph = ti.ph;
      L.s = ti.s;
      L.nk = P.K / kBK;
      L.need = mt * NB0;  // phase-0 tiles of the segment, all of which store h
      const int e = seg_exp[ti.s];
      L.row_a = seg_off[ti.s] + ti.m_blk * kBM;
      L.small = any_small && small_tile(p, seg_off, seg_end, ti.s, ti.m_blk);
      // a weight tile read by this m-block only need not stay in L2; one
      // that the segment's other m-blocks read too should
      L.wpol = mt >= 2 ? policy_evict_last() : policy_evict_first();
      // B rows of k-block 0; packed: [e][n_blk][kb][half][128 rows][64 cols],
      // so one k-block of the tile is 32 contiguous KiB.
      const int64_t packed0 = (int64_t)(e * NB + ti.n_blk) * L.nk * 256;
      L.row_b0 = p.b_packed ? (int)packed0 : e * P.b_rows_per_expert + ti.n_blk * P.b_nblk_stride;
      L.row_b1 = p.b_packed ? L.row_b0 + 128 : L.row_b0 + P.b_second_off;
      L.b_x_step = p.b_packed ? 0 : kBK;
      L.b_y_step = p.b_packed ? 256 : 0;
      return L;
    };
    // A phase-1 tile reads h rows: every phase-0 tile of its segment must
    // have stored them (bounded wait on the segment's counter).
    auto wait_h = [&](const Loads &L) {
      if (!wait_counter(p.ready + L.s, L.need, abort_flag, p.status, kid)) return false;
      fence_proxy_async_global();
      return true;
    };
    // k-block kb of a tile into the next ring stage (lane 0; tiled A rows).
    auto load_stage = [&](const Loads &L, int kb) {
      if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, p.status, kid)) return false;
      const CUtensorMap *ma =
          L.ph ? (L.small ? &tmap_a1s : &tmap_a1) : (L.small ? &tmap_a0s : &tmap_a0);
      const CUtensorMap *mb = L.ph ? &tmap_b1 : &tmap_b0;
      uint8_t *sa = smem + (size_t)stage * kStageBytes;
      if (any_small && kb == 0) tile_small[tile_seq++ & 7u] = L.small ? 1 : 0;
      mbar_arrive_expect_tx(&bars->full[stage],
                            L.small ? kStageBytes - kABytes / 2 : kStageBytes);
      tma_load_2d(sa, ma, kb * kBK, L.row_a, &bars->full[stage]);
      tma_load_2d_hint(sa + kABytes, mb, kb * L.b_x_step, L.row_b0 + kb * L.b_y_step,
                       &bars->full[stage], L.wpol);
      tma_load_2d_hint(sa + kABytes + kBHalfBytes, mb, kb * L.b_x_step,
                       L.row_b1 + kb * L.b_y_step, &bars->full[stage], L.wpol);
      armed |= 1u << stage;
      armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
      return true;
    };
    TileWalk walk;
    walk.start(Mh, Mc, NB0, NB1, p.ph1_shift);
    if (p.gather_src == nullptr) {
      // Lane 0 alone.  The next tile's loads are prepared right after the
      // current tile's first stage is issued, while the ring is full, so
      // that its first stage goes out as soon as a slot frees.
      if (lane == 0 && walk.valid()) {
        Loads cur = prepare(walk.info(pre_h, pre_c, p.S));
        for (;;) {
          if (cur.ph == 1 && !wait_h(cur)) {
            ok = false;
            break;
          }
          Loads nxt = cur;
          bool more = false;
          for (int kb = 0; kb < cur.nk; ++kb) {
            if (!load_stage(cur, kb)) {
              ok = false;
              break;
            }
            if (kb == 0) {
              walk.next();
              more = walk.valid();
              if (more) nxt = prepare(walk.info(pre_h, pre_c, p.S));
            }
          }
          if (!ok || !more) break;
          cur = nxt;
        }
      }
    } else {
      // Gathered A rows: the whole warp stages each phase-0 tile's 128
      // token indices; in every stage of such a tile each lane issues one
      // four-row gather (the TMA requests go out in parallel, not from one
      // thread in turn), lane 0 the two weight loads.  Phase-1 tiles load as
      // above, from lane 0.
      for (; walk.valid(); walk.next()) {
        const TileInfo ti = walk.info(pre_h, pre_c, p.S);
        const Loads L = prepare(ti);
        if (ti.ph == 1) {
          if (lane == 0) {
            if (!wait_h(L)) ok = false;
            for (int kb = 0; kb < L.nk && ok; ++kb)
              if (!load_stage(L, kb)) ok = false;
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          // the other lanes follow lane 0's ring position
          stage = __shfl_sync(0xffffffffu, stage, 0);
          phase = __shfl_sync(0xffffffffu, phase, 0);
          if (!ok) break;
          continue;
        }
        // token row of each of the tile's 128 rows (token 0 past the end)
        const int row0 = seg_off[ti.s] + ti.m_blk * kBM;
        const int row_end = seg_end[ti.s];
        for (int j = lane; j < kBM; j += 32) {
          int tok = 0;
          if (row0 + j < row_end) {
            tok = __ldg(p.gather_src + row0 + j) / p.gather_k;
            if (tok < 0 || tok >= p.gather_T) tok = 0;
          }
          gidx[j] = tok;
        }
        __syncwarp();
        for (int kb = 0; kb < L.nk; ++kb) {
          int got = 0;
          if (lane == 0)
            got = mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, p.status, kid) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + (size_t)stage * kStageBytes;
          if (lane == 0) mbar_arrive_expect_tx(&bars->full[stage], kStageBytes);
          __syncwarp();  // the transaction count is armed before any copy lands
          tma_gather4(sa + lane * 512, &tmap_a0, kb * kBK, gidx[4 * lane], gidx[4 * lane + 1],
                      gidx[4 * lane + 2], gidx[4 * lane + 3], &bars->full[stage]);
          if (lane == 0) {
            tma_load_2d_hint(sa + kABytes, &tmap_b0, kb * L.b_x_step, L.row_b0 + kb * L.b_y_step,
                             &bars->full[stage], L.wpol);
            tma_load_2d_hint(sa + kABytes + kBHalfBytes, &tmap_b0, kb * L.b_x_step,
                             L.row_b1 + kb * L.b_y_step, &bars->full[stage], L.wpol);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        __syncwarp();  // gidx is rewritten for the next tile only after every lane issued
      }
    }
    if (lane == 0)
      for (int i = 0; i < kStages; ++i)  // own copies land before the CTA exits
        if ((armed >> i) & 1u) mbar_wait_drain(&bars->full[i], (armed_par >> i) & 1u);
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      uint32_t tile_seq = 0;
      TileWalk walk;
      walk.start(Mh, Mc, NB0, NB1, p.ph1_shift);
      for (; walk.valid() && ok; walk.next()) {
        const int nk = p.ph[walk.phase()].K / kBK;
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort_flag, p.status, kid)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        if (!any_small) {
          ok = mma_tile<kIdesc, true>(nk, d_tmem, smem, bars, stage, phase, abort_flag, p.status,
                                      kid);
        } else {
          // the first stage has landed, so the producer's flag for this tile is visible
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, p.status, kid)) break;
          ok = tile_small[tile_seq++ & 7u]
                   ? mma_tile<kIdescSmall, false>(nk, d_tmem, smem, bars, stage, phase,
                                                  abort_flag, p.status, kid)
                   : mma_tile<kIdesc, false>(nk, d_tmem, smem, bars, stage, phase, abort_flag,
                                             p.status, kid);
        }
        if (!ok) break;
        umma_commit(&bars->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(&bars->drain);  // every MMA of this thread has finished
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // -------------------------------------------------- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    TileWalk walk;
    walk.start(Mh, Mc, NB0, NB1, p.ph1_shift);
    for (; walk.valid(); walk.next()) {
      const TileInfo ti = walk.info(pre_h, pre_c, p.S);
      const Phase &P = p.ph[ti.ph];
      // tile row held by this thread's TMEM lane (M = 64 tiles: lanes 0..15
      // of each quadrant; kBM, past every segment's end, for the others)
      const int r_in = !(any_small && small_tile(p, seg_off, seg_end, ti.s, ti.m_blk))
                           ? q * 32 + lane
                       : lane < 16 ? q * 16 + lane
                                   : kBM;
      const int row = seg_off[ti.s] + ti.m_blk * kBM + r_in;
      const bool valid = row < seg_end[ti.s];
      // One thread waits for the accumulator; all 128 then act on its verdict,
      // so the named barriers below are always reached by every epilogue warp.
      if (warp == 2 && lane == 0)
        epi_ok[acc] = mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, p.status, kid) ? 1 : 0;
      epilogue_bar();
      if (!epi_ok[acc]) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
      uint16_t *orow = valid ? P.out + (int64_t)row * P.out_ld + (int64_t)ti.n_blk * P.out_nblk_stride
                             : nullptr;
      if (P.mode == 0) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + 128 + c * 32, u);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(silu_mul(g[2 * i], u[2 * i]), silu_mul(g[2 * i + 1], u[2 * i + 1]));
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->tempty[acc]);
      if (p.n_phases > 1 && ti.ph == 0) {
        // publish this tile's h rows to the phase-1 TMA loads of any CTA
        fence_proxy_async_global();
        __threadfence();
        epilogue_bar();
        if (warp == 2 && lane == 0) atomicAdd(p.ready + ti.s, 1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // Every wait on and increment of a readiness counter is behind each CTA
  // that has finished: the last one to finish clears them for the next
  // launch on this workspace (no memset between the permute and this kernel).
  if (threadIdx.x == 0) {
    __threadfence();
    *last_cta = atomicAdd(p.exit_count, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (*last_cta) {
    for (int s = threadIdx.x; s < p.S; s += kThreads) p.ready[s] = 0;
    if (threadIdx.x == 0) *p.exit_count = 0u;
  }
}

// ------------------------------------------------------------------ host
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

// 2-D bf16 row-major [rows, cols] map with a 64-column x box_rows box
// (128 for tiled loads, 1 for tile::gather4).
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
              uint32_t box_rows = 128) {
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

bool ensure_smem_attr() {
  constexpr int kMaxDevices = 64;
  static bool done[kMaxDevices] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return true;
  if (cudaFuncSetAttribute(grouped_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes) != cudaSuccess)
    return false;
  if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return true;
}

// Cooperative launch: every CTA is resident at once, so a phase-1 tile that
// waits for phase-0 tiles of other CTAs can always be satisfied.  With
// programmatic dependent launch, so that the launch and the set-up overlap
// the tail of the kernel before it (the permute).
moe_status launch(const CUtensorMap &a0, const CUtensorMap &b0, const CUtensorMap &a1,
                  const CUtensorMap &b1, const CUtensorMap &a0s, const CUtensorMap &a1s,
                  const FfnParams &p, int64_t max_tiles, cudaStream_t st) {
  int64_t grid = moe_host::sm_count();
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) return MOE_OK;
  return moe_host::launch_coop_pdl(grouped_ffn_kernel, dim3((unsigned)grid), dim3(kThreads),
                                   kSmemBytes, st, a0, b0, a1, b1, a0s, a1s, p);
}

// Pack kernel: W[e][row][k] -> P[e][nb][kb][half][128][64] in 16-byte units.
// Source row of (nb, half, r): gate/up (mode 0) half*I + nb*128 + r; down
// (mode 1) nb*256 + half*128 + r.
__global__ void pack_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t total16,
                            int NB, int nk, int rows_per_expert, int K8, int mode, int I) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t d = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; d < total16; d += stride) {
    int64_t q = d;
    const int c16 = (int)(q % 8);
    q /= 8;
    const int r = (int)(q % 128);
    q /= 128;
    const int half = (int)(q % 2);
    q /= 2;
    const int kb = (int)(q % nk);
    q /= nk;
    const int nb = (int)(q % NB);
    const int64_t e = q / NB;
    const int row = mode == 0 ? half * I + nb * 128 + r : nb * 256 + half * 128 + r;
    dst[d] = __ldg(src + (e * rows_per_expert + row) * K8 + kb * 8 + c16);
  }
}

moe_status check_ffn_args(const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets,
                          const int32_t *seg_expert, int32_t S, int32_t E,
                          const uint16_t *w_gate_up, const uint16_t *w_down, int32_t H, int32_t I,
                          uint16_t *h, uint16_t *y_perm, void *ws, size_t ws_bytes) {
  if (n_rows < 0 || S < 1 || E < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (S > kMaxSegs || H % 256 != 0 || I % 128 != 0 || n_rows >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if ((int64_t)E * 2 * I * (int64_t)H / 64 >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  // tile indices, and a segment's tiles, are split in 32-bit arithmetic
  if (((n_rows + kBM - 1) / kBM + S) * (int64_t)(I / 128 + H / 256) >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!seg_offsets || !seg_expert || !w_gate_up || !w_down) return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, kReadyOff + (size_t)S * sizeof(int32_t)))
    return s;
  if (n_rows == 0) return MOE_OK;
  if (!x_perm || !h || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(x_perm) || !moe_host::aligned16(h) || !moe_host::aligned16(y_perm) ||
      !moe_host::aligned16(w_gate_up) || !moe_host::aligned16(w_down))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// gather_src == nullptr: x_perm holds the n_rows dispatched rows.  Otherwise
// x_perm is the token matrix x [gather_T, H] and dispatched row r is token
// gather_src[r] / gather_k (read with tile::gather4, no permuted copy).
moe_status run_ffn(const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets,
                   const int32_t *seg_expert, int32_t S, int32_t E, const uint16_t *w_gate_up,
                   const uint16_t *w_down, int32_t H, int32_t I, uint16_t *h, uint16_t *y_perm,
                   void *ws, size_t ws_bytes, void *stream, bool packed,
                   const int32_t *gather_src = nullptr, int32_t gather_k = 1,
                   int64_t gather_T = 0, const int32_t *masked_m = nullptr, int32_t cap = 0,
                   int64_t extra_lo = 0, int64_t extra_rows = 0, int32_t extra_expert = 0,
                   const moe_ffn_schedule *sched = nullptr) {
  // an extra segment (a shared expert) is appended after the S listed ones
  const int32_t S_listed = S;
  if (extra_rows > 0) S = S + 1;
  if (moe_status s = check_ffn_args(x_perm, n_rows, masked_m ? masked_m : seg_offsets, seg_expert,
                                    S, E, w_gate_up, w_down, H, I, h, y_perm, ws, ws_bytes))
    return s;
  if (n_rows == 0) return MOE_OK;
  if (!ensure_smem_attr()) return MOE_ERR_CUDA;

  CUtensorMap m_x, m_wgu, m_h, m_wd, m_xs, m_hs;
  const uint64_t gu_rows = packed ? (uint64_t)E * 2 * I * H / kBK : (uint64_t)E * 2 * I;
  const uint64_t gu_cols = packed ? (uint64_t)kBK : (uint64_t)H;
  const uint64_t d_rows = packed ? (uint64_t)E * H * I / kBK : (uint64_t)E * H;
  const uint64_t d_cols = packed ? (uint64_t)kBK : (uint64_t)I;
  const bool ok_x = gather_src ? make_map(&m_x, x_perm, (uint64_t)gather_T, (uint64_t)H, 1)
                               : make_map(&m_x, x_perm, (uint64_t)n_rows, (uint64_t)H);
  if (!ok_x ||
      !make_map(&m_wgu, w_gate_up, gu_rows, gu_cols) ||
      !make_map(&m_h, h, (uint64_t)n_rows, (uint64_t)I) ||
      !make_map(&m_xs, x_perm, gather_src ? (uint64_t)gather_T : (uint64_t)n_rows, (uint64_t)H,
                kBMSmall) ||
      !make_map(&m_hs, h, (uint64_t)n_rows, (uint64_t)I, kBMSmall) ||
      !make_map(&m_wd, w_down, d_rows, d_cols))
    return MOE_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t m_tiles_max = (n_rows + kBM - 1) / kBM + S;  // sum of ceil(count/128)
  int32_t *ready = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kReadyOff);

  // packed weights and rows from a dispatched buffer: SM pairs when the
  // schedule asks for them (measured slower than single-SM tiles on every
  // layer here, so not the default)
  if (packed && gather_src == nullptr && sched != nullptr && sched->cta_pairs) {
    // this kernel leaves its counters set: clear them before and after
    if (cudaMemsetAsync(ready, 0, (size_t)S * sizeof(int32_t), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    moe_pair::PairRun r{};
    r.x_perm = x_perm;
    r.n_rows = n_rows;
    r.seg_offsets = seg_offsets;
    r.masked_m = masked_m;
    r.cap = cap;
    r.seg_expert = seg_expert;
    r.S = S;
    r.n_listed = S_listed;
    r.E = E;
    r.H = H;
    r.I = I;
    r.extra_lo = extra_lo;
    r.extra_hi = extra_lo + extra_rows;
    r.extra_expert = extra_expert;
    r.w_gate_up_packed = w_gate_up;
    r.w_down_packed = w_down;
    r.h = h;
    r.y_perm = y_perm;
    r.ready = ready;
    r.status = moe_host::status_ptr(ws);
    r.interleave = sched ? sched->interleave : 1;
    r.ph1_shift = (sched && sched->ph1_shift >= 0) ? sched->ph1_shift : (H + I / 2) / I;
    r.max_pair_tiles = ((n_rows + 255) / 256 + S) * (int64_t)(I / 128 + H / 256);
    if (moe_status s = moe_pair::run(r, st)) return s;
    return cudaMemsetAsync(ready, 0, (size_t)S * sizeof(int32_t), st) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }

  FfnParams p{};
  p.seg_offsets = seg_offsets;
  p.seg_expert = seg_expert;
  p.S = S;
  p.n_listed = S_listed;
  p.extra_lo = (int32_t)extra_lo;
  p.extra_hi = (int32_t)(extra_lo + extra_rows);
  p.extra_expert = extra_expert;
  p.E = E;
  p.n_rows = (int32_t)n_rows;
  p.b_packed = packed ? 1 : 0;
  p.n_phases = 2;
  p.ready = ready;
  p.status = moe_host::status_ptr(ws);
  p.exit_count = reinterpret_cast<uint32_t *>(ws) + moe::kFfnExitWord;
  // schedule: which CTA runs which tile, never a row's arithmetic
  p.interleave = sched ? sched->interleave : 1;
  // a gate/up tile (depth H) takes about H/I down tiles' time (depth I)
  p.ph1_shift = (sched && sched->ph1_shift >= 0) ? sched->ph1_shift : (H + I / 2) / I;
  p.small_rows = (sched == nullptr || sched->small_tiles) ? kBMSmall : 0;
  p.gather_src = gather_src;
  p.gather_k = gather_k;
  p.gather_T = (int32_t)gather_T;
  p.masked_m = masked_m;
  p.cap = cap;
  Phase &g = p.ph[0];  // gate/up + SwiGLU -> h
  g.K = H;
  g.n_blocks = I / 128;
  g.b_rows_per_expert = 2 * I;
  g.b_nblk_stride = 128;
  g.b_second_off = I;
  g.out = h;
  g.out_ld = I;
  g.out_nblk_stride = 128;
  g.mode = 0;
  Phase &d = p.ph[1];  // down -> y_perm
  d.K = I;
  d.n_blocks = H / 256;
  d.b_rows_per_expert = H;
  d.b_nblk_stride = 256;
  d.b_second_off = 128;
  d.out = y_perm;
  d.out_ld = H;
  d.out_nblk_stride = 256;
  d.mode = 1;
  return launch(m_x, m_wgu, m_h, m_wd, m_xs, m_hs, p, m_tiles_max * (g.n_blocks + d.n_blocks),
                st);
}

}  // namespace

extern "C" moe_status moe_grouped_ffn(const uint16_t *x_perm, int64_t n_rows,
                                      const int32_t *seg_offsets, const int32_t *seg_expert,
                                      int32_t S, int32_t E, const uint16_t *w_gate_up,
                                      const uint16_t *w_down, int32_t H, int32_t I, uint16_t *h,
                                      uint16_t *y_perm, void *ws, size_t ws_bytes, void *stream) {
  return run_ffn(x_perm, n_rows, seg_offsets, seg_expert, S, E, w_gate_up, w_down, H, I, h, y_perm,
                 ws, ws_bytes, stream, false);
}

extern "C" moe_status moe_grouped_ffn_packed(const uint16_t *x_perm, int64_t n_rows,
                                             const int32_t *seg_offsets, const int32_t *seg_expert,
                                             int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                             const uint16_t *w_down_packed, int32_t H, int32_t I,
                                             uint16_t *h, uint16_t *y_perm, void *ws,
                                             size_t ws_bytes, void *stream) {
  return run_ffn(x_perm, n_rows, seg_offsets, seg_expert, S, E, w_gate_up_packed, w_down_packed, H,
                 I, h, y_perm, ws, ws_bytes, stream, true);
}

extern "C" moe_status moe_grouped_ffn_packed_shared(
    const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets, const int32_t *seg_expert,
    int32_t S, int32_t E, const uint16_t *w_gate_up_packed, const uint16_t *w_down_packed, int32_t H,
    int32_t I, int64_t shared_row0, int64_t shared_rows, int32_t shared_expert, uint16_t *h,
    uint16_t *y_perm, void *ws, size_t ws_bytes, void *stream) {
  if (shared_row0 < 0 || shared_rows < 0 || shared_row0 + shared_rows > n_rows)
    return MOE_ERR_INVALID_ARG;
  if (shared_rows > 0 && (shared_expert < 0 || shared_expert >= E)) return MOE_ERR_INVALID_ARG;
  return run_ffn(x_perm, n_rows, seg_offsets, seg_expert, S, E, w_gate_up_packed, w_down_packed, H,
                 I, h, y_perm, ws, ws_bytes, stream, true, nullptr, 1, 0, nullptr, 0, shared_row0,
                 shared_rows, shared_expert);
}

extern "C" moe_status moe_grouped_ffn_packed_scheduled(
    const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets, const int32_t *seg_expert,
    int32_t S, int32_t E, const uint16_t *w_gate_up_packed, const uint16_t *w_down_packed, int32_t H,
    int32_t I, int64_t shared_row0, int64_t shared_rows, int32_t shared_expert,
    const moe_ffn_schedule *schedule, uint16_t *h, uint16_t *y_perm, void *ws, size_t ws_bytes,
    void *stream) {
  if (shared_row0 < 0 || shared_rows < 0 || shared_row0 + shared_rows > n_rows)
    return MOE_ERR_INVALID_ARG;
  if (shared_rows > 0 && (shared_expert < 0 || shared_expert >= E)) return MOE_ERR_INVALID_ARG;
  if (schedule && (schedule->ph1_shift < -1 || (schedule->interleave & ~1) != 0 ||
                   (schedule->small_tiles & ~1) != 0 || (schedule->cta_pairs & ~1) != 0))
    return MOE_ERR_INVALID_ARG;
  return run_ffn(x_perm, n_rows, seg_offsets, seg_expert, S, E, w_gate_up_packed, w_down_packed, H,
                 I, h, y_perm, ws, ws_bytes, stream, true, nullptr, 1, 0, nullptr, 0, shared_row0,
                 shared_rows, shared_expert, schedule);
}

extern "C" moe_status moe_grouped_ffn_gather(const uint16_t *x, int64_t T, int32_t k,
                                             const int32_t *src_assign, int64_t n_rows,
                                             const int32_t *seg_offsets, const int32_t *seg_expert,
                                             int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                             const uint16_t *w_down_packed, int32_t H, int32_t I,
                                             uint16_t *h, uint16_t *y_perm, void *ws,
                                             size_t ws_bytes, void *stream) {
  if (T < 0 || k < 1 || (n_rows > 0 && (!src_assign || T == 0))) return MOE_ERR_INVALID_ARG;
  if (T >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  return run_ffn(x, n_rows, seg_offsets, seg_expert, S, E, w_gate_up_packed, w_down_packed, H, I,
                 h, y_perm, ws, ws_bytes, stream, true, src_assign, k, T);
}

extern "C" moe_status moe_grouped_ffn_masked(const uint16_t *x_perm, int32_t cap,
                                             const int32_t *masked_m, const int32_t *seg_expert,
                                             int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                             const uint16_t *w_down_packed, int32_t H, int32_t I,
                                             uint16_t *h, uint16_t *y_perm, void *ws,
                                             size_t ws_bytes, void *stream) {
  if (cap < 1 || S < 1 || !masked_m) return MOE_ERR_INVALID_ARG;
  const int64_t n_rows = (int64_t)S * cap;
  return run_ffn(x_perm, n_rows, nullptr, seg_expert, S, E, w_gate_up_packed, w_down_packed, H, I,
                 h, y_perm, ws, ws_bytes, stream, true, nullptr, 1, 0, masked_m, cap);
}

extern "C" moe_status moe_pack_expert_weights(const uint16_t *w_gate_up, const uint16_t *w_down,
                                              int32_t E, int32_t H, int32_t I,
                                              uint16_t *w_gate_up_packed, uint16_t *w_down_packed,
                                              void *stream) {
  if (E < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!w_gate_up || !w_down || !w_gate_up_packed || !w_down_packed) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(w_gate_up) || !moe_host::aligned16(w_down) ||
      !moe_host::aligned16(w_gate_up_packed) || !moe_host::aligned16(w_down_packed))
    return MOE_ERR_INVALID_ARG;
  if (w_gate_up == w_gate_up_packed || w_down == w_down_packed) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t grid = (int64_t)moe_host::sm_count() * 8;
  const int64_t gu16 = (int64_t)E * 2 * I * H / 8;
  pack_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(w_gate_up),
                                               reinterpret_cast<uint4 *>(w_gate_up_packed), gu16,
                                               I / 128, H / kBK, 2 * I, H / 8, 0, I);
  if (moe_status s = moe_host::launch_status()) return s;
  const int64_t d16 = (int64_t)E * H * I / 8;
  pack_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(w_down),
                                               reinterpret_cast<uint4 *>(w_down_packed), d16,
                                               H / 256, I / kBK, H, I / 8, 1, I);
  return moe_host::launch_status();
}

// ------------------------------------------------------ L2 prefetch of weights
namespace {

// "Mixture-of-Experts Inference", "Memory pressure" (EP size in prefill and
// decode): in a decode step the expert work is dominated by loading the
// expert weights.  Once routing is known, so are the weight tiles the
// grouped FFN's first wave of CTAs streams first.  One warp per first-wave
// tile derives the FFN's segments and tile order from the routed ids (an
// expert's rows land in its first slot, exact for placements without
// replicas) and asks L2 for the first k-blocks of its tile's gate/up
// weights.  The fetches run beside the layout and the permute, while HBM is
// otherwise idle.  They are spread over every SM's TMA unit, and each CTA
// holds a few KiB of shared memory and exits within microseconds, so it
// never keeps the cooperative FFN launch from finding room on an SM.
// Prefetches are hints: no result depends on them.
constexpr int kPrefetchMaxSegs = 256;

struct PrefetchArgs {
  const int32_t *topk_ids;
  int64_t A;
  const int32_t *rep_offsets, *rep_slots, *slot_expert;
  int32_t E, S;
  const uint16_t *w_gu;  // packed [e][n_blk][kb][half][128][64]
  int32_t NB, nk;        // gate/up n-blocks (I/128) and k-blocks (H/64)
  int32_t kblocks;       // k-blocks fetched per first-wave tile (<= 32)
  int32_t interleave;
};

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// grid = the FFN's persistent grid (its first-wave tiles), one warp each;
// dynamic shared memory: 3 * (S + 1) int32.
__global__ void __launch_bounds__(32) prefetch_ffn_weights_kernel(PrefetchArgs a) {
  extern __shared__ int32_t pf_smem[];
  int32_t *cnt = pf_smem;               // [S]
  int32_t *pre_h = cnt + (a.S + 1);     // [S+1]
  int32_t *pre_c = pre_h + (a.S + 1);   // [S+1]
  const int lane = threadIdx.x;
  for (int i = lane; i < a.S; i += 32) cnt[i] = 0;
  __syncwarp();
  for (int64_t i = lane; i < a.A; i += 32) {
    const int e = __ldg(a.topk_ids + i);
    if (e < 0 || e >= a.E) continue;
    const int r0 = __ldg(a.rep_offsets + e);
    if (r0 < 0 || r0 >= a.S || r0 >= __ldg(a.rep_offsets + e + 1)) continue;
    const int s = __ldg(a.rep_slots + r0);
    if (s >= 0 && s < a.S) atomicAdd(&cnt[s], 1);
  }
  __syncwarp();
  for (int s = lane; s < a.S; s += 32) {  // as the FFN's prologue
    const int mt = (cnt[s] + kBM - 1) / kBM;
    const bool hot = a.interleave && mt >= 2;
    pre_h[s] = hot ? mt : 0;
    pre_c[s] = hot ? 0 : mt;
  }
  __syncwarp();
  warp_exclusive_scan(pre_h, a.S, lane);
  __syncwarp();
  warp_exclusive_scan(pre_c, a.S, lane);
  __syncwarp();
  const int64_t Mh = pre_h[a.S], Mc = pre_c[a.S];
  const int64_t t = blockIdx.x;  // the FFN's CTA blockIdx.x takes this tile first
  if (t >= (Mh + Mc) * a.NB || lane >= a.kblocks) return;
  int s, nb, mb;
  tile_order::merged(t, pre_h, pre_c, a.S, a.NB, Mh, Mc, s, nb, mb);
  // m-blocks of one (segment, n-block) share their weight tile, and the
  // earlier ones sit earlier in the wave: fetch it once, for m-block 0
  const int e = __ldg(a.slot_expert + s);
  if (mb != 0 || e < 0 || e >= a.E) return;
  prefetch_l2(a.w_gu + (((int64_t)e * a.NB + nb) * a.nk + lane) * 256 * kBK, 256 * kBK * 2);
}

}  // namespace

extern "C" moe_status moe_prefetch_ffn_weights(const int32_t *topk_ids, int64_t T, int32_t k,
                                               const moe_placement *pl,
                                               const uint16_t *w_gate_up_packed, int32_t H,
                                               int32_t I, int64_t max_bytes, void *stream) {
  if (T < 0 || k < 1 || pl == nullptr || H < 1 || I < 1 || max_bytes < 0)
    return MOE_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0 || pl->n_slots < 1 || pl->n_slots > kMaxSegs ||
      pl->n_experts < 1)
    return MOE_ERR_UNSUPPORTED;
  if ((int64_t)pl->n_experts * 2 * I * (int64_t)H / 64 >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!topk_ids || !w_gate_up_packed || !pl->slot_expert || !pl->rep_offsets || !pl->rep_slots)
    return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(w_gate_up_packed)) return MOE_ERR_INVALID_ARG;
  const int64_t tile_bytes = 256 * kBK * 2;  // one k-block of a gate/up weight tile
  // nothing to do: no rows, a budget below one k-block, or more segments
  // than the few KiB of shared memory a prefetching CTA may hold
  if (T == 0 || max_bytes < tile_bytes || pl->n_slots > kPrefetchMaxSegs) return MOE_OK;
  const int wave = moe_host::sm_count();
  if (wave < 1) return MOE_ERR_CUDA;
  PrefetchArgs a{};
  a.topk_ids = topk_ids;
  a.A = T * (int64_t)k;
  a.rep_offsets = pl->rep_offsets;
  a.rep_slots = pl->rep_slots;
  a.slot_expert = pl->slot_expert;
  a.E = pl->n_experts;
  a.S = pl->n_slots;
  a.w_gu = w_gate_up_packed;
  a.NB = I / 128;
  a.nk = H / kBK;
  a.interleave = 1;  // the FFN's default tile order
  int64_t kb = max_bytes / ((int64_t)wave * tile_bytes);
  if (kb > a.nk) kb = a.nk;
  if (kb > 32) kb = 32;  // one k-block per lane
  a.kblocks = (int32_t)kb;
  if (a.kblocks < 1) return MOE_OK;
  const size_t smem = (size_t)3 * (a.S + 1) * sizeof(int32_t);
  prefetch_ffn_weights_kernel<<<wave, 32, smem, static_cast<cudaStream_t>(stream)>>>(a);
  return moe_host::launch_status();
}

// ------------------------------------------------------------ watchdog self-test
namespace {

__device__ int32_t g_never_set = 0;  // no code writes this word

// One thread runs the two kinds of wait the grouped FFN uses, on conditions
// nothing will ever satisfy: an mbarrier phase that expects an arrival
// nobody makes, and a global counter nobody increments.  Each gives up at
// its deadline and records MOE_ERR_DEVICE_TIMEOUT; the kernel then returns.
__global__ void wait_selftest_kernel(int32_t *status, uint64_t limit_ns, int32_t *waited_us) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_barrier_init();
  const uint64_t t0 = moe::global_timer_ns();
  const bool a = mbar_wait(&bar, 0, &abort_flag, status, moe::K_SELFTEST, limit_ns);
  const uint64_t t1 = moe::global_timer_ns();
  abort_flag = 0;  // the second wait must run to its own deadline
  const bool b = wait_counter(&g_never_set, 1, &abort_flag, status, moe::K_SELFTEST, limit_ns);
  const uint64_t t2 = moe::global_timer_ns();
  if (waited_us != nullptr) {
    waited_us[0] = a ? -1 : (int32_t)((t1 - t0) / 1000);
    waited_us[1] = b ? -1 : (int32_t)((t2 - t1) / 1000);
  }
}

}  // namespace

extern "C" moe_status moe_selftest_wait_timeout(void *ws, size_t ws_bytes, int32_t limit_us,
                                                int32_t *waited_us, void *stream) {
  if (limit_us < 1 || (int64_t)limit_us * 1000 > (int64_t)moe::kWaitLimitNs)
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      moe_host::status_ptr(ws), (uint64_t)limit_us * 1000, waited_us);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
