// Internal interface between the grouped FFN entry points (grouped_ffn.cu)
// and the SM-pair kernel (grouped_ffn_pair.cu).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe_pair {

// One grouped FFN launch on packed weights (moe_pack_expert_weights), with
// the segments of the caller's layout; see grouped_ffn_pair.cu.
struct PairRun {
  const uint16_t *x_perm;
  int64_t n_rows;
  const int32_t *seg_offsets;  // contiguous layout, or
  const int32_t *masked_m;     // fixed capacity: segment s is rows [s*cap, s*cap + masked_m[s])
  int32_t cap;
  const int32_t *seg_expert;
  int32_t S, n_listed, E, H, I;
  int64_t extra_lo, extra_hi;  // an appended segment (a shared expert), if S > n_listed
  int32_t extra_expert;
  const uint16_t *w_gate_up_packed, *w_down_packed;
  uint16_t *h, *y_perm;
  int32_t *ready;   // [S] zeroed readiness counters
  int32_t *status;  // workspace status word
  int32_t interleave, ph1_shift;
  int64_t max_pair_tiles;  // upper bound on the tiles of both phases
};

moe_status run(const PairRun &r, cudaStream_t st);

}  // namespace moe_pair
