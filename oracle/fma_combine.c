/* CPU oracle, TEST INFRASTRUCTURE ONLY: the combine step with its fp32
 * rounding order written out.
 *
 * "14. Serving Mixture-of-Experts Models", "Follow one token through an MoE
 * layer", step 4: the expert outputs return through the inverse permutation
 * and are summed with the router weights.  Per output element:
 *     acc = shared[t] (or 0);  for j = 0..k-1: acc = fmaf(w[t,j], y_j, acc);
 *     out = bf16(acc)  (round to nearest, ties to even)
 * where y_j is row dest_row[t*k+j] of the expert outputs; a term whose
 * dest_row is -1 (an assignment dropped by a fixed-capacity layout, whose
 * output is zero: same chapter, "Capacity, padding, and the drop
 * decision") is skipped.  bf16 values are passed as their 16-bit patterns.
 * Shares no code with the CUDA library. */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* nearest-even rounding of a finite fp32 value to bf16 by integer arithmetic */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

void oracle_combine_fma32(const uint16_t *y_perm, const int32_t *dest_row,
                          const float *topk_w, const uint16_t *shared,
                          int64_t T, int32_t k, int32_t H, uint16_t *out) {
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t h = 0; h < H; ++h) {
      float acc = shared ? bf16_to_f32(shared[t * (int64_t)H + h]) : 0.0f;
      for (int32_t j = 0; j < k; ++j) {
        int64_t row = dest_row[t * k + j];
        if (row < 0) continue; /* dropped by a fixed-capacity layout: adds nothing */
        acc = fmaf(topk_w[t * k + j], bf16_to_f32(y_perm[row * H + h]), acc);
      }
      out[t * (int64_t)H + h] = f32_to_bf16(acc);
    }
  }
}

/* The combine with node-local pre-reduction ("Zepp", Section 4.2, "Merge":
 * the weighted expert outputs of one token on one node are summed there
 * and only that partial sum returns; Algorithm 1's PreReduce and Reduce).
 * Per token and element: for each destination node n in ascending order,
 * part_n = bf16(fmaf chain over its assignments j in ascending order,
 * from 0); then acc = shared[t] (or 0), acc = acc + part_n over the nodes in
 * ascending order, out = bf16(acc).  node[t*k + j] is assignment j's
 * destination node. */
void oracle_combine_merged_fma32(const uint16_t *y_perm, const int32_t *dest_row,
                                 const float *topk_w, const int32_t *node,
                                 const uint16_t *shared, int64_t T, int32_t k, int32_t H,
                                 uint16_t *out) {
  for (int64_t t = 0; t < T; ++t) {
    const int32_t *nd = node + t * k;
    for (int32_t h = 0; h < H; ++h) {
      float acc = shared ? bf16_to_f32(shared[t * (int64_t)H + h]) : 0.0f;
      int32_t prev = -2147483647 - 1;
      for (;;) {
        /* next node id above prev among this token's assignments */
        int32_t n = 2147483647;
        int found = 0;
        for (int32_t j = 0; j < k; ++j)
          if (nd[j] > prev && nd[j] <= n) {
            n = nd[j];
            found = 1;
          }
        if (!found) break;
        float part = 0.0f;
        for (int32_t j = 0; j < k; ++j) {
          if (nd[j] != n) continue;
          int64_t row = dest_row[t * k + j];
          part = fmaf(topk_w[t * k + j], bf16_to_f32(y_perm[row * H + h]), part);
        }
        acc = acc + bf16_to_f32(f32_to_bf16(part));
        prev = n;
      }
      out[t * (int64_t)H + h] = f32_to_bf16(acc);
    }
  }
}
