/*
 * moe.h -- C ABI of the single-GPU MoE-layer hot path for GB300 (sm_103a).
 *
 * The six compute calls follow the four runtime steps of an MoE layer as
 * "14. Serving Mixture-of-Experts Models" states them ("Follow one token
 * through an MoE layer"): the router picks expert ids and weights; tokens
 * are packed into contiguous per-expert segments by a histogram and a
 * permutation; a grouped GEMM runs every expert's segment with its own row
 * count; the inverse permutation and a weighted sum combine the outputs.
 * The balancedness statistic is the one of "The slowest expert sets the
 * pace" in the same chapter.  Expert-parallel ranks are simulated: a rank's
 * share of the dispatched rows is a contiguous run of segments in one
 * device buffer.
 *
 * Conventions for every call:
 *  - Pointers named *device* point to GPU global memory of the current
 *    device; pointers named *host* to host memory.  The caller allocates and
 *    owns every buffer; the library allocates nothing and keeps no state
 *    beyond per-device attribute caches.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, rows
 *    contiguous.  All bf16 pointers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous on that stream and never synchronises the host,
 *    except moe_check_device_status.  Route, layout, permute, combine and
 *    balance use programmatic dependent launch: each kernel may start while
 *    its predecessor on the stream drains and waits (griddepcontrol.wait)
 *    before reading anything.
 *  - Errors found on the host (bad sizes, NULL pointers, unsupported shapes)
 *    return a status at once and launch nothing.  Errors found on the
 *    device (an expert id or row index out of range, a bounded wait that
 *    expired) never trap: the kernel records the first one in the status
 *    word at the start of the workspace, skips the bad access, and returns;
 *    moe_check_device_status reports it.
 *  - `ws` is a device workspace of at least moe_workspace_size() bytes,
 *    16-byte aligned, zeroed once by moe_workspace_init before first use.
 *    Calls that share a workspace must be ordered on one stream.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* NULL pointer, negative or inconsistent size */
  MOE_ERR_UNSUPPORTED = 2,    /* shape outside the kernels' limits (see each call) */
  MOE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_INDEX = 4,   /* device: expert id, slot or row index out of range */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* device: a bounded wait expired; outputs are invalid */
  MOE_ERR_WORKSPACE = 6,      /* workspace NULL, misaligned or too small */
  MOE_ERR_PLACEMENT = 7       /* device: placement tables inconsistent */
} moe_status;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };

/* Router configuration.
 *  score_fn     MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID.
 *  k            experts per token, 1 <= k <= 16, k <= E.
 *  n_groups     1 = no group limit; else E % n_groups == 0, n_groups <= 32.
 *  topk_groups  groups kept (1..n_groups); k <= topk_groups * E / n_groups.
 *  group_topn   experts summed into a group's score (1..E/n_groups). */
typedef struct moe_route_cfg {
  int32_t score_fn;
  int32_t k;
  int32_t n_groups;
  int32_t topk_groups;
  int32_t group_topn;
} moe_route_cfg;

/* Expert placement over simulated ranks (all arrays are *device* int32).
 *  slot_expert[S], slot_rank[S]: physical expert slot s hosts expert
 *      slot_expert[s] on rank slot_rank[s]; slots are sorted by (rank,
 *      expert) strictly increasing, so segment s of the dispatched buffer is
 *      slot s and each rank's segments are contiguous.
 *  rep_offsets[E+1], rep_slots[S]: CSR list of each expert's slots, in
 *      ascending rank order; every expert has at least one and every slot
 *      appears once (rep_offsets[E] == S).
 *  token_src_rank[T] or NULL: the rank each token lives on (NULL: t mod R).
 *  ranks_per_node: ranks of one node; node(r) = r / ranks_per_node. */
typedef struct moe_placement {
  int32_t n_experts;
  int32_t n_slots;
  int32_t n_ranks;
  int32_t ranks_per_node;
  const int32_t *slot_expert;
  const int32_t *slot_rank;
  const int32_t *rep_offsets;
  const int32_t *rep_slots;
  const int32_t *token_src_rank;
} moe_placement;

/* Bytes of device workspace needed by moe_dispatch_layout for T tokens,
 * top-k and n_slots slots (a 256-byte status block plus the scan's tile
 * flags); it also covers moe_grouped_ffn with up to n_slots segments.
 * Route, permute, combine and balance need only the status block
 * (MOE_WS_STATUS_BYTES).  Returns 0 for invalid sizes. */
#define MOE_WS_STATUS_BYTES 256
size_t moe_workspace_size(int64_t T, int32_t k, int32_t n_slots);

/* Zero the workspace (device, `ws_bytes` bytes) on `stream`. */
moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, read the status word of `ws`, clear it, and return
 * the first device-side error recorded since the last check (MOE_OK if
 * none).  *info_host (may be NULL) receives a code-specific detail (the
 * offending index, or for MOE_ERR_DEVICE_TIMEOUT the microseconds the
 * expired wait lasted). */
moe_status moe_check_device_status(void *ws, void *stream, int32_t *info_host);

/* L2 prefetch of the grouped FFN's first weight tiles.  "Mixture-of-Experts
 * Inference", "Memory pressure" (EP size in prefill and decode): a decode
 * step's expert work is dominated by loading the expert weights.  One warp
 * per CTA of the FFN's first wave derives, from the routed ids (device
 * int32 [T,k]) and the placement, the segments and tile order of
 * moe_grouped_ffn_packed (an expert's rows land in its first slot, exact
 * without replicas) and asks L2 for the first k-blocks of the gate/up
 * weight tile that CTA takes first: at most max_bytes in all, at most 32
 * k-blocks a tile.  Issued on a second stream right after moe_route, the
 * fetches run while the layout and the permute leave HBM idle; each CTA
 * holds 12*(n_slots+1) bytes of shared memory and exits at once, so the
 * cooperative FFN launch still finds room on every SM.  The fetches are
 * hints: no output depends on them and the call writes nothing.
 * w_gate_up_packed: the packed gate/up weights (moe_pack_expert_weights),
 * 16-byte aligned.  Limits as moe_grouped_ffn_packed; T == 0, a budget
 * below one 32 KiB k-block, or n_slots > 256 launches nothing. */
moe_status moe_prefetch_ffn_weights(const int32_t *topk_ids, int64_t T, int32_t k,
                                    const moe_placement *pl, const uint16_t *w_gate_up_packed,
                                    int32_t H, int32_t I, int64_t max_bytes, void *stream);

/* Watchdog self-test of the device-side waits.  Launches one thread that
 * runs the grouped FFN's two kinds of bounded wait on conditions nothing
 * will satisfy: an mbarrier phase that expects an arrival nobody makes,
 * and a global counter nobody increments.  Each gives up after limit_us
 * microseconds of %globaltimer and records MOE_ERR_DEVICE_TIMEOUT in the
 * status word of `ws` (the first one is kept; read it with
 * moe_check_device_status).  The kernel then returns normally, so the
 * context stays usable.  waited_us (device, 2 int32, may be NULL) receives
 * how long each wait lasted (-1 if it completed).  Nothing faults, traps
 * or hangs: the production kernels use the same waits with a 2 s limit.
 * 1 <= limit_us <= 2,000,000; ws: at least MOE_WS_STATUS_BYTES. */
moe_status moe_selftest_wait_timeout(void *ws, size_t ws_bytes, int32_t limit_us,
                                     int32_t *waited_us, void *stream);

/* Router: per token, the k experts with the largest scores and their
 * weights.  "14. Serving Mixture-of-Experts Models", "Follow one token
 * through an MoE layer" (the router produces expert ids and weights for
 * every token); "Zepp", Section 2 (a learned router selects the top-k
 * experts); group-limited selection per "Mixture-of-Experts Inference",
 * "MoE architecture recap" (pick a limited number of expert groups, then
 * the top experts within them).
 *  logits   device fp32 [T, E] row-major (finite values).
 *  topk_ids device int32 [T, k]: descending score, ties to the lower id.
 *  topk_w   device fp32 [T, k]: softmax -- exp(l_j - l_max) renormalised
 *           over the selected k; sigmoid -- sigmoid(l_j) / sum over the
 *           selected k.  fp32 with compensated sums: within a few fp32
 *           ulps of the exact value.
 *  Group-limited (n_groups > 1, sigmoid scores only): groups are E /
 *  n_groups contiguous experts; a group's score is the fp64 sum of the fp64
 *  sigmoids of its group_topn largest logits; the topk_groups best groups
 *  (ties: lower group id) are kept and the k experts are chosen among them.
 *  Limits: 1 <= E <= 512, k <= 16, n_groups <= 32, group_topn <= 8.
 *  ws may be NULL (no device errors). */
moe_status moe_route(const float *logits, int64_t T, int32_t E, const moe_route_cfg *cfg,
                     int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                     void *stream);

/* Dispatch layout: map every assignment a = t*k + j to a physical slot and
 * build the stable permutation into contiguous per-slot segments.
 * "14. Serving Mixture-of-Experts Models", "Follow one token", step 1 (a
 * permutation built from a histogram over the expert ids into contiguous
 * per-expert segments) and step 2 (each row goes to the rank that owns the
 * expert); replica choice per "The network topology is visible in every MoE
 * layer" (prefer a copy on the token's own node, else spread).
 *  Slot rule: one copy -> its slot; several -> the lowest-rank copy on the
 *  node of the token's source rank, else copy (t mod n_copies).
 *  Outputs (device int32, caller-allocated):
 *   slot[A]            slot of each assignment;
 *   seg_counts[S]      assignments per slot (histogram);
 *   seg_offsets[S+1]   exclusive prefix sum of seg_counts;
 *   dest_row[A]        row of assignment a in the dispatched buffer:
 *                      seg_offsets[slot[a]] + #{a' < a : slot[a'] == slot[a]};
 *   src_assign[A]      inverse permutation: src_assign[dest_row[a]] == a;
 *   rank_counts[R]     assignments per simulated rank.
 *  Device errors: MOE_ERR_DEVICE_INDEX (expert id outside [0,E)),
 *  MOE_ERR_PLACEMENT (tables inconsistent), MOE_ERR_DEVICE_TIMEOUT.
 *  Limits: n_slots <= 1024, n_ranks <= 1024, n_experts <= 4096, T*k < 2^30.
 *  ws: moe_workspace_size(T,k,S).  The scan's ticket and flags in ws must be
 *  zero on entry; moe_workspace_init makes them so and every call leaves
 *  them zero again (no per-call memset). */
moe_status moe_dispatch_layout(const int32_t *topk_ids, int64_t T, int32_t k,
                               const moe_placement *placement, int32_t *slot,
                               int32_t *seg_counts, int32_t *seg_offsets,
                               int32_t *dest_row, int32_t *src_assign,
                               int32_t *rank_counts, void *ws, size_t ws_bytes,
                               void *stream);

/* Locality-preferred replica routing under relaxed load bounds: choose,
 * for every assignment, which copy of its expert serves it.  "Zepp",
 * Section 4.1, "Locality-preferred token routing" (Eq. 1: keep each
 * source's expert selections, keep each replica's load within C * q_j of
 * its balanced share q_j, minimise inter-node traffic) and Section 5,
 * "Routing" (greedy water-filling: the source's own GPU first, then its
 * node, then remote nodes, each allocation limited by the replica's
 * remaining capacity while reserving enough demand for the other replicas'
 * lower bounds).  Readings fixed here:
 *  - per expert with several replicas, demand d_i = its assignments whose
 *    token lives on rank i (token_src_rank, or t mod R);
 *  - integer targets q_p = floor(D/n) + (p < D mod n) over the replicas in
 *    ascending rank; bounds q_p -+ floor(C*D/n), lower bound >= 0, with
 *    C = c_num / c_den;
 *  - sources in ascending rank; passes own GPU, own node, remote, each
 *    over replicas in ascending rank; then a completion pass (replicas
 *    below their lower bound first, then any with capacity);
 *  - a source's assignments, in ascending assignment order, fill its
 *    destinations in locality order (own GPU, own node, remote).
 *  The refinement that consolidates a token's remote requests onto fewer
 *  nodes is a separate call on this call's output, moe_route_refine.
 *  slot        device int32 [T*k] (output): the chosen slot per assignment.
 *  inter_node  device int32 scalar (output): assignments whose slot is on a
 *              node other than their token's.
 *  ws: moe_route_replicas_workspace_size(T, k, E, S, R) bytes (it also
 *  covers moe_dispatch_layout_routed and moe_grouped_ffn on the same
 *  workspace).  Limits: (n_slots - n_experts) * n_ranks <= 1024, at most 16
 *  copies of an expert.  Device errors: MOE_ERR_DEVICE_INDEX,
 *  MOE_ERR_PLACEMENT, MOE_ERR_DEVICE_TIMEOUT. */
size_t moe_route_replicas_workspace_size(int64_t T, int32_t k, int32_t n_experts,
                                         int32_t n_slots, int32_t n_ranks);
moe_status moe_route_replicas(const int32_t *topk_ids, int64_t T, int32_t k,
                              const moe_placement *placement, int32_t c_num, int32_t c_den,
                              int32_t *slot, int32_t *inter_node, void *ws, size_t ws_bytes,
                              void *stream);

/* Greedy refinement of a replica routing: consolidate each token's remote
 * expert requests onto fewer nodes within the same load bounds.  "Zepp",
 * Section 5, "Routing" (starting from the water-filling's feasible
 * assignments, a greedy refinement moves a token's remote requests onto
 * fewer nodes while the load bounds still hold) and Section 1 (remaining
 * requests consolidated onto fewer remote nodes); the merged dispatch of
 * Section 4.2 then sends a token once per remote node.  Readings fixed
 * here:
 *  - every source rank keeps its count of assignments per copy, so each
 *    copy's load, the bounds of Eq. 1 and the number of inter-node
 *    assignments are exactly those of the input routing; only which of a
 *    source's requests that went to a remote copy of a replicated expert
 *    takes which remote copy changes (node-local choices and experts with
 *    one copy keep their slot);
 *  - per source rank, tokens in ascending order; a token covers its open
 *    requests node by node: a node it already sends to first, then the
 *    node covering the most open requests, ties to the lower node id; a
 *    request takes the lowest-rank copy on that node whose count for the
 *    source is not used up;
 *  - a source rank keeps the refined choices only if its number of
 *    distinct (token, remote node) pairs does not rise.
 *  slot      device int32 [T*k], in/out: a routing in which every slot hosts
 *            its assignment's expert (for example moe_route_replicas's).
 *  messages  device int32 [2] (output): distinct (token, remote node) pairs
 *            before and after, i.e. the inter-node dispatch messages after
 *            merging.
 *  ws: moe_route_replicas_workspace_size(T, k, E, S, R) bytes (the same
 *  workspace as moe_route_replicas; this call uses its last 4*T*k bytes).
 *  Limits: k <= 32, the placement limits of moe_dispatch_layout.  Device
 *  errors: MOE_ERR_PLACEMENT when a request finds no copy (input slots
 *  that do not host their expert). */
moe_status moe_route_refine(const int32_t *topk_ids, int64_t T, int32_t k,
                            const moe_placement *placement, int32_t *slot, int32_t *messages,
                            void *ws, size_t ws_bytes, void *stream);

/* moe_dispatch_layout with each assignment's slot already chosen (for
 * example by moe_route_replicas) instead of the fixed replica rule; same
 * outputs and passage ("14. Serving Mixture-of-Experts Models", "Follow one
 * token", steps 1-2).  slot_in[a] must host topk_ids[a]'s expert, else
 * MOE_ERR_PLACEMENT is recorded and the assignment is skipped. */
moe_status moe_dispatch_layout_routed(const int32_t *topk_ids, const int32_t *slot_in, int64_t T,
                                      int32_t k, const moe_placement *placement,
                                      int32_t *seg_counts, int32_t *seg_offsets,
                                      int32_t *dest_row, int32_t *src_assign,
                                      int32_t *rank_counts, void *ws, size_t ws_bytes,
                                      void *stream);

/* moe_dispatch_layout without a workspace: for callers that cannot
 * allocate device memory when they run the layout, such as a serving engine
 * that has handed all free HBM to its weight and KV-cache pools, or a plugin
 * hosted by another runtime that gives it no workspace and does not let it
 * call cudaMalloc.  The pages have no counterpart: this is a packaging
 * variant of moe_dispatch_layout with identical inputs, outputs and results.
 *  Scratch: a fixed 1 MiB device array inside the library (one per GPU that
 *  loads it, held until the process exits).  Nothing is allocated per call:
 *  no cudaMalloc, cudaFree or allocating library routine.
 *  Limit: 64 + ceil(T*k / 1024) * n_slots <= 262144 (32-bit words);
 *  larger requests return MOE_ERR_UNSUPPORTED without launching.
 *  The first call on each device looks up the array's device address (with
 *  that device current) and caches it; make that first call before any
 *  stream capture.
 *  Every call clears the part of the array it uses and then reuses it, and
 *  all calls on one GPU share the array: calls that may overlap on the same
 *  GPU (for example on two streams) race.  Order them on one stream.
 *  status: device int32[3] (code, detail, kernel id) for device-side errors,
 *  written like the workspace status word of the other calls.  It may be
 *  NULL, but then a device-side error (an expert id out of range, an
 *  inconsistent placement, an expired look-back wait) is dropped: the call
 *  still returns MOE_OK and the outputs cannot be checked.  Pass a status
 *  array whenever the inputs are not known to be valid. */
moe_status moe_dispatch_layout_noalloc(const int32_t *topk_ids, int64_t T, int32_t k,
                                       const moe_placement *placement, int32_t *slot,
                                       int32_t *seg_counts, int32_t *seg_offsets,
                                       int32_t *dest_row, int32_t *src_assign,
                                       int32_t *rank_counts, int32_t *status, void *stream);

/* Fixed-capacity ("masked") dispatch layout: every slot owns `cap` rows of
 * the dispatched buffer whatever its load, so buffer shapes, kernel grids
 * and addresses are the same every step.  "Mixture-of-Experts Inference",
 * "Communication pressure" (decode pads tokens into fixed-size masked
 * layouts so that one captured CUDA graph can be replayed); "14. Serving
 * Mixture-of-Experts Models", "Capacity, padding, and the drop decision"
 * (a fixed per-expert capacity; assignments beyond it are dropped and
 * their output for the layer is zero).
 *  Slot choice as moe_dispatch_layout.  Slot s owns rows [s*cap, (s+1)*cap);
 *  its assignments in ascending order a take rows s*cap, s*cap + 1, ...;
 *  those after the first `cap` are dropped.
 *  Outputs (device int32, caller-allocated):
 *   slot[A]           slot of each assignment;
 *   seg_counts[S]     assignments per slot (the demand, before dropping);
 *   masked_m[S]       rows used in each slot: min(seg_counts[s], cap);
 *   dest_row[A]       s*cap + rank within the slot, or -1 if dropped;
 *   src_assign[S*cap] assignment held by each row, -1 on unused rows;
 *   rank_counts[R]    rows each rank executes (sum of its slots' masked_m);
 *   n_dropped[1]      assignments dropped.
 *  Limits: those of moe_dispatch_layout, cap >= 1, S*cap < 2^31.
 *  ws: moe_workspace_size(T, k, S), same zero-on-entry rule. */
moe_status moe_dispatch_layout_masked(const int32_t *topk_ids, int64_t T, int32_t k,
                                      const moe_placement *placement, int32_t cap,
                                      int32_t *slot, int32_t *seg_counts, int32_t *masked_m,
                                      int32_t *dest_row, int32_t *src_assign,
                                      int32_t *rank_counts, int32_t *n_dropped, void *ws,
                                      size_t ws_bytes, void *stream);

/* Permute: x_perm[dest_row[t*k + j], :] = x[t, :] for every j (a byte
 * copy).  "14. Serving Mixture-of-Experts Models", "Price one dispatch"
 * (each assignment carries its token's hidden row: 2 * H bytes).
 *  x       device bf16 [T, H];  x_perm device bf16 [T*k, H].
 *  Limits: H % 8 == 0.  Rows whose dest_row is out of range are skipped and
 *  reported as MOE_ERR_DEVICE_INDEX. */
moe_status moe_permute(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                       const int32_t *dest_row, uint16_t *x_perm, void *ws,
                       size_t ws_bytes, void *stream);

/* moe_permute that also copies every token row t to row T*k + t, so that a
 * shared expert can run on those T rows inside the same grouped FFN launch
 * (moe_grouped_ffn_packed_shared).  "Mixture-of-Experts Inference", "MoE
 * architecture recap" (the shared expert processes every token) and
 * "Communication pressure" (shared-expert work is independent of the
 * routed path until the outputs are merged, so it can overlap with it).
 *  x_perm device bf16 [T*k + T, H].  Limits as moe_permute. */
moe_status moe_permute_shared(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                              const int32_t *dest_row, uint16_t *x_perm, void *ws,
                              size_t ws_bytes, void *stream);

/* moe_permute into a buffer of n_rows rows (a fixed-capacity layout:
 * n_rows = S*cap) where dest_row -1 marks a dropped assignment, which moves
 * nothing.  Other out-of-range rows are skipped and reported as
 * MOE_ERR_DEVICE_INDEX.  Rows no assignment lands on are left unwritten. */
moe_status moe_permute_masked(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                              const int32_t *dest_row, int64_t n_rows, uint16_t *x_perm,
                              void *ws, size_t ws_bytes, void *stream);

/* FP8 dispatch, sending side: quantize each token row once and write the
 * codes to its k destination rows.  "Mixture-of-Experts Inference",
 * "Communication pressure" (token activations can be quantized, for example
 * to FP8, before dispatch, to cut the bytes the all-to-all moves).
 *  Format (a reading; the pages name only "FP8"): OCP E4M3 codes; one fp32
 *  scale 2^e per (token, 128 consecutive channels), e the smallest integer
 *  with max|x| <= 448 * 2^e over the block, clamped to [-126, 127], e = 0
 *  for an all-zero block; code = E4M3(x / 2^e), nearest, ties to even.
 *  x        device bf16 [T, H];  dest_row device int32 [T*k] (-1: dropped);
 *  xq       device uint8 [n_rows, H] (codes, row r = dispatched row r);
 *  x_scale  device fp32 [n_rows, H/128].
 *  Limits: H % 128 == 0; x and xq 16-byte aligned. */
moe_status moe_permute_fp8(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                           const int32_t *dest_row, int64_t n_rows, uint8_t *xq, float *x_scale,
                           void *ws, size_t ws_bytes, void *stream);

/* FP8 dispatch, receiving side: x_perm[r, c] = bf16(E4M3 value of
 * xq[r, c] * x_scale[r, c/128]) (the product is exact in fp32; one rounding
 * to bf16, nearest even).  With masked_m (device int32 [n_rows / cap], a
 * fixed-capacity layout) row r is restored only if r mod cap <
 * masked_m[r / cap]; otherwise every row is.  ws may be NULL.
 *  Limits: H % 128 == 0; xq and x_perm 16-byte aligned. */
moe_status moe_dequant_fp8(const uint8_t *xq, const float *x_scale, int64_t n_rows, int32_t H,
                           int32_t cap, const int32_t *masked_m, uint16_t *x_perm, void *ws,
                           size_t ws_bytes, void *stream);

/* Grouped SwiGLU expert FFN over contiguous segments.  "14. Serving
 * Mixture-of-Experts Models", "Follow one token", step 3 (a grouped matrix
 * multiplication: one kernel processes every expert's segment with its own
 * row count); "Mixture-of-Experts Inference", "Optimized kernels for MoE"
 * (grouped GEMM, contiguous layout).  For segment s with expert
 * e = seg_expert[s] and rows [seg_offsets[s], seg_offsets[s+1]):
 *     G = X Wg_e^T,  U = X Wu_e^T            (fp32 accumulation)
 *     h = bf16(silu(G) * U),  silu(g) = g / (1 + e^-g)   (fp32)
 *     y = bf16(h Wd_e^T)                     (fp32 accumulation)
 *  x_perm     device bf16 [n_rows, H]
 *  seg_offsets device int32 [S+1], non-decreasing, seg_offsets[S] <= n_rows
 *  seg_expert device int32 [S], values in [0, E)
 *  w_gate_up  device bf16 [E, 2I, H]: rows 0..I-1 gate, I..2I-1 up (K-major)
 *  w_down     device bf16 [E, H, I] (K-major)
 *  h          device bf16 [n_rows, I] (intermediate, written)
 *  y_perm     device bf16 [n_rows, H]
 *  Rows outside every segment are left unwritten.  Uses tcgen05 tensor
 *  cores with TMA-fed shared memory and TMEM accumulators; both GEMMs run
 *  in one cooperative launch, a segment's down-projection tiles starting
 *  as soon as all its gate/up tiles have stored h.
 *  ws: at least 256 + 4*S bytes (moe_workspace_size(T, k, S) is enough).
 *  Its per-segment readiness counters (bytes [256, 256 + 4*S)) and the
 *  finished-CTA counter (status-block word 16) must be zero on entry:
 *  moe_workspace_init makes them so, and the last CTA of every launch
 *  clears them again (no per-call memset).  The launch uses programmatic
 *  dependent launch: it may begin while the previous kernel on the stream
 *  drains, and reads nothing before that kernel has finished.
 *  Limits: H % 256 == 0, I % 128 == 0, S <= 1024, n_rows < 2^31,
 *  E*2I*H/64 < 2^31, and a tile list of (ceil(n_rows/128) + S) *
 *  (I/128 + H/256) < 2^31 tiles.
 *  Device errors: MOE_ERR_DEVICE_INDEX (expert id), MOE_ERR_DEVICE_TIMEOUT. */
moe_status moe_grouped_ffn(const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets,
                           const int32_t *seg_expert, int32_t S, int32_t E,
                           const uint16_t *w_gate_up, const uint16_t *w_down, int32_t H,
                           int32_t I, uint16_t *h, uint16_t *y_perm, void *ws,
                           size_t ws_bytes, void *stream);

/* moe_grouped_ffn_packed on a fixed-capacity layout: segment s is rows
 * [s*cap, s*cap + masked_m[s]) of x_perm [S*cap, H], with expert
 * seg_expert[s]; h is [S*cap, I] and y_perm [S*cap, H].  Only the rows in
 * use are computed and stored, so padding costs memory but no tensor-core
 * time.  The launch's shape depends on S and cap only, so it can be
 * captured once in a CUDA graph and replayed for any routing.
 *  masked_m device int32 [S] (moe_dispatch_layout_masked); a value outside
 *  [0, cap] is clamped and reported as MOE_ERR_DEVICE_INDEX.
 *  Limits as moe_grouped_ffn, and S*cap < 2^31. */
moe_status moe_grouped_ffn_masked(const uint16_t *x_perm, int32_t cap, const int32_t *masked_m,
                                  const int32_t *seg_expert, int32_t S, int32_t E,
                                  const uint16_t *w_gate_up_packed, const uint16_t *w_down_packed,
                                  int32_t H, int32_t I, uint16_t *h, uint16_t *y_perm, void *ws,
                                  size_t ws_bytes, void *stream);

/* Expert weights rearranged for streaming: each 128-row x 64-column block
 * that the grouped GEMM loads per pipeline stage becomes one contiguous
 * 16 KiB run, so the weight stream is sequential in HBM.  Expert execution
 * with few tokens per expert is dominated by loading the expert weights
 * ("Mixture-of-Experts Inference", "Memory pressure"); the layout itself is
 * this library's own.  Done once per set of weights.
 *  Packed gate/up, index (e, nb, kb, half, r, c) with nb < I/128, kb < H/64,
 *  half < 2, r < 128, c < 64, holds w_gate_up[e][half*I + nb*128 + r][kb*64 + c].
 *  Packed down, (e, nb, kb, half, r, c) with nb < H/256, kb < I/64 holds
 *  w_down[e][nb*256 + half*128 + r][kb*64 + c].
 *  Outputs have the sizes of the inputs and must not alias them.
 *  Limits: H % 256 == 0, I % 128 == 0. */
moe_status moe_pack_expert_weights(const uint16_t *w_gate_up, const uint16_t *w_down, int32_t E,
                                   int32_t H, int32_t I, uint16_t *w_gate_up_packed,
                                   uint16_t *w_down_packed, void *stream);

/* moe_grouped_ffn on weights packed by moe_pack_expert_weights: same
 * arguments, same results bit for bit. */
moe_status moe_grouped_ffn_packed(const uint16_t *x_perm, int64_t n_rows,
                                  const int32_t *seg_offsets, const int32_t *seg_expert,
                                  int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                  const uint16_t *w_down_packed, int32_t H, int32_t I,
                                  uint16_t *h, uint16_t *y_perm, void *ws, size_t ws_bytes,
                                  void *stream);

/* moe_grouped_ffn_packed with one more segment after the S listed ones:
 * rows [shared_row0, shared_row0 + shared_rows) of x_perm with expert
 * shared_expert of the packed weights.  This runs a shared expert in the
 * routed experts' launch, so that its tensor-bound tiles overlap the
 * routed experts' weight streaming instead of following them.  Per row the
 * arithmetic is that of a separate call: the results are bit-identical.
 *  Requires 0 <= shared_row0, shared_row0 + shared_rows <= n_rows,
 *  0 <= shared_expert < E, S + 1 <= 1024; ws: 256 + 4*(S+1) bytes. */
moe_status moe_grouped_ffn_packed_shared(const uint16_t *x_perm, int64_t n_rows,
                                         const int32_t *seg_offsets, const int32_t *seg_expert,
                                         int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                         const uint16_t *w_down_packed, int32_t H, int32_t I,
                                         int64_t shared_row0, int64_t shared_rows,
                                         int32_t shared_expert, uint16_t *h, uint16_t *y_perm,
                                         void *ws, size_t ws_bytes, void *stream);

/* The tile schedule of the grouped FFN.  It decides which CTA runs which
 * tile and in what order, never the arithmetic of a row: every setting gives
 * the same output bits.  The pages fix no schedule; this is the library's own
 * (an ordering of the pages' grouped GEMM over per-expert segments).
 *  ph1_shift    phase-1 (down-projection) positions first given to the CTAs
 *               that took one gate/up tile fewer, per such CTA; -1 for the
 *               default round(H / I), 0 for plain round-robin.
 *  interleave   1: merge the tiles of segments with several 128-row blocks
 *               and of one-block segments in proportion to their counts (the
 *               default); 0: plain segment order.
 *  small_tiles  single-SM tiles only: 1, a tile whose segment ends within 64
 *               rows of its first row runs as an M = 64 tile (the default);
 *               0, every tile M = 128.
 *  cta_pairs    0: one SM per tile (the default); 1: tiles of 256 rows run on
 *               pairs of SMs (tcgen05 cta_group::2, a cluster of two CTAs;
 *               each SM stages its own rows and half of every weight tile).
 *               Same bits; slower on the layers measured here. */
typedef struct {
  int32_t ph1_shift;
  int32_t interleave;
  int32_t small_tiles;
  int32_t cta_pairs;
} moe_ffn_schedule;

/* moe_grouped_ffn_packed_shared with an explicit tile schedule (NULL: the
 * default one, {-1, 1, 1, 0}).  Same arguments and results otherwise;
 * MOE_ERR_INVALID_ARG for ph1_shift < -1 or flags outside {0, 1}. */
moe_status moe_grouped_ffn_packed_scheduled(
    const uint16_t *x_perm, int64_t n_rows, const int32_t *seg_offsets,
    const int32_t *seg_expert, int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
    const uint16_t *w_down_packed, int32_t H, int32_t I, int64_t shared_row0,
    int64_t shared_rows, int32_t shared_expert, const moe_ffn_schedule *schedule, uint16_t *h,
    uint16_t *y_perm, void *ws, size_t ws_bytes, void *stream);

/* moe_grouped_ffn_packed without the permuted copy: dispatched row r of
 * the gate/up GEMM is read straight from token row src_assign[r] / k of x
 * with TMA tile::gather4 loads (four rows per instruction), so moe_permute
 * and x_perm are not needed.  "Mixture-of-Experts Inference", "Optimized
 * kernels for MoE" (a fused MoE kernel combines token permutation with the
 * expert GEMMs); "Zepp", Section 5, "Transport" (expert GEMMs select their
 * rows through gather indices instead of repacking).  Results are bit-
 * identical to permute + moe_grouped_ffn_packed.
 *  x          device bf16 [T, H]; src_assign device int32 [n_rows] (from
 *             moe_dispatch_layout); other arguments as moe_grouped_ffn_packed. */
moe_status moe_grouped_ffn_gather(const uint16_t *x, int64_t T, int32_t k,
                                  const int32_t *src_assign, int64_t n_rows,
                                  const int32_t *seg_offsets, const int32_t *seg_expert,
                                  int32_t S, int32_t E, const uint16_t *w_gate_up_packed,
                                  const uint16_t *w_down_packed, int32_t H, int32_t I,
                                  uint16_t *h, uint16_t *y_perm, void *ws, size_t ws_bytes,
                                  void *stream);

/* Combine: y[t] = bf16(acc) with acc = shared[t] (or 0) and, for j = 0..k-1
 * in order, acc = fmaf(topk_w[t,j], y_perm[dest_row[t*k+j]], acc) in fp32.
 * "14. Serving Mixture-of-Experts Models", "Follow one token", step 4 (the
 * inverse permutation followed by a weighted sum); shared experts per
 * "Mixture-of-Experts Inference", "MoE architecture recap" (they process
 * every token; weight one here).
 *  y_perm device bf16 [T*k, H]; topk_w device fp32 [T, k];
 *  shared device bf16 [T, H] or NULL; y device bf16 [T, H].
 *  Limits: H % 8 == 0. */
moe_status moe_combine(const uint16_t *y_perm, const int32_t *dest_row, const float *topk_w,
                       int64_t T, int32_t k, int32_t H, const uint16_t *shared, uint16_t *y,
                       void *ws, size_t ws_bytes, void *stream);

/* moe_combine on a buffer of n_rows rows (a fixed-capacity layout: n_rows =
 * S*cap) where dest_row -1 marks a dropped assignment: its term is skipped,
 * so it adds nothing ("14. Serving Mixture-of-Experts Models", "Capacity,
 * padding, and the drop decision": a dropped token's output is zero). */
moe_status moe_combine_masked(const uint16_t *y_perm, int64_t n_rows, const int32_t *dest_row,
                              const float *topk_w, int64_t T, int32_t k, int32_t H,
                              const uint16_t *shared, uint16_t *y, void *ws, size_t ws_bytes,
                              void *stream);

/* Combine with node-local pre-reduction, the combine side of "Zepp"'s
 * merge (Section 4.2, "Merge": the weighted expert outputs of one token on
 * one node are accumulated there and only that partial sum returns;
 * Algorithm 1's PreReduce and Reduce), simulated on one GPU.  Per token and
 * element: for each destination node n of its k assignments, in ascending
 * node order, part_n = bf16(fmaf chain over that node's assignments in j
 * order, from 0) -- the bf16 payload that would cross the network; then
 * acc = shared[t] (or 0), acc += part_n in node order, y = bf16(acc).
 * Also counts the step's inter-node dispatch messages (Section 3.2,
 * "Redundant Tokens"): messages[0] = assignments whose copy is on another
 * node than their token, messages[1] = distinct (token, remote node) pairs,
 * i.e. the transfers left after merge.
 *  slot     device int32 [T*k]: each assignment's slot (moe_dispatch_layout).
 *  messages device int32 [2] (output, cleared by the call).
 *  Other arguments as moe_combine.  Limits: H % 8 == 0, k <= 16. */
moe_status moe_combine_merged(const uint16_t *y_perm, const int32_t *dest_row, const float *topk_w,
                              const int32_t *slot, const moe_placement *placement, int64_t T,
                              int32_t k, int32_t H, const uint16_t *shared, uint16_t *y,
                              int32_t *messages, void *ws, size_t ws_bytes, void *stream);

/* Balancedness of one step: mean per-rank load over the busiest rank's
 * load, total / (R * max) in fp64; 1.0 when total is 0.  "14. Serving
 * Mixture-of-Experts Models", "The slowest expert sets the pace" (loads
 * count assignments, "Price one dispatch").
 *  rank_counts device int32 [R]; outputs are device scalars.
 *  ws may be NULL. */
moe_status moe_balance_stats(const int32_t *rank_counts, int32_t R, double *balancedness,
                             int32_t *max_count, int64_t *total, void *ws, size_t ws_bytes,
                             void *stream);

/* Balancedness of a step over L MoE layers.  "14. Serving Mixture-of-Experts
 * Models", "The slowest expert sets the pace": avg_tokens / max_tokens,
 * "summed across layers".  Reading: both are summed over the layers -- the
 * sum of each layer's mean per-rank load over the sum of each layer's
 * busiest-rank load, computed as total / (R * max_sum) in fp64; 1.0 when
 * total is 0.  With L = 1 this is moe_balance_stats.
 *  rank_counts device int32 [L][R] (row l: one layer's rank_counts).
 *  balancedness device double, max_sum device int64 (sum over layers of the
 *  busiest rank's load), total device int64 (all assignments).
 *  Limits: L >= 1, R >= 1. */
moe_status moe_balance_stats_layers(const int32_t *rank_counts, int32_t L, int32_t R,
                                    double *balancedness, int64_t *max_sum, int64_t *total,
                                    void *stream);

/* Static text for a status code. */
const char *moe_status_string(moe_status status);

/* Library version string. */
const char *moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
