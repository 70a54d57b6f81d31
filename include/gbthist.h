/*
 * gbthist: level-batched (gradient, hessian) histogram construction for
 * histogram gradient-boosted trees on one GB300 (sm_103a).
 *
 * C ABI. Plain pointers and sizes; no C++ or framework types cross it. Every
 * call returns a gbt_status; nothing throws or aborts. Work is enqueued
 * asynchronously on the stream given to gbt_create; device-side faults (a bin
 * or row out of range, a quantisation overflow, a bounded wait that ran out,
 * an inconsistent subtraction) set bits in a device error word that
 * gbt_sync() reads and clears. There is no CPU fallback: every step of the
 * path runs in this library's CUDA kernels.
 *
 * Pointer kinds. Arguments documented "host or device" are inspected with
 * cudaPointerGetAttributes: device (or managed) memory is read in place, host
 * memory is copied on the context stream first (pinned host memory keeps that
 * copy asynchronous; pageable host memory makes it synchronous). Pinned host
 * inputs of up to 4 MiB, and pinned host split outputs, are read and written
 * in place by the kernels instead (keep them unchanged, or unread, until
 * gbt_sync, as for a copy). Arguments documented "device" must be device
 * memory.
 *
 * Histogram layout (the one global contiguous bin array of "GBDT engine
 * engineering deep-dive" (ybb.press), section 1): int64
 * hist[node][feature][slot][2] = (G, H), slot in [0, n_bins] where slot n_bins
 * holds the rows whose bin is the missing sentinel. B = n_bins + 1 slots per
 * feature. G and H are exact sums of fixed-point values (bonsai "9.
 * Parallelism & determinism", "The idea": int64 cells give one integer in any
 * order), so results are bit-identical run to run and to the serial oracle.
 */
#ifndef GBTHIST_H
#define GBTHIST_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gbt_ctx gbt_ctx;

typedef enum {
  GBT_OK = 0,
  GBT_ERR_INVALID_ARG = 1,    /* a NULL, negative size, misaligned pointer or wrong pointer kind */
  GBT_ERR_STATE = 2,          /* call out of order (no bins uploaded, no tree begun, sizes mismatch) */
  GBT_ERR_OOM = 3,            /* a device or pinned allocation failed */
  GBT_ERR_CUDA = 4,           /* a CUDA runtime call failed; gbt_last_error has the text */
  GBT_ERR_BIN_RANGE = 5,      /* device: a bin value was neither < n_bins nor the sentinel */
  GBT_ERR_ROW_RANGE = 6,      /* device: a row index was outside [0, n_rows), or offsets not ascending */
  GBT_ERR_QUANT_OVERFLOW = 7, /* device: a quantised value beyond this library's limit |q| <= 2^21-1, or not finite */
  GBT_ERR_UNSUPPORTED = 8,    /* a size beyond this library's limits */
  GBT_ERR_TIMEOUT = 9,        /* device: a bounded wait ran out */
  GBT_ERR_INCONSISTENT = 10   /* device: subtraction produced a negative hessian cell */
} gbt_status;

/* The best split of one node. feature = -1 (and gain = -inf, sums 0) when no
 * candidate is valid. Rows with slot <= bin go left; the missing slot goes
 * left iff default_left = 1. Sums are the fixed-point left/right totals. */
typedef struct {
  int32_t feature;
  int32_t bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
} gbt_split; /* 56 bytes */

/* The best split of one node in the float-cell mode: as gbt_split, with the
 * left/right sums as doubles. */
typedef struct {
  int32_t feature;
  int32_t bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  double g_left, h_left, g_right, h_right;
} gbt_split_f64; /* 56 bytes */

/* lambda: L2 regulariser; gamma: per-split penalty; min_child_weight: minimum
 * converted hessian on each side (0 disables). */
typedef struct {
  double lambda, gamma, min_child_weight;
} gbt_params;

/* Create a context on `device`, enqueuing on `cuda_stream` (a cudaStream_t;
 * NULL = the legacy default stream). The context owns the binned-matrix
 * mirror, the quantised gradients and scratch; the caller owns every input,
 * output and histogram buffer. */
gbt_status gbt_create(int device, void *cuda_stream, gbt_ctx **out);

/* Synchronise the stream and free everything the context owns. NULL is a no-op. */
gbt_status gbt_destroy(gbt_ctx *ctx);

/* Text of the last host-side error on this context ("" if none). The pointer
 * stays valid until the next call on the same context. Not thread-safe. */
const char *gbt_last_error(const gbt_ctx *ctx);

/* Wait for all enqueued work, then read and clear the device error word.
 * Returns the first device error (in the order of the enum) or GBT_OK. */
gbt_status gbt_sync(gbt_ctx *ctx);

/* Upload the binned matrix once per dataset [bonsai "10: CUDA histogram
 * backend", "The kernel": feature-major, uint8 when every feature fits 256
 * bins, uint16 otherwise].
 *   bins: host or device, feature-major [n_features][n_rows], bin_bytes each.
 *   bin_bytes: 1 (then n_bins <= 255) or 2 (then n_bins <= 65535).
 *   n_bins: real bins per feature; the histogram has n_bins + 1 slots.
 *   missing_sentinel: the width's missing value [hessboost PR #163, "Change"]
 *     (0xFF / 0xFFFF usually); must be >= n_bins and fit the width.
 * The library copies the data into its own tiled row-major mirror (64-byte
 * row strips per tile of features), validating every value on the device
 * (GBT_ERR_BIN_RANGE), and keeps a feature-major copy of the validated slots
 * for the row partition (device memory: about 2 x n_rows x n_features x
 * bin_bytes in all). The caller may free `bins` after the call returns
 * (device pointer) or after gbt_sync (host pointer).
 * Limits: n_rows < 2^31, n_features < 2^24. */
gbt_status gbt_upload_bins(gbt_ctx *ctx, const void *bins, int bin_bytes, int64_t n_rows, int32_t n_features,
                           int32_t n_bins, uint32_t missing_sentinel);

/* Begin a tree [bonsai "10: CUDA histogram backend", "The device context
 * lifecycle": begin_tree takes the tree's gradients; "GBDT engine engineering
 * deep-dive", section 7: gradients are quantised to fixed point for integer
 * atomics].
 *   gpair: host or device, packed float32 (g, h) pairs [n_rows][2].
 *   scale_g, scale_h: fixed-point scales; q = round-half-even(float32(x * s)).
 *     The definition admits any q with |x * s| < 2^31 (one 32-bit half of
 *     the page's packed (g, h) word); this library accepts |q| <= 2^21 - 1
 *     per row and reports GBT_ERR_QUANT_OVERFLOW on the device word for
 *     larger (or non-finite) values. That limit is the kernels' own: it lets
 *     them sum any 1024 rows exactly in 32-bit shared-memory partials.
 *     Histogram cells are exact int64 sums.
 * Read only during the call's stream work. The call also brings max|q| back
 * to the host (asynchronously) to size the build's scratch. */
gbt_status gbt_begin_tree(gbt_ctx *ctx, const float *gpair, float scale_g, float scale_h);

/* Suggest power-of-two scales such that `rows_per_partial` rows of the
 * largest |g| (|h|) sum below 2^31 (the width of the kernels' per-chunk
 * partial sums); rows_per_partial <= 0 means 65536, values below 1024 are
 * raised to 1024. A larger scale (up to |q| <= 2^21 - 1) is always correct; it
 * only makes the build split nodes into more row chunks. */
gbt_status gbt_suggest_scales(int64_t rows_per_partial, float max_abs_g, float max_abs_h, float *scale_g,
                              float *scale_h);

/* Build the histograms of a batch of nodes in one pass [bonsai "10: CUDA
 * histogram backend", "Level batching": every smaller sibling of a level in
 * one pass; "GBDT engine engineering deep-dive", section 1: for each row add
 * (g, h) into its bin of every feature].
 *   rows: host or device int32 [node_offsets[n_nodes]] row ids of the batch,
 *     node segments concatenated; rows within a node are unique, any order.
 *     NULL = the identity list (position k is row k).
 *   node_offsets: host or device int64 [n_nodes + 1], ascending, offsets[0] = 0.
 *   hist_out: device, 16-byte aligned, [n_nodes][n_features][B][2] int64,
 *     overwritten.
 * Limits: n_nodes <= 65535; total rows < 2^31. */
gbt_status gbt_build_level(gbt_ctx *ctx, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                           int64_t *hist_out);

/* Sibling subtraction ["GBDT engine engineering deep-dive", section 3:
 * hist(right) = hist(parent) - hist(left)]: large[p] = parent[parent_of[p]] -
 * small[p] cell by cell, exact in int64. A negative hessian cell (impossible
 * for consistent inputs) sets GBT_ERR_INCONSISTENT instead of being clamped.
 *   parent_hist, small_hist, large_hist: device [..][n_features][B][2] int64,
 *     16-byte aligned; large_hist may not alias the others.
 *   parent_of: host or device int32 [n_pairs]; NULL = identity. */
gbt_status gbt_subtract_siblings(gbt_ctx *ctx, const int64_t *parent_hist, const int32_t *parent_of,
                                 const int64_t *small_hist, int64_t *large_hist, int32_t n_pairs);

/* Best split per node ["GBDT engine engineering deep-dive", section 1: gain
 * = 1/2 [GL^2/(HL+lambda) + GR^2/(HR+lambda) - (GL+GR)^2/(HL+HR+lambda)] -
 * gamma, cuts on bin boundaries; section 4: missing goes wholly left or right,
 * the larger gain wins; bonsai "9. Parallelism & determinism", "In bonsai":
 * ties break as a serial scan in feature order].
 * Candidates: cut t in [0, n_bins-1] (slots <= t left) x {missing right,
 * missing left}; valid iff both sides' quantised H > 0 and both converted
 * H >= min_child_weight; values convert as (double)x * (1/(double)scale);
 * the first strictly larger gain in (feature, t, right-before-left) order wins.
 *   hist: device [n_nodes][n_features][B][2] int64.
 *   out: host or device gbt_split [n_nodes] (host: valid after gbt_sync). */
gbt_status gbt_find_splits(gbt_ctx *ctx, const int64_t *hist, int32_t n_nodes, const gbt_params *params,
                           gbt_split *out);

/* Multi-output (vector-leaf) trees [hessboost PR #163 "perf(multi): sweep
 * vector-leaf histograms by feature on sparse indexes", "Summary" and
 * "Change": each row carries one (g, h) per target and a bin read serves all
 * of them]. Quantises the k pairs of every row, target t with its own scales:
 * q = round-half-even(fl32(x * scale)), |q| <= 2^21 - 1 (else
 * GBT_ERR_QUANT_OVERFLOW at gbt_sync), as gbt_begin_tree does for one target.
 *   gpair: host or device float32 [n_rows][n_targets][2], read during the call's
 *   stream work. scales_g, scales_h: host float [n_targets], finite and > 0.
 *   n_targets: 1 .. 16 (else GBT_ERR_UNSUPPORTED). Independent of gbt_begin_tree. */
gbt_status gbt_begin_tree_multi(gbt_ctx *ctx, const float *gpair, int32_t n_targets, const float *scales_g,
                                const float *scales_h);

/* Histograms of every target for the nodes of one level, in one pass over the
 * bins: hist_out[t] is exactly gbt_build_level's histogram of target t's
 * quantised pairs (int64 (G, H) cells, bit-identical in any order).
 *   rows, node_offsets: as gbt_build_level. hist_out: device, 16-byte aligned,
 *   [n_targets][n_nodes][n_features][n_bins + 1][2] int64, target-major, so each
 *   target's block is a histogram that gbt_subtract_siblings and
 *   gbt_find_splits accept. u8 bins only (else GBT_ERR_UNSUPPORTED). */
gbt_status gbt_build_level_multi(gbt_ctx *ctx, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                                 int64_t *hist_out);

/* Float-cell mode [bonsai "10: CUDA histogram backend", "The kernel": float
 * shared-memory cells merged into double global cells; "GBDT engine
 * engineering deep-dive", section 7 listing; section 3: the hessian is
 * clamped at zero after subtraction]. Cells are double sums of the
 * unquantised float32 (g, h); the order of the additions is not fixed, so
 * cells agree with a serial double sum to rounding (the tests use
 * |a - b| <= 1e-5 * (sum of |g| over the cell's rows)), not bit for bit.
 *   gpair: host or device float32 [n_rows][2], read during the call's stream work.
 *   rows, node_offsets: as gbt_build_level. hist_out: device, 16-byte aligned,
 *   [n_nodes][n_features][B][2] double, overwritten. Needs gbt_upload_bins
 *   only (no gbt_begin_tree). Limits: as gbt_build_level; u16 n_bins <= 5119. */
gbt_status gbt_build_level_f64(gbt_ctx *ctx, const float *gpair, const int32_t *rows, const int64_t *node_offsets,
                               int32_t n_nodes, double *hist_out);

/* large[p] = parent[parent_of[p]] - small[p] in double, a negative hessian
 * cell clamped to 0. Histograms: device [..][F][B][2] double, 16-byte aligned. */
gbt_status gbt_subtract_siblings_f64(gbt_ctx *ctx, const double *parent_hist, const int32_t *parent_of,
                                     const double *small_hist, double *large_hist, int32_t n_pairs);

/* gbt_find_splits on double cells: the same candidates, gain formula and
 * tie-break, values used as they are (no scale), a candidate valid iff both
 * sides' H > 0 and >= min_child_weight; every candidate evaluated in double.
 *   hist: device [n_nodes][F][B][2] double. out: host or device gbt_split_f64. */
gbt_status gbt_find_splits_f64(gbt_ctx *ctx, const double *hist, int32_t n_nodes, const gbt_params *params,
                               gbt_split_f64 *out);

/* The split of an oblivious (symmetric) tree level: one feature, cut and
 * missing direction for every node ["GBDT engine engineering deep-dive",
 * section 5: an oblivious tree uses the same feature and threshold across a
 * level; bonsai "10: CUDA histogram backend", "The device context lifecycle":
 * find_level_split]. The pages give no level gain; this library's reading: a
 * candidate (feature, t, direction) scores the sum over the nodes, ascending,
 * of each node's gbt_find_splits gain at that candidate (each node's own
 * feature totals, gamma included per node), a node for which the candidate
 * is not valid adding nothing; it is valid when valid for at least one node;
 * the first strictly larger sum in (feature, t, right-before-left) order wins.
 * The sum is evaluated in double in node order (bit-identical to the oracle).
 *   hist: device [n_nodes][n_features][B][2] int64, 16-byte aligned.
 *   out: host or device, ONE gbt_split: feature, bin, default_left, the level
 *     gain, and the left/right sums over all nodes. feature = -1 (gain -inf)
 *     when no candidate is valid for any node. */
gbt_status gbt_find_level_split(gbt_ctx *ctx, const int64_t *hist, int32_t n_nodes, const gbt_params *params,
                                gbt_split *out);

/* gbt_find_splits without a context and without any allocation. The paper
 * has no counterpart: this exists for callers that may not allocate device
 * memory themselves or through a library, e.g. a host application that hands
 * out all device memory from its own pool, or code that must not let a
 * cudaMalloc synchronise the device in the middle of stream-ordered work.
 * Same candidates, tie-break and result as gbt_find_splits with a context
 * whose tree began with these scales.
 *   hist: device [n_nodes][n_features][n_bins + 1][2] int64, 16-byte aligned.
 *   out: DEVICE gbt_split [n_nodes] (no host staging: that would allocate).
 *   scale_g, scale_h: the scales the histogram was quantised with (> 0, finite).
 *   cuda_stream: a cudaStream_t of the calling thread's current device.
 * Scratch: one fixed 4 MiB + 32 KiB array inside the library, present on
 * every device that loads it until the process exits. Limits per call:
 * n_nodes <= 4096 and n_nodes * ceil(n_features / 8) <= 32768; beyond them
 * the call returns GBT_ERR_UNSUPPORTED before touching the device. The first
 * call on each device looks up that array's device address; the address is
 * looked up again when the calling thread's current context is another one
 * than at the last lookup, e.g. after cudaDeviceReset created the device's
 * primary context anew. Every call uses the same array and clears only its
 * arrival counters: calls whose work overlaps on the GPU (other streams,
 * other threads) race on it, so order them on one stream or synchronise.
 * Errors: GBT_ERR_INVALID_ARG (NULL, bad sizes or scales, host or misaligned
 * buffers), GBT_ERR_UNSUPPORTED (limits), GBT_ERR_CUDA (launch failed). */
gbt_status gbt_find_splits_noalloc(const int64_t *hist, int32_t n_nodes, int32_t n_features, int32_t n_bins,
                                   float scale_g, float scale_h, const gbt_params *params, gbt_split *out,
                                   void *cuda_stream);

/* One level of a depth-wise grower in three kernels: build the histograms of
 * the smaller siblings of every pair (as gbt_build_level), derive the larger
 * siblings from their parents (as gbt_subtract_siblings) and find the best
 * split of both (as gbt_find_splits) [bonsai "10: CUDA histogram backend",
 * "The device context lifecycle": advance_level builds the smaller siblings
 * in one pass and derives the larger by subtraction; "Level batching"].
 * Pair p = the p-th node segment of `rows`/`node_offsets` (its smaller
 * sibling) and parent parent_of[p] (NULL = p).
 *   rows, node_offsets: as gbt_build_level, n_pairs segments.
 *   parent_hist: device [..][F][B][2] int64.
 *   small_hist, large_hist: device [n_pairs][F][B][2] int64, written.
 *   small_out, large_out: host or device gbt_split [n_pairs].
 * Results equal gbt_build_level + gbt_subtract_and_find; the partial sums of
 * the build go straight into the subtraction, with no int64 round trip. */
gbt_status gbt_level_step(gbt_ctx *ctx, const int32_t *rows, const int64_t *node_offsets, int32_t n_pairs,
                          const int64_t *parent_hist, const int32_t *parent_of, int64_t *small_hist,
                          int64_t *large_hist, const gbt_params *params, gbt_split *small_out,
                          gbt_split *large_out);

/* gbt_subtract_siblings and gbt_find_splits for both siblings in one pass
 * over the parent and small histograms: small_out[p] is the split of
 * small_hist[p], large_out[p] of large_hist[p]. Outputs as above. */
gbt_status gbt_subtract_and_find(gbt_ctx *ctx, const int64_t *parent_hist, const int32_t *parent_of,
                                 const int64_t *small_hist, int64_t *large_hist, int32_t n_pairs,
                                 const gbt_params *params, gbt_split *small_out, gbt_split *large_out);

/* Route each node's rows to its children [bonsai "10: CUDA histogram
 * backend", "The device context lifecycle": partition_level routes each parent
 * segment into stable left and right child segments]. Node i's rows go to
 * child 2i (slot(bin[feature][row]) <= bin, or missing with default_left) or
 * 2i+1 (otherwise), keeping their order; a node with feature = -1 sends every
 * row left.
 *   rows: host or device int32 [node_offsets[n_nodes]]; NULL = identity.
 *   node_offsets: host or device int64 [n_nodes + 1], offsets[0] = 0.
 *   splits: host or device gbt_split [n_nodes].
 *   out_rows: device int32 [node_offsets[n_nodes]]; must not alias rows.
 *   out_offsets: device int64 [2 * n_nodes + 1]. */
gbt_status gbt_partition_level(gbt_ctx *ctx, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                               const gbt_split *splits, int32_t *out_rows, int64_t *out_offsets);

/* gbt_partition_level that also lists every pair's smaller child for the
 * next level's build [bonsai "10: CUDA histogram backend", "The device
 * context lifecycle": partition_level, then advance_level builds the smaller
 * siblings in one pass]. Outputs as gbt_partition_level, plus:
 *   small_side: device uint8 [n_nodes]: 0 when child 2i (left) has no more
 *     rows than child 2i + 1, else 1 (the smaller sibling; ties go left).
 *   small_offsets: device int64 [n_nodes + 1]: small_offsets[0] = 0,
 *     small_offsets[i + 1] - small_offsets[i] = rows of node i's smaller child.
 *   small_rows: device int32 [small_offsets[n_nodes]] (at most half the
 *     level's rows): node i's smaller child's rows in their order, node by
 *     node. All three must be device memory (else GBT_ERR_INVALID_ARG). */
gbt_status gbt_partition_level_pairs(gbt_ctx *ctx, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                                     const gbt_split *splits, int32_t *out_rows, int64_t *out_offsets,
                                     int32_t *small_rows, int64_t *small_offsets, uint8_t *small_side);

/* One level of a depth-wise grower in node order [bonsai "10: CUDA histogram
 * backend", "The device context lifecycle": advance_level builds the smaller
 * siblings in one pass, derives the larger by subtraction and flips the
 * buffers so that the children become the next frontier]. Pair p is nodes
 * (2p, 2p + 1) with parent p: its smaller child 2p + small_side[p] is built
 * from segment p of small_rows / small_offsets (as gbt_build_level), the
 * other is parent_hist[p] minus it (as gbt_subtract_siblings), and both
 * splits are found (as gbt_find_splits). Results are written in node order,
 * so that level_hist is the next level's parent_hist and level_splits the
 * next gbt_partition_level_pairs's splits.
 *   small_rows, small_offsets, small_side: as gbt_partition_level_pairs
 *     writes them (host or device; small_side NULL = all 0).
 *   parent_hist: device [n_pairs][F][B][2] int64 (the previous level).
 *   level_hist: device [2 n_pairs][F][B][2] int64, written; must not alias
 *     parent_hist.
 *   level_splits: host or device gbt_split [2 n_pairs], written.
 * Limits: n_pairs <= 32767. */
gbt_status gbt_advance_level(gbt_ctx *ctx, const int32_t *small_rows, const int64_t *small_offsets,
                             const uint8_t *small_side, int32_t n_pairs, const int64_t *parent_hist,
                             int64_t *level_hist, const gbt_params *params, gbt_split *level_splits);

/* Per-kernel device-time accounting for diagnostics. When enabled, every
 * kernel this context launches is bracketed by a pair of CUDA events on the
 * context stream. gbt_profile_read synchronises the stream, adds up the
 * elapsed times of the recorded launches of `kernel` (a kernel name such as
 * "k_hist_u8"; NULL = all kernels), returns them in total_ms / launches and
 * forgets those launches (records of other kernels are kept). */
gbt_status gbt_profile_enable(gbt_ctx *ctx, int on);
gbt_status gbt_profile_read(gbt_ctx *ctx, const char *kernel, double *total_ms, int64_t *launches);

/* B = n_bins + 1 of the uploaded matrix, or -1 before gbt_upload_bins. */
int32_t gbt_slots_per_feature(const gbt_ctx *ctx);

/* Number of CUDA kernels this context has launched (for launch accounting). */
int64_t gbt_kernel_launches(const gbt_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* GBTHIST_H */
