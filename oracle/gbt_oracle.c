/*
 * Serial CPU oracle for the level-batched (gradient, hessian) histogram path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or helper with the CUDA library;
 * it is the plain definition of what the library computes, written out in the
 * most obvious serial order so that a reader can check it against the pages.
 *
 * Compile with -O2 -ffp-contract=off (no fused multiply-add anywhere) so that
 * every double operation below is one IEEE round-to-nearest operation.
 *
 * Sources (page title, section):
 *  [P1] bonsai "10: CUDA histogram backend" - "The kernel", "The device context
 *       lifecycle" (feature-major binned matrix, u8/u16 widths, packed (g,h),
 *       level batching of the smaller siblings, subtraction for the larger).
 *  [P2] bonsai "9. Parallelism & determinism" - "The idea" (GPU cells are int64
 *       fixed point, one integer in any order); "In bonsai" (split scan merges
 *       per-feature winners in feature order so ties break like a serial scan).
 *  [P4] "GBDT engine engineering deep-dive" (ybb.press) - section 1 (split gain
 *       formula; histogram algorithm enumerates cuts on bin boundaries; the
 *       per-row loop adding (g,h) into each entry's bin), section 3 (histogram
 *       subtraction hist(right) = hist(parent) - hist(left)), section 4
 *       (missing values: try all-missing-left and all-missing-right, keep the
 *       larger gain, store the direction), section 7 (fixed-point quantised
 *       gradients packed for integer atomics).
 *  [P5] hessboost PR #163 "sweep vector-leaf histograms by feature on sparse
 *       indexes" - "Change" (the width's missing sentinel is skipped from the
 *       real bins; here it is routed to its own slot).
 *  [P1] also: "The device context lifecycle" names find_level_split, the
 *       oblivious grower's scan of the frontier histograms; [P4] section 5
 *       defines the oblivious (symmetric) tree: every node of a level uses the
 *       same feature and the same threshold.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *  R1 cells are int64 fixed point: q = round-half-even(x * s) of the float32
 *     product, an error unless |x * s| < 2^31 (so q fits the 32 bits per
 *     component that the pages' packed atomics give each of g and h), cell =
 *     exact int64 sum (no overflow: fewer than 2^31 rows of |q| < 2^31).
 *  R2 slot(b) = b for a real bin b < n_bins, slot(sentinel) = n_bins (the
 *     missing slot); any other value is an error.
 *  R3 a cut t in [0, n_bins-1] sends slots <= t left; missing goes wholly left
 *     or wholly right; the candidate order is (feature asc, t asc, missing
 *     right before missing left) and the first strictly larger gain wins.
 *  R4 a candidate is valid iff both sides have quantised hessian > 0 and both
 *     converted hessians are >= min_child_weight.
 *  R5 fixed-point values are converted as (double)x * inv_s, inv_s = 1/(double)s.
 *  R6 gain = 0.5 * (GL^2/(HL+l) + GR^2/(HR+l) - G^2/(H+l)) - gamma, evaluated
 *     left to right. G, H stand for GL+GR, HL+HR of the formula, i.e. the
 *     feature's own total over all its slots (missing included); for any
 *     histogram built from rows every feature's total is the node's total.
 *  R7 after subtraction a negative hessian cell cannot arise from consistent
 *     inputs; the oracle reports it instead of clamping.
 *  R9 the float-cell mode [P1 "The kernel": float shared cells merged into
 *     double global cells; P4 s7 listing; P4 s3: clamp the hessian at zero
 *     after subtraction]: cells are double sums of the unquantised float32
 *     g and h, added per bin in the given row order (one chain per bin);
 *     subtraction clamps a negative H cell to 0 (G is left as is); the split
 *     find uses R3/R4/R6 on these double cells with inv_s = 1 (values are
 *     not scaled), prefixes summed left to right.
 *  R8 the level split of an oblivious tree: candidate (f, t, direction) scores
 *     the sum over the level's nodes, ascending, of each node's R6 gain at that
 *     candidate (node totals of feature f); a node for which the candidate is
 *     not valid (R4) adds nothing; the candidate is valid iff it is valid for
 *     at least one node; the sum starts from 0.0 and adds in node order; the
 *     order and tie-break are R3's. The reported sums are the candidate's
 *     left/right totals over all nodes.
 *  R10 multi-output (vector-leaf) histograms [P5 "Summary", "Change": each
 *     row carries k gradient pairs, one per target, and a bin read serves all
 *     of them]: target t's histogram is R1-R2's histogram of the t-th pairs;
 *     each target's pairs are quantised with that target's own scales. The
 *     pages build vector-leaf cells as f64 chains; here, as for one target,
 *     the cells are exact int64 sums of the quantised pairs (R1).
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_BIN 2
#define OR_ERR_ROW 3
#define OR_ERR_QUANT 4
#define OR_ERR_INCONSISTENT 5

typedef struct {
  int32_t feature;      /* -1: no valid split */
  int32_t bin;          /* cut t: slots <= t go left */
  uint8_t default_left; /* 1: missing slot goes left */
  uint8_t pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
} oracle_split;

/* [P4 s7], [P2 "The idea"]: quantise one float to fixed point, R1. */
static int quantise_one(float x, float s, int32_t *q) {
  float p = x * s; /* one IEEE float32 multiply, round to nearest even */
  if (!(fabsf(p) < 2147483648.0f)) return OR_ERR_QUANT; /* |p| < 2^31; also catches NaN/inf */
  long long r = llrintf(p); /* current mode: round to nearest, ties to even */
  if (r <= -2147483648LL || r >= 2147483648LL) return OR_ERR_QUANT;
  *q = (int32_t)r;
  return OR_OK;
}

/* Quantise a packed (g, h) float pair array [n][2] into int32 pairs [n][2]. */
int oracle_quantise(const float *gpair, int64_t n, float scale_g, float scale_h, int32_t *q) {
  if (n < 0 || (n > 0 && (!gpair || !q))) return OR_ERR_ARG;
  int st = OR_OK;
  for (int64_t i = 0; i < n; ++i) {
    int32_t a = 0, b = 0;
    int e1 = quantise_one(gpair[2 * i], scale_g, &a);
    int e2 = quantise_one(gpair[2 * i + 1], scale_h, &b);
    if (e1 != OR_OK || e2 != OR_OK) st = OR_ERR_QUANT;
    q[2 * i] = a;
    q[2 * i + 1] = b;
  }
  return st;
}

/* Largest |q| over all rows and both components (used by tests for headroom). */
int64_t oracle_max_abs_q(const int32_t *q, int64_t n) {
  int64_t m = 0;
  for (int64_t i = 0; i < 2 * n; ++i) {
    int64_t v = q[i] < 0 ? -(int64_t)q[i] : (int64_t)q[i];
    if (v > m) m = v;
  }
  return m;
}

/* R2: bin value -> histogram slot, or -1 on a value that is neither. */
static int64_t slot_of(uint32_t b, int32_t n_bins, uint32_t sentinel) {
  if (b == sentinel) return n_bins;
  if (b < (uint32_t)n_bins) return b;
  return -1;
}

/*
 * Histogram build [P4 s1 per-row loop; P1 "The kernel"; P1 "Level batching"].
 * bins: feature-major [n_features][n_rows], 1 or 2 bytes per entry.
 * q: quantised pairs [n_rows][2].
 * rows: level row list [node_offsets[n_nodes]] (row ids), or NULL meaning the
 *       identity (position k is row k).
 * node_offsets: [n_nodes + 1], node i owns rows[node_offsets[i] .. node_offsets[i+1]).
 * hist: out [n_nodes][n_features][n_bins + 1][2] int64 (G, H), overwritten.
 * For each node, rows in the given order, then features: add (qg, qh) into
 * the row's slot of every feature's histogram.
 */
int oracle_build_hist(const void *bins, int bin_bytes, int64_t n_rows, int32_t n_features, int32_t n_bins,
                      uint32_t sentinel, const int32_t *q, const int32_t *rows, const int64_t *node_offsets,
                      int32_t n_nodes, int64_t *hist) {
  if (bin_bytes != 1 && bin_bytes != 2) return OR_ERR_ARG;
  if (n_rows < 0 || n_features < 0 || n_nodes < 0 || n_bins < 1) return OR_ERR_ARG;
  if (!node_offsets || (n_nodes > 0 && !hist)) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  for (int64_t i = 0; i < (int64_t)n_nodes * per_node; ++i) hist[i] = 0;
  const uint8_t *b8 = (const uint8_t *)bins;
  const uint16_t *b16 = (const uint16_t *)bins;
  int st = OR_OK;
  for (int32_t n = 0; n < n_nodes; ++n) {
    int64_t *hn = hist + (int64_t)n * per_node;
    for (int64_t k = node_offsets[n]; k < node_offsets[n + 1]; ++k) {
      int64_t r = rows ? (int64_t)rows[k] : k;
      if (r < 0 || r >= n_rows) { st = OR_ERR_ROW; continue; }
      int64_t qg = q[2 * r], qh = q[2 * r + 1];
      for (int32_t f = 0; f < n_features; ++f) {
        uint32_t b = bin_bytes == 1 ? b8[(int64_t)f * n_rows + r] : b16[(int64_t)f * n_rows + r];
        int64_t s = slot_of(b, n_bins, sentinel);
        if (s < 0) { st = OR_ERR_BIN; continue; }
        hn[((int64_t)f * B + s) * 2 + 0] += qg;
        hn[((int64_t)f * B + s) * 2 + 1] += qh;
      }
    }
  }
  return st;
}

/*
 * Multi-output histograms (R10). q: quantised pairs [n_rows][k][2] (target t
 * of row r at q[(r * k + t) * 2]). hist: out [k][n_nodes][n_features][n_bins
 * + 1][2] int64, target-major, overwritten. For each node, rows in the given
 * order, then features, then targets: add target t's (qg, qh) into the row's
 * slot of feature f in target t's histogram.
 */
int oracle_build_hist_multi(const void *bins, int bin_bytes, int64_t n_rows, int32_t n_features, int32_t n_bins,
                            uint32_t sentinel, const int32_t *q, int32_t k, const int32_t *rows,
                            const int64_t *node_offsets, int32_t n_nodes, int64_t *hist) {
  if (bin_bytes != 1 && bin_bytes != 2) return OR_ERR_ARG;
  if (n_rows < 0 || n_features < 0 || n_nodes < 0 || n_bins < 1 || k < 1) return OR_ERR_ARG;
  if (!node_offsets || (n_nodes > 0 && !hist)) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  const int64_t per_target = (int64_t)n_nodes * per_node;
  for (int64_t i = 0; i < (int64_t)k * per_target; ++i) hist[i] = 0;
  const uint8_t *b8 = (const uint8_t *)bins;
  const uint16_t *b16 = (const uint16_t *)bins;
  int st = OR_OK;
  for (int32_t n = 0; n < n_nodes; ++n) {
    for (int64_t j = node_offsets[n]; j < node_offsets[n + 1]; ++j) {
      int64_t r = rows ? (int64_t)rows[j] : j;
      if (r < 0 || r >= n_rows) { st = OR_ERR_ROW; continue; }
      for (int32_t f = 0; f < n_features; ++f) {
        uint32_t b = bin_bytes == 1 ? b8[(int64_t)f * n_rows + r] : b16[(int64_t)f * n_rows + r];
        int64_t s = slot_of(b, n_bins, sentinel);
        if (s < 0) { st = OR_ERR_BIN; continue; }
        for (int32_t t = 0; t < k; ++t) {
          int64_t *cell = hist + t * per_target + (int64_t)n * per_node + ((int64_t)f * B + s) * 2;
          cell[0] += q[(r * k + t) * 2 + 0];
          cell[1] += q[(r * k + t) * 2 + 1];
        }
      }
    }
  }
  return st;
}

/*
 * Sibling subtraction [P4 s3]: large[p] = parent[parent_of[p]] - small[p], cell by
 * cell, exact in int64. parent_of NULL means parent_of[p] = p. A negative
 * hessian cell in the result is reported (R7), not clamped.
 */
int oracle_subtract(const int64_t *parent, const int32_t *parent_of, const int64_t *small, int64_t *large,
                    int32_t n_pairs, int32_t n_features, int32_t n_slots) {
  if (n_pairs < 0 || n_features < 0 || n_slots < 1) return OR_ERR_ARG;
  const int64_t per_node = (int64_t)n_features * n_slots * 2;
  int st = OR_OK;
  for (int32_t p = 0; p < n_pairs; ++p) {
    int64_t par = parent_of ? parent_of[p] : p;
    for (int64_t c = 0; c < per_node; ++c) {
      int64_t v = parent[par * per_node + c] - small[(int64_t)p * per_node + c];
      large[(int64_t)p * per_node + c] = v;
      if ((c & 1) && v < 0) st = OR_ERR_INCONSISTENT;
    }
  }
  return st;
}

/* R6: the split gain of [P4 s1], every operation one IEEE double op. */
double oracle_gain(double gl, double hl, double gr, double hr, double g, double h, double lambda, double gamma) {
  double left = (gl * gl) / (hl + lambda);
  double right = (gr * gr) / (hr + lambda);
  double parent = (g * g) / (h + lambda);
  double s = left + right;
  s = s - parent;
  return 0.5 * s - gamma;
}

/*
 * Split find [P4 s1 enumeration on bin boundaries; P4 s4 default direction;
 * P2 "In bonsai" serial tie-break]. hist: [n_nodes][n_features][n_bins + 1][2].
 */
int oracle_find_splits(const int64_t *hist, int32_t n_nodes, int32_t n_features, int32_t n_bins, double lambda,
                       double gamma, double min_child_weight, double inv_sg, double inv_sh, oracle_split *out) {
  if (n_nodes < 0 || n_features < 0 || n_bins < 1 || (n_nodes > 0 && (!hist || !out))) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  for (int32_t n = 0; n < n_nodes; ++n) {
    const int64_t *hn = hist + (int64_t)n * per_node;
    oracle_split best;
    best.feature = -1;
    best.bin = -1;
    best.default_left = 0;
    for (int i = 0; i < 7; ++i) best.pad[i] = 0;
    best.gain = -INFINITY;
    best.g_left = best.h_left = best.g_right = best.h_right = 0;
    for (int32_t f = 0; f < n_features; ++f) {
      const int64_t *hf = hn + (int64_t)f * B * 2;
      /* G = GL + GR and H = HL + HR: this feature's total, missing slot included */
      int64_t G = 0, H = 0;
      for (int64_t s = 0; s < B; ++s) { G += hf[s * 2]; H += hf[s * 2 + 1]; }
      const double Gd = (double)G * inv_sg, Hd = (double)H * inv_sh;
      const int64_t Gm = hf[(int64_t)n_bins * 2], Hm = hf[(int64_t)n_bins * 2 + 1];
      int64_t pg = 0, ph = 0; /* prefix over real slots 0..t */
      for (int32_t t = 0; t < n_bins; ++t) {
        pg += hf[(int64_t)t * 2];
        ph += hf[(int64_t)t * 2 + 1];
        for (int dir = 0; dir < 2; ++dir) { /* 0: missing right, 1: missing left */
          int64_t GL = pg + (dir ? Gm : 0), HL = ph + (dir ? Hm : 0);
          int64_t GR = G - GL, HR = H - HL;
          if (!(HL > 0 && HR > 0)) continue;
          double gld = (double)GL * inv_sg, hld = (double)HL * inv_sh;
          double grd = (double)GR * inv_sg, hrd = (double)HR * inv_sh;
          if (!(hld >= min_child_weight && hrd >= min_child_weight)) continue;
          double gain = oracle_gain(gld, hld, grd, hrd, Gd, Hd, lambda, gamma);
          if (gain > best.gain) {
            best.feature = f;
            best.bin = t;
            best.default_left = (uint8_t)dir;
            best.gain = gain;
            best.g_left = GL;
            best.h_left = HL;
            best.g_right = GR;
            best.h_right = HR;
          }
        }
      }
    }
    out[n] = best;
  }
  return OR_OK;
}

/*
 * Float-cell mode (R9). gpair: float32 [n_rows][2]. hist: out
 * [n_nodes][n_features][n_bins + 1][2] double; abs_out (may be NULL): the same
 * shape, the sums of |g| and |h| per cell (the tolerance scale).
 */
int oracle_build_hist_f64(const void *bins, int bin_bytes, int64_t n_rows, int32_t n_features, int32_t n_bins,
                          uint32_t sentinel, const float *gpair, const int32_t *rows, const int64_t *node_offsets,
                          int32_t n_nodes, double *hist, double *abs_out) {
  if (bin_bytes != 1 && bin_bytes != 2) return OR_ERR_ARG;
  if (n_rows < 0 || n_features < 0 || n_nodes < 0 || n_bins < 1) return OR_ERR_ARG;
  if (!node_offsets || (n_nodes > 0 && !hist)) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  for (int64_t i = 0; i < (int64_t)n_nodes * per_node; ++i) {
    hist[i] = 0.0;
    if (abs_out) abs_out[i] = 0.0;
  }
  const uint8_t *b8 = (const uint8_t *)bins;
  const uint16_t *b16 = (const uint16_t *)bins;
  int st = OR_OK;
  for (int32_t n = 0; n < n_nodes; ++n) {
    double *hn = hist + (int64_t)n * per_node;
    double *an = abs_out ? abs_out + (int64_t)n * per_node : NULL;
    for (int64_t k = node_offsets[n]; k < node_offsets[n + 1]; ++k) {
      int64_t r = rows ? (int64_t)rows[k] : k;
      if (r < 0 || r >= n_rows) { st = OR_ERR_ROW; continue; }
      const double g = (double)gpair[2 * r], h = (double)gpair[2 * r + 1];
      for (int32_t f = 0; f < n_features; ++f) {
        uint32_t b = bin_bytes == 1 ? b8[(int64_t)f * n_rows + r] : b16[(int64_t)f * n_rows + r];
        int64_t s = slot_of(b, n_bins, sentinel);
        if (s < 0) { st = OR_ERR_BIN; continue; }
        hn[((int64_t)f * B + s) * 2 + 0] += g;
        hn[((int64_t)f * B + s) * 2 + 1] += h;
        if (an) {
          an[((int64_t)f * B + s) * 2 + 0] += fabs(g);
          an[((int64_t)f * B + s) * 2 + 1] += fabs(h);
        }
      }
    }
  }
  return st;
}

/* Float-cell subtraction (R9): large = parent - small, a negative H cell clamped to 0. */
int oracle_subtract_f64(const double *parent, const int32_t *parent_of, const double *small, double *large,
                        int32_t n_pairs, int32_t n_features, int32_t n_slots) {
  if (n_pairs < 0 || n_features < 0 || n_slots < 1) return OR_ERR_ARG;
  const int64_t per_node = (int64_t)n_features * n_slots * 2;
  for (int32_t p = 0; p < n_pairs; ++p) {
    const int64_t pp = parent_of ? parent_of[p] : p;
    for (int64_t i = 0; i < per_node; i += 2) {
      large[p * per_node + i] = parent[pp * per_node + i] - small[p * per_node + i];
      const double h = parent[pp * per_node + i + 1] - small[p * per_node + i + 1];
      large[p * per_node + i + 1] = h < 0.0 ? 0.0 : h;
    }
  }
  return OR_OK;
}

typedef struct {
  int32_t feature;
  int32_t bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  double g_left, h_left, g_right, h_right;
} oracle_split_f64;

/* Float-cell split find (R9): R3/R4/R6 on double cells, unscaled. */
int oracle_find_splits_f64(const double *hist, int32_t n_nodes, int32_t n_features, int32_t n_bins, double lambda,
                           double gamma, double min_child_weight, oracle_split_f64 *out) {
  if (n_nodes < 0 || n_features < 0 || n_bins < 1 || (n_nodes > 0 && (!hist || !out))) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  for (int32_t n = 0; n < n_nodes; ++n) {
    const double *hn = hist + (int64_t)n * per_node;
    oracle_split_f64 best;
    best.feature = -1;
    best.bin = -1;
    best.default_left = 0;
    for (int i = 0; i < 7; ++i) best.pad[i] = 0;
    best.gain = -INFINITY;
    best.g_left = best.h_left = best.g_right = best.h_right = 0.0;
    for (int32_t f = 0; f < n_features; ++f) {
      const double *hf = hn + (int64_t)f * B * 2;
      double G = 0.0, H = 0.0;
      for (int64_t s = 0; s < B; ++s) { G += hf[s * 2]; H += hf[s * 2 + 1]; }
      const double Gm = hf[(int64_t)n_bins * 2], Hm = hf[(int64_t)n_bins * 2 + 1];
      double pg = 0.0, ph = 0.0;
      for (int32_t t = 0; t < n_bins; ++t) {
        pg += hf[(int64_t)t * 2];
        ph += hf[(int64_t)t * 2 + 1];
        for (int dir = 0; dir < 2; ++dir) {
          const double GL = pg + (dir ? Gm : 0.0), HL = ph + (dir ? Hm : 0.0);
          const double GR = G - GL, HR = H - HL;
          if (!(HL > 0.0 && HR > 0.0 && HL >= min_child_weight && HR >= min_child_weight)) continue;
          const double gain = oracle_gain(GL, HL, GR, HR, G, H, lambda, gamma);
          if (gain > best.gain) {
            best.feature = f;
            best.bin = t;
            best.default_left = (uint8_t)dir;
            best.gain = gain;
            best.g_left = GL;
            best.h_left = HL;
            best.g_right = GR;
            best.h_right = HR;
          }
        }
      }
    }
    out[n] = best;
  }
  return OR_OK;
}

/*
 * Oblivious level split [P1 "The device context lifecycle": find_level_split;
 * P4 s5: one feature and threshold for every node of a level], reading R8.
 * hist: [n_nodes][n_features][n_bins + 1][2]; out: one record.
 */
int oracle_find_level_split(const int64_t *hist, int32_t n_nodes, int32_t n_features, int32_t n_bins, double lambda,
                            double gamma, double min_child_weight, double inv_sg, double inv_sh, oracle_split *out) {
  if (n_nodes < 0 || n_features < 0 || n_bins < 1 || !out || (n_nodes > 0 && !hist)) return OR_ERR_ARG;
  const int64_t B = (int64_t)n_bins + 1;
  const int64_t per_node = (int64_t)n_features * B * 2;
  oracle_split best;
  best.feature = -1;
  best.bin = -1;
  best.default_left = 0;
  for (int i = 0; i < 7; ++i) best.pad[i] = 0;
  best.gain = -INFINITY;
  best.g_left = best.h_left = best.g_right = best.h_right = 0;
  for (int32_t f = 0; f < n_features; ++f) {
    for (int32_t t = 0; t < n_bins; ++t) {
      for (int dir = 0; dir < 2; ++dir) { /* 0: missing right, 1: missing left */
        double sum = 0.0;
        int any = 0;
        int64_t sgl = 0, shl = 0, sgr = 0, shr = 0;
        for (int32_t n = 0; n < n_nodes; ++n) {
          const int64_t *hf = hist + (int64_t)n * per_node + (int64_t)f * B * 2;
          int64_t G = 0, H = 0, pg = 0, ph = 0;
          for (int64_t s = 0; s < B; ++s) { G += hf[s * 2]; H += hf[s * 2 + 1]; }
          for (int64_t s = 0; s <= t; ++s) { pg += hf[s * 2]; ph += hf[s * 2 + 1]; }
          const int64_t GL = pg + (dir ? hf[(int64_t)n_bins * 2] : 0);
          const int64_t HL = ph + (dir ? hf[(int64_t)n_bins * 2 + 1] : 0);
          const int64_t GR = G - GL, HR = H - HL;
          sgl += GL; shl += HL; sgr += GR; shr += HR;
          if (!(HL > 0 && HR > 0)) continue;
          const double gld = (double)GL * inv_sg, hld = (double)HL * inv_sh;
          const double grd = (double)GR * inv_sg, hrd = (double)HR * inv_sh;
          if (!(hld >= min_child_weight && hrd >= min_child_weight)) continue;
          sum = sum + oracle_gain(gld, hld, grd, hrd, (double)G * inv_sg, (double)H * inv_sh, lambda, gamma);
          any = 1;
        }
        if (any && sum > best.gain) {
          best.feature = f;
          best.bin = t;
          best.default_left = (uint8_t)dir;
          best.gain = sum;
          best.g_left = sgl;
          best.h_left = shl;
          best.g_right = sgr;
          best.h_right = shr;
        }
      }
    }
  }
  *out = best;
  return OR_OK;
}

/*
 * Row partition of one level [P1 "The device context lifecycle": each parent
 * segment is routed into stable left and right child segments]. For parent
 * node i with split (feature f, cut t, default_left d): a row goes left iff
 * slot(bin[f][row]) <= t, or it is missing and d = 1. Children are written in
 * level order: left child of node i is node 2i, right child 2i+1. A node with
 * no valid split (feature < 0) sends every row left and leaves the right
 * child empty. rows NULL means the identity list.
 * out_rows: [node_offsets[n_nodes] - node_offsets[0]]; out_offsets: [2*n_nodes + 1].
 */
int oracle_partition(const void *bins, int bin_bytes, int64_t n_rows, int32_t n_bins, uint32_t sentinel,
                     const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes, const oracle_split *splits,
                     int32_t *out_rows, int64_t *out_offsets) {
  if (bin_bytes != 1 && bin_bytes != 2) return OR_ERR_ARG;
  const uint8_t *b8 = (const uint8_t *)bins;
  const uint16_t *b16 = (const uint16_t *)bins;
  int64_t w = 0;
  int st = OR_OK;
  out_offsets[0] = 0;
  for (int32_t n = 0; n < n_nodes; ++n) {
    const oracle_split *sp = &splits[n];
    for (int side = 0; side < 2; ++side) { /* 0: left pass, 1: right pass */
      for (int64_t k = node_offsets[n]; k < node_offsets[n + 1]; ++k) {
        int64_t r = rows ? (int64_t)rows[k] : k;
        if (r < 0 || r >= n_rows) { st = OR_ERR_ROW; continue; }
        int left;
        if (sp->feature < 0) {
          left = 1;
        } else {
          uint32_t b = bin_bytes == 1 ? b8[(int64_t)sp->feature * n_rows + r]
                                      : b16[(int64_t)sp->feature * n_rows + r];
          int64_t s = slot_of(b, n_bins, sentinel);
          if (s < 0) { st = OR_ERR_BIN; s = n_bins; }
          left = (s == n_bins) ? (sp->default_left != 0) : (s <= sp->bin);
        }
        if (left == (side == 0)) out_rows[w++] = (int32_t)r;
      }
      out_offsets[2 * n + side + 1] = w;
    }
  }
  return st;
}
