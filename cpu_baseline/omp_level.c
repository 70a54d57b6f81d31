/*
 * All-core CPU baseline of one tree level: an OpenMP feature-parallel
 * histogram fill, sibling subtraction, then a serial split scan.
 *
 * This is a measured comparison point for the benchmark, not the oracle and
 * not the product: it shares no code with either. Its shape follows the CPU
 * engine the pages describe: bonsai "9. Parallelism & determinism", "In
 * bonsai" (fill_columns: one thread owns a feature and walks the rows in
 * order; the split scan merges per-feature winners in feature order) and
 * bonsai "E6. The wide-data wall", "Two fills" (the feature-parallel fill).
 * The arithmetic is the method's: exact int64 cells of quantised (g, h) pairs
 * ("GBDT engine engineering deep-dive", section 1 loop and gain formula;
 * section 3 subtraction; section 4 missing direction).
 *
 * Build: gcc -O3 -fopenmp -ffp-contract=off -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <omp.h>

typedef struct {
  int32_t feature, bin;
  uint8_t default_left, pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
} level_split;

int omp_threads(void) { return omp_get_max_threads(); }

/* Fill hist [n_nodes][F][B][2] for the level's built nodes. Features are
 * dealt to threads; each thread walks every node's rows in order. */
static void fill(const void *bins, int width, int64_t n_rows, int32_t F, int32_t n_bins, uint32_t missing,
                 const int32_t *q, const int32_t *rows, const int64_t *offs, int32_t n_nodes, int64_t *hist) {
  const int64_t B = (int64_t)n_bins + 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t f = 0; f < F; ++f) {
    const uint8_t *c8 = (const uint8_t *)bins + (int64_t)f * n_rows;
    const uint16_t *c16 = (const uint16_t *)bins + (int64_t)f * n_rows;
    for (int32_t n = 0; n < n_nodes; ++n) {
      int64_t *h = hist + ((int64_t)n * F + f) * B * 2;
      memset(h, 0, (size_t)B * 2 * sizeof(int64_t));
      for (int64_t k = offs[n]; k < offs[n + 1]; ++k) {
        const int64_t r = rows ? rows[k] : k;
        const uint32_t b = width == 1 ? c8[r] : c16[r];
        const int64_t s = b == missing ? n_bins : (int64_t)b;
        h[2 * s] += q[2 * r];
        h[2 * s + 1] += q[2 * r + 1];
      }
    }
  }
}

static double gain_of(double gl, double hl, double gr, double hr, double lam, double gamma) {
  const double g = gl + gr, h = hl + hr;
  const double a = gl * gl / (hl + lam);
  const double b = gr * gr / (hr + lam);
  const double c = g * g / (h + lam);
  return 0.5 * (a + b - c) - gamma;
}

/* Serial scan of every node's features: cut t, missing right then left. */
static void scan(const int64_t *hist, int32_t n_nodes, int32_t F, int32_t n_bins, double lam, double gamma,
                 double mcw, double inv_sg, double inv_sh, level_split *out) {
  const int64_t B = (int64_t)n_bins + 1;
  for (int32_t n = 0; n < n_nodes; ++n) {
    level_split best;
    memset(&best, 0, sizeof best);
    best.feature = -1;
    best.bin = -1;
    best.gain = -INFINITY;
    for (int32_t f = 0; f < F; ++f) {
      const int64_t *h = hist + ((int64_t)n * F + f) * B * 2;
      int64_t G = 0, H = 0;
      for (int64_t s = 0; s < B; ++s) {
        G += h[2 * s];
        H += h[2 * s + 1];
      }
      const int64_t mg = h[2 * n_bins], mh = h[2 * n_bins + 1];
      int64_t pg = 0, ph = 0;
      for (int32_t t = 0; t < n_bins; ++t) {
        pg += h[2 * t];
        ph += h[2 * t + 1];
        for (int d = 0; d < 2; ++d) {
          const int64_t gl = pg + (d ? mg : 0), hl = ph + (d ? mh : 0);
          const int64_t gr = G - gl, hr = H - hl;
          if (hl <= 0 || hr <= 0) continue;
          const double hld = (double)hl * inv_sh, hrd = (double)hr * inv_sh;
          if (hld < mcw || hrd < mcw) continue;
          const double v = gain_of((double)gl * inv_sg, hld, (double)gr * inv_sg, hrd, lam, gamma);
          if (v > best.gain) {
            best.feature = f;
            best.bin = t;
            best.default_left = (uint8_t)d;
            best.gain = v;
            best.g_left = gl;
            best.h_left = hl;
            best.g_right = gr;
            best.h_right = hr;
          }
        }
      }
    }
    out[n] = best;
  }
}

/* One level: fill the built nodes, derive large[p] = parent[p] - small[p]
 * when parent is given (n_nodes pairs), then scan small (and large). */
int omp_level(const void *bins, int width, int64_t n_rows, int32_t F, int32_t n_bins, uint32_t missing,
              const int32_t *q, const int32_t *rows, const int64_t *offs, int32_t n_nodes, const int64_t *parent,
              int64_t *small, int64_t *large, double lam, double gamma, double mcw, double inv_sg, double inv_sh,
              level_split *small_out, level_split *large_out) {
  if ((width != 1 && width != 2) || n_nodes < 0 || F < 1 || n_bins < 1) return 1;
  fill(bins, width, n_rows, F, n_bins, missing, q, rows, offs, n_nodes, small);
  if (parent) {
    const int64_t cells = (int64_t)n_nodes * F * ((int64_t)n_bins + 1) * 2;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cells; ++i) large[i] = parent[i] - small[i];
  }
  scan(small, n_nodes, F, n_bins, lam, gamma, mcw, inv_sg, inv_sh, small_out);
  if (parent) scan(large, n_nodes, F, n_bins, lam, gamma, mcw, inv_sg, inv_sh, large_out);
  return 0;
}
