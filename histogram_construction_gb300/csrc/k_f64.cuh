// Float-cell mode: histograms of the unquantised (g, h), merged in double
// [bonsai "10: CUDA histogram backend", "The kernel": float shared-memory
// cells per chunk of at most 32k rows, merged into double global cells;
// "GBDT engine engineering deep-dive", section 7 listing; section 3: the
// hessian is clamped at zero after subtraction].
//
// The histogram pass is the fixed-point kernels' float-cell instantiation
// (k_hist_u8<true>, k_hist_u16<TS, true>): same plan, same shared layouts,
// red.shared.add.f32 instead of the integer reductions, one double image per
// (node, feature group). This file holds the passes after it: the images to
// the [n][F][B][2] double histogram, the clamped subtraction and the split
// find on double cells.
#pragma once

#include "common.cuh"
#include "k_hist.cuh"
#include "k_split.cuh"

namespace gbt {

// Group images ([image][sub-block][slot][sbw][G, H] double; feature fl of an
// item's group is sub-block fl / sbw, column fl % sbw) -> hist_out
// [n][F][B][2] double, summing a node's group images.
__global__ void __launch_bounds__(256) k_finalize_f64(double *__restrict__ partial,
                                                      const int32_t *__restrict__ group_prefix,
                                                      const int32_t *__restrict__ img_first, int64_t r_cap,
                                                      int64_t image_doubles,
                                                      int32_t n_fgroups, int32_t item_feats, int32_t sbw,
                                                      int32_t n_nodes, int32_t n_features, int32_t B,
                                                      double *__restrict__ hist_out, const DevState *st) {
  pdl_wait();
  if (!st->plan_ok) return;
  const int64_t units = (int64_t)n_nodes * n_features * B;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int s = (int)(u % B);  // consecutive threads: consecutive slots of one feature (contiguous writes)
    const int64_t r = u / B;
    const int f = (int)(r % n_features);
    const int n = (int)(r / n_features);
    const int fg = f / item_feats, fl = f - fg * item_feats;
    const int sb = fl / sbw, c = fl - sb * sbw;
    const int64_t cell = (((int64_t)sb * B + s) * sbw + c) * 2;
    double g = 0.0, h = 0.0;
    const int32_t i0 = img_first[n];
    const bool zero = i0 < r_cap;  // reduce-region images are zeroed as they are read
    const int32_t ng = group_prefix[n + 1] - group_prefix[n];
    double *src0 = partial + ((int64_t)i0 * n_fgroups + fg) * image_doubles + cell;
    const int64_t gstride = (int64_t)n_fgroups * image_doubles;
    for (int32_t k = 0; k < ng; ++k) {  // loads first, then the zeroing stores
      const double2 x = __ldcg(reinterpret_cast<const double2 *>(src0 + k * gstride));
      g += x.x;
      h += x.y;
    }
    if (zero)
      for (int32_t k = 0; k < ng; ++k) __stcg(reinterpret_cast<double2 *>(src0 + k * gstride), make_double2(0.0, 0.0));
    double *d = hist_out + (((int64_t)n * n_features + f) * B + s) * 2;
    d[0] = g;
    d[1] = h;
  }
}

// large = parent - small per cell; a negative H cell is clamped to 0.
__global__ void __launch_bounds__(256) k_subtract_f64(const double *__restrict__ parent,
                                                      const int32_t *__restrict__ parent_of,
                                                      const double *__restrict__ small, double *__restrict__ large,
                                                      int32_t n_pairs, int64_t cells_per_node) {
  const int64_t cells = (int64_t)n_pairs * cells_per_node;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < cells; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = u / cells_per_node, w = u - p * cells_per_node;
    const int64_t pp = parent_of ? (int64_t)parent_of[p] : p;
    const double2 a = reinterpret_cast<const double2 *>(parent)[pp * cells_per_node + w];
    const double2 b = reinterpret_cast<const double2 *>(small)[u];
    const double h = __dsub_rn(a.y, b.y);
    reinterpret_cast<double2 *>(large)[u] = make_double2(__dsub_rn(a.x, b.x), h < 0.0 ? 0.0 : h);
  }
}

// ----------------------------------------------------------------------------
// Split find on double cells. On GB300 an FP64 add has about 65 cycles of
// latency and about 1/64 of the FP32 throughput, a division about 560 cycles,
// and a double -> float conversion is as slow as an FP64 add (measured), so
// the scan screens every candidate with integer and FP32 work and touches
// FP64 only for the few features whose candidates can still be the best.
//
// Screen. Per strip (one feature of one node) the cells are put on a common
// fixed-point grid, from their bit patterns: with E the largest biased
// exponent among the strip's g (or h) cells, a cell becomes the int64 number
// of units 2^-k below it in magnitude (truncation), k = 62 - ceil(log2 B) -
// (E - 1022), so that every prefix sums exactly in int64. Each of a
// candidate's sums S (G_L, H_L, G_R, H_R, and the totals) is then known up to
//   |S_float - S_double| <= 2.02 u |S_float| + B 2^-k + 2 B^2 2^-52 2^(E-1022)
// (u = 2^-24: the int64 -> float conversion; the truncation of at most B
// cells; the rounding of the double values that phase 2 uses, with a wide
// margin), and each gain
// term x^2 / (d + lambda) is bounded from the endpoints of these intervals,
// widened by 16u for the float operations that form it; the gain interval is
// widened by 2^-19 (a + b + c + |gamma|) for the final sums. A candidate is
// certainly valid when both sides' H intervals lie above 0 and above
// min_child_weight; only certainly valid candidates lend their lower bound to
// the threshold; certainly invalid ones are dropped. Strips whose exponents
// leave the usable range, and quantities outside [2^-60, 2^60], get infinite
// intervals (evaluated in double).
constexpr float F64_U = 5.9604644775390625e-08f;  // 2^-24
constexpr int F64_TOT_U = 8;                       // strip loads in flight per lane in the totals passes

// Units of 2^-k in x, truncated toward zero, from the bit pattern (integer
// ALU only). Exact for zero; for a normal x with |x| 2^k < 2^61, |result
// 2^-k - x| < 2^-k; subnormals give 0 (below 2^-1022 <= 2^-k for the k used).
__device__ __forceinline__ int64_t dbl_to_fixed(double x, int k) {
  const long long b = __double_as_longlong(x);
  const int e = (int)((b >> 52) & 0x7ff);
  if (e == 0) return 0;
  const long long mant = (b & 0xfffffffffffffLL) | (1LL << 52);
  const int sh = e - 1075 + k;  // x 2^k = mant 2^sh
  long long q = 0;
  if (sh >= 0) q = mant << sh;  // sh <= 8 by the choice of k
  else if (sh > -63) q = mant >> (-sh);
  return b < 0 ? -q : q;
}

// Largest biased exponent of a double (0 for zero and subnormals, 2047 for inf/NaN).
__device__ __forceinline__ int dbl_exp(double x) { return (int)((__double_as_longlong(x) >> 52) & 0x7ff); }

// Both components exactly zero (either sign), from the bit patterns.
__device__ __forceinline__ bool dbl2_zero(double2 v) {
  return ((unsigned long long)(__double_as_longlong(v.x) | __double_as_longlong(v.y)) << 1) == 0ull;
}

struct F64Screen {
  float lam, gam, gam_abs, mcw_hi;  // lambda, gamma, |gamma| in float; min_child_weight rounded up
  int filter;                        // 0: every valid candidate is evaluated in double
};

// Per-strip fixed-point grid of one component.
struct FixGrid {
  int k;       // units of 2^-k
  float p2;    // 2^-k as a float
  float eabs;  // absolute part of the error radius of a sum
};

__device__ __forceinline__ bool make_grid(int E, int B, int L, FixGrid &g) {
  E = max(E, 1023 - 60);                // all cells below 2^-60 (or zero): the grid of 2^-60 cells
  if (E > 1022 + 100) return false;     // cells of 2^100 and more (or inf, NaN): no screen
  g.k = 62 - L - (E - 1022);
  g.p2 = __int_as_float((127 - g.k) << 23);
  const float mx = __int_as_float((E - 1022 + 127) << 23);  // 2^(E-1022) >= every |cell|
  const float fb = (float)B;
  g.eabs = __fadd_ru(__fadd_ru(__fmul_ru(fb, g.p2), __fmul_ru(__fmul_ru(__fmul_ru(fb, fb), mx), 4.440892098500626e-16f)),
                     7.52316384526264e-37f);  // B 2^-k + 2 B^2 2^-52 max + 2^-120
  return true;
}

// float value of an exact fixed-point sum and its error radius
__device__ __forceinline__ void fix_to_f32(int64_t q, const FixGrid &g, float &v, float &e) {
  v = __fmul_rn(i64_to_f32(q), g.p2);
  e = __fmaf_ru(fabsf(v), 2.02f * F64_U, g.eabs);
}

// Bounds [lo_t, hi_t] of x^2 / (d + lambda) for x in [xf - ex, xf + ex], d in
// [df - ed, df + ed]; false when the interval is unusable (denominator not
// certainly positive, or out of range).
__device__ __forceinline__ bool term_bounds(float xf, float ex, float df, float ed, float lam, float &lo_t,
                                            float &hi_t) {
  const float rlo = 8.673617379884035e-19f, rhi = 1.152921504606847e+18f;  // 2^-60, 2^60
  const float ax = fabsf(xf);
  const float gmin = fmaxf(0.f, __fsub_rd(ax, ex)), gmax = __fadd_ru(ax, ex);
  const float dmin = __fsub_rd(__fadd_rd(df, lam), ed), dmax = __fadd_ru(__fadd_ru(df, lam), ed);
  if (!(dmin > rlo && dmax < rhi && gmax < rhi)) return false;
  hi_t = __fmul_ru(__fdividef(__fmul_ru(gmax, gmax), dmin), 1.0f + 16.f * F64_U);
  lo_t = (gmin > rlo) ? __fmul_rd(__fdividef(__fmul_rd(gmin, gmin), dmax), 1.0f - 16.f * F64_U) : 0.f;
  if (!(hi_t < rhi)) return false;
  if (lo_t < rlo) lo_t = 0.f;
  return true;
}

// One candidate from its fixed-point sums. Returns false when it is certainly
// invalid; else up (and, when certainly valid, lo) bound its double gain.
__device__ __forceinline__ bool screen_fix(int64_t GLq, int64_t HLq, int64_t TG, int64_t TH, const FixGrid &gg,
                                          const FixGrid &gh, float c_lo, float c_hi, bool c_ok, const F64Screen &sc,
                                          float &up, float &lo) {
  float GLf, eGL, HLf, eHL, GRf, eGR, HRf, eHR;
  fix_to_f32(GLq, gg, GLf, eGL);
  fix_to_f32(HLq, gh, HLf, eHL);
  fix_to_f32(TG - GLq, gg, GRf, eGR);
  fix_to_f32(TH - HLq, gh, HRf, eHR);
  const float hl_lo = __fsub_rd(HLf, eHL), hl_hi = __fadd_ru(HLf, eHL);
  const float hr_lo = __fsub_rd(HRf, eHR), hr_hi = __fadd_ru(HRf, eHR);
  if (!(hl_hi > 0.f) || !(hr_hi > 0.f)) return false;
  const bool sure = hl_lo > 0.f && hr_lo > 0.f && hl_lo >= sc.mcw_hi && hr_lo >= sc.mcw_hi;
  up = INFINITY;
  lo = -INFINITY;
  if (!sc.filter || !c_ok) return true;
  float a_lo, a_hi, b_lo, b_hi;
  if (!term_bounds(GLf, eGL, HLf, eHL, sc.lam, a_lo, a_hi) || !term_bounds(GRf, eGR, HRf, eHR, sc.lam, b_lo, b_hi))
    return true;
  const float mag = __fadd_ru(__fadd_ru(__fadd_ru(a_hi, b_hi), c_hi), sc.gam_abs);
  const float slack = __fmul_ru(mag, 1.9073486328125e-06f);  // 2^-19
  const float g_hi = __fsub_ru(__fmul_ru(0.5f, __fsub_ru(__fadd_ru(a_hi, b_hi), c_lo)), sc.gam);
  const float g_lo = __fsub_rd(__fmul_rd(0.5f, __fsub_rd(__fadd_rd(a_lo, b_lo), c_hi)), sc.gam);
  if (!(g_hi == g_hi) || !(g_lo == g_lo) || !(mag < 1.152921504606847e+18f)) return true;
  up = __fadd_ru(g_hi, slack);
  if (sure) lo = __fsub_rd(g_lo, slack);
  return true;
}

// Fixed-point prefixes of chunk [c0, c0 + 128): lane-local inclusive
// prefixes and the exclusive prefix of the lane's first slot (carry: the sums
// before the chunk, updated).
__device__ __forceinline__ void scan_chunk_fix(const double2 *strip, int n_bins, int c0, int kg, int kh,
                                               int64_t (&carry)[2], int64_t (&pg)[SCAN_SPL],
                                               int64_t (&ph)[SCAN_SPL], int64_t &eg, int64_t &eh) {
  const int lane = threadIdx.x & 31;
  double2 v[SCAN_SPL];
#pragma unroll
  for (int i = 0; i < SCAN_SPL; ++i) {
    const int s = c0 + SCAN_SPL * lane + i;
    v[i] = s < n_bins ? __ldg(strip + s) : make_double2(0.0, 0.0);
  }
  int64_t ag = 0, ah = 0;
#pragma unroll
  for (int i = 0; i < SCAN_SPL; ++i) {
    ag += dbl_to_fixed(v[i].x, kg);
    ah += dbl_to_fixed(v[i].y, kh);
    pg[i] = ag;
    ph[i] = ah;
  }
  int64_t x = ag, y = ah;
  warp_incl_scan(x, y);
  const int64_t tx = shfl_i64(x, 31), ty = shfl_i64(y, 31);
  eg = x - ag + carry[0];
  eh = y - ah + carry[1];
  carry[0] += tx;
  carry[1] += ty;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// An exact fixed-point sum as a double (one rounding; the scaling by 2^-k is exact).
__device__ __forceinline__ double fix_to_f64(int64_t q, const FixGrid &g) {
  return __dmul_rn(__ll2double_rn((long long)q), __longlong_as_double((long long)(1023 - g.k) << 52));
}

// Validity and gain of one candidate in double; keeps the better of it and best.
__device__ __forceinline__ void f64_consider(double GL, double HL, double GR, double HR, double parent, double mcw,
                                             const SplitParams &sp, int f, int t, int dir, Cand &best) {
  if (!(HL > 0.0 && HR > 0.0 && HL >= mcw && HR >= mcw)) return;
  const double l2 = __ddiv_rn(__dmul_rn(GL, GL), __dadd_rn(HL, sp.lambda));
  const double r2 = __ddiv_rn(__dmul_rn(GR, GR), __dadd_rn(HR, sp.lambda));
  const double gain = __dsub_rn(__dmul_rn(0.5, __dsub_rn(__dadd_rn(l2, r2), parent)), sp.gamma);
  Cand c;
  set_exact(c, gain);
  c.t = t;
  c.dir = dir;
  c.f = f;
  c.gl = __double_as_longlong(GL);
  c.hl = __double_as_longlong(HL);
  c.gr = __double_as_longlong(GR);
  c.hr = __double_as_longlong(HR);
  if (cand_better(c, best)) best = c;
}

constexpr int F64_MAX_CHUNKS = 80;  // 128-slot chunks per strip (n_bins <= 10240, the u16 limit)

// What phase 2 needs of a warp's strip.
struct F64Strip {
  int64_t TG, TH, mq_g, mq_h;
  FixGrid gg, gh;
  float c_lo, c_hi;
  int c_ok, ok, no_missing;
};

// grid (ceil(F / 8), n_nodes), 256 threads. Phase 1: warp w screens feature
// blockIdx.x * 8 + w of node blockIdx.y, keeping its best certain lower bound
// and, per 128-slot chunk, the largest upper bound and the fixed-point sums
// before the chunk. The CTA's threshold is the largest lower bound of its
// warps. Phase 2: every (feature, chunk) whose largest upper bound reaches
// the threshold is a task; the tasks are dealt round-robin to the CTA's warps,
// which rescan the chunk and evaluate in double each candidate whose upper
// bound reaches the threshold. A feature without a usable grid is scanned
// wholly in double by its own warp. The CTA's best goes to
// cand[node][blockIdx.x]; the node's last CTA writes the split. The double
// sums travel as bit patterns in the candidate's 64-bit fields, so the output
// record is a gbt_split whose four sums are doubles.
__global__ void __launch_bounds__(SCAN_THREADS, 2) k_find_f64(const double *__restrict__ hist, int32_t n_features,
                                                              int32_t n_bins, SplitParams sp, double mcw,
                                                              Cand *__restrict__ cand,
                                                              uint32_t *__restrict__ counters,
                                                              SplitOut *__restrict__ out) {
  __shared__ Cand s_best[SCAN_WARPS];
  __shared__ float s_lo[SCAN_WARPS];
  __shared__ F64Strip s_strip[SCAN_WARPS];
  __shared__ float s_cup[SCAN_WARPS][F64_MAX_CHUNKS];
  __shared__ int64_t s_carry[SCAN_WARPS][F64_MAX_CHUNKS][2];
  __shared__ uint32_t s_last;
  pdl_wait();
  const int node = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * SCAN_WARPS + warp;
  const int B = n_bins + 1;
  const int L = 32 - __clz(B - 1);  // ceil(log2 B)
  const int n_chunks = (n_bins + 32 * SCAN_SPL - 1) / (32 * SCAN_SPL);
  F64Screen sc;
  sc.lam = sp.lambda_f;
  sc.gam = sp.gamma_f;
  sc.gam_abs = sp.gamma_abs_f;
  sc.mcw_hi = __double2float_ru(mcw);
  sc.filter = sp.filter;
  const bool active = f < n_features;
  float run_lo = -INFINITY;
  Cand best = no_cand();
  // ---- phase 1
  {
    const double2 *strip = reinterpret_cast<const double2 *>(hist) + ((int64_t)node * n_features + f) * B;
    F64Strip st;
    st.TG = st.TH = st.mq_g = st.mq_h = 0;
    st.c_lo = st.c_hi = 0.f;
    st.c_ok = st.ok = st.no_missing = 0;
    if (active) {
      int Eg = 0, Eh = 0;
      for (int s0 = lane; s0 < B; s0 += 32 * F64_TOT_U) {
        double2 v[F64_TOT_U];
#pragma unroll
        for (int u = 0; u < F64_TOT_U; ++u) {
          const int s = s0 + 32 * u;
          v[u] = s < B ? __ldg(strip + s) : make_double2(0.0, 0.0);
        }
#pragma unroll
        for (int u = 0; u < F64_TOT_U; ++u) {
          Eg = max(Eg, dbl_exp(v[u].x));
          Eh = max(Eh, dbl_exp(v[u].y));
        }
      }
      Eg = (int)__reduce_max_sync(0xffffffffu, (unsigned)Eg);
      Eh = (int)__reduce_max_sync(0xffffffffu, (unsigned)Eh);
      const double2 m = __ldg(strip + n_bins);
      st.no_missing = dbl2_zero(m);
      st.ok = make_grid(Eg, B, L, st.gg) && make_grid(Eh, B, L, st.gh) && sc.filter;
      if (st.ok) {
        int64_t TG = 0, TH = 0;
        for (int s0 = lane; s0 < B; s0 += 32 * F64_TOT_U) {
          double2 v[F64_TOT_U];
#pragma unroll
          for (int u = 0; u < F64_TOT_U; ++u) {
            const int s = s0 + 32 * u;
            v[u] = s < B ? __ldg(strip + s) : make_double2(0.0, 0.0);
          }
#pragma unroll
          for (int u = 0; u < F64_TOT_U; ++u) {
            TG += dbl_to_fixed(v[u].x, st.gg.k);
            TH += dbl_to_fixed(v[u].y, st.gh.k);
          }
        }
        warp_sum2(TG, TH);
        st.TG = TG;
        st.TH = TH;
        st.mq_g = dbl_to_fixed(m.x, st.gg.k);
        st.mq_h = dbl_to_fixed(m.y, st.gh.k);
        float Gf, eG, Hf, eH;
        fix_to_f32(TG, st.gg, Gf, eG);
        fix_to_f32(TH, st.gh, Hf, eH);
        st.c_ok = term_bounds(Gf, eG, Hf, eH, sc.lam, st.c_lo, st.c_hi);
        int64_t carry[2] = {0, 0};
        for (int c = 0; c < n_chunks; ++c) {
          const int c0 = c * 32 * SCAN_SPL;
          if (lane == 0) {
            s_carry[warp][c][0] = carry[0];
            s_carry[warp][c][1] = carry[1];
          }
          int64_t pg[SCAN_SPL], ph[SCAN_SPL], eg, eh;
          scan_chunk_fix(strip, n_bins, c0, st.gg.k, st.gh.k, carry, pg, ph, eg, eh);
          float cup = -INFINITY;
#pragma unroll
          for (int i = 0; i < SCAN_SPL; ++i) {
            if (c0 + SCAN_SPL * lane + i >= n_bins) continue;
#pragma unroll
            for (int dir = 0; dir < 2; ++dir) {
              if (dir && st.no_missing) continue;  // empty missing slot: same sums, missing-right comes first
              float u, l;
              if (!screen_fix(eg + pg[i] + (dir ? st.mq_g : 0), eh + ph[i] + (dir ? st.mq_h : 0), TG, TH, st.gg,
                              st.gh, st.c_lo, st.c_hi, st.c_ok, sc, u, l))
                continue;
              cup = fmaxf(cup, u);
              run_lo = fmaxf(run_lo, l);
            }
          }
          cup = warp_max_f(cup);
          if (lane == 0) s_cup[warp][c] = cup;
        }
        run_lo = warp_max_f(run_lo);
      }
    }
    if (lane == 0) {
      s_lo[warp] = run_lo;
      s_strip[warp] = st;
    }
  }
  __syncthreads();
  float thr = -INFINITY;
#pragma unroll
  for (int w = 0; w < SCAN_WARPS; ++w) thr = fmaxf(thr, s_lo[w]);
  // ---- phase 2a: a strip without a usable grid, wholly in double, by its own warp
  if (active && !s_strip[warp].ok) {
    const double2 *strip = reinterpret_cast<const double2 *>(hist) + ((int64_t)node * n_features + f) * B;
    const double2 m = __ldg(strip + n_bins);
    const bool no_missing = s_strip[warp].no_missing;
    double G = 0.0, H = 0.0;
    for (int s = lane; s < B; s += 32) {
      const double2 v = __ldg(strip + s);
      G += v.x;
      H += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      G += __shfl_xor_sync(0xffffffffu, G, o);
      H += __shfl_xor_sync(0xffffffffu, H, o);
    }
    const double parent = __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, sp.lambda));
    double cg = 0.0, ch = 0.0;
    for (int c0 = 0; c0 < n_bins; c0 += 32 * SCAN_SPL) {
      double pg[SCAN_SPL], ph[SCAN_SPL], ag = 0.0, ah = 0.0;
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) {
        const int s = c0 + SCAN_SPL * lane + i;
        const double2 v = s < n_bins ? __ldg(strip + s) : make_double2(0.0, 0.0);
        ag += v.x;
        ah += v.y;
        pg[i] = ag;
        ph[i] = ah;
      }
      double eg = ag, eh = ah;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double yg = __shfl_up_sync(0xffffffffu, eg, o), yh = __shfl_up_sync(0xffffffffu, eh, o);
        if (lane >= o) {
          eg += yg;
          eh += yh;
        }
      }
      const double tg = __shfl_sync(0xffffffffu, eg, 31), th = __shfl_sync(0xffffffffu, eh, 31);
      eg = eg - ag + cg;
      eh = eh - ah + ch;
      cg += tg;
      ch += th;
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) {
        if (c0 + SCAN_SPL * lane + i >= n_bins) continue;
#pragma unroll
        for (int dir = 0; dir < 2; ++dir) {
          if (dir && no_missing) continue;
          const double GL = eg + pg[i] + (dir ? m.x : 0.0), HL = eh + ph[i] + (dir ? m.y : 0.0);
          f64_consider(GL, HL, G - GL, H - HL, parent, mcw, sp, f, c0 + SCAN_SPL * lane + i, dir, best);
        }
      }
    }
  }
  // ---- phase 2b: tasks (feature, chunk) whose upper bound reaches the threshold, dealt to the warps. The
  // candidates' sums are the exact fixed-point sums (cells truncated to the strip's grid, summed without
  // rounding in int64) rounded once to double: within B 2^-k + 2^-53 |S| of the exact sums of the double
  // cells, and equal to them whenever the cells lie on the grid.
  {
    int task = 0;
    for (int w = 0; w < SCAN_WARPS; ++w) {
      if (blockIdx.x * SCAN_WARPS + w >= n_features || !s_strip[w].ok) continue;
      for (int c = 0; c < n_chunks; ++c) {
        if (!(s_cup[w][c] >= thr)) continue;
        if ((task++ % SCAN_WARPS) != warp) continue;
        const F64Strip &st = s_strip[w];
        const int fw = blockIdx.x * SCAN_WARPS + w;
        const double2 *strip = reinterpret_cast<const double2 *>(hist) + ((int64_t)node * n_features + fw) * B;
        const int c0 = c * 32 * SCAN_SPL;
        int64_t carry[2] = {s_carry[w][c][0], s_carry[w][c][1]};
        int64_t pg[SCAN_SPL], ph[SCAN_SPL], eg, eh;
        scan_chunk_fix(strip, n_bins, c0, st.gg.k, st.gh.k, carry, pg, ph, eg, eh);
        double G = 0.0, H = 0.0, parent = 0.0;
        bool have_parent = false;
#pragma unroll
        for (int i = 0; i < SCAN_SPL; ++i) {
          if (c0 + SCAN_SPL * lane + i >= n_bins) continue;
#pragma unroll
          for (int dir = 0; dir < 2; ++dir) {
            if (dir && st.no_missing) continue;
            const int64_t GLq = eg + pg[i] + (dir ? st.mq_g : 0), HLq = eh + ph[i] + (dir ? st.mq_h : 0);
            float u, l;
            if (!screen_fix(GLq, HLq, st.TG, st.TH, st.gg, st.gh, st.c_lo, st.c_hi, st.c_ok, sc, u, l) || u < thr)
              continue;
            if (!have_parent) {
              G = fix_to_f64(st.TG, st.gg);
              H = fix_to_f64(st.TH, st.gh);
              parent = __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, sp.lambda));
              have_parent = true;
            }
            f64_consider(fix_to_f64(GLq, st.gg), fix_to_f64(HLq, st.gh), fix_to_f64(st.TG - GLq, st.gg),
                         fix_to_f64(st.TH - HLq, st.gh), parent, mcw, sp, fw, c0 + SCAN_SPL * lane + i, dir, best);
          }
        }
      }
    }
  }
  best = warp_best_cand(best);
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  const int nfb = gridDim.x;
  Cand *cn = cand + (int64_t)node * nfb;
  if (threadIdx.x == 0) {
    Cand b = s_best[0];
    for (int w = 1; w < SCAN_WARPS; ++w)
      if (cand_better(s_best[w], b)) b = s_best[w];
    cn[blockIdx.x] = b;
    __threadfence();
    const uint32_t done = atomicAdd(counters + node, 1u);
    s_last = (done == (uint32_t)nfb - 1) ? 1u : 0u;
    if (s_last) {
      counters[node] = 0;
      __threadfence();
    }
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  Cand b = no_cand();
  for (int i = lane; i < nfb; i += 32) {
    const Cand c = load_cand(cn + i);
    if (cand_better(c, b)) b = c;
  }
  b = warp_best_cand(b);
  if (lane == 0) {
    SplitOut o = cand_to_split(b);
    if (b.f == INT32_MAX) o.g_left = o.h_left = o.g_right = o.h_right = __double_as_longlong(0.0);
    out[node] = o;
  }
}

}  // namespace gbt
