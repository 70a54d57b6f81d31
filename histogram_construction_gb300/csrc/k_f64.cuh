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
__global__ void __launch_bounds__(256) k_finalize_f64(const double *__restrict__ partial,
                                                      const int32_t *__restrict__ group_prefix, int64_t image_doubles,
                                                      int32_t n_fgroups, int32_t item_feats, int32_t sbw,
                                                      int32_t n_nodes, int32_t n_features, int32_t B,
                                                      double *__restrict__ hist_out, const DevState *st) {
  pdl_wait();
  if (!st->plan_ok) return;
  const int64_t units = (int64_t)n_nodes * n_features * B;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int f = (int)(u % n_features);  // consecutive threads: consecutive features of one slot
    int64_t r = u / n_features;
    const int s = (int)(r % B);
    const int n = (int)(r / B);
    const int fg = f / item_feats, fl = f - fg * item_feats;
    const int sb = fl / sbw, c = fl - sb * sbw;
    const int64_t cell = (((int64_t)sb * B + s) * sbw + c) * 2;
    double g = 0.0, h = 0.0;
    for (int32_t k = group_prefix[n]; k < group_prefix[n + 1]; ++k) {
      const double *src = partial + ((int64_t)k * n_fgroups + fg) * image_doubles + cell;
      g += __ldcg(src);
      h += __ldcg(src + 1);
    }
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

// FP32 screen of a float-cell candidate from its double sums: (up, lo) with
// lo <= gain_fp64 <= up. Each double converts to float with relative error
// u = 2^-24, within the 4u per input that the fixed-point screen's error
// budget (screen_f32) assumes, so its bound 2^-19 (a + b + c + |gamma|)
// holds; values outside [2^-60, 2^60] give an infinite bound (evaluated in
// double).
__device__ __forceinline__ void screen_dbl(double GL, double HL, double GR, double HR, float Gf2den,
                                           const SplitParams &sp, float &up, float &lo) {
  const float gl = __double2float_rn(GL), hl = __double2float_rn(HL);
  const float gr = __double2float_rn(GR), hr = __double2float_rn(HR);
  const float dl = __fadd_rn(hl, sp.lambda_f), dr = __fadd_rn(hr, sp.lambda_f);
  const float a = __fdividef(__fmul_rn(gl, gl), dl);
  const float b = __fdividef(__fmul_rn(gr, gr), dr);
  const float g = __fsub_rn(__fmul_rn(0.5f, __fsub_rn(__fadd_rn(a, b), Gf2den)), sp.gamma_f);
  const float mag = __fadd_rn(__fadd_rn(__fadd_rn(a, b), Gf2den), sp.gamma_abs_f);
  const float err = __fmul_rn(mag, 1.9073486328125e-06f);  // 2^-19
  const float rlo = 8.673617379884035e-19f, rhi = 1.152921504606847e+18f;  // 2^-60, 2^60
  const float ag = fabsf(gl), ar = fabsf(gr);
  const bool ok = (ag == 0.f || (ag > rlo && ag < rhi)) && (ar == 0.f || (ar > rlo && ar < rhi)) && dl > rlo &&
                  dr > rlo && dl < rhi && dr < rhi && mag < rhi && (a == 0.f || a > rlo) && (b == 0.f || b > rlo) &&
                  g == g;
  up = ok ? __fadd_rn(g, err) : INFINITY;
  lo = ok ? __fsub_rn(g, err) : -INFINITY;
}

// Parent term G^2 / (H + lambda) in FP32 from the double totals; NaN (every
// candidate then unscreened) outside the checked range.
__device__ __forceinline__ float parent_dbl(double G, double H, const SplitParams &sp) {
  const float Gf = __double2float_rn(G), Hf = __double2float_rn(H);
  const float den = __fadd_rn(Hf, sp.lambda_f);
  const float rlo = 8.673617379884035e-19f, rhi = 1.152921504606847e+18f;
  const float ag = fabsf(Gf);
  if (den > rlo && den < rhi && (ag == 0.f || (ag > rlo && ag < rhi))) {
    const float c = __fdividef(__fmul_rn(Gf, Gf), den);
    if (c == 0.f || (c > rlo && c < rhi)) return c;
  }
  return __int_as_float(0x7fc00000);
}

// Split find on double cells: grid (ceil(F / 8), n_nodes), 256 threads; warp w
// scans feature blockIdx.x * 8 + w of node blockIdx.y. Prefix sums are double;
// each valid candidate is screened in FP32 with a rigorous bound and only
// those whose upper bound reaches the warp's running best lower bound are
// evaluated in double (the best candidate and every candidate tied with it
// always are; FP64 is a small fraction of the FP32 rate on this part). The
// CTA's best goes to cand[node][blockIdx.x]; the node's last CTA writes the
// split. The double sums travel as bit patterns in the candidate's 64-bit
// fields, so the output record is a gbt_split whose four sums are doubles.
__global__ void __launch_bounds__(SCAN_THREADS) k_find_f64(const double *__restrict__ hist, int32_t n_features,
                                                           int32_t n_bins, SplitParams sp, double mcw,
                                                           Cand *__restrict__ cand, uint32_t *__restrict__ counters,
                                                           SplitOut *__restrict__ out) {
  __shared__ Cand s_best[SCAN_WARPS];
  __shared__ uint32_t s_last;
  pdl_wait();
  const int node = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * SCAN_WARPS + warp;
  const int B = n_bins + 1;
  Cand best = no_cand();
  if (f < n_features) {
    const double2 *strip = reinterpret_cast<const double2 *>(hist) + ((int64_t)node * n_features + f) * B;
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
    const double2 m = __ldg(strip + n_bins);
    const double parent = __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, sp.lambda));
    const float Gf2den = sp.filter ? parent_dbl(G, H, sp) : 0.f;
    float run_lo = -INFINITY;
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
      float up[SCAN_SPL][2];
      uint32_t vmask = 0;
      float l = -INFINITY;
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) {
        const int s = c0 + SCAN_SPL * lane + i;
#pragma unroll
        for (int dir = 0; dir < 2; ++dir) {
          up[i][dir] = -INFINITY;
          if (s >= n_bins) continue;
          const double GL = eg + pg[i] + (dir ? m.x : 0.0), HL = eh + ph[i] + (dir ? m.y : 0.0);
          const double GR = G - GL, HR = H - HL;
          if (!(HL > 0.0 && HR > 0.0 && HL >= mcw && HR >= mcw)) continue;
          float u = INFINITY, lw = -INFINITY;
          if (sp.filter) screen_dbl(GL, HL, GR, HR, Gf2den, sp, u, lw);
          up[i][dir] = u;
          vmask |= 1u << (2 * i + dir);
          l = fmaxf(l, lw);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
      run_lo = fmaxf(run_lo, l);
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) {
#pragma unroll
        for (int dir = 0; dir < 2; ++dir) {
          if (!((vmask >> (2 * i + dir)) & 1u) || up[i][dir] < run_lo) continue;  // invalid, or below a lower bound
          const double GL = eg + pg[i] + (dir ? m.x : 0.0), HL = eh + ph[i] + (dir ? m.y : 0.0);
          const double GR = G - GL, HR = H - HL;
          const double l2 = __ddiv_rn(__dmul_rn(GL, GL), __dadd_rn(HL, sp.lambda));
          const double r2 = __ddiv_rn(__dmul_rn(GR, GR), __dadd_rn(HR, sp.lambda));
          const double gain = __dsub_rn(__dmul_rn(0.5, __dsub_rn(__dadd_rn(l2, r2), parent)), sp.gamma);
          Cand c;
          set_exact(c, gain);
          c.t = c0 + SCAN_SPL * lane + i;
          c.dir = dir;
          c.f = f;
          c.gl = __double_as_longlong(GL);
          c.hl = __double_as_longlong(HL);
          c.gr = __double_as_longlong(GR);
          c.hr = __double_as_longlong(HR);
          if (cand_better(c, best)) best = c;
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
