// Sibling subtraction and split finding.
//
// Subtraction ["GBDT engine engineering deep-dive" (ybb.press), section 3]:
//   Large[p] = Parent[parent_of[p]] - Small[p], exact int64, a pure streaming op.
// Split find [same page, section 1 gain and bin-boundary cuts; section 4
// default direction; bonsai "9. Parallelism & determinism", "In bonsai": serial
// feature-order tie-break]: per node and feature an inclusive int64 prefix over
// the real slots, two candidates per cut t (missing right, missing left), gain
// in IEEE double with no contraction, first strictly larger gain in (feature,
// t, right-before-left) order.
#pragma once

#include <float.h>

#include "common.cuh"

namespace gbt {

struct SplitParams {
  double lambda, gamma, mcw, inv_sg, inv_sh;
};

// gain = 0.5 * (GL^2/(HL+lambda) + GR^2/(HR+lambda) - G^2/(H+lambda)) - gamma,
// every operation one IEEE double op in this order (no fused multiply-add).
__device__ __forceinline__ double split_gain(double gl, double hl, double gr, double hr, double g, double h,
                                             const SplitParams &sp) {
  const double left = __ddiv_rn(__dmul_rn(gl, gl), __dadd_rn(hl, sp.lambda));
  const double right = __ddiv_rn(__dmul_rn(gr, gr), __dadd_rn(hr, sp.lambda));
  const double parent = __ddiv_rn(__dmul_rn(g, g), __dadd_rn(h, sp.lambda));
  double s = __dadd_rn(left, right);
  s = __dsub_rn(s, parent);
  return __dsub_rn(__dmul_rn(0.5, s), sp.gamma);
}

struct Best {
  double gain;
  int32_t t, dir;
};

__device__ __forceinline__ bool better(const Best &a, const Best &b) {
  return a.gain > b.gain || (a.gain == b.gain && (a.t < b.t || (a.t == b.t && a.dir < b.dir)));
}

// Evaluate both directions of cut t with prefix (pg, ph), missing (gm, hm),
// totals (G, H); update the lane's best (t ascending per lane, strict >).
__device__ __forceinline__ void eval_cut(Best &best, int32_t t, int64_t pg, int64_t ph, int64_t gm, int64_t hm,
                                         int64_t G, int64_t H, double Gd, double Hd, const SplitParams &sp) {
#pragma unroll
  for (int dir = 0; dir < 2; ++dir) {
    const int64_t GL = pg + (dir ? gm : 0), HL = ph + (dir ? hm : 0);
    const int64_t GR = G - GL, HR = H - HL;
    if (!(HL > 0 && HR > 0)) continue;
    const double gld = __dmul_rn(__ll2double_rn(GL), sp.inv_sg);
    const double hld = __dmul_rn(__ll2double_rn(HL), sp.inv_sh);
    const double grd = __dmul_rn(__ll2double_rn(GR), sp.inv_sg);
    const double hrd = __dmul_rn(__ll2double_rn(HR), sp.inv_sh);
    if (!(hld >= sp.mcw && hrd >= sp.mcw)) continue;
    const double g = split_gain(gld, hld, grd, hrd, Gd, Hd, sp);
    if (g > best.gain) {
      best.gain = g;
      best.t = t;
      best.dir = dir;
    }
  }
}

__device__ __forceinline__ int64_t shfl_i64(int64_t v, int src) {
  return (int64_t)__shfl_sync(0xffffffffu, (long long)v, src);
}
__device__ __forceinline__ int64_t shfl_up_i64(int64_t v, int d) {
  return (int64_t)__shfl_up_sync(0xffffffffu, (long long)v, d);
}
__device__ __forceinline__ int64_t shfl_xor_i64(int64_t v, int m) {
  return (int64_t)__shfl_xor_sync(0xffffffffu, (long long)v, m);
}

// One warp scans one feature strip (B cells of (G,H) int64, reads via ld).
// The strip was fully loaded/written by this warp (or is read-only input).
__device__ __forceinline__ Best warp_scan_strip(const longlong2 *strip, int n_bins, const SplitParams &sp) {
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  // totals and missing cell
  int64_t tg = 0, th = 0;
  for (int s = lane; s < B; s += 32) {
    const longlong2 c = strip[s];
    tg += c.x;
    th += c.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tg += shfl_xor_i64(tg, o);
    th += shfl_xor_i64(th, o);
  }
  const longlong2 m = strip[n_bins];
  const double Gd = __dmul_rn(__ll2double_rn(tg), sp.inv_sg);
  const double Hd = __dmul_rn(__ll2double_rn(th), sp.inv_sh);
  Best best{-INFINITY, INT32_MAX, 1};
  int64_t cg = 0, ch = 0;  // carry of previous rounds
  for (int s0 = 0; s0 < n_bins; s0 += 32) {
    const int s = s0 + lane;
    longlong2 c = make_longlong2(0, 0);
    if (s < n_bins) c = strip[s];
    int64_t pg = c.x, ph = c.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t yg = shfl_up_i64(pg, o), yh = shfl_up_i64(ph, o);
      if (lane >= o) {
        pg += yg;
        ph += yh;
      }
    }
    pg += cg;
    ph += ch;
    if (s < n_bins) eval_cut(best, s, pg, ph, m.x, m.y, tg, th, Gd, Hd, sp);
    cg = shfl_i64(pg, 31);
    ch = shfl_i64(ph, 31);
  }
  // warp argmax
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best other;
    other.gain = __shfl_xor_sync(0xffffffffu, best.gain, o);
    other.t = __shfl_xor_sync(0xffffffffu, best.t, o);
    other.dir = __shfl_xor_sync(0xffffffffu, best.dir, o);
    if (better(other, best)) best = other;
  }
  return best;
}

// Find: one warp per (node, feature) of `hist`; writes cand[node][f].
constexpr int SCAN_THREADS = 256;

__global__ void __launch_bounds__(SCAN_THREADS) k_find(const int64_t *__restrict__ hist, int32_t n_nodes,
                                                       int32_t n_features, int32_t n_bins, SplitParams sp,
                                                       Cand *__restrict__ cand) {
  const int64_t units = (int64_t)n_nodes * n_features;
  const int64_t wglobal = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int B = n_bins + 1;
  for (int64_t u = wglobal; u < units; u += nw) {
    const longlong2 *strip = reinterpret_cast<const longlong2 *>(hist) + u * B;
    const Best b = warp_scan_strip(strip, n_bins, sp);
    if ((threadIdx.x & 31) == 0) cand[u] = Cand{b.gain, b.t, b.dir};
  }
}

// Subtract and find: one warp per (pair, feature): Large = Parent - Small
// (stored), then the scan of both strips. cand[2p][f] small, cand[2p+1][f] large.
__global__ void __launch_bounds__(SCAN_THREADS) k_subtract_find(const int64_t *__restrict__ parent,
                                                                const int32_t *__restrict__ parent_of,
                                                                const int64_t *__restrict__ small,
                                                                int64_t *__restrict__ large, int32_t n_pairs,
                                                                int32_t n_features, int32_t n_bins, SplitParams sp,
                                                                Cand *__restrict__ cand, DevState *st) {
  const int64_t units = (int64_t)n_pairs * n_features;
  const int64_t wglobal = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  for (int64_t u = wglobal; u < units; u += nw) {
    const int64_t p = u / n_features, f = u - p * n_features;
    const int64_t pp = parent_of ? (int64_t)parent_of[p] : p;
    const longlong2 *P = reinterpret_cast<const longlong2 *>(parent) + (pp * n_features + f) * B;
    const longlong2 *S = reinterpret_cast<const longlong2 *>(small) + u * B;
    longlong2 *L = reinterpret_cast<longlong2 *>(large) + u * B;
    bool neg = false;
    for (int s = lane; s < B; s += 32) {
      const longlong2 a = P[s], b = S[s];
      const longlong2 d = make_longlong2(a.x - b.x, a.y - b.y);
      neg |= d.y < 0;
      L[s] = d;
    }
    if (neg) raise_err(st, ERRBIT_INCONSISTENT);
    __syncwarp();
    const Best bs = warp_scan_strip(S, n_bins, sp);
    const Best bl = warp_scan_strip(L, n_bins, sp);
    if (lane == 0) {
      cand[(2 * p) * n_features + f] = Cand{bs.gain, bs.t, bs.dir};
      cand[(2 * p + 1) * n_features + f] = Cand{bl.gain, bl.t, bl.dir};
    }
  }
}

// Plain subtraction (no split find): 16-byte units.
__global__ void __launch_bounds__(256) k_subtract(const int64_t *__restrict__ parent, const int32_t *__restrict__ parent_of,
                                                  const int64_t *__restrict__ small, int64_t *__restrict__ large,
                                                  int32_t n_pairs, int64_t units_per_node, DevState *st) {
  const int64_t units = (int64_t)n_pairs * units_per_node;
  bool neg = false;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = u / units_per_node, w = u - p * units_per_node;
    const int64_t pp = parent_of ? (int64_t)parent_of[p] : p;
    const longlong2 a = reinterpret_cast<const longlong2 *>(parent)[pp * units_per_node + w];
    const longlong2 b = reinterpret_cast<const longlong2 *>(small)[u];
    const longlong2 d = make_longlong2(a.x - b.x, a.y - b.y);
    neg |= d.y < 0;
    reinterpret_cast<longlong2 *>(large)[u] = d;
  }
  if (neg) raise_err(st, ERRBIT_INCONSISTENT);
}

// Per node: the best candidate over features (gain desc, feature asc), then
// the winner's left/right sums from its strip. One block per node.
// hist_of(node) selects the strip source: mode 0 -> hist[node]; mode 1 ->
// node 2p from small[p], node 2p+1 from large[p].
struct SplitOut {
  int32_t feature, bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
};

__global__ void __launch_bounds__(256) k_reduce_splits(const Cand *__restrict__ cand, int32_t n_nodes,
                                                       int32_t n_features, int32_t n_bins, int mode,
                                                       const int64_t *__restrict__ hist_a,
                                                       const int64_t *__restrict__ hist_b, SplitOut *out_a,
                                                       SplitOut *out_b) {
  const int node = blockIdx.x;
  if (node >= n_nodes) return;
  const Cand *cn = cand + (int64_t)node * n_features;
  double bg = -INFINITY;
  int32_t bf = INT32_MAX;
  for (int f = threadIdx.x; f < n_features; f += blockDim.x) {
    const Cand c = cn[f];
    if (c.t != INT32_MAX && (c.gain > bg || (c.gain == bg && f < bf))) {
      bg = c.gain;
      bf = f;
    }
  }
  __shared__ double s_g[256];
  __shared__ int32_t s_f[256];
  s_g[threadIdx.x] = bg;
  s_f[threadIdx.x] = bf;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      const double og = s_g[threadIdx.x + w];
      const int32_t of = s_f[threadIdx.x + w];
      if (og > s_g[threadIdx.x] || (og == s_g[threadIdx.x] && of < s_f[threadIdx.x])) {
        s_g[threadIdx.x] = og;
        s_f[threadIdx.x] = of;
      }
    }
    __syncthreads();
  }
  const int32_t f = s_f[0];
  SplitOut o;
  for (int i = 0; i < 7; ++i) o.pad[i] = 0;
  if (f == INT32_MAX) {
    o.feature = -1;
    o.bin = -1;
    o.default_left = 0;
    o.gain = -INFINITY;
    o.g_left = o.h_left = o.g_right = o.h_right = 0;
  } else {
    const Cand c = cn[f];
    const int B = n_bins + 1;
    const int64_t *src;
    if (mode == 0) src = hist_a + ((int64_t)node * n_features + f) * B * 2;
    else src = ((node & 1) ? hist_b : hist_a) + ((int64_t)(node >> 1) * n_features + f) * B * 2;
    int64_t lg = 0, lh = 0, tg = 0, th = 0;
    for (int s = threadIdx.x; s < B; s += blockDim.x) {
      const int64_t g = src[2 * s], h = src[2 * s + 1];
      tg += g;
      th += h;
      const bool left = (s < n_bins) ? (s <= c.t) : (c.dir == 1);
      if (left) {
        lg += g;
        lh += h;
      }
    }
    __shared__ long long s_v[4][256];
    s_v[0][threadIdx.x] = lg;
    s_v[1][threadIdx.x] = lh;
    s_v[2][threadIdx.x] = tg;
    s_v[3][threadIdx.x] = th;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w)
        for (int k = 0; k < 4; ++k) s_v[k][threadIdx.x] += s_v[k][threadIdx.x + w];
      __syncthreads();
    }
    o.feature = f;
    o.bin = c.t;
    o.default_left = (uint8_t)c.dir;
    o.gain = c.gain;
    o.g_left = s_v[0][0];
    o.h_left = s_v[1][0];
    o.g_right = s_v[2][0] - s_v[0][0];
    o.h_right = s_v[3][0] - s_v[1][0];
  }
  if (threadIdx.x == 0) {
    if (mode == 0) out_a[node] = o;
    else if (node & 1) out_b[node >> 1] = o;
    else out_a[node >> 1] = o;
  }
}

}  // namespace gbt
