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
//
// GB300 has little FP64 throughput, so every candidate is first evaluated in
// FP32 together with a rigorous bound on |gain_fp32 - gain_fp64|; a candidate
// whose upper bound falls below the best lower bound seen so far cannot be
// the double-precision argmax and is dropped; the rest are evaluated in
// double exactly as the definition says. The result is bit-identical to
// evaluating every candidate in double.
#pragma once

#include <float.h>

#include "common.cuh"

namespace gbt {

struct SplitParams {
  double lambda, gamma, inv_sg, inv_sh;
  int64_t h_min;   // smallest quantised H with (double)H * inv_sh >= min_child_weight (and >= 1)
  float lambda_f, gamma_f, gamma_abs_f, inv_sg_f, inv_sh_f;
  int32_t filter;  // 1: FP32 pre-filter enabled (lambda >= 0, finite parameters)
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

// FP32 estimate of the gain and an upper bound of its distance to the double
// value. Each of the three non-negative terms carries a relative error below
// 13 u (u = 2^-24) in FP32; after the sum, difference, halving and the
// subtraction of gamma the error is below 8 u (a + b + c) + 2 u |gamma|. The bound used is 2^-20 (a + b + c +
// |gamma|), i.e. 16 u with a factor-of-two margin for the rounding of the
// bound itself and the double path's own (2^-53-scale) errors. Values outside
// [2^-60, 2^60] (possible underflow / overflow) get an infinite bound, which
// forces the double evaluation.
__device__ __forceinline__ void gain_f32(int64_t GL, int64_t HL, int64_t GR, int64_t HR, float Gf2den,
                                         const SplitParams &sp, float &g, float &err) {
  const float gl = __fmul_rn(__ll2float_rn(GL), sp.inv_sg_f);
  const float hl = __fmul_rn(__ll2float_rn(HL), sp.inv_sh_f);
  const float gr = __fmul_rn(__ll2float_rn(GR), sp.inv_sg_f);
  const float hr = __fmul_rn(__ll2float_rn(HR), sp.inv_sh_f);
  const float dl = __fadd_rn(hl, sp.lambda_f), dr = __fadd_rn(hr, sp.lambda_f);
  const float a = __fdiv_rn(__fmul_rn(gl, gl), dl);
  const float b = __fdiv_rn(__fmul_rn(gr, gr), dr);
  const float s = __fsub_rn(__fadd_rn(a, b), Gf2den);
  g = __fsub_rn(__fmul_rn(0.5f, s), sp.gamma_f);
  const float mag = __fadd_rn(__fadd_rn(__fadd_rn(a, b), Gf2den), sp.gamma_abs_f);
  err = __fmul_rn(mag, 9.5367431640625e-07f);  // 2^-20
  const float lo = 8.673617379884035e-19f, hi = 1.152921504606847e+18f;  // 2^-60, 2^60
  const float ag = fabsf(gl), ar = fabsf(gr);
  const bool ok = (ag == 0.f || (ag > lo && ag < hi)) && (ar == 0.f || (ar > lo && ar < hi)) && dl > lo &&
                  dr > lo && dl < hi && dr < hi && mag < hi && (a == 0.f || a > lo) && (b == 0.f || b > lo);
  if (!ok) err = INFINITY;
}

// Candidate of a block of features (pre-reduced per CTA). 64 bytes, 16-byte
// aligned, so it can be read back with four 16-byte loads.
struct __align__(16) Cand {
  double gain;
  int32_t t, dir;
  int32_t f, pad;
  int64_t gl, hl, gr, hr;
  int64_t pad2;
};
static_assert(sizeof(Cand) == 64, "Cand is read as four 16-byte words");

struct SplitOut {
  int32_t feature, bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
};

// Per-lane best candidate (exact double gain) with its left sums.
struct Best {
  double gain;
  int32_t t, dir;
  int64_t gl, hl;
};

__device__ __forceinline__ bool better(const Best &a, const Best &b) {
  return a.gain > b.gain || (a.gain == b.gain && (a.t < b.t || (a.t == b.t && a.dir < b.dir)));
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

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best other;
    other.gain = __shfl_xor_sync(0xffffffffu, b.gain, o);
    other.t = __shfl_xor_sync(0xffffffffu, b.t, o);
    other.dir = __shfl_xor_sync(0xffffffffu, b.dir, o);
    other.gl = shfl_xor_i64(b.gl, o);
    other.hl = shfl_xor_i64(b.hl, o);
    if (better(other, b)) b = other;
  }
  return b;
}

// Warp inclusive scan of (G, H) int64.
__device__ __forceinline__ void warp_incl_scan(int64_t &pg, int64_t &ph) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t yg = shfl_up_i64(pg, o), yh = shfl_up_i64(ph, o);
    if (lane >= o) {
      pg += yg;
      ph += yh;
    }
  }
}

__device__ __forceinline__ void warp_sum2(int64_t &a, int64_t &b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += shfl_xor_i64(a, o);
    b += shfl_xor_i64(b, o);
  }
}

// Per-strip constants of the FP32 filter.
struct StripInfo {
  int64_t tg, th;  // feature totals
  int64_t mg, mh;  // missing cell
  float Gf2den;    // parent term in FP32
};

__device__ __forceinline__ float parent_f32(int64_t tg, int64_t th, const SplitParams &sp) {
  const float Gf = __fmul_rn(__ll2float_rn(tg), sp.inv_sg_f);
  const float Hf = __fmul_rn(__ll2float_rn(th), sp.inv_sh_f);
  return __fdiv_rn(__fmul_rn(Gf, Gf), __fadd_rn(Hf, sp.lambda_f));
}

// FP32 bounds of the two candidates of cut s (missing right / left) with
// inclusive prefix (pg, ph). Invalid candidates get (-inf, -inf).
__device__ __forceinline__ void cut_bounds(int s, int n_bins, int64_t pg, int64_t ph, const StripInfo &si,
                                           const SplitParams &sp, float (&up)[2], float (&lo)[2]) {
#pragma unroll
  for (int dir = 0; dir < 2; ++dir) {
    const int64_t GL = pg + (dir ? si.mg : 0), HL = ph + (dir ? si.mh : 0);
    const int64_t HR = si.th - HL;
    up[dir] = -INFINITY;
    lo[dir] = -INFINITY;
    if (s < n_bins && HL >= sp.h_min && HR >= sp.h_min) {
      if (sp.filter) {
        float g, e;
        gain_f32(GL, HL, si.tg - GL, HR, si.Gf2den, sp, g, e);
        up[dir] = __fadd_rn(g, e);
        lo[dir] = __fsub_rn(g, e);
        if (!(up[dir] == up[dir])) up[dir] = INFINITY;  // NaN: keep for the double pass
        if (!(lo[dir] == lo[dir])) lo[dir] = -INFINITY;
      } else {
        up[dir] = INFINITY;
      }
    }
  }
}

// A candidate that survived the FP32 filter; evaluated in double later.
struct Surv {
  int64_t gl, hl, tg, th;
  int32_t t;
  int16_t f;     // feature offset within the CTA
  int8_t dir;
  int8_t node;   // 0: first strip set (small / hist), 1: second (large)
};

constexpr int SURV_CAP = 256;

// Exact double gain of a survivor.
__device__ __forceinline__ double surv_gain(const Surv &v, const SplitParams &sp) {
  const double gld = __dmul_rn(__ll2double_rn(v.gl), sp.inv_sg);
  const double hld = __dmul_rn(__ll2double_rn(v.hl), sp.inv_sh);
  const double grd = __dmul_rn(__ll2double_rn(v.tg - v.gl), sp.inv_sg);
  const double hrd = __dmul_rn(__ll2double_rn(v.th - v.hl), sp.inv_sh);
  const double Gd = __dmul_rn(__ll2double_rn(v.tg), sp.inv_sg);
  const double Hd = __dmul_rn(__ll2double_rn(v.th), sp.inv_sh);
  return split_gain(gld, hld, grd, hrd, Gd, Hd, sp);
}

// Shared state of the CTA-batched split evaluation.
struct SurvPool {
  Surv v[SURV_CAP];
  double gain[SURV_CAP];
  float warp_lo[2][32];
  Cand best[2];  // the CTA's best candidate per strip set, written by pool_eval
  int n;
};

// Strip access: cells in registers (NR rounds of 32 slots) ...
template <int NR>
struct RegStrip {
  const longlong2 (&c)[NR];
  __device__ __forceinline__ longlong2 cell(int r) const { return c[r]; }
};

// Pass A over a register strip: totals, missing cell, and the warp's best
// lower bound. Returns the strip constants.
template <int NR>
__device__ __forceinline__ StripInfo regs_pass_a(const longlong2 (&c)[NR], int n_bins, const SplitParams &sp,
                                                 float &wlo) {
  const int lane = threadIdx.x & 31;
  StripInfo si;
  si.tg = 0;
  si.th = 0;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    si.tg += c[r].x;
    si.th += c[r].y;
  }
  warp_sum2(si.tg, si.th);
  const int rm = n_bins >> 5, lm = n_bins & 31;
  si.mg = 0;
  si.mh = 0;
#pragma unroll
  for (int r = 0; r < NR; ++r)
    if (r == rm) {
      si.mg = shfl_i64(c[r].x, lm);
      si.mh = shfl_i64(c[r].y, lm);
    }
  si.Gf2den = parent_f32(si.tg, si.th, sp);
  float l = -INFINITY;
  int64_t cg = 0, ch = 0;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r * 32 >= n_bins) break;
    const int s = r * 32 + lane;
    int64_t pg = s < n_bins ? c[r].x : 0, ph = s < n_bins ? c[r].y : 0;
    warp_incl_scan(pg, ph);
    pg += cg;
    ph += ch;
    cg = shfl_i64(pg, 31);
    ch = shfl_i64(ph, 31);
    float up[2], lo[2];
    cut_bounds(s, n_bins, pg, ph, si, sp, up, lo);
    l = fmaxf(l, fmaxf(lo[0], lo[1]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
  wlo = l;
  return si;
}

// Append the candidates of cut s whose upper bound reaches `thr`.
__device__ __forceinline__ void push_survivors(SurvPool &pool, int s, int n_bins, int64_t pg, int64_t ph,
                                               const StripInfo &si, const SplitParams &sp, float thr, int f_off,
                                               int node, int &overflow) {
  float up[2], lo[2];
  cut_bounds(s, n_bins, pg, ph, si, sp, up, lo);
#pragma unroll
  for (int dir = 0; dir < 2; ++dir) {
    if (!(up[dir] >= thr) || up[dir] == -INFINITY) continue;
    const int idx = atomicAdd(&pool.n, 1);
    if (idx >= SURV_CAP) {
      overflow = 1;
      continue;
    }
    Surv v;
    v.gl = pg + (dir ? si.mg : 0);
    v.hl = ph + (dir ? si.mh : 0);
    v.tg = si.tg;
    v.th = si.th;
    v.t = s;
    v.f = (int16_t)f_off;
    v.dir = (int8_t)dir;
    v.node = (int8_t)node;
    pool.v[idx] = v;
  }
}

template <int NR>
__device__ __forceinline__ void regs_pass_b(const longlong2 (&c)[NR], int n_bins, const StripInfo &si,
                                            const SplitParams &sp, float thr, int f_off, int node, SurvPool &pool,
                                            int &overflow) {
  const int lane = threadIdx.x & 31;
  int64_t cg = 0, ch = 0;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r * 32 >= n_bins) break;
    const int s = r * 32 + lane;
    int64_t pg = s < n_bins ? c[r].x : 0, ph = s < n_bins ? c[r].y : 0;
    warp_incl_scan(pg, ph);
    pg += cg;
    ph += ch;
    cg = shfl_i64(pg, 31);
    ch = shfl_i64(ph, 31);
    push_survivors(pool, s, n_bins, pg, ph, si, sp, thr, f_off, node, overflow);
  }
}

// Streaming variants (strip in global memory, any B): two reads of the strip.
__device__ __forceinline__ StripInfo stream_pass_a(const longlong2 *strip, int n_bins, const SplitParams &sp,
                                                   float &wlo) {
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  StripInfo si;
  si.tg = 0;
  si.th = 0;
  for (int s0 = 0; s0 < B; s0 += 256) {
    longlong2 c[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int s = s0 + r * 32 + lane;
      c[r] = s < B ? strip[s] : make_longlong2(0, 0);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      si.tg += c[r].x;
      si.th += c[r].y;
    }
  }
  warp_sum2(si.tg, si.th);
  const longlong2 m = strip[n_bins];
  si.mg = m.x;
  si.mh = m.y;
  si.Gf2den = parent_f32(si.tg, si.th, sp);
  float l = -INFINITY;
  int64_t cg = 0, ch = 0;
  for (int s0 = 0; s0 < n_bins; s0 += 256) {
    longlong2 c[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int s = s0 + r * 32 + lane;
      c[r] = s < n_bins ? strip[s] : make_longlong2(0, 0);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (s0 + r * 32 >= n_bins) break;
      const int s = s0 + r * 32 + lane;
      int64_t pg = c[r].x, ph = c[r].y;
      warp_incl_scan(pg, ph);
      pg += cg;
      ph += ch;
      cg = shfl_i64(pg, 31);
      ch = shfl_i64(ph, 31);
      float up[2], lo[2];
      cut_bounds(s, n_bins, pg, ph, si, sp, up, lo);
      l = fmaxf(l, fmaxf(lo[0], lo[1]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
  wlo = l;
  return si;
}

__device__ __forceinline__ void stream_pass_b(const longlong2 *strip, int n_bins, const StripInfo &si,
                                              const SplitParams &sp, float thr, int f_off, int node, SurvPool &pool,
                                              int &overflow) {
  const int lane = threadIdx.x & 31;
  int64_t cg = 0, ch = 0;
  for (int s0 = 0; s0 < n_bins; s0 += 256) {
    longlong2 c[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int s = s0 + r * 32 + lane;
      c[r] = s < n_bins ? strip[s] : make_longlong2(0, 0);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (s0 + r * 32 >= n_bins) break;
      const int s = s0 + r * 32 + lane;
      int64_t pg = c[r].x, ph = c[r].y;
      warp_incl_scan(pg, ph);
      pg += cg;
      ph += ch;
      cg = shfl_i64(pg, 31);
      ch = shfl_i64(ph, 31);
      push_survivors(pool, s, n_bins, pg, ph, si, sp, thr, f_off, node, overflow);
    }
  }
}

constexpr int SCAN_THREADS = 256;
constexpr int SCAN_FEATS = SCAN_THREADS / 32;  // features per CTA, one per warp

__device__ __forceinline__ bool cand_better(const Cand &c, const Cand &best) {
  return c.f != INT32_MAX && (best.f == INT32_MAX || c.gain > best.gain || (c.gain == best.gain && c.f < best.f));
}

__device__ __forceinline__ Cand make_cand(const Best &b, int f, int64_t tg, int64_t th) {
  Cand c;
  c.gain = b.gain;
  c.t = b.t;
  c.dir = b.dir;
  c.f = (b.t == INT32_MAX) ? INT32_MAX : f;
  c.pad = 0;
  c.pad2 = 0;
  c.gl = b.gl;
  c.hl = b.hl;
  c.gr = tg - b.gl;
  c.hr = th - b.hl;
  return c;
}

__device__ __forceinline__ SplitOut cand_to_split(const Cand &best) {
  SplitOut o;
  for (int i = 0; i < 7; ++i) o.pad[i] = 0;
  if (best.f == INT32_MAX) {
    o.feature = -1;
    o.bin = -1;
    o.default_left = 0;
    o.gain = -INFINITY;
    o.g_left = o.h_left = o.g_right = o.h_right = 0;
  } else {
    o.feature = best.f;
    o.bin = best.t;
    o.default_left = (uint8_t)best.dir;
    o.gain = best.gain;
    o.g_left = best.gl;
    o.h_left = best.hl;
    o.g_right = best.gr;
    o.h_right = best.hr;
  }
  return o;
}

// Reduce the per-CTA candidates of `nodes` nodes (n_cand each, stored node
// after node) with one warp per node and write their splits.
__device__ __forceinline__ void reduce_nodes_warp(const Cand *cand, int n_cand, SplitOut *out) {
  const int lane = threadIdx.x & 31;
  Cand best;
  best.f = INT32_MAX;
  best.gain = -INFINITY;
  for (int i = lane; i < n_cand; i += 32) {
    Cand c;
    const int4 *src = reinterpret_cast<const int4 *>(cand + i);  // L2 reads: written by other CTAs
    int4 *dst = reinterpret_cast<int4 *>(&c);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = __ldcg(src + k);
    if (cand_better(c, best)) best = c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand c;
    c.gain = __shfl_xor_sync(0xffffffffu, best.gain, o);
    c.f = __shfl_xor_sync(0xffffffffu, best.f, o);
    c.t = __shfl_xor_sync(0xffffffffu, best.t, o);
    c.dir = __shfl_xor_sync(0xffffffffu, best.dir, o);
    c.gl = shfl_xor_i64(best.gl, o);
    c.hl = shfl_xor_i64(best.hl, o);
    c.gr = shfl_xor_i64(best.gr, o);
    c.hr = shfl_xor_i64(best.hr, o);
    if (cand_better(c, best)) best = c;
  }
  if (lane == 0) *out = cand_to_split(best);
}

// CTA epilogue of the batched evaluation: every survivor of the CTA is
// evaluated in double by one thread, then the CTA's best candidate of each
// node set (0/1) is formed (gain desc, feature asc, t asc, dir asc).
// Survivors that did not fit the pool (overflow) were evaluated by their
// warps directly and arrive in `extra[node][warp]`.
__device__ __forceinline__ void pool_eval(SurvPool &pool, const SplitParams &sp, int f_base, int n_sets,
                                          const Cand (*extra)[SCAN_FEATS]) {
  const int n = min(pool.n, SURV_CAP);
  for (int i = threadIdx.x; i < n; i += blockDim.x) pool.gain[i] = surv_gain(pool.v[i], sp);
  __syncthreads();
  if (threadIdx.x < n_sets) {
    const int node = threadIdx.x;
    Cand best;
    best.f = INT32_MAX;
    best.gain = -INFINITY;
    best.t = INT32_MAX;
    best.dir = 1;
    for (int i = 0; i < n; ++i) {
      const Surv &v = pool.v[i];
      if (v.node != node) continue;
      const double g = pool.gain[i];
      const int f = f_base + v.f;
      const bool take = best.f == INT32_MAX || g > best.gain ||
                        (g == best.gain && (f < best.f || (f == best.f && (v.t < best.t ||
                                                                           (v.t == best.t && v.dir < best.dir)))));
      if (take) {
        best.gain = g;
        best.f = f;
        best.t = v.t;
        best.dir = v.dir;
        best.gl = v.gl;
        best.hl = v.hl;
        best.gr = v.tg - v.gl;
        best.hr = v.th - v.hl;
      }
    }
    for (int w = 0; w < SCAN_FEATS; ++w) {
      const Cand &c = extra[node][w];
      if (c.f == INT32_MAX) continue;
      const bool take = best.f == INT32_MAX || c.gain > best.gain ||
                        (c.gain == best.gain && (c.f < best.f || (c.f == best.f && (c.t < best.t ||
                                                                                    (c.t == best.t && c.dir < best.dir)))));
      if (take) best = c;
    }
    best.pad = 0;
    best.pad2 = 0;
    pool.best[node] = best;
  }
  __syncthreads();
}

// Overflow path (more survivors than the pool holds, e.g. many exact ties):
// the warp evaluates its own survivors in double, serially per lane.
__device__ __forceinline__ Cand warp_direct_best(const longlong2 *strip, int n_bins, const StripInfo &si,
                                                 const SplitParams &sp, float thr, int f) {
  const int lane = threadIdx.x & 31;
  Best best{-INFINITY, INT32_MAX, 1, 0, 0};
  int64_t cg = 0, ch = 0;
  for (int s0 = 0; s0 < n_bins; s0 += 32) {
    const int s = s0 + lane;
    int64_t pg = s < n_bins ? strip[s].x : 0, ph = s < n_bins ? strip[s].y : 0;
    warp_incl_scan(pg, ph);
    pg += cg;
    ph += ch;
    cg = shfl_i64(pg, 31);
    ch = shfl_i64(ph, 31);
    float up[2], lo[2];
    cut_bounds(s, n_bins, pg, ph, si, sp, up, lo);
#pragma unroll
    for (int dir = 0; dir < 2; ++dir) {
      if (!(up[dir] >= thr) || up[dir] == -INFINITY) continue;
      Surv v;
      v.gl = pg + (dir ? si.mg : 0);
      v.hl = ph + (dir ? si.mh : 0);
      v.tg = si.tg;
      v.th = si.th;
      const double g = surv_gain(v, sp);
      if (g > best.gain) {
        best.gain = g;
        best.t = s;
        best.dir = dir;
        best.gl = v.gl;
        best.hl = v.hl;
      }
    }
  }
  best = warp_best(best);
  Cand c;
  c.gain = best.gain;
  c.t = best.t;
  c.dir = best.dir;
  c.f = best.t == INT32_MAX ? INT32_MAX : f;
  c.pad = 0;
  c.pad2 = 0;
  c.gl = best.gl;
  c.hl = best.hl;
  c.gr = si.tg - best.gl;
  c.hr = si.th - best.hl;
  return c;
}

// Thread 0 stores the CTA's candidate(s) and counts the CTA in; returns true
// in the last CTA of the group (which resets the counter). No CTA waits.
__device__ __forceinline__ bool cta_publish(const Cand *c, int n_sets, Cand *dst0, Cand *dst1,
                                            uint32_t *counter, uint32_t group_ctas) {
  __shared__ uint32_t s_last;
  if (threadIdx.x == 0) {
    *dst0 = c[0];
    if (n_sets > 1) *dst1 = c[1];
    __threadfence();
    const uint32_t done = atomicAdd(counter, 1u);
    s_last = (done == group_ctas - 1) ? 1u : 0u;
    if (s_last) {
      *counter = 0;
      __threadfence();
    }
  }
  __syncthreads();
  return s_last != 0;
}

__device__ __forceinline__ void pool_init(SurvPool &pool, Cand (*extra)[SCAN_FEATS]) {
  if (threadIdx.x == 0) pool.n = 0;
  if (threadIdx.x < 2 * SCAN_FEATS) {
    Cand c;
    c.f = INT32_MAX;
    c.gain = -INFINITY;
    c.t = INT32_MAX;
    c.dir = 1;
    c.gl = c.hl = c.gr = c.hr = 0;
    c.pad = 0;
    c.pad2 = 0;
    extra[threadIdx.x / SCAN_FEATS][threadIdx.x % SCAN_FEATS] = c;
  }
}

// Find: grid (ceil(F / SCAN_FEATS), n_nodes); warp w scans feature
// blockIdx.x * SCAN_FEATS + w of node blockIdx.y; the last CTA of a node
// writes its split.
template <int NR>
__global__ void __launch_bounds__(SCAN_THREADS) k_find(const int64_t *__restrict__ hist, int32_t n_features,
                                                       int32_t n_bins, SplitParams sp, Cand *__restrict__ cand,
                                                       uint32_t *__restrict__ counters, SplitOut *__restrict__ out) {
  __shared__ SurvPool pool;
  __shared__ Cand extra[2][SCAN_FEATS];
  const int node = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = blockIdx.x * SCAN_FEATS;
  const int f = f0 + warp;
  const int B = n_bins + 1;
  pool_init(pool, extra);
  constexpr int R = (NR > 0) ? NR : 1;
  longlong2 c[R];
  StripInfo si{};
  float wlo = -INFINITY;
  const longlong2 *strip = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)node * n_features + f) * B;
  if (f < n_features) {
    if (NR > 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int s = r * 32 + lane;
        c[r] = s < B ? __ldg(strip + s) : make_longlong2(0, 0);
      }
      si = regs_pass_a<R>(c, n_bins, sp, wlo);
    } else {
      si = stream_pass_a(strip, n_bins, sp, wlo);
    }
  }
  if (lane == 0) pool.warp_lo[0][warp] = wlo;
  __syncthreads();
  float thr = -INFINITY;
  for (int w = 0; w < SCAN_FEATS; ++w) thr = fmaxf(thr, pool.warp_lo[0][w]);
  int overflow = 0;
  if (f < n_features) {
    if (NR > 0) regs_pass_b<R>(c, n_bins, si, sp, thr, warp, 0, pool, overflow);
    else stream_pass_b(strip, n_bins, si, sp, thr, warp, 0, pool, overflow);
    if (__any_sync(0xffffffffu, overflow)) {
      const Cand d = warp_direct_best(strip, n_bins, si, sp, thr, f);
      if (lane == 0) extra[0][warp] = d;
    }
  }
  __syncthreads();
  pool_eval(pool, sp, f0, 1, extra);
  const int nfb = gridDim.x;
  Cand *cn = cand + (int64_t)node * nfb;
  if (cta_publish(pool.best, 1, cn + blockIdx.x, nullptr, counters + node, nfb)) {
    __threadfence();
    if (warp == 0) reduce_nodes_warp(cn, nfb, out + node);
  }
}

// Subtract and find: grid (ceil(F / SCAN_FEATS), n_pairs). Large = Parent -
// Small (stored), then the scan of both strips. Candidates of node 2p
// (small) and 2p+1 (large); the last CTA of pair p writes small_out[p] and
// large_out[p].
template <int NR>
__global__ void __launch_bounds__(SCAN_THREADS) k_subtract_find(
    const int64_t *__restrict__ parent, const int32_t *__restrict__ parent_of, const int64_t *__restrict__ small,
    int64_t *__restrict__ large, int32_t n_features, int32_t n_bins, SplitParams sp, Cand *__restrict__ cand,
    uint32_t *__restrict__ counters, SplitOut *__restrict__ small_out, SplitOut *__restrict__ large_out,
    DevState *st) {
  __shared__ SurvPool pool;
  __shared__ Cand extra[2][SCAN_FEATS];
  const int p = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = blockIdx.x * SCAN_FEATS;
  const int f = f0 + warp;
  const int B = n_bins + 1;
  pool_init(pool, extra);
  constexpr int R = (NR > 0) ? NR : 1;
  longlong2 cs[R], cl[R];
  StripInfo ss{}, sl{};
  float wlo_s = -INFINITY, wlo_l = -INFINITY;
  const int64_t pp = parent_of ? (int64_t)parent_of[p] : p;
  const longlong2 *P = reinterpret_cast<const longlong2 *>(parent) + (pp * n_features + f) * B;
  const longlong2 *S = reinterpret_cast<const longlong2 *>(small) + ((int64_t)p * n_features + f) * B;
  longlong2 *L = reinterpret_cast<longlong2 *>(large) + ((int64_t)p * n_features + f) * B;
  if (f < n_features) {
    bool neg = false;
    if (NR > 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int s = r * 32 + lane;
        cs[r] = s < B ? __ldg(S + s) : make_longlong2(0, 0);
        cl[r] = s < B ? __ldg(P + s) : make_longlong2(0, 0);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int s = r * 32 + lane;
        cl[r] = make_longlong2(cl[r].x - cs[r].x, cl[r].y - cs[r].y);
        neg |= cl[r].y < 0;
        if (s < B) L[s] = cl[r];
      }
      ss = regs_pass_a<R>(cs, n_bins, sp, wlo_s);
      sl = regs_pass_a<R>(cl, n_bins, sp, wlo_l);
    } else {
      for (int s0 = 0; s0 < B; s0 += 256) {
        longlong2 a[8], b[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int s = s0 + r * 32 + lane;
          a[r] = s < B ? __ldg(P + s) : make_longlong2(0, 0);
          b[r] = s < B ? __ldg(S + s) : make_longlong2(0, 0);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int s = s0 + r * 32 + lane;
          const longlong2 d = make_longlong2(a[r].x - b[r].x, a[r].y - b[r].y);
          neg |= d.y < 0;
          if (s < B) L[s] = d;
        }
      }
      __syncwarp();
      ss = stream_pass_a(S, n_bins, sp, wlo_s);
      sl = stream_pass_a(L, n_bins, sp, wlo_l);
    }
    if (neg) raise_err(st, ERRBIT_INCONSISTENT);
  }
  if (lane == 0) {
    pool.warp_lo[0][warp] = wlo_s;
    pool.warp_lo[1][warp] = wlo_l;
  }
  __syncthreads();
  float thr_s = -INFINITY, thr_l = -INFINITY;
  for (int w = 0; w < SCAN_FEATS; ++w) {
    thr_s = fmaxf(thr_s, pool.warp_lo[0][w]);
    thr_l = fmaxf(thr_l, pool.warp_lo[1][w]);
  }
  int ovf_s = 0, ovf_l = 0;
  if (f < n_features) {
    if (NR > 0) {
      regs_pass_b<R>(cs, n_bins, ss, sp, thr_s, warp, 0, pool, ovf_s);
      regs_pass_b<R>(cl, n_bins, sl, sp, thr_l, warp, 1, pool, ovf_l);
    } else {
      stream_pass_b(S, n_bins, ss, sp, thr_s, warp, 0, pool, ovf_s);
      stream_pass_b(L, n_bins, sl, sp, thr_l, warp, 1, pool, ovf_l);
    }
    if (__any_sync(0xffffffffu, ovf_s | ovf_l)) {
      const Cand ds = warp_direct_best(S, n_bins, ss, sp, thr_s, f);
      const Cand dl = warp_direct_best(L, n_bins, sl, sp, thr_l, f);
      if (lane == 0) {
        extra[0][warp] = ds;
        extra[1][warp] = dl;
      }
    }
  }
  __syncthreads();
  pool_eval(pool, sp, f0, 2, extra);
  const int nfb = gridDim.x;
  Cand *cs_base = cand + (int64_t)(2 * p) * nfb;
  Cand *cl_base = cand + (int64_t)(2 * p + 1) * nfb;
  if (cta_publish(pool.best, 2, cs_base + blockIdx.x, cl_base + blockIdx.x, counters + p, nfb)) {
    __threadfence();
    if (warp == 0) reduce_nodes_warp(cs_base, nfb, small_out + p);
    if (warp == 1) reduce_nodes_warp(cl_base, nfb, large_out + p);
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

}  // namespace gbt
