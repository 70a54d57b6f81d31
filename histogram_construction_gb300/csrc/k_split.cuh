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
// GB300 executes FP64 (and 64-bit integer conversions) at a small fraction of
// its FP32 rate, so every candidate is screened in FP32 first, with an upper
// bound on |gain_fp32 - gain_fp64|: a candidate whose upper bound lies below
// another candidate's lower bound cannot be the double-precision argmax and is
// dropped. The few survivors of a CTA are evaluated in double, exactly as the
// definition says, one per thread. The result is bit-identical to evaluating
// every candidate in double.
#pragma once

#include <float.h>

#include "common.cuh"
#include "k_hist.cuh"

namespace gbt {

struct SplitParams {
  double lambda, gamma, inv_sg, inv_sh;
  int64_t h_min;  // smallest quantised H with (double)H * inv_sh >= min_child_weight (and >= 1)
  float lambda_f, gamma_f, gamma_abs_f, inv_sg_f, inv_sh_f;
  int32_t filter;  // 1: FP32 screen enabled (lambda >= 0, finite parameters)
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

// Non-negative 64-bit integer -> float with FP32/integer ALU work only: the
// value is split into three 23-bit chunks, each converted exactly by the
// 2^23 magic-number construction, and recombined by two FMAs (each rounding
// once): relative error below 2 u, u = 2^-24.
__device__ __forceinline__ float u64_to_f32(uint64_t x) {
  const uint32_t c = (uint32_t)x & 0x7FFFFFu;
  const uint32_t b = (uint32_t)(x >> 23) & 0x7FFFFFu;
  const uint32_t a = (uint32_t)(x >> 46);  // < 2^18
  const float fc = __fsub_rn(__int_as_float(0x4B000000u | c), 8388608.0f);
  const float fb = __fsub_rn(__int_as_float(0x4B000000u | b), 8388608.0f);
  const float fa = __fsub_rn(__int_as_float(0x4B000000u | a), 8388608.0f);
  return __fmaf_rn(fa, 70368744177664.0f, __fmaf_rn(fb, 8388608.0f, fc));  // 2^46, 2^23
}

__device__ __forceinline__ float i64_to_f32(int64_t x) {
  const float f = u64_to_f32(x < 0 ? (uint64_t)(-x) : (uint64_t)x);
  return x < 0 ? -f : f;
}

// Signed 64-bit integer -> float for |x| < 2^45: x = hi * 2^23 + lo with
// hi = x >> 23 in [-2^22, 2^22) and lo in [0, 2^23), both converted exactly
// by magic-number constructions (1.5 * 2^23 and 2^23); the FMA rounds once,
// so the relative error is at most u = 2^-24.
__device__ __forceinline__ float i45_to_f32(int64_t x) {
  const int32_t hi = (int32_t)(x >> 23);
  const uint32_t lo = (uint32_t)x & 0x7FFFFFu;
  const float fh = __fsub_rn(__int_as_float(0x4B400000 + hi), 12582912.0f);
  const float fl = __fsub_rn(__int_as_float(0x4B000000u | lo), 8388608.0f);
  return __fmaf_rn(fh, 8388608.0f, fl);
}

// FP32 screen of one candidate: returns (up, lo) with lo <= gain_fp64 <= up.
// Error budget (u = 2^-24): an int64 value converts with relative error 2u,
// the scale product adds u and the float scale u, so each converted value is
// within 4u; a square is within 9u; a denominator (H + lambda, both >= 0)
// within 5u; __fdividef adds at most 2 ulp (4u), so each of the three
// non-negative terms a, b, c is within 18u. The sum, difference, halving and
// subtraction of gamma then stay below 10 u (a + b + c) + 2 u |gamma|. The
// bound used is 2^-19 (a + b + c + |gamma|) = 32 u (...), three times that,
// which also covers the rounding of the bound itself and the double path's
// own 2^-53-scale errors. Values outside [2^-60, 2^60] (possible underflow
// or overflow, __fdividef range) give an infinite bound: such candidates are
// always evaluated in double.
__device__ __forceinline__ void screen_f32(int64_t GL, int64_t HL, int64_t GR, int64_t HR, float Gf2den,
                                           const SplitParams &sp, float &up, float &lo) {
  const float gl = __fmul_rn(i64_to_f32(GL), sp.inv_sg_f);
  const float hl = __fmul_rn(i64_to_f32(HL), sp.inv_sh_f);
  const float gr = __fmul_rn(i64_to_f32(GR), sp.inv_sg_f);
  const float hr = __fmul_rn(i64_to_f32(HR), sp.inv_sh_f);
  const float dl = __fadd_rn(hl, sp.lambda_f), dr = __fadd_rn(hr, sp.lambda_f);
  const float a = __fdividef(__fmul_rn(gl, gl), dl);
  const float b = __fdividef(__fmul_rn(gr, gr), dr);
  const float s = __fsub_rn(__fadd_rn(a, b), Gf2den);
  const float g = __fsub_rn(__fmul_rn(0.5f, s), sp.gamma_f);
  const float mag = __fadd_rn(__fadd_rn(__fadd_rn(a, b), Gf2den), sp.gamma_abs_f);
  const float err = __fmul_rn(mag, 1.9073486328125e-06f);  // 2^-19
  const float rlo = 8.673617379884035e-19f, rhi = 1.152921504606847e+18f;  // 2^-60, 2^60
  const float ag = fabsf(gl), ar = fabsf(gr);
  const bool ok = (ag == 0.f || (ag > rlo && ag < rhi)) && (ar == 0.f || (ar > rlo && ar < rhi)) && dl > rlo &&
                  dr > rlo && dl < rhi && dr < rhi && mag < rhi && (a == 0.f || a > rlo) &&
                  (b == 0.f || b > rlo) && g == g;
  if (ok) {
    up = __fadd_rn(g, err);
    lo = __fsub_rn(g, err);
  } else {
    up = INFINITY;
    lo = -INFINITY;
  }
}

// Parent term G^2/(H+lambda) of the screen in FP32. Outside the checked
// range it is NaN, which gives every candidate of the strip an infinite bound
// (all of them are then evaluated in double).
__device__ __forceinline__ float parent_f32(int64_t tg, int64_t th, const SplitParams &sp) {
  const bool small = tg > -(1LL << 45) && tg < (1LL << 45) && th > -(1LL << 45) && th < (1LL << 45);
  const float Gf = __fmul_rn(small ? i45_to_f32(tg) : i64_to_f32(tg), sp.inv_sg_f);  // both round once
  const float Hf = __fmul_rn(small ? i45_to_f32(th) : i64_to_f32(th), sp.inv_sh_f);
  const float den = __fadd_rn(Hf, sp.lambda_f);
  const float rlo = 8.673617379884035e-19f, rhi = 1.152921504606847e+18f;
  const float ag = fabsf(Gf);
  if (den > rlo && den < rhi && (ag == 0.f || (ag > rlo && ag < rhi))) {
    const float c = __fdividef(__fmul_rn(Gf, Gf), den);
    if (c == 0.f || (c > rlo && c < rhi)) return c;
  }
  return __int_as_float(0x7fc00000);  // NaN: screen_f32 then yields an infinite bound
}


// Whether every candidate of a strip can use screen_fast: all its quantised
// sums are below 2^45 in magnitude (|G| sums are bounded by sabs, the sum of
// |G| over the strip's slots, H sums by th) and every float quantity the
// screen forms stays within [2^-59, 2^59] or is zero: nonzero |gl| >= inv_sg,
// denominators in [inv_sh + lambda, th * inv_sh + lambda] (valid candidates
// have H >= h_min >= 1 on both sides), terms a, b in
// [inv_sg^2 / dmax, gmax^2 / dmin]. The error analysis of screen_f32 then
// holds for every candidate without per-candidate checks.
__device__ __forceinline__ bool strip_fast(int64_t sabs, int64_t th, float Gf2den, const SplitParams &sp) {
  if (!sp.filter || sabs >= (1LL << 45) || th >= (1LL << 45) || !(Gf2den == Gf2den)) return false;
  const float rlo = 1.7347234759768071e-18f, rhi = 5.764607523034235e+17f;  // 2^-59, 2^59
  const float gmax = __fmul_rn(i45_to_f32(sabs), sp.inv_sg_f);
  const float dmax = __fadd_rn(__fmul_rn(i45_to_f32(th), sp.inv_sh_f), sp.lambda_f);
  const float dmin = __fadd_rn(sp.inv_sh_f, sp.lambda_f);
  // range checks with a factor 2 of margin: the approximate division (2 ulp for denominators in
  // [2^-126, 2^126]; a larger dmax already fails its own check) decides nothing differently
  const float amax = __fdividef(__fmul_rn(gmax, gmax), dmin);
  const float amin = __fdividef(__fmul_rn(sp.inv_sg_f, sp.inv_sg_f), dmax);
  return sp.inv_sg_f > rlo && dmin > rlo && gmax < rhi && dmax < rhi && amax < rhi && amin > rlo &&
         __fadd_rn(__fmul_rn(3.0f, amax), sp.gamma_abs_f) < rhi;
}

// Integer -> float, rounded once (relative error at most u): a 32-bit value
// by the conversion instruction, a 64-bit one below 2^45 by i45_to_f32.
__device__ __forceinline__ float to_f32(int32_t x) { return __int2float_rn(x); }
__device__ __forceinline__ float to_f32(int64_t x) { return i45_to_f32(x); }

// screen_f32 for a strip that passed strip_fast (same bound, no range checks).
// I: the integer type of the sums (int32_t when every partial sum of the
// strip fits, which the caller has checked).
template <typename I>
__device__ __forceinline__ void screen_fast(I GL, I HL, I GR, I HR, float Gf2den, const SplitParams &sp, float &up,
                                            float &lo) {
  const float gl = __fmul_rn(to_f32(GL), sp.inv_sg_f);
  const float hl = __fmul_rn(to_f32(HL), sp.inv_sh_f);
  const float gr = __fmul_rn(to_f32(GR), sp.inv_sg_f);
  const float hr = __fmul_rn(to_f32(HR), sp.inv_sh_f);
  const float a = __fdividef(__fmul_rn(gl, gl), __fadd_rn(hl, sp.lambda_f));
  const float b = __fdividef(__fmul_rn(gr, gr), __fadd_rn(hr, sp.lambda_f));
  const float ab = __fadd_rn(a, b);
  const float g = __fsub_rn(__fmul_rn(0.5f, __fsub_rn(ab, Gf2den)), sp.gamma_f);
  const float err = __fmul_rn(__fadd_rn(__fadd_rn(ab, Gf2den), sp.gamma_abs_f), 1.9073486328125e-06f);  // 2^-19
  up = __fadd_rn(g, err);
  lo = __fsub_rn(g, err);
}

// Upper bound on the gain of every valid candidate (HL, HR >= h_min) of a run
// of consecutive cuts of one missing direction in a strip that passed
// strip_fast: gl_mn, gl_mx bound GL over the run (int64, the missing slot
// already added for missing-left), HL rises from hl_a to hl_b. The gain
// term GL^2/(HL + lambda) is largest at the largest |GL| and the smallest
// valid HL, the right term likewise at the largest |G - GL| and the
// smallest valid HR, so screen_fast's upper bound of that (possibly
// unreal) corner candidate bounds every candidate of the run: its inputs
// are sums of subsets of the strip's slots, within strip_fast's ranges.
// I as in screen_fast; hm: h_min in I.
template <typename I>
__device__ __forceinline__ float run_bound(I gl_mn, I gl_mx, I hl_a, I hl_b, I tg, I th, I hm, float Gf2den,
                                           const SplitParams &sp) {
  const I ga = max(gl_mn < 0 ? -gl_mn : gl_mn, gl_mx < 0 ? -gl_mx : gl_mx);
  const I r1 = tg - gl_mn, r2 = tg - gl_mx;
  const I gb = max(r1 < 0 ? -r1 : r1, r2 < 0 ? -r2 : r2);
  const I hl = max(hl_a, hm), hr = max(th - hl_b, hm);
  float up, lo;
  screen_fast<I>(ga, hl, gb, hr, Gf2den, sp, up, lo);
  return up;
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

__device__ __forceinline__ int32_t shfl_i64(int32_t v, int src) { return __shfl_sync(0xffffffffu, v, src); }
__device__ __forceinline__ int32_t shfl_up_i64(int32_t v, int d) { return __shfl_up_sync(0xffffffffu, v, d); }
__device__ __forceinline__ int32_t shfl_xor_i64(int32_t v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }

template <typename I>
__device__ __forceinline__ void warp_incl_scan(I &pg, I &ph) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const I yg = shfl_up_i64(pg, o), yh = shfl_up_i64(ph, o);
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

__device__ __forceinline__ void warp_sum3(int64_t &a, int64_t &b, int64_t &c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += shfl_xor_i64(a, o);
    b += shfl_xor_i64(b, o);
    c += shfl_xor_i64(c, o);
  }
}

// Candidate record (per CTA and node), 64 bytes, 16-byte aligned so that it
// can be read back with four 16-byte loads. An exact candidate carries its
// double gain; a bounded one only the FP32 bounds lo <= gain <= up (for an
// exact one they are the gain rounded down and up).
struct __align__(16) Cand {
  double gain;
  int32_t t, dir;
  int32_t f, exact;
  int64_t gl, hl, gr, hr;
  float up, lo;
};
static_assert(sizeof(Cand) == 64, "Cand is read as four 16-byte words");

struct SplitOut {
  int32_t feature, bin;
  uint8_t default_left;
  uint8_t pad[7];
  double gain;
  int64_t g_left, h_left, g_right, h_right;
};

__device__ __forceinline__ Cand no_cand() {
  Cand c;
  c.gain = -INFINITY;
  c.t = INT32_MAX;
  c.dir = 1;
  c.f = INT32_MAX;
  c.exact = 1;
  c.gl = c.hl = c.gr = c.hr = 0;
  c.up = c.lo = -INFINITY;
  return c;
}

// Fills the bounds of an exact candidate from its double gain.
__device__ __forceinline__ void set_exact(Cand &c, double gain) {
  c.gain = gain;
  c.exact = 1;
  c.lo = __double2float_rd(gain);
  c.up = __double2float_ru(gain);
}

// Total order of candidates: gain desc, then (feature, t, dir) asc.
__device__ __forceinline__ bool cand_better(const Cand &c, const Cand &b) {
  if (c.f == INT32_MAX) return false;
  if (b.f == INT32_MAX) return true;
  if (c.gain != b.gain) return c.gain > b.gain;
  if (c.f != b.f) return c.f < b.f;
  if (c.t != b.t) return c.t < b.t;
  return c.dir < b.dir;
}

__device__ __forceinline__ Cand shfl_xor_cand(const Cand &b, int o) {
  Cand c;
  c.gain = __shfl_xor_sync(0xffffffffu, b.gain, o);
  c.f = __shfl_xor_sync(0xffffffffu, b.f, o);
  c.t = __shfl_xor_sync(0xffffffffu, b.t, o);
  c.dir = __shfl_xor_sync(0xffffffffu, b.dir, o);
  c.gl = shfl_xor_i64(b.gl, o);
  c.hl = shfl_xor_i64(b.hl, o);
  c.gr = shfl_xor_i64(b.gr, o);
  c.hr = shfl_xor_i64(b.hr, o);
  c.exact = __shfl_xor_sync(0xffffffffu, b.exact, o);
  c.up = __shfl_xor_sync(0xffffffffu, b.up, o);
  c.lo = __shfl_xor_sync(0xffffffffu, b.lo, o);
  return c;
}

__device__ __forceinline__ Cand warp_best_cand(Cand b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Cand c = shfl_xor_cand(b, o);
    if (cand_better(c, b)) b = c;
  }
  return b;
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

// A candidate that passed its warp's running screen.
struct Surv {
  int64_t gl, hl, tg, th;
  float up, lo;
  int32_t t;
  int32_t f;
  int16_t dir;
  int16_t node;  // strip set: 0 (small / hist) or 1 (large)
};

constexpr int SCAN_THREADS = 256;
constexpr int SCAN_WARPS = SCAN_THREADS / 32;
constexpr int SURV_CAP = 256;
constexpr int SCAN_SPL = 4;  // consecutive slots per lane in the warp scan
constexpr int PUB_K = 2;     // candidates a CTA publishes per node set before it resorts to double
constexpr int STAGE_SLOTS = 256;  // strips with B <= 256 are staged in shared memory

// Position of slot s in a staged strip: slots are permuted within aligned
// blocks of 8 cells (16 bytes each) so that both shared-memory access
// patterns of a warp are free of bank conflicts: lane l reading slot 4l + i
// (the scan: four consecutive slots per lane) and lane l reading slot l + 32k.
__device__ __forceinline__ int swz(int s) { return (s & ~7) | ((s & 7) ^ ((s >> 3) & 7)); }

struct ScanShared {
  longlong2 cells[SCAN_WARPS][STAGE_SLOTS];
  Surv pool[SURV_CAP];
  double gain[SURV_CAP];
  float warp_lo[SCAN_WARPS];
  int warp_overflow[SCAN_WARPS];
  Cand extra[SCAN_WARPS];
  Cand pub[2][PUB_K];
  int sel[2][PUB_K];
  int cnt[2];
  float red[SCAN_WARPS];
  int rcnt[2];  // candidates evaluated by each half's node reduce
  int64_t ptot[SCAN_WARPS][4][4];  // long strips: each warp's share of the small strips' (G, H, |G|, H < 0)
  int n;
  uint32_t last;
};

// Warp scan of one strip of `cells` (shared or global memory; missing cell at
// n_bins) with totals (tg, th): screens every candidate and pushes into the
// CTA pool those whose upper bound reaches the best lower bound seen so far.
// Lane l takes the SCAN_SPL consecutive slots of each (32 * SCAN_SPL)-slot
// chunk: prefix sums run in registers, with one warp scan of the lane totals
// per chunk. ND: directions scanned (1 when the missing slot is empty: both
// directions then give the same sums, and missing-right comes first, so the
// left direction can never win); mode 0: screen_fast, 1: screen_f32, 2: no
// screen (every valid candidate pushed with an infinite upper bound); MODE
// fixes it at compile time, or -1 takes `mode`.

// Lane partial sums (G, H, |G|) of a strip in global memory, FIN_BATCH loads
// in flight per lane (a loop that used each load at once would wait for every
// one of them in turn).
constexpr int FIN_BATCH = 8;
__device__ __forceinline__ void strip_totals(const longlong2 *cells, int B, int64_t &tg, int64_t &th, int64_t &sa,
                                             bool &hneg) {
  const int lane = threadIdx.x & 31;
  for (int s0 = lane; s0 < B; s0 += 32 * FIN_BATCH) {
    longlong2 c[FIN_BATCH];
#pragma unroll
    for (int u = 0; u < FIN_BATCH; ++u) {
      const int s = s0 + 32 * u;
      c[u] = s < B ? cells[s] : make_longlong2(0, 0);
    }
#pragma unroll
    for (int u = 0; u < FIN_BATCH; ++u) {
      tg += c[u].x;
      th += c[u].y;
      sa += c[u].x < 0 ? -c[u].x : c[u].x;
      hneg |= c[u].y < 0;
    }
  }
}

// A cut t > 0 whose own cell is empty has the sums of cut t - 1 (in both
// missing directions), so its gain equals that earlier candidate's and the
// serial order never picks it: such cuts are skipped (runs of empty bins would
// otherwise flood the survivor pool with exact ties).
//
// SKIP (long strips under the fast screen): a chunk is skipped whole when an
// upper bound on all its candidates (run_bound) lies below the best lower
// bound found so far by the warps of the same node set in this CTA
// (set_warps warps from the set's first, each publishing its running bound
// in sh.warp_lo). Every skipped candidate's gain is then strictly below
// another candidate's, so it cannot be chosen.
// I: the integer type of the prefix sums (int32_t only under the fast screen,
// when every partial sum of the strip fits: fewer instructions per cut).
template <int ND, int MODE, bool SKIP, typename I>
__device__ __forceinline__ float scan_push_impl(const longlong2 *cells, bool sw, int n_bins, int64_t tg64, int64_t th64,
                                                longlong2 m64, float Gf2den, const SplitParams &sp, int f, int node,
                                                ScanShared &sh, int &overflow, int mode, int set_warps, float lo0) {
  if (MODE >= 0) mode = MODE;
  const I tg = (I)tg64, th = (I)th64, h_min = (I)sp.h_min;  // exact: the caller checked the range for int32_t
  struct {
    I x, y;
  } m = {(I)m64.x, (I)m64.y};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sw0 = warp - warp % set_warps;
  volatile float *vlo = sh.warp_lo;
  float run_lo = lo0;  // a lower bound of a candidate of the same node set, found earlier (or -inf)
  I carry_g = 0, carry_h = 0;
  if (!__isShared(cells))
    asm volatile("prefetch.global.L1 [%0];" ::"l"(cells + min(32 * SCAN_SPL + SCAN_SPL * lane, n_bins)));
  for (int c0 = 0; c0 < n_bins; c0 += 32 * SCAN_SPL) {
    // the next chunk's cells on their way to L1 while this chunk is screened
    // (strips in global memory: u16 bins)
    // (clamped to the strip's missing slot: the address stays inside the strip)
    if (c0 + 32 * SCAN_SPL < n_bins && !__isShared(cells))
      asm volatile("prefetch.global.L1 [%0];" ::"l"(cells + min(c0 + 2 * 32 * SCAN_SPL + SCAN_SPL * lane, n_bins)));
    I pg[SCAN_SPL], ph[SCAN_SPL];
    I ag = 0, ah = 0;
    uint32_t nzmask = 0;  // slots of the lane whose cell is not empty
#pragma unroll
    for (int i = 0; i < SCAN_SPL; ++i) {
      const int s = c0 + SCAN_SPL * lane + i;
      longlong2 c = make_longlong2(0, 0);
      if (s < n_bins) c = cells[sw ? swz(s) : s];
      const I cx = (I)c.x, cy = (I)c.y;
      ag += cx;
      ah += cy;
      pg[i] = ag;
      ph[i] = ah;
      nzmask |= ((cx | cy) != 0 || s == 0) ? (1u << i) : 0u;  // cut 0 has no earlier twin
    }
    I eg = ag, eh = ah;
    warp_incl_scan<I>(eg, eh);
    const I tot_g = shfl_i64(eg, 31), tot_h = shfl_i64(eh, 31);
    eg += carry_g - ag;  // exclusive prefix of the lane's first slot
    eh += carry_h - ah;
    const I h_a = carry_h;  // HL over the chunk's cuts lies in [h_a, h_b]
    carry_g += tot_g;
    carry_h += tot_h;
    if (SKIP && MODE == 0) {
      float sthr = run_lo;
      for (int w = 0; w < set_warps; ++w) sthr = fmaxf(sthr, vlo[sw0 + w]);
      if (sthr > -INFINITY) {
        I mn = eg + pg[0], mx = mn;
#pragma unroll
        for (int i = 1; i < SCAN_SPL; ++i) {
          mn = min(mn, eg + pg[i]);
          mx = max(mx, eg + pg[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          mn = min(mn, shfl_xor_i64(mn, o));
          mx = max(mx, shfl_xor_i64(mx, o));
        }
        float ub = run_bound<I>(mn, mx, h_a, carry_h, tg, th, h_min, Gf2den, sp);
        if (ND == 2)
          ub = fmaxf(ub, run_bound<I>(mn + m.x, mx + m.x, h_a + m.y, carry_h + m.y, tg, th, h_min, Gf2den, sp));
        if (ub < sthr) continue;  // no candidate of the chunk can reach the set's best
      }
    }
    float up[SCAN_SPL][ND], lo[SCAN_SPL][ND];
    uint32_t vmask = 0;
    float l = -INFINITY;
#pragma unroll
    for (int i = 0; i < SCAN_SPL; ++i) {
      const int s = c0 + SCAN_SPL * lane + i;
#pragma unroll
      for (int dir = 0; dir < ND; ++dir) {
        const I GL = eg + pg[i] + (dir ? m.x : 0), HL = eh + ph[i] + (dir ? m.y : 0);
        const I HR = th - HL;
        const bool valid = s < n_bins && ((nzmask >> i) & 1u) && HL >= h_min && HR >= h_min &&
                           !(ND == 2 && dir && m.x == 0 && m.y == 0);
        float u = -INFINITY, lw = -INFINITY;
        if (valid) {
          if (mode == 0) screen_fast<I>(GL, HL, tg - GL, HR, Gf2den, sp, u, lw);
          else if (mode == 1) screen_f32(GL, HL, tg - GL, HR, Gf2den, sp, u, lw);
          else u = INFINITY;
          vmask |= 1u << (2 * i + dir);
        }
        up[i][dir] = u;
        lo[i][dir] = lw;
        l = fmaxf(l, lw);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
    if (l > run_lo) {
      run_lo = l;
      if (SKIP && MODE == 0 && lane == 0) vlo[warp] = run_lo;  // the other warps of the set may skip by it
    }
#pragma unroll
    for (int i = 0; i < SCAN_SPL; ++i) {
#pragma unroll
      for (int dir = 0; dir < ND; ++dir) {
        if (!((vmask >> (2 * i + dir)) & 1u) || up[i][dir] < run_lo) continue;
        const int idx = atomicAdd(&sh.n, 1);
        if (idx >= SURV_CAP) {
          overflow = 1;
          continue;
        }
        Surv v;
        v.gl = (int64_t)(eg + pg[i] + (dir ? m.x : 0));
        v.hl = (int64_t)(eh + ph[i] + (dir ? m.y : 0));
        v.tg = tg64;
        v.th = th64;
        v.up = up[i][dir];
        v.lo = lo[i][dir];
        v.t = c0 + SCAN_SPL * lane + i;
        v.f = f;
        v.dir = (int16_t)dir;
        v.node = (int16_t)node;
        sh.pool[idx] = v;
      }
    }
  }
  return run_lo;
}

// sabs: the sum of |G| over the strip's slots (for the range check of the fast screen).
// sw: a staged strip (shared memory, slot s at swz(s)).
// The checked screen and the unscreened scan (rare: extreme ranges, lambda < 0), out of line so that
// their registers do not weigh on the common copies.
__device__ __noinline__ float scan_push_checked(const longlong2 *cells, bool sw, int n_bins, int64_t tg, int64_t th,
                                                longlong2 m, float Gf2den, const SplitParams &sp, int f, int node,
                                                ScanShared &sh, int &overflow, int set_warps, float lo0) {
  return scan_push_impl<2, -1, false, int64_t>(cells, sw, n_bins, tg, th, m, Gf2den, sp, f, node, sh, overflow,
                                               sp.filter ? 1 : 2, set_warps, lo0);
}

// h_ok: no H cell of the strip is negative (then every partial sum of H lies
// in [0, th] and of G in [-sabs, sabs], and the 32-bit scan is exact when
// th, sabs and h_min are below 2^31).
__device__ __forceinline__ float warp_scan_push(const longlong2 *cells, bool sw, int n_bins, int64_t tg, int64_t th,
                                                int64_t sabs, bool h_ok, const SplitParams &sp, int f, int node,
                                                ScanShared &sh, int &overflow, int set_warps,
                                                float lo0 = -INFINITY) {
  const longlong2 m = cells[sw ? swz(n_bins) : n_bins];
  const bool no_missing = (m.x == 0 && m.y == 0);
  const float Gf2den = parent_f32(tg, th, sp);
  const bool fast = strip_fast(sabs, th, Gf2den, sp);
  const bool i32 = h_ok && sabs < (1LL << 31) && th < (1LL << 31) && sp.h_min < (1LL << 31);
  // the common cases (fast screen, with or without missing values) get their own copies; chunk
  // skipping only pays on long strips (in global memory): a staged strip has two chunks
#define GBT_SCAN(ND, MODE, SKIP, I, mode) \
  scan_push_impl<ND, MODE, SKIP, I>(cells, sw, n_bins, tg, th, m, Gf2den, sp, f, node, sh, overflow, mode, set_warps, \
                                    lo0)
  if (fast && no_missing) {
    if (sw) return i32 ? GBT_SCAN(1, 0, false, int32_t, 0) : GBT_SCAN(1, 0, false, int64_t, 0);
    return i32 ? GBT_SCAN(1, 0, true, int32_t, 0) : GBT_SCAN(1, 0, true, int64_t, 0);
  }
  if (fast) {
    if (sw) return i32 ? GBT_SCAN(2, 0, false, int32_t, 0) : GBT_SCAN(2, 0, false, int64_t, 0);
    return i32 ? GBT_SCAN(2, 0, true, int32_t, 0) : GBT_SCAN(2, 0, true, int64_t, 0);
  }
  return scan_push_checked(cells, sw, n_bins, tg, th, m, Gf2den, sp, f, node, sh, overflow, set_warps, lo0);
#undef GBT_SCAN
}

__device__ __forceinline__ double surv_gain(int64_t gl, int64_t hl, int64_t tg, int64_t th, const SplitParams &sp) {
  const double gld = __dmul_rn(__ll2double_rn(gl), sp.inv_sg);
  const double hld = __dmul_rn(__ll2double_rn(hl), sp.inv_sh);
  const double grd = __dmul_rn(__ll2double_rn(tg - gl), sp.inv_sg);
  const double hrd = __dmul_rn(__ll2double_rn(th - hl), sp.inv_sh);
  const double Gd = __dmul_rn(__ll2double_rn(tg), sp.inv_sg);
  const double Hd = __dmul_rn(__ll2double_rn(th), sp.inv_sh);
  return split_gain(gld, hld, grd, hrd, Gd, Hd, sp);
}

// Overflow path (more pushes than the pool holds, e.g. very many exact
// ties): the warp re-scans its strip and evaluates every candidate whose
// upper bound reaches thr in double itself.
__device__ __noinline__ Cand warp_direct_best(const longlong2 *cells, bool sw, int n_bins, int64_t tg, int64_t th,
                                              const SplitParams &sp, float thr, int f) {
  const int lane = threadIdx.x & 31;
  const longlong2 m = cells[sw ? swz(n_bins) : n_bins];
  const float Gf2den = parent_f32(tg, th, sp);
  Cand best = no_cand();
  int64_t cg = 0, ch = 0;
  for (int s0 = 0; s0 < n_bins; s0 += 32) {
    const int s = s0 + lane;
    int64_t pg = 0, ph = 0;
    if (s < n_bins) {
      const longlong2 c = cells[sw ? swz(s) : s];
      pg = c.x;
      ph = c.y;
    }
    warp_incl_scan(pg, ph);
    pg += cg;
    ph += ch;
    cg = shfl_i64(pg, 31);
    ch = shfl_i64(ph, 31);
#pragma unroll
    for (int dir = 0; dir < 2; ++dir) {
      const int64_t GL = pg + (dir ? m.x : 0), HL = ph + (dir ? m.y : 0);
      const int64_t HR = th - HL;
      if (!(s < n_bins && HL >= sp.h_min && HR >= sp.h_min)) continue;
      float up = INFINITY, lo = -INFINITY;
      if (sp.filter) screen_f32(GL, HL, tg - GL, HR, Gf2den, sp, up, lo);
      if (up < thr) continue;
      Cand c;
      set_exact(c, surv_gain(GL, HL, tg, th, sp));
      c.t = s;
      c.dir = dir;
      c.f = f;
      c.gl = GL;
      c.hl = HL;
      c.gr = tg - GL;
      c.hr = th - HL;
      if (cand_better(c, best)) best = c;
    }
  }
  return warp_best_cand(best);
}

__device__ __forceinline__ Cand surv_cand(const Surv &v) {
  Cand c;
  c.gain = -INFINITY;
  c.t = v.t;
  c.dir = v.dir;
  c.f = v.f;
  c.exact = 0;
  c.gl = v.gl;
  c.hl = v.hl;
  c.gr = v.tg - v.gl;
  c.hr = v.th - v.hl;
  c.up = v.up;
  c.lo = v.lo;
  return c;
}

// What a CTA publishes for each node set, after the scan and the overflow
// pass (thr[set]: the set's best lower bound in the CTA). Candidates that can
// still be the node's best are the pool survivors with up >= thr plus the
// exact results of warps whose pushes overflowed the pool. Up to PUB_K of
// them are published with their bounds, with no double work in this CTA;
// with more, they are evaluated in double and the exact best is published.
// All threads call it; sh.pub[set][0 .. PUB_K-1] holds the result. Warp w
// scanned a strip of set w >> set_shift. The thresholds come by value: an
// array whose address a call takes lives in local memory, whose lines the
// long strips' streaming evicts (each access then a DRAM round trip).
__device__ __noinline__ void cta_select(ScanShared &sh, const SplitParams &sp, int n_sets, float thr0, float thr1,
                                        int set_shift) {
  const int n = min(sh.n, SURV_CAP);
  if (threadIdx.x < 2) sh.cnt[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const Surv &v = sh.pool[i];
    if (v.up >= (v.node == 0 ? thr0 : thr1)) {
      const int k = atomicAdd(&sh.cnt[v.node], 1);
      if (k < PUB_K) sh.sel[v.node][k] = i;
    }
  }
  if (threadIdx.x < SCAN_WARPS && sh.warp_overflow[threadIdx.x] && sh.extra[threadIdx.x].f != INT32_MAX) {
    const int set = (int)threadIdx.x >> set_shift;
    const int k = atomicAdd(&sh.cnt[set], 1);
    if (k < PUB_K) sh.sel[set][k] = -1 - (int)threadIdx.x;
  }
  __syncthreads();
  const bool dbl0 = sh.cnt[0] > PUB_K, dbl1 = n_sets > 1 && sh.cnt[1] > PUB_K;
  if (dbl0 || dbl1) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const Surv &v = sh.pool[i];
      const bool need = (v.node == 0 ? dbl0 : dbl1) && v.up >= (v.node == 0 ? thr0 : thr1);
      sh.gain[i] = need ? surv_gain(v.gl, v.hl, v.tg, v.th, sp) : -INFINITY;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < n_sets && (warp == 0 ? dbl0 : dbl1)) {
      Cand best = no_cand();
      for (int i = lane; i < n; i += 32) {
        const Surv &v = sh.pool[i];
        if (v.node != warp || !(v.up >= (warp == 0 ? thr0 : thr1))) continue;
        Cand c = surv_cand(v);
        set_exact(c, sh.gain[i]);
        if (cand_better(c, best)) best = c;
      }
      for (int w = lane; w < SCAN_WARPS; w += 32)
        if ((w >> set_shift) == warp && sh.warp_overflow[w] && cand_better(sh.extra[w], best)) best = sh.extra[w];
      best = warp_best_cand(best);
      if (lane < PUB_K) sh.pub[warp][lane] = lane == 0 ? best : no_cand();
    }
  }
  if (threadIdx.x < n_sets * PUB_K) {
    const int set = threadIdx.x / PUB_K, k = threadIdx.x % PUB_K;
    if (!(set == 0 ? dbl0 : dbl1)) {
      Cand c = no_cand();
      if (k < sh.cnt[set]) {
        const int i = sh.sel[set][k];
        c = i >= 0 ? surv_cand(sh.pool[i]) : sh.extra[-1 - i];
      }
      sh.pub[set][k] = c;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ Cand load_cand(const Cand *p) {
  Cand c;
  const int4 *src = reinterpret_cast<const int4 *>(p);  // L2 reads: written by other CTAs
  int4 *dst = reinterpret_cast<int4 *>(&c);
#pragma unroll
  for (int k = 0; k < 4; ++k) dst[k] = __ldcg(src + k);
  return c;
}

// Order-preserving key of a float (larger float, larger key; 0 is below every
// finite or infinite value) for atomicMax over lower bounds.
__device__ __forceinline__ uint32_t lo_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_lo(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp argmax in the order of cand_better on the keys alone (gain bits,
// feature, slot and direction); returns the lane holding the best record.
__device__ __forceinline__ int warp_argmax_lane(const Cand &best) {
  double g = best.gain;
  int f = best.f, td = best.f == INT32_MAX ? INT32_MAX : best.t * 2 + best.dir;
  const int my_td = td;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double og = __shfl_xor_sync(0xffffffffu, g, o);
    const int of = __shfl_xor_sync(0xffffffffu, f, o), otd = __shfl_xor_sync(0xffffffffu, td, o);
    const bool better = of != INT32_MAX &&
                        (f == INT32_MAX || (og != g ? og > g : (of != f ? of < f : otd < td)));
    if (better) {
      g = og;
      f = of;
      td = otd;
    }
  }
  const bool mine = best.f == f && my_td == td && __double_as_longlong(best.gain) == __double_as_longlong(g);
  return __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
}

// Node reduce by the nthr threads from t0 (whole warps, named barrier `bar`)
// over the n_ent published candidates of one node. The node threshold is the
// best published lower bound; candidates whose upper bound reaches it are
// evaluated in double (unless exact already) and the best one is written to
// out. slot: nthr / 32 Cand of shared scratch, sthr: nthr / 32 floats.
// With rcnt (a shared counter) and at most one entry per thread, each thread reads its record once, the
// block settles the threshold, and a short list takes the argmax of the few evaluated records.
__device__ __forceinline__ void reduce_node(const Cand *cand, int n_ent, const SplitParams &sp, SplitOut *out,
                                            int t0, int nthr, int bar, Cand *slot, float *sthr, int *rcnt = nullptr) {
  const int t = threadIdx.x - t0, lane = threadIdx.x & 31, w = t >> 5, nw = nthr >> 5;
  if (rcnt && n_ent <= nthr) {
    Cand c = t < n_ent ? load_cand(cand + t) : no_cand();
    float thr = c.lo;  // -inf for no record
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, o));
    if (lane == 0) sthr[w] = thr;
    if (t == 0) *rcnt = 0;
    named_sync(bar, nthr);
    for (int k = 0; k < nw; ++k) thr = fmaxf(thr, sthr[k]);
    const bool take = c.f != INT32_MAX && c.up >= thr;
    if (take) {
      if (!c.exact) set_exact(c, surv_gain(c.gl, c.hl, c.gl + c.gr, c.hl + c.hr, sp));
      const int k = atomicAdd(rcnt, 1);
      if (k < nw) slot[k] = c;
    }
    named_sync(bar, nthr);
    const int nc = *rcnt;
    if (nc <= nw) {
      if (t == 0) {
        Cand b = no_cand();
        for (int k = 0; k < nc; ++k)
          if (cand_better(slot[k], b)) b = slot[k];
        *out = cand_to_split(b);
      }
      return;
    }
    named_sync(bar, nthr);  // every thread has read the count before the list is overwritten
    const Cand best = take ? c : no_cand();
    if (lane == warp_argmax_lane(best)) slot[w] = best;
    named_sync(bar, nthr);
    if (w == 0) {
      const Cand b = lane < nw ? slot[lane] : no_cand();
      if (lane == warp_argmax_lane(b)) *out = cand_to_split(b);
    }
    return;
  }
  constexpr int RB = 8;  // loads in flight per thread
  float thr = -INFINITY;
  for (int i0 = t; i0 < n_ent; i0 += nthr * RB) {
    float v[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int i = i0 + u * nthr;
      v[u] = i < n_ent ? __int_as_float(__ldcg(reinterpret_cast<const int4 *>(cand + i) + 3).w) : -INFINITY;  // lo
    }
#pragma unroll
    for (int u = 0; u < RB; ++u) thr = fmaxf(thr, v[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, o));
  if (lane == 0) sthr[w] = thr;
  named_sync(bar, nthr);
  for (int k = 0; k < nw; ++k) thr = fmaxf(thr, sthr[k]);
  Cand best = no_cand();
  for (int i0 = t; i0 < n_ent; i0 += nthr * RB) {
    float up[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int i = i0 + u * nthr;
      // past the node's entries: NaN, which never passes the test below (no load beyond the entries)
      up[u] = i < n_ent ? __int_as_float(__ldcg(reinterpret_cast<const int4 *>(cand + i) + 3).z)
                        : __int_as_float(0x7fc00000);
    }
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      if (!(up[u] >= thr)) continue;
      Cand c = load_cand(cand + i0 + u * nthr);
      if (c.f == INT32_MAX) continue;
      if (!c.exact) set_exact(c, surv_gain(c.gl, c.hl, c.gl + c.gr, c.hl + c.hr, sp));
      if (cand_better(c, best)) best = c;
    }
  }
  if (lane == warp_argmax_lane(best)) slot[w] = best;
  named_sync(bar, nthr);
  if (w == 0) {
    const Cand b = lane < nw ? slot[lane] : no_cand();
    if (lane == warp_argmax_lane(b)) *out = cand_to_split(b);
  }
}

// reduce_node for published entries whose bounds are also stored compactly,
// cb[i] = (lo, up) of entry i (n_ent even, cb 16-byte aligned): both passes
// read 8 bytes per entry, two entries per 16-byte load, and only the entries
// whose upper bound reaches the threshold are read in full.
// BAR, the named barrier, is a compile-time constant so that a kernel reserves only the barriers it
// uses, also when the call stays out of line (reduce_node_cb_ool).
template <int BAR>
__device__ __forceinline__ void reduce_node_cb(const Cand *cand, const float2 *cb, int n_ent, const SplitParams &sp,
                                               SplitOut *out, int t0, int nthr, Cand *slot, float *sthr, int *rcnt) {
  constexpr int bar = BAR;
  const int t = threadIdx.x - t0, lane = threadIdx.x & 31, w = t >> 5, nw = nthr >> 5;
  constexpr int RB = 8;  // 16-byte loads in flight per thread
  const float4 *cb4 = reinterpret_cast<const float4 *>(cb);
  const int n4 = n_ent >> 1;
  const bool one = n4 <= nthr;  // each thread holds at most one pair of entries: kept in registers
  float thr = -INFINITY;
  float4 v1 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  if (one) {
    if (t < n4) v1 = __ldcg(cb4 + t);
    thr = fmaxf(v1.x, v1.z);
  } else {
    for (int i0 = t; i0 < n4; i0 += nthr * RB) {
      float4 v[RB];
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        const int i = i0 + u * nthr;
        v[u] = i < n4 ? __ldcg(cb4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < RB; ++u) thr = fmaxf(thr, fmaxf(v[u].x, v[u].z));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, o));
  // the entry of this pair with the larger upper bound, read in full already if it reaches the warp's
  // best lower bound (the node's threshold is at least that): the load overlaps the barrier
  const int se = v1.w > v1.y ? 1 : 0;
  const bool spec = one && t < n4 && (se ? v1.w : v1.y) >= thr;
  Cand cs;
  if (spec) cs = load_cand(cand + 2 * t + se);
  if (lane == 0) sthr[w] = thr;
  if (t == 0) *rcnt = 0;
  named_sync(bar, nthr);
  for (int k = 0; k < nw; ++k) thr = fmaxf(thr, sthr[k]);
  Cand best = no_cand();
  auto consider = [&](Cand c) {
    if (c.f == INT32_MAX) return;
    if (!c.exact) set_exact(c, surv_gain(c.gl, c.hl, c.gl + c.gr, c.hl + c.hr, sp));
    if (cand_better(c, best)) best = c;
  };
  if (one) {
    if (t < n4)
      for (int e = 0; e < 2; ++e)
        if ((e ? v1.w : v1.y) >= thr) consider(spec && e == se ? cs : load_cand(cand + 2 * t + e));
  } else {
    for (int i0 = t; i0 < n4; i0 += nthr * RB) {
      uint32_t pass = 0;  // bit 2u + e: entry 2 (i0 + u nthr) + e reaches the threshold
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        const int i = i0 + u * nthr;
        if (i < n4) {
          const float4 x = __ldcg(cb4 + i);
          pass |= (x.y >= thr ? 1u : 0u) << (2 * u);
          pass |= (x.w >= thr ? 1u : 0u) << (2 * u + 1);
        }
      }
      // one copy of the evaluation, however many entries pass
      while (pass) {
        const int b = __ffs(pass) - 1;
        pass &= pass - 1u;
        consider(load_cand(cand + 2 * (i0 + (b >> 1) * nthr) + (b & 1)));
      }
    }
  }
  // the argmax: a short list when few candidates were evaluated (the usual case), else warp shuffles
  if (best.f != INT32_MAX) {
    const int k = atomicAdd(rcnt, 1);
    if (k < nw) slot[k] = best;
  }
  named_sync(bar, nthr);
  const int nc = *rcnt;
  if (nc <= nw) {
    if (t == 0) {
      Cand b = no_cand();
      for (int k = 0; k < nc; ++k)
        if (cand_better(slot[k], b)) b = slot[k];
      *out = cand_to_split(b);
    }
    return;
  }
  named_sync(bar, nthr);  // every thread has read the count before the list is overwritten
  if (lane == warp_argmax_lane(best)) slot[w] = best;
  named_sync(bar, nthr);
  if (w == 0) {
    const Cand b = lane < nw ? slot[lane] : no_cand();
    if (lane == warp_argmax_lane(b)) *out = cand_to_split(b);
  }
}

// reduce_node_cb out of line: only the last CTA of a node runs it, so in a kernel budgeted for many
// CTAs per SM its registers need not weigh on the other CTAs (a one-wave grid keeps it inline: the
// call would lengthen the critical path).
template <int BAR>
__device__ __noinline__ void reduce_node_cb_ool(const Cand *cand, const float2 *cb, int n_ent, const SplitParams &sp,
                                                SplitOut *out, int t0, int nthr, Cand *slot, float *sthr, int *rcnt) {
  reduce_node_cb<BAR>(cand, cb, n_ent, sp, out, t0, nthr, slot, sthr, rcnt);
}

// Stores the CTA's published candidates (dst[set] + 0 .. PUB_K-1), and their
// bounds (lo, up) in cb[set] + 0 .. PUB_K-1 when cb0 is given, and counts the
// CTA in; returns true in the last CTA of the group, which resets the
// counter. No CTA waits. Ordering: the stores precede the block barrier,
// which precedes thread 0's acquire-release increment (a release that covers
// what the barrier ordered before it); in the last CTA that increment
// acquires every other CTA's release, and the second barrier orders the
// block's later reads after it.
__device__ __forceinline__ bool cta_publish(ScanShared &sh, int n_sets, Cand *dst0, Cand *dst1, uint32_t *counter,
                                            uint32_t group_ctas, float2 *cb0 = nullptr, float2 *cb1 = nullptr) {
  if (threadIdx.x < n_sets * PUB_K) {
    const int set = threadIdx.x / PUB_K, k = threadIdx.x % PUB_K;
    const Cand &c = sh.pub[set][k];
    (set == 0 ? dst0 : dst1)[k] = c;
    if (cb0) (set == 0 ? cb0 : cb1)[k] = make_float2(c.lo, c.up);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t done;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(done) : "l"(counter) : "memory");
    sh.last = (done == group_ctas - 1) ? 1u : 0u;
    if (sh.last) *counter = 0;  // every CTA of the group has counted in
  }
  __syncthreads();
  return sh.last != 0;
}

__device__ __forceinline__ void scan_init(ScanShared &sh) {
  if (threadIdx.x == 0) sh.n = 0;
  if (threadIdx.x < SCAN_WARPS) {
    sh.extra[threadIdx.x] = no_cand();
    sh.warp_overflow[threadIdx.x] = 0;
    sh.warp_lo[threadIdx.x] = -INFINITY;
  }
  __syncthreads();
}

// Find: grid (ceil(F / SCAN_WARPS), n_nodes); warp w scans feature
// blockIdx.x * SCAN_WARPS + w of node blockIdx.y; the last CTA of a node
// writes its split.
__global__ void __launch_bounds__(SCAN_THREADS, 3) k_find(const int64_t *__restrict__ hist, int32_t n_features,
                                                       int32_t n_bins, SplitParams sp, Cand *__restrict__ cand,
                                                       uint32_t *__restrict__ counters, SplitOut *__restrict__ out) {
  __shared__ ScanShared sh;
  pdl_wait();  // the kernel that wrote hist, when launched as its dependent (a no-op otherwise)
  const int node = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * SCAN_WARPS + warp;
  const int B = n_bins + 1;
  const bool staged = B <= STAGE_SLOTS;
  scan_init(sh);
  const longlong2 *strip = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)node * n_features + f) * B;
  const longlong2 *cells = staged ? sh.cells[warp] : strip;
  int64_t tg = 0, th = 0;
  if (f < n_features) {
    int64_t sa = 0;
    bool hneg = false;
    if (staged) {
      for (int s = lane; s < B; s += 32) {
        const longlong2 c = __ldg(strip + s);
        sh.cells[warp][swz(s)] = c;
        tg += c.x;
        th += c.y;
        sa += c.x < 0 ? -c.x : c.x;
        hneg |= c.y < 0;
      }
    } else {
      strip_totals(strip, B, tg, th, sa, hneg);
    }
    warp_sum3(tg, th, sa);
    const bool h_ok = !__any_sync(0xffffffffu, hneg);
    __syncwarp();
    int ovf = 0;
    const float wlo = warp_scan_push(cells, staged, n_bins, tg, th, sa, h_ok, sp, f, 0, sh, ovf, SCAN_WARPS);
    ovf = __any_sync(0xffffffffu, ovf);
    if (lane == 0) {
      sh.warp_lo[warp] = wlo;
      sh.warp_overflow[warp] = ovf;
    }
  }
  __syncthreads();
  float thr0 = -INFINITY;
#pragma unroll
  for (int w = 0; w < SCAN_WARPS; ++w) thr0 = fmaxf(thr0, sh.warp_lo[w]);
  if (f < n_features && sh.warp_overflow[warp]) {
    const Cand d = warp_direct_best(cells, staged, n_bins, tg, th, sp, thr0, f);
    if (lane == 0) sh.extra[warp] = d;
  }
  __syncthreads();
  cta_select(sh, sp, 1, thr0, -INFINITY, 3);
  const int nfb = gridDim.x;
  Cand *cn = cand + (int64_t)node * nfb * PUB_K;
  if (cta_publish(sh, 1, cn + blockIdx.x * PUB_K, nullptr, counters + node, nfb)) {
    reduce_node(cn, nfb * PUB_K, sp, out + node, 0, SCAN_THREADS, 1, sh.extra, sh.red, sh.rcnt);
  }
}

// Where the small sibling's histogram comes from in the level-finish kernel.
struct SmallSource {
  const int64_t *hist;  // complete small histograms [n_pairs][F][B][2] (FROM_PARTIALS = false)
  // group images of the level build (FROM_PARTIALS = true); the summed small
  // histogram is also written to `hist_out`
  PartialView view;
  int32_t item_feats;
  int32_t pad;
  int64_t *hist_out;
};

// Level finish: grid (ceil(F / (4 PASSES)), n_pairs), 8 warps. In pass k,
// warp w takes feature (blockIdx.x * PASSES + k) * 4 + (w & 3) of pair
// blockIdx.y; warps 0-3 form the small sibling's strip (read, or summed from
// the build's chunk partials and written out), warps 4-7 load the parent
// strip and form Large = Parent - Small (written out). Every warp then scans
// its strip; after the last pass the CTA selects and publishes once, and the
// last CTA of pair p writes small_out[p] and large_out[p]. With node_side (node order), pair
// p's outputs go to node 2p + node_side[p] (small) and 2p + 1 - node_side[p] (large) of
// one level array instead (the small histogram's own index, small_out and
// hist_out, and large / large_out then name the same arrays).
// STAGED: the instance for B <= STAGE_SLOTS (strips in shared memory), compiled
// without the long-strip paths. CTAS: resident CTAs per SM the registers are
// budgeted for (4 pays when the grid is several waves: more warps hide the
// latency of each CTA's chain; 3 keeps a one-wave grid's chains shorter).
// PASSES: groups of four features per CTA, taken one after the other (the
// selection, publication and node-reduce entries are then paid once for all).
template <bool FROM_PARTIALS, bool STAGED, int CTAS, int PASSES>
__global__ void __launch_bounds__(SCAN_THREADS, CTAS) k_level_finish(
    SmallSource src, const int64_t *__restrict__ parent, const int32_t *__restrict__ parent_of,
    int64_t *__restrict__ large, int32_t n_features, int32_t n_bins, SplitParams sp, Cand *__restrict__ cand,
    float2 *__restrict__ cbounds, uint32_t *__restrict__ counters, SplitOut *__restrict__ small_out,
    SplitOut *__restrict__ large_out, DevState *st, const uint8_t *__restrict__ node_side) {
  __shared__ ScanShared sh;
  const int p = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int fo = warp & 3, side = warp >> 2;
  const int B = n_bins + 1;
  const bool staged = STAGED;  // B <= STAGE_SLOTS (the host picks the instance)
  const int64_t pp = parent_of ? (int64_t)parent_of[p] : p;
  const int fcta = blockIdx.x * 4 * PASSES;  // the CTA's first feature: PASSES groups of four, one per pass
  // The parent strips (and parent_of) were complete before the kernel this one
  // waits for started, so warps 4-7 stage the first pass's while that kernel finishes.
  if (side == 1 && fcta + fo < n_features && staged) {
    const longlong2 *P0 = reinterpret_cast<const longlong2 *>(parent) + (pp * n_features + fcta + fo) * B;
    for (int s = lane; s < B; s += 32) sh.cells[warp][swz(s)] = __ldg(P0 + s);
  }
  pdl_wait();  // the histogram kernel (or whatever ran before on the stream)
  // the plan's verdict and this pair's groups in one round trip (the arrays exist whatever the verdict;
  // no image address is formed from them unless the plan is valid)
  int32_t g0 = 0, g1 = 0, i0 = 0;  // the small sibling's exclusive groups and first group image
  uint32_t plan_ok = 1;
  if (FROM_PARTIALS) {
    plan_ok = st->plan_ok;
    g0 = src.view.group_prefix[p];
    g1 = src.view.group_prefix[p + 1];
    i0 = src.view.img_first[p];
  }
  if (!plan_ok) return;
  scan_init(sh);
  int64_t si = p, li = p;  // output indices of the small and the large sibling
  if (node_side) {
    const int sd = node_side[p] & 1;
    si = 2 * (int64_t)p + sd;
    li = 2 * (int64_t)p + 1 - sd;
  }
  float wlo = -INFINITY;  // this warp's best lower bound over its passes
  int ovf_any = 0;        // some pass of this warp overflowed the pool
  for (int pass = 0; pass < PASSES; ++pass) {
  const int f = fcta + 4 * pass + fo;
  const bool active = f < n_features;
  const longlong2 *P = reinterpret_cast<const longlong2 *>(parent) + (pp * n_features + f) * B;
  if (pass > 0) {
    __syncthreads();  // every warp is done with the previous pass's staged strips
    if (side == 1 && active && staged)
      for (int s = lane; s < B; s += 32) sh.cells[warp][swz(s)] = __ldg(P + s);
  }
  if (STAGED && pass + 1 < PASSES && fcta + 4 * pass + 4 < n_features) {
    // the next pass's parent strips (four strips of 16-byte cells, one 128-byte line per thread) and
    // group image rows (one sector per slot and group) on their way to L2 while this pass runs
    const int fn = fcta + 4 * pass + 4;
    const int64_t ncells = (int64_t)min(4, n_features - fn) * B;
    if ((int64_t)threadIdx.x * 8 < ncells)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const longlong2 *>(parent) +
                                                    (pp * n_features + fn) * B + threadIdx.x * 8));
    if (FROM_PARTIALS && (int)threadIdx.x < B) {
      const int2 *img = image_cell(src.view, i0, fn, src.item_feats, (int)threadIdx.x);
      const int64_t stride = src.view.n_fgroups * src.view.image_int4s * 2;
      for (int32_t k = g0; k < g1; ++k, img += stride) asm volatile("prefetch.global.L2 [%0];" ::"l"(img));
    }
  }
  longlong2 *L = reinterpret_cast<longlong2 *>(large) + (li * n_features + f) * B;
  longlong2 *Sout = FROM_PARTIALS ? reinterpret_cast<longlong2 *>(src.hist_out) + (si * n_features + f) * B
                                  : nullptr;
  const longlong2 *Sin = FROM_PARTIALS ? Sout
                                       : reinterpret_cast<const longlong2 *>(src.hist) + ((int64_t)p * n_features + f) * B;
  // phase A: small strips; the parent strips (warps 4-7) are staged above
  if (FROM_PARTIALS) {
    // all 256 threads sum the group images of the four features: thread t
    // takes feature t & 3 and slots (t >> 2) + 64 u, eight loads in flight,
    // so each warp load covers 8 slots x 4 features (whole 32-byte sectors)
    constexpr int PA = STAGED ? STAGE_SLOTS / 64 : 8;  // a staged strip has at most 4 slots per thread
    const int t = threadIdx.x, fi = t & 3, ff = fcta + 4 * pass + fi;
    int64_t pg = 0, ph = 0, pa = 0;  // long strips: this thread's part of feature fi's totals
    bool pn = false;
    if (ff < n_features) {
      const bool zero = i0 < src.view.r_cap;  // reduce-region images are zeroed as they are read
      const int64_t stride = src.view.n_fgroups * src.view.image_int4s * 2;
      int2 *img0 = image_cell(src.view, i0, ff, src.item_feats, 0);
      const int64_t sstride = src.view.sbw;  // int2 between slots
      longlong2 *So = reinterpret_cast<longlong2 *>(src.hist_out) + (si * n_features + ff) * B;
      for (int s0 = t >> 2; s0 < B; s0 += 64 * PA) {
        int64_t ag[PA], ah[PA];
#pragma unroll
        for (int u = 0; u < PA; ++u) ag[u] = ah[u] = 0;
        int2 *img = img0;
        for (int32_t k = g0; k < g1; ++k, img += stride) {
          int2 x[PA];
#pragma unroll
          for (int u = 0; u < PA; ++u) {
            const int s = s0 + 64 * u;
            x[u] = s < B ? __ldcg(img + s * sstride) : make_int2(0, 0);
          }
#pragma unroll
          for (int u = 0; u < PA; ++u) {
            ag[u] += x[u].x;
            ah[u] += x[u].y;
          }
        }
        if (zero) {  // after all the loads (a store would hold back the loads after it)
          img = img0;
          for (int32_t k = g0; k < g1; ++k, img += stride) {
#pragma unroll
            for (int u = 0; u < PA; ++u)
              if (s0 + 64 * u < B) __stcg(img + (s0 + 64 * u) * sstride, make_int2(0, 0));
          }
        }
#pragma unroll
        for (int u = 0; u < PA; ++u) {
          const int s = s0 + 64 * u;
          if (s < B) {
            const longlong2 c = make_longlong2(ag[u], ah[u]);
            So[s] = c;
            if (staged) {
              sh.cells[fi][swz(s)] = c;
            } else {
              pg += c.x;
              ph += c.y;
              pa += c.x < 0 ? -c.x : c.x;
              pn |= c.y < 0;
            }
          }
        }
      }
    }
    if (!staged) {  // the small strips' totals as they are written: the scan then reads each strip once
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {  // lanes of equal fi
        pg += shfl_xor_i64(pg, o);
        ph += shfl_xor_i64(ph, o);
        pa += shfl_xor_i64(pa, o);
        pn |= __shfl_xor_sync(0xffffffffu, (int)pn, o) != 0;
      }
      if (lane < 4) {
        sh.ptot[warp][lane][0] = pg;
        sh.ptot[warp][lane][1] = ph;
        sh.ptot[warp][lane][2] = pa;
        sh.ptot[warp][lane][3] = pn ? 1 : 0;
      }
    }
  } else if (side == 0 && active && staged) {
    for (int s = lane; s < B; s += 32) sh.cells[warp][swz(s)] = __ldg(Sin + s);
  }
  __syncthreads();
  // phase B: large = parent - small
  int64_t bg = 0, bh = 0, ba = 0;  // long strips: this lane's part of the large strip's totals as it is written
  bool bn = false;
  if (active && side == 1) {
    bool neg = false;
    if (staged) {
      for (int s = lane; s < B; s += 32) {
        const int q = swz(s);
        const longlong2 a = sh.cells[warp][q], b = sh.cells[warp - 4][q];
        const longlong2 d = make_longlong2(a.x - b.x, a.y - b.y);
        neg |= d.y < 0;
        L[s] = d;
        sh.cells[warp][q] = d;
      }
    } else {
      // FIN_BATCH loads of each operand in flight per lane before the stores
      for (int s0 = lane; s0 < B; s0 += 32 * FIN_BATCH) {
        longlong2 a[FIN_BATCH], b[FIN_BATCH];
#pragma unroll
        for (int u = 0; u < FIN_BATCH; ++u) {
          const int s = s0 + 32 * u;
          a[u] = s < B ? __ldg(P + s) : make_longlong2(0, 0);
          b[u] = s < B ? (FROM_PARTIALS ? __ldcg(Sin + s) : __ldg(Sin + s)) : make_longlong2(0, 0);
        }
#pragma unroll
        for (int u = 0; u < FIN_BATCH; ++u) {
          const int s = s0 + 32 * u;
          if (s < B) {
            const longlong2 d = make_longlong2(a[u].x - b[u].x, a[u].y - b[u].y);
            neg |= d.y < 0;
            L[s] = d;
            bg += d.x;
            bh += d.y;
            ba += d.x < 0 ? -d.x : d.x;
          }
        }
      }
    }
    if (neg) raise_err(st, ERRBIT_INCONSISTENT);
    bn = neg;
  }
  __syncwarp();
  // phase C: scan
  const longlong2 *cells = staged ? sh.cells[warp] : (side ? L : Sin);
  int64_t tg = 0, th = 0;
  if (active) {
    int64_t sa = 0;
    bool hneg = false;
    if (staged) {
      for (int s = lane; s < B; s += 32) {
        const longlong2 c = cells[swz(s)];
        tg += c.x;
        th += c.y;
        sa += c.x < 0 ? -c.x : c.x;
        hneg |= c.y < 0;
      }
      warp_sum3(tg, th, sa);
    } else if (side == 1) {  // summed by this warp in phase B
      tg = bg;
      th = bh;
      sa = ba;
      hneg = bn;
      warp_sum3(tg, th, sa);
    } else if (FROM_PARTIALS) {  // summed by the block in phase A
      for (int w = 0; w < SCAN_WARPS; ++w) {
        tg += sh.ptot[w][fo][0];
        th += sh.ptot[w][fo][1];
        sa += sh.ptot[w][fo][2];
        hneg |= sh.ptot[w][fo][3] != 0;
      }
    } else {
      strip_totals(cells, B, tg, th, sa, hneg);
      warp_sum3(tg, th, sa);
    }
    const bool h_ok = !__any_sync(0xffffffffu, hneg);
    int ovf = 0;
    wlo = warp_scan_push(cells, staged, n_bins, tg, th, sa, h_ok, sp, f, side, sh, ovf, 4, wlo);
    ovf = __any_sync(0xffffffffu, ovf);
    ovf_any |= ovf;
    if (lane == 0) {
      sh.warp_lo[warp] = wlo;
      sh.warp_overflow[warp] = ovf;
    }
  }
  __syncthreads();
  float thr0 = -INFINITY, thr1 = -INFINITY;  // the small and the large set's best lower bound so far
#pragma unroll
  for (int w = 0; w < SCAN_WARPS / 2; ++w) {
    thr0 = fmaxf(thr0, sh.warp_lo[w]);
    thr1 = fmaxf(thr1, sh.warp_lo[w + SCAN_WARPS / 2]);
  }
  if (active && sh.warp_overflow[warp]) {  // this pass's strip overflowed: the warp rescans it now
    const Cand d = warp_direct_best(cells, staged, n_bins, tg, th, sp, side ? thr1 : thr0, f);
    if (lane == 0 && cand_better(d, sh.extra[warp])) sh.extra[warp] = d;
  }
  }  // passes
  if (lane == 0) sh.warp_overflow[warp] = ovf_any;  // the select takes sh.extra of every warp that overflowed
  __syncthreads();
  float thr0 = -INFINITY, thr1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < SCAN_WARPS / 2; ++w) {
    thr0 = fmaxf(thr0, sh.warp_lo[w]);
    thr1 = fmaxf(thr1, sh.warp_lo[w + SCAN_WARPS / 2]);
  }
  cta_select(sh, sp, 2, thr0, thr1, 2);
  const int nfb = gridDim.x;
  const int64_t es = (int64_t)(2 * p) * nfb * PUB_K, el = es + (int64_t)nfb * PUB_K;  // the siblings' first entries
  if (cta_publish(sh, 2, cand + es + blockIdx.x * PUB_K, cand + el + blockIdx.x * PUB_K, counters + p, nfb,
                  cbounds + es + blockIdx.x * PUB_K, cbounds + el + blockIdx.x * PUB_K)) {
    // warps 0-3 reduce the small sibling, warps 4-7 the large one
    if (CTAS >= 4) {
      if (threadIdx.x < 128)
        reduce_node_cb_ool<1>(cand + es, cbounds + es, nfb * PUB_K, sp, small_out + si, 0, 128, sh.extra, sh.red,
                              sh.rcnt);
      else
        reduce_node_cb_ool<2>(cand + el, cbounds + el, nfb * PUB_K, sp, large_out + li, 128, 128, sh.extra + 4,
                              sh.red + 4, sh.rcnt + 1);
    } else {
      if (threadIdx.x < 128)
        reduce_node_cb<1>(cand + es, cbounds + es, nfb * PUB_K, sp, small_out + si, 0, 128, sh.extra, sh.red,
                          sh.rcnt);
      else
        reduce_node_cb<2>(cand + el, cbounds + el, nfb * PUB_K, sp, large_out + li, 128, 128, sh.extra + 4,
                          sh.red + 4, sh.rcnt + 1);
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

}  // namespace gbt
