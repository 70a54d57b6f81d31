// Oblivious level split: one (feature, cut, missing direction) for every node
// of a level ["GBDT engine engineering deep-dive" (ybb.press), section 5: an
// oblivious tree uses the same feature and threshold across a level; bonsai
// "10: CUDA histogram backend", "The device context lifecycle":
// find_level_split scans the frontier histograms].
//
// A candidate's level gain is the sum, over the nodes in ascending order, of
// each node's split gain at that candidate (its own feature totals); a node
// for which the candidate is not valid adds nothing; the candidate is valid
// when it is valid for at least one node. The first strictly larger level gain
// in (feature, cut, missing-right before missing-left) order wins.
//
// GB300 design: each warp owns one feature and walks its slots in chunks of
// 32 * SCAN_SPL (lane l: SCAN_SPL consecutive slots). For every node it forms
// the FP32 screen bounds of each candidate (the node split's rigorous bound)
// and adds them into per-candidate level bounds with directed rounding (down
// for the lower bound, up for the upper), so [lo, up] still encloses the
// double-precision level gain. Candidates whose level upper bound reaches the
// best level lower bound are published; the last CTA evaluates the few that
// reach the level-wide threshold exactly (per-node gains in double, summed in
// node order) and writes the split. Per-node totals and the running prefix of
// each (node, feature) live in a global scratch between chunks.
#pragma once

#include "common.cuh"
#include "k_split.cuh"

namespace gbt {

// Per (node, feature) scratch: totals G, H, sum |G|, missing cell (G, H) and
// the running prefix (G, H) before the current chunk.
struct LevelTot {
  int64_t tg, th, sabs, mg, mh, cg, ch, pad;
};

// Exact level gains by one warp, in the oracle's arithmetic: lane k takes
// nodes k, k + 32, ...; each node's gain meets in `gbuf` ([n_nodes] doubles,
// global) and lane 0 sums them in node order.

// Node-gain slot value for "this candidate is not valid for this node".
__device__ __forceinline__ double no_gain() { return __longlong_as_double(0x7ff8000000000001LL); }

__device__ __forceinline__ double ordered_sum(const double *gbuf, int n_nodes) {
  double sum = 0.0;
  if ((threadIdx.x & 31) == 0)
    for (int n = 0; n < n_nodes; ++n) {
      const double g = gbuf[n];
      if (!(g != g)) sum = __dadd_rn(sum, g);
    }
  return __shfl_sync(0xffffffffu, sum, 0);
}

// Exact level gain and left/right totals of candidate (f, t, dir); false when
// no node makes it valid.
__device__ __forceinline__ bool level_exact(const int64_t *hist, int n_nodes, int n_features, int n_bins, int f, int t,
                                            int dir, const SplitParams &sp, double *gbuf, double &gain, int64_t &sgl,
                                            int64_t &shl, int64_t &sgr, int64_t &shr) {
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  int64_t agl = 0, ahl = 0, agr = 0, ahr = 0;
  int any = 0;
  for (int n = lane; n < n_nodes; n += 32) {
    const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)n * n_features + f) * B;
    int64_t G = 0, H = 0, pg = 0, ph = 0;
    for (int s = 0; s < B; ++s) {
      const longlong2 v = __ldcg(c + s);
      G += v.x;
      H += v.y;
      if (s <= t) {
        pg += v.x;
        ph += v.y;
      }
    }
    const longlong2 m = __ldcg(c + n_bins);
    const int64_t GL = pg + (dir ? m.x : 0), HL = ph + (dir ? m.y : 0), GR = G - GL, HR = H - HL;
    agl += GL;
    ahl += HL;
    agr += GR;
    ahr += HR;
    const bool valid = HL >= sp.h_min && HR >= sp.h_min;
    gbuf[n] = valid ? surv_gain(GL, HL, G, H, sp) : no_gain();
    any |= valid;
  }
  __syncwarp();
  warp_sum2(agl, ahl);
  warp_sum2(agr, ahr);
  any = __any_sync(0xffffffffu, any);
  gain = ordered_sum(gbuf, n_nodes);
  __syncwarp();
  sgl = agl;
  shl = ahl;
  sgr = agr;
  shr = ahr;
  return any != 0;
}

// Exact best over every cut of feature f in direction dir: the fallback when a
// CTA's survivors overflow its pool (many near-equal level gains). Slow
// (every cut re-reads its nodes' strips) but only taken in that case.
__device__ __forceinline__ Cand level_exact_feature(const int64_t *hist, int n_nodes, int n_features, int n_bins,
                                                    int f, int dir, const SplitParams &sp, double *gbuf, Cand best) {
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  for (int t = 0; t < n_bins; ++t) {
    int64_t agl = 0, ahl = 0, agr = 0, ahr = 0;
    int any = 0;
    for (int n = lane; n < n_nodes; n += 32) {
      const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)n * n_features + f) * B;
      int64_t G = 0, H = 0, pg = 0, ph = 0;
      for (int s = 0; s < B; ++s) {
        const longlong2 v = __ldcg(c + s);
        G += v.x;
        H += v.y;
        if (s <= t) {
          pg += v.x;
          ph += v.y;
        }
      }
      const longlong2 m = __ldcg(c + n_bins);
      const int64_t GL = pg + (dir ? m.x : 0), HL = ph + (dir ? m.y : 0), GR = G - GL, HR = H - HL;
      agl += GL;
      ahl += HL;
      agr += GR;
      ahr += HR;
      const bool valid = HL >= sp.h_min && HR >= sp.h_min;
      gbuf[n] = valid ? surv_gain(GL, HL, G, H, sp) : no_gain();
      any |= valid;
    }
    __syncwarp();
    warp_sum2(agl, ahl);
    warp_sum2(agr, ahr);
    any = __any_sync(0xffffffffu, any);
    const double gain = ordered_sum(gbuf, n_nodes);
    __syncwarp();
    if (any) {
      Cand cc;
      set_exact(cc, gain);
      cc.f = f;
      cc.t = t;
      cc.dir = dir;
      cc.gl = agl;
      cc.hl = ahl;
      cc.gr = agr;
      cc.hr = ahr;
      if (cand_better(cc, best)) best = cc;
    }
  }
  return best;
}

struct LevelShared {
  Surv pool[SURV_CAP];
  int n;
  int overflow;
  float warp_lo[SCAN_WARPS];
  Cand pub[PUB_K];
  Cand best[SCAN_WARPS];
  uint32_t last;
  float thr;
};

// grid ceil(F / SCAN_WARPS), SCAN_THREADS threads; warp w takes feature
// blockIdx.x * SCAN_WARPS + w. cand: [gridDim.x][PUB_K]; counters[0] arrival
// count and counters[1] threshold key (zero before and after); gbuf:
// [SCAN_WARPS + gridDim.x][n_nodes] doubles (exact-evaluation buffers: the
// last CTA's warps use slices 0..7, a CTA resolving its own survivors slice
// SCAN_WARPS + blockIdx.x); scratch: [n_nodes][n_features] LevelTot.
__global__ void __launch_bounds__(SCAN_THREADS, 3) k_level_split(const int64_t *__restrict__ hist, int32_t n_nodes,
                                                              int32_t n_features, int32_t n_bins, SplitParams sp,
                                                              LevelTot *__restrict__ scratch, Cand *__restrict__ cand,
                                                              uint32_t *__restrict__ counters, double *gbuf,
                                                              SplitOut *__restrict__ out) {
  __shared__ LevelShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * SCAN_WARPS + warp;
  const int B = n_bins + 1;
  if (threadIdx.x == 0) {
    sh.n = 0;
    sh.overflow = 0;
  }
  if (threadIdx.x < SCAN_WARPS) sh.warp_lo[threadIdx.x] = -INFINITY;
  __syncthreads();
  float run_lo = -INFINITY;
  if (f < n_features) {
    // per-node totals of this feature
    for (int n = 0; n < n_nodes; ++n) {
      const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)n * n_features + f) * B;
      int64_t tg = 0, th = 0, sa = 0;
      for (int s = lane; s < B; s += 32) {
        const longlong2 v = __ldg(c + s);
        tg += v.x;
        th += v.y;
        sa += v.x < 0 ? -v.x : v.x;
      }
      warp_sum3(tg, th, sa);
      if (lane == 0) {
        const longlong2 m = __ldg(c + n_bins);
        LevelTot lt;
        lt.tg = tg;
        lt.th = th;
        lt.sabs = sa;
        lt.mg = m.x;
        lt.mh = m.y;
        lt.cg = 0;
        lt.ch = 0;
        lt.pad = 0;
        scratch[(int64_t)n * n_features + f] = lt;
      }
    }
    __syncwarp();
    for (int c0 = 0; c0 < n_bins; c0 += 32 * SCAN_SPL) {
      float lo[SCAN_SPL][2], up[SCAN_SPL][2];
      uint32_t vmask = 0;
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) lo[i][0] = lo[i][1] = up[i][0] = up[i][1] = 0.f;
      for (int n = 0; n < n_nodes; ++n) {
        LevelTot *ltp = scratch + (int64_t)n * n_features + f;
        const LevelTot lt = *ltp;
        const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + ((int64_t)n * n_features + f) * B;
        int64_t pg[SCAN_SPL], ph[SCAN_SPL], ag = 0, ah = 0;
#pragma unroll
        for (int i = 0; i < SCAN_SPL; ++i) {
          const int s = c0 + SCAN_SPL * lane + i;
          longlong2 v = make_longlong2(0, 0);
          if (s < n_bins) v = __ldg(c + s);
          ag += v.x;
          ah += v.y;
          pg[i] = ag;
          ph[i] = ah;
        }
        int64_t eg = ag, eh = ah;
        warp_incl_scan(eg, eh);
        const int64_t tot_g = shfl_i64(eg, 31), tot_h = shfl_i64(eh, 31);
        eg += lt.cg - ag;  // exclusive prefix of the lane's first slot
        eh += lt.ch - ah;
        const float Gf2den = parent_f32(lt.tg, lt.th, sp);
        const bool fast = strip_fast(lt.sabs, lt.th, Gf2den, sp);
#pragma unroll
        for (int i = 0; i < SCAN_SPL; ++i) {
          const int s = c0 + SCAN_SPL * lane + i;
#pragma unroll
          for (int dir = 0; dir < 2; ++dir) {
            const int64_t GL = eg + pg[i] + (dir ? lt.mg : 0), HL = eh + ph[i] + (dir ? lt.mh : 0);
            const int64_t HR = lt.th - HL;
            if (!(s < n_bins && HL >= sp.h_min && HR >= sp.h_min)) continue;  // adds nothing
            float u = INFINITY, w = -INFINITY;
            if (fast) screen_fast(GL, HL, lt.tg - GL, HR, Gf2den, sp, u, w);
            else if (sp.filter) screen_f32(GL, HL, lt.tg - GL, HR, Gf2den, sp, u, w);
            lo[i][dir] = __fadd_rd(lo[i][dir], w);
            up[i][dir] = __fadd_ru(up[i][dir], u);
            vmask |= 1u << (2 * i + dir);
          }
        }
        if (lane == 0) {
          ltp->cg = lt.cg + tot_g;
          ltp->ch = lt.ch + tot_h;
        }
        __syncwarp();
      }
      float l = -INFINITY;
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i)
#pragma unroll
        for (int dir = 0; dir < 2; ++dir)
          if ((vmask >> (2 * i + dir)) & 1u) l = fmaxf(l, lo[i][dir]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
      run_lo = fmaxf(run_lo, l);
#pragma unroll
      for (int i = 0; i < SCAN_SPL; ++i) {
#pragma unroll
        for (int dir = 0; dir < 2; ++dir) {
          if (!((vmask >> (2 * i + dir)) & 1u) || up[i][dir] < run_lo) continue;
          const int idx = atomicAdd(&sh.n, 1);
          if (idx >= SURV_CAP) {
            sh.overflow = 1;
            continue;
          }
          Surv v;
          v.gl = v.hl = v.tg = v.th = 0;
          v.up = up[i][dir];
          v.lo = lo[i][dir];
          v.t = c0 + SCAN_SPL * lane + i;
          v.f = f;
          v.dir = (int16_t)dir;
          v.node = 0;
          sh.pool[idx] = v;
        }
      }
    }
    if (lane == 0) sh.warp_lo[warp] = run_lo;
  }
  __syncthreads();
  float thr = -INFINITY;
  for (int w = 0; w < SCAN_WARPS; ++w) thr = fmaxf(thr, sh.warp_lo[w]);
  // publish up to PUB_K survivors with their bounds; with more, or when the
  // pool overflowed, warp 0 resolves the CTA's best exactly
  const int n = min(sh.n, SURV_CAP);
  if (threadIdx.x == 0) {
    int k = 0;
    for (int i = 0; i < n && k <= PUB_K; ++i)
      if (sh.pool[i].up >= thr) ++k;
    sh.last = (k > PUB_K || sh.overflow) ? 1u : 0u;
  }
  __syncthreads();
  if (sh.last) {
    if (warp == 0) {
      double *buf = gbuf + (int64_t)(SCAN_WARPS + blockIdx.x) * n_nodes;
      Cand best = no_cand();
      if (sh.overflow) {
        for (int w = 0; w < SCAN_WARPS; ++w) {
          const int ff = blockIdx.x * SCAN_WARPS + w;
          if (ff >= n_features) break;
          best = level_exact_feature(hist, n_nodes, n_features, n_bins, ff, 0, sp, buf, best);
          best = level_exact_feature(hist, n_nodes, n_features, n_bins, ff, 1, sp, buf, best);
        }
      } else {
        for (int i = 0; i < n; ++i) {
          const Surv v = sh.pool[i];
          if (!(v.up >= thr)) continue;
          double gain;
          int64_t a, b, c2, d;
          if (!level_exact(hist, n_nodes, n_features, n_bins, v.f, v.t, v.dir, sp, buf, gain, a, b, c2, d)) continue;
          Cand cc;
          set_exact(cc, gain);
          cc.f = v.f;
          cc.t = v.t;
          cc.dir = v.dir;
          cc.gl = a;
          cc.hl = b;
          cc.gr = c2;
          cc.hr = d;
          if (cand_better(cc, best)) best = cc;
        }
      }
      if (lane < PUB_K) sh.pub[lane] = lane == 0 ? best : no_cand();
    }
  } else if (threadIdx.x < PUB_K) {
    int k = 0, pick = -1;
    for (int i = 0; i < n; ++i)
      if (sh.pool[i].up >= thr) {
        if (k == (int)threadIdx.x) {
          pick = i;
          break;
        }
        ++k;
      }
    Cand c = no_cand();
    if (pick >= 0) {
      const Surv &v = sh.pool[pick];
      c.t = v.t;
      c.dir = v.dir;
      c.f = v.f;
      c.exact = 0;
      c.up = v.up;
      c.lo = v.lo;
    }
    sh.pub[threadIdx.x] = c;
  }
  __syncthreads();
  // store, raise the level threshold key, count in
  Cand *dst = cand + (int64_t)blockIdx.x * PUB_K;
  if (threadIdx.x < PUB_K) {
    const Cand c = sh.pub[threadIdx.x];
    dst[threadIdx.x] = c;
    if (c.f != INT32_MAX) atomicMax(&counters[1], lo_key(c.lo));
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t done = atomicAdd(&counters[0], 1u);
    sh.last = (done == gridDim.x - 1) ? 1u : 0u;
    if (sh.last) {
      __threadfence();
      const uint32_t k = atomicExch(&counters[1], 0u);
      sh.thr = k ? key_lo(k) : -INFINITY;
      counters[0] = 0;
      __threadfence();
    }
  }
  __syncthreads();
  if (!sh.last) return;
  // last CTA: warp w takes published candidates w, w + 8, ...
  const float lthr = sh.thr;
  const int n_ent = gridDim.x * PUB_K;
  Cand best = no_cand();
  double *buf = gbuf + (int64_t)warp * n_nodes;
  for (int i = warp; i < n_ent; i += SCAN_WARPS) {
    Cand c = load_cand(cand + i);
    if (c.f == INT32_MAX || !(c.up >= lthr)) continue;
    if (!c.exact) {
      double gain;
      int64_t a, b, c2, d;
      if (!level_exact(hist, n_nodes, n_features, n_bins, c.f, c.t, c.dir, sp, buf, gain, a, b, c2, d)) continue;
      set_exact(c, gain);
      c.gl = a;
      c.hl = b;
      c.gr = c2;
      c.hr = d;
    }
    if (cand_better(c, best)) best = c;
  }
  if (lane == 0) sh.best[warp] = best;
  __syncthreads();
  if (warp == 0) {
    Cand b = lane < SCAN_WARPS ? sh.best[lane] : no_cand();
    b = warp_best_cand(b);
    if (lane == 0) *out = cand_to_split(b);
  }
}

}  // namespace gbt
