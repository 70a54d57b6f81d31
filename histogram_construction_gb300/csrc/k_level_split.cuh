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
// GB300 design, two kernels:
//  * k_level_totals: one warp per (node, feature) sums the strip's slots into
//    its totals and the prefix carried into each 128-slot chunk;
//  * k_level_split: one CTA per (feature, chunk); its warps share the nodes.
//    Lane l takes 4 consecutive slots of the chunk. For every node a warp
//    forms the FP32 screen bounds of each candidate (the node split's rigorous
//    bound) and adds them into per-candidate level bounds with directed
//    rounding (down for the lower bound, up for the upper), so [lo, up] still
//    encloses the double-precision level gain; the warps' bounds are combined
//    the same way. Candidates whose level upper bound reaches the CTA's best
//    level lower bound are published (at most two; with more the CTA resolves
//    them exactly); the last CTA evaluates in double the published candidates
//    that reach the level-wide threshold (per-node gains summed in node order)
//    and writes the split.
#pragma once

#include "common.cuh"
#include "k_split.cuh"

namespace gbt {

constexpr int LS_CHUNK = 32 * SCAN_SPL;  // slots per chunk (128)

// Per (node, feature): totals G, H, sum |G|, missing cell (G, H).
struct LevelTot {
  int64_t tg, th, sabs, mg, mh, pad0, pad1, pad2;
};

// k_level_totals: grid ceil(n_nodes * F / 8), 256 threads; warp -> (node, feature).
// carry: [n_nodes][F][n_chunks] prefix (G, H) of the slots before each chunk.
__global__ void __launch_bounds__(256) k_level_totals(const int64_t *__restrict__ hist, int32_t n_nodes,
                                                     int32_t n_features, int32_t n_bins, LevelTot *__restrict__ tot,
                                                     longlong2 *__restrict__ carry) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (int64_t)n_nodes * n_features) return;
  const int B = n_bins + 1;
  const int n_chunks = (n_bins + LS_CHUNK - 1) / LS_CHUNK;
  const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + wid * B;
  int64_t cg = 0, ch = 0, sa = 0;
  for (int k = 0; k < n_chunks; ++k) {
    if (lane == 0) carry[wid * n_chunks + k] = make_longlong2(cg, ch);
    int64_t g = 0, h = 0;
    for (int s = k * LS_CHUNK + lane; s < min((k + 1) * LS_CHUNK, n_bins); s += 32) {
      const longlong2 v = __ldg(c + s);
      g += v.x;
      h += v.y;
      sa += v.x < 0 ? -v.x : v.x;
    }
    warp_sum2(g, h);
    cg += g;
    ch += h;
  }
  const longlong2 m = __ldg(c + n_bins);
  sa += (m.x < 0 ? -m.x : m.x) * (lane == 0);
  int64_t z0 = 0, z1 = 0;
  warp_sum3(sa, z0, z1);
  if (lane == 0) {
    LevelTot lt;
    lt.tg = cg + m.x;
    lt.th = ch + m.y;
    lt.sabs = sa;
    lt.mg = m.x;
    lt.mh = m.y;
    lt.pad0 = lt.pad1 = lt.pad2 = 0;
    tot[wid] = lt;
  }
}

// Node-gain slot value for "this candidate is not valid for this node".
__device__ __forceinline__ double no_gain() { return __longlong_as_double(0x7ff8000000000001LL); }

// Exact level gain and left/right totals of candidate (f, t, dir), by one warp
// in the oracle's arithmetic: lane k takes nodes k, k + 32, ...; the node gains
// meet in gbuf ([n_nodes] doubles, global) and lane 0 sums them in node order.
// Returns false when no node makes the candidate valid.
__device__ __forceinline__ bool level_exact(const int64_t *hist, const LevelTot *tot, const longlong2 *carry,
                                            int n_nodes, int n_features, int n_bins, int f, int t, int dir,
                                            const SplitParams &sp, double *gbuf, Cand &out) {
  const int lane = threadIdx.x & 31;
  const int B = n_bins + 1;
  const int n_chunks = (n_bins + LS_CHUNK - 1) / LS_CHUNK;
  const int k = t / LS_CHUNK;
  int64_t agl = 0, ahl = 0, agr = 0, ahr = 0;
  int any = 0;
  for (int n = lane; n < n_nodes; n += 32) {
    const int64_t nf = (int64_t)n * n_features + f;
    const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + nf * B;
    const LevelTot lt = tot[nf];
    const longlong2 cc = carry[nf * n_chunks + k];
    int64_t pg = cc.x, ph = cc.y;
    for (int s = k * LS_CHUNK; s <= t; ++s) {
      const longlong2 v = __ldcg(c + s);
      pg += v.x;
      ph += v.y;
    }
    const int64_t GL = pg + (dir ? lt.mg : 0), HL = ph + (dir ? lt.mh : 0), GR = lt.tg - GL, HR = lt.th - HL;
    agl += GL;
    ahl += HL;
    agr += GR;
    ahr += HR;
    const bool valid = HL >= sp.h_min && HR >= sp.h_min;
    gbuf[n] = valid ? surv_gain(GL, HL, lt.tg, lt.th, sp) : no_gain();
    any |= valid;
  }
  __syncwarp();
  warp_sum2(agl, ahl);
  warp_sum2(agr, ahr);
  any = __any_sync(0xffffffffu, any);
  double sum = 0.0;
  if (lane == 0)
    for (int n = 0; n < n_nodes; ++n) {
      const double g = gbuf[n];
      if (!(g != g)) sum = __dadd_rn(sum, g);
    }
  sum = __shfl_sync(0xffffffffu, sum, 0);
  __syncwarp();
  set_exact(out, sum);
  out.f = f;
  out.t = t;
  out.dir = dir;
  out.gl = agl;
  out.hl = ahl;
  out.gr = agr;
  out.hr = ahr;
  return any != 0;
}

struct LevelShared {
  float lo[SCAN_WARPS][LS_CHUNK][2];
  float up[SCAN_WARPS][LS_CHUNK][2];
  uint8_t valid[SCAN_WARPS][LS_CHUNK][2];
  float red[SCAN_WARPS];
  int surv[SCAN_WARPS * 2 * LS_CHUNK];
  int n_surv;
  int list[2 * LS_CHUNK];  // last CTA: published entries reaching the level threshold
  int n_list;
  Cand pub[PUB_K];
  Cand best[SCAN_WARPS];
  uint32_t last;
  float thr;
};

// k_level_split: grid (ceil(F / fpc), n_chunks), SCAN_THREADS threads; the CTA
// takes fpc = 8 / wpf features of one chunk, wpf warps per feature sharing its
// nodes (wpf from the node count, so that small levels pack more features per
// CTA). cand: [grid][PUB_K];
// counters[0] arrival count and counters[1] threshold key (zero before and
// after); gbuf: [SCAN_WARPS + F * n_chunks][n_nodes] doubles (slices 0..7 for
// the last CTA's warps, slice SCAN_WARPS + cta for a CTA resolving its own).
__global__ void __launch_bounds__(SCAN_THREADS, 2) k_level_split(const int64_t *__restrict__ hist, int32_t n_nodes,
                                                              int32_t n_features, int32_t n_bins, SplitParams sp,
                                                              const LevelTot *__restrict__ tot,
                                                              const longlong2 *__restrict__ carry,
                                                              Cand *__restrict__ cand, uint32_t *__restrict__ counters,
                                                              double *gbuf, int32_t wpf,
                                                              SplitOut *__restrict__ out) {
  __shared__ LevelShared sh;
  pdl_wait();  // the totals
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int fpc = SCAN_WARPS / wpf;
  const int lf = warp / wpf, wj = warp - lf * wpf;  // local feature, rank among its warps
  const int f = blockIdx.x * fpc + lf, k = blockIdx.y;
  const int n_chunks = gridDim.y;
  const int cta = blockIdx.y * gridDim.x + blockIdx.x;
  const int B = n_bins + 1;
  const int c0 = k * LS_CHUNK;
  float lo[SCAN_SPL][2], up[SCAN_SPL][2];
  uint32_t vmask = 0;
#pragma unroll
  for (int i = 0; i < SCAN_SPL; ++i) lo[i][0] = lo[i][1] = up[i][0] = up[i][1] = 0.f;
  for (int n = wj; f < n_features && n < n_nodes; n += wpf) {
    const int64_t nf = (int64_t)n * n_features + f;
    const LevelTot lt = tot[nf];
    const longlong2 cc = carry[nf * n_chunks + k];
    const longlong2 *c = reinterpret_cast<const longlong2 *>(hist) + nf * B;
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
    eg += cc.x - ag;  // exclusive prefix of the lane's first slot
    eh += cc.y - ah;
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
  }
#pragma unroll
  for (int i = 0; i < SCAN_SPL; ++i)
#pragma unroll
    for (int dir = 0; dir < 2; ++dir) {
      sh.lo[warp][SCAN_SPL * lane + i][dir] = lo[i][dir];
      sh.up[warp][SCAN_SPL * lane + i][dir] = up[i][dir];
      sh.valid[warp][SCAN_SPL * lane + i][dir] = (vmask >> (2 * i + dir)) & 1u;
    }
  if (threadIdx.x == 0) sh.n_surv = 0;
  __syncthreads();
  // combine each feature's warps: thread -> (slot, direction), for every local feature
  const int cs = threadIdx.x >> 1, cd = threadIdx.x & 1;
  float L[SCAN_WARPS], U[SCAN_WARPS];
  uint32_t V = 0;
  float l = -INFINITY;
  for (int q = 0; q < fpc; ++q) {
    L[q] = 0.f;
    U[q] = 0.f;
    for (int j = 0; j < wpf; ++j) {
      const int w = q * wpf + j;
      if (!sh.valid[w][cs][cd]) continue;
      L[q] = __fadd_rd(L[q], sh.lo[w][cs][cd]);
      U[q] = __fadd_ru(U[q], sh.up[w][cs][cd]);
      V |= 1u << q;
    }
    if ((V >> q) & 1u) l = fmaxf(l, L[q]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
  if (lane == 0) sh.red[warp] = l;
  __syncthreads();
  float thr = -INFINITY;
  for (int w = 0; w < SCAN_WARPS; ++w) thr = fmaxf(thr, sh.red[w]);
  // survivors: (local feature, slot, direction); their bounds go to warp q*wpf's slots
  for (int q = 0; q < fpc; ++q) {
    if (!((V >> q) & 1u)) continue;
    sh.lo[q * wpf][cs][cd] = L[q];
    sh.up[q * wpf][cs][cd] = U[q];
    if (U[q] >= thr) sh.surv[atomicAdd(&sh.n_surv, 1)] = (q << 8) | (cs << 1) | cd;
  }
  __syncthreads();
  const int ns = sh.n_surv;
  if (ns > PUB_K) {
    // resolve here: warp 0 evaluates the survivors exactly
    if (warp == 0) {
      double *buf = gbuf + (int64_t)(SCAN_WARPS + cta) * n_nodes;
      Cand best = no_cand();
      for (int i = 0; i < ns; ++i) {
        const int e = sh.surv[i];
        const int ff = blockIdx.x * fpc + (e >> 8), ss = (e >> 1) & 127;
        Cand cc;
        if (level_exact(hist, tot, carry, n_nodes, n_features, n_bins, ff, c0 + ss, e & 1, sp, buf, cc) &&
            cand_better(cc, best))
          best = cc;
      }
      if (lane < PUB_K) sh.pub[lane] = lane == 0 ? best : no_cand();
    }
  } else if (threadIdx.x < PUB_K) {
    Cand c = no_cand();
    if ((int)threadIdx.x < ns) {
      const int e = sh.surv[threadIdx.x];
      const int q = e >> 8, ss = (e >> 1) & 127;
      c.t = c0 + ss;
      c.dir = e & 1;
      c.f = blockIdx.x * fpc + q;
      c.exact = 0;
      c.lo = sh.lo[q * wpf][ss][e & 1];
      c.up = sh.up[q * wpf][ss][e & 1];
    }
    sh.pub[threadIdx.x] = c;
  }
  __syncthreads();
  // store, raise the level threshold key, count in
  Cand *dst = cand + (int64_t)cta * PUB_K;
  if (threadIdx.x < PUB_K) {
    const Cand c = sh.pub[threadIdx.x];
    dst[threadIdx.x] = c;
    if (c.f != INT32_MAX) atomicMax(&counters[1], lo_key(c.lo));
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t done = atomicAdd(&counters[0], 1u);
    sh.last = (done == gridDim.x * n_chunks - 1) ? 1u : 0u;
    if (sh.last) {
      __threadfence();
      const uint32_t kk = atomicExch(&counters[1], 0u);
      sh.thr = kk ? key_lo(kk) : -INFINITY;
      counters[0] = 0;
      __threadfence();
    }
  }
  __syncthreads();
  if (!sh.last) return;
  // last CTA: every thread filters published entries by their upper bound
  // (two 16-byte reads each); the few that reach the level threshold are then
  // taken by the warps (w, w + 8, ...) and evaluated exactly
  const float lthr = sh.thr;
  const int n_ent = gridDim.x * n_chunks * PUB_K;
  if (threadIdx.x == 0) sh.n_list = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_ent; i += blockDim.x) {
    const int4 w1 = __ldcg(reinterpret_cast<const int4 *>(cand + i) + 1);  // f, exact, gl
    const int4 w3 = __ldcg(reinterpret_cast<const int4 *>(cand + i) + 3);  // hr, up, lo
    if (w1.x == INT32_MAX || !(__int_as_float(w3.z) >= lthr)) continue;
    const int j = atomicAdd(&sh.n_list, 1);
    if (j < 2 * LS_CHUNK) sh.list[j] = i;
  }
  __syncthreads();
  const bool listed = sh.n_list <= 2 * LS_CHUNK;  // else (mass ties) every entry is examined
  const int n_take = listed ? sh.n_list : n_ent;
  Cand best = no_cand();
  double *buf = gbuf + (int64_t)warp * n_nodes;
  for (int j = warp; j < n_take; j += SCAN_WARPS) {
    Cand c = load_cand(cand + (listed ? sh.list[j] : j));
    if (c.f == INT32_MAX || !(c.up >= lthr)) continue;
    if (!c.exact && !level_exact(hist, tot, carry, n_nodes, n_features, n_bins, c.f, c.t, c.dir, sp, buf, c))
      continue;
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
