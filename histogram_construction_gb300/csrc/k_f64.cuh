// Float-cell mode: histograms of the unquantised (g, h) in double [bonsai "10:
// CUDA histogram backend", "The kernel": float shared-memory cells merged into
// double global cells; "GBDT engine engineering deep-dive", section 7 listing;
// section 3: the hessian is clamped at zero after subtraction].
//
// GB300 design: the same device plan and persistent work items as the
// fixed-point build, with double cells. A work item holds TS features (TS a
// power of two, 32 for u8) as a [slot][TS][G, H] double image in shared
// memory; lane l takes feature l % TS of row l / TS of each group of 32/TS
// rows and adds (g, h) with two 64-bit shared atomics. Missing entries (u16:
// up to 40%) are summed in registers and added once per item. Items of one
// node add their images into one double image with TMA bulk reduce-adds (the
// plan zeroes it), or store it when they are its only chunk. Addition order
// is not fixed: cells agree with a serial double sum to rounding, not bit for
// bit.
#pragma once

#include "common.cuh"
#include "k_hist.cuh"
#include "k_split.cuh"

namespace gbt {

constexpr int HF_THREADS = 512;
constexpr int HF_SMEM_MAX = 160 * 1024;

__device__ __forceinline__ void bulk_reduce_add_f64(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f64 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}

struct HistF64Params {
  LevelParams lv;
  const unsigned char *mirror;  // tile pairs (see mirror_offset)
  const float2 *gpair;          // [n_rows] (g, h)
  int32_t n_features;
  int32_t n_slots;              // B
  int32_t n_bins;
  int32_t tile_feats;           // features per 64-byte mirror strip (64 u8, 32 u16)
};

template <typename T, int TS>
__global__ void __launch_bounds__(HF_THREADS, 1) k_hist_f64(HistF64Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  double *hist = reinterpret_cast<double *>(smem);  // [B][TS][2]
  __shared__ int32_t s_item;
  constexpr int RPI = 32 / TS;  // rows per warp instruction
  const LevelParams &p = P.lv;
  pdl_wait();
  pdl_trigger();
  if (!p.st->plan_ok) return;
  const int64_t chunk = p.st->chunk_rows;
  const int32_t cpg = p.st->chunks_per_group;
  const int32_t n_items = p.st->n_items;
  const int B = P.n_slots;
  const int64_t N = p.n_rows;
  const bool ident = (p.rows == nullptr);
  const uint32_t miss = (uint32_t)P.n_bins;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int fl = lane % TS, rho = lane / TS;
  uint32_t bad = 0;
  for (;;) {
    if (threadIdx.x == 0) s_item = (int32_t)atomicAdd(&p.st->work_next, 1u);
    __syncthreads();
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = decode_item(id, p, chunk, cpg);
    for (int i = threadIdx.x; i < B * TS * 2; i += blockDim.x) hist[i] = 0.0;
    __syncthreads();
    const int f = it.fgroup * TS + fl;
    const bool f_on = f < P.n_features;
    const int tile = f / P.tile_feats, ft = f - tile * P.tile_feats;
    const T *strip = reinterpret_cast<const T *>(P.mirror + mirror_offset(tile, 0, N)) + ft;
    double mg = 0.0, mh = 0.0;
    for (int64_t k = it.k0 + (int64_t)warp * RPI + rho; k < it.k1; k += (int64_t)nwarps * RPI) {
      const int32_t r = ident ? (int32_t)k : __ldg(p.rows + k);
      if (r < 0 || r >= N) {
        bad = 1;
        continue;
      }
      if (!f_on) continue;
      const float2 gh = __ldg(P.gpair + r);
      const uint32_t slot = __ldg(reinterpret_cast<const T *>(reinterpret_cast<const unsigned char *>(strip) +
                                                               (int64_t)r * MIRROR_ROW_BYTES));
      if (slot == miss) {
        mg += (double)gh.x;
        mh += (double)gh.y;
      } else {
        atomicAdd(&hist[(slot * TS + fl) * 2], (double)gh.x);
        atomicAdd(&hist[(slot * TS + fl) * 2 + 1], (double)gh.y);
      }
    }
#pragma unroll
    for (int o = TS; o < 32; o <<= 1) {
      mg += __shfl_xor_sync(0xffffffffu, mg, o);
      mh += __shfl_xor_sync(0xffffffffu, mh, o);
    }
    if (rho == 0 && f_on) {
      atomicAdd(&hist[(miss * TS + fl) * 2], mg);
      atomicAdd(&hist[(miss * TS + fl) * 2 + 1], mh);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned char *dst = reinterpret_cast<unsigned char *>(p.partial + it.image * p.image_int4s * 4);
      const unsigned char *src = reinterpret_cast<const unsigned char *>(hist);
      const uint32_t total = (uint32_t)B * TS * 16u;
      for (uint32_t off = 0; off < total; off += 65536u) {
        if (it.multi) bulk_reduce_add_f64(dst + off, src + off, min(65536u, total - off));
        else bulk_store(dst + off, src + off, min(65536u, total - off));
      }
      bulk_commit();
      bulk_wait_read_all();
    }
    __syncthreads();
  }
  if (bad) raise_err(p.st, ERRBIT_ROW);
  if (threadIdx.x == 0) bulk_wait_all();
}

// Group images ([image][slot][TS][2] double) -> hist_out [n][F][B][2] double.
__global__ void __launch_bounds__(256) k_finalize_f64(const double *__restrict__ partial,
                                                      const int32_t *__restrict__ group_prefix, int64_t image_doubles,
                                                      int32_t n_fgroups, int32_t ts, int32_t n_nodes,
                                                      int32_t n_features, int32_t B, double *__restrict__ hist_out,
                                                      const DevState *st) {
  pdl_wait();
  if (!st->plan_ok) return;
  const int64_t units = (int64_t)n_nodes * n_features * B;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int f = (int)(u % n_features);  // consecutive threads: consecutive features of one slot
    int64_t r = u / n_features;
    const int s = (int)(r % B);
    const int n = (int)(r / B);
    const int fg = f / ts, fl = f - fg * ts;
    double g = 0.0, h = 0.0;
    for (int32_t k = group_prefix[n]; k < group_prefix[n + 1]; ++k) {
      const double *c = partial + ((int64_t)k * n_fgroups + fg) * image_doubles + ((int64_t)s * ts + fl) * 2;
      g += __ldcg(c);
      h += __ldcg(c + 1);
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

// Split find on double cells: grid (ceil(F / 8), n_nodes), 256 threads; warp w
// scans feature blockIdx.x * 8 + w of node blockIdx.y, every candidate in
// double; the CTA's best goes to cand[node][blockIdx.x]; the node's last CTA
// writes the split. The double sums travel as bit patterns in the candidate's
// 64-bit fields, so the output record is a gbt_split whose four sums are doubles.
__global__ void __launch_bounds__(SCAN_THREADS) k_find_f64(const double *__restrict__ hist, int32_t n_features,
                                                           int32_t n_bins, double lambda, double gamma, double mcw,
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
    const double parent = __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, lambda));
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
        const int s = c0 + SCAN_SPL * lane + i;
        if (s >= n_bins) continue;
#pragma unroll
        for (int dir = 0; dir < 2; ++dir) {
          const double GL = eg + pg[i] + (dir ? m.x : 0.0), HL = eh + ph[i] + (dir ? m.y : 0.0);
          const double GR = G - GL, HR = H - HL;
          if (!(HL > 0.0 && HR > 0.0 && HL >= mcw && HR >= mcw)) continue;
          const double l = __ddiv_rn(__dmul_rn(GL, GL), __dadd_rn(HL, lambda));
          const double r = __ddiv_rn(__dmul_rn(GR, GR), __dadd_rn(HR, lambda));
          const double gain = __dsub_rn(__dmul_rn(0.5, __dsub_rn(__dadd_rn(l, r), parent)), gamma);
          Cand c;
          set_exact(c, gain);
          c.t = s;
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
