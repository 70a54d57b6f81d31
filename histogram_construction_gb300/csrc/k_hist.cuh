// Level-batched histogram build: level plan, the persistent shared-memory
// histogram kernels (exact int32 partials per work item) and the finalize
// kernel that adds the partials of each node into its int64 histogram.
//
// What is computed [bonsai "10: CUDA histogram backend", "Level batching" and
// "The kernel"; "GBDT engine engineering deep-dive" (ybb.press), section 1
// per-row loop and section 7 shared-memory histograms]: for every node n of the
// batch, every feature f and slot s,
//   Hist[n][f][s] = sum over rows k of node n with slot(bins[f][row_k]) == s of (qg, qh).
//
// GB300 design (differs from the pages' (feature, node, row-chunk) grid with
// float shared cells and double global atomics):
//  * work items (node, 64-feature tile, row chunk), about one per SM and
//    decoded by the level plan, go to a persistent grid (one 1024-thread CTA
//    per SM): the first by block index, later ones through an atomic counter;
//  * each warp streams its rows' 16-byte strip quarters into a shared ring
//    with cp.async, two steps ahead of the step whose reductions it issues;
//  * a CTA holds the tile's histogram as int32 (G, H) pairs in shared memory,
//    in 16-feature sub-blocks of [256 slots][16 features]; each lane adds
//    (qg, qh) with two 32-bit shared atomics, and lanes are assigned to
//    (row, feature, component) so that the 32 lanes of every atomic
//    instruction hit 32 different banks whatever the bin values;
//  * a chunk never holds more rows than keep every int32 partial exact
//    (rows * max|q| < 2^31);
//  * the item's shared image leaves as is with TMA bulk stores, or bulk
//    reduce-adds into a group image the plan zeroed when several chunks of a
//    node share it (no transposition, no global atomics); the images of a
//    node's groups are added in int64 afterwards (finalize kernel, or the
//    fused subtract + split-find kernel).
#pragma once

#include <type_traits>

#include "common.cuh"

namespace gbt {

constexpr int CHUNK_MIN_ROWS = 1024;

// A work item: node, feature group, row range [k0, k1) in level order and
// the group image it adds into. Item ids run chunk-major, feature group
// fastest; the plan writes every item's record, so that a claim is one load.
struct Item {
  int32_t node, fgroup;
  int64_t k0, k1;
  int64_t image;  // group image index
  int32_t multi;  // the group has more than one chunk: reduce-add, else store
  int32_t pad;
};

struct LevelParams {
  const int32_t *rows;    // level row list or nullptr (identity)
  const int64_t *offs;    // [n_nodes + 1]
  int32_t n_nodes;
  int32_t n_fgroups;      // feature groups per node chunk (work items per chunk)
  int32_t target_items;   // load-balance target for the item count
  int32_t item_feats;     // features per work item (64 for u8, TS for u16)
  int64_t n_rows;
  const int2 *q;          // quantised gpair [n_rows]
  int32_t *group_prefix;  // [n_nodes + 1] exactness groups before each node (written by the plan)
  int32_t *img_first;     // [n_nodes] first group image of each node (written by the plan)
  int64_t r_cap_groups;   // size of the reduce region in group images; store node n owns r_cap_groups + n
  int32_t *partial;       // int32 group images (see PartialView)
  int64_t image_int4s;    // 16-byte units per image
  int32_t sbw;            // features per sub-block of the image (16 for u8, TS for u16)
  int32_t nsb;            // sub-blocks per image (4 for u8, 1 for u16)
  uint32_t qmax_plan;     // if nonzero, the plan's exactness bound uses it instead of the tree's max|q|
  int32_t chunk_cap;      // if nonzero, no chunk holds more rows (float cells: rounding per chunk)
  Item *items;            // [items] decoded work items (written by the plan kernel)
  int32_t fold;           // 1: the histogram kernel plans the level itself (n_nodes <= FOLD_MAX_NODES)
  int32_t pad_;
  DevState *st;
  const int2 *qpos = nullptr;  // if set: q of the level's rows in level order, qpos[k] = q[rows[k]] (k_gather_q)
};

// The level's (qg, qh) pairs in level order, qpos[k] = q[rows[k]] (zero for an
// id outside [0, n_rows), which the histogram kernel reports). With many
// feature tiles every work item of a row would otherwise gather its pair by
// row id, one sector per row and tile; in level order eight rows share one
// 64-byte load. Grid-stride over the level's positions.
__global__ void __launch_bounds__(256) k_gather_q(const int32_t *__restrict__ rows, const int64_t *__restrict__ offs,
                                                  int32_t n_nodes, int64_t n_rows, const int2 *__restrict__ q,
                                                  int2 *__restrict__ qpos) {
  pdl_wait();  // the kernel that wrote the row list
  pdl_trigger();
  const int64_t R = min(max(offs[n_nodes], (int64_t)0), n_rows);
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < R; k += (int64_t)gridDim.x * blockDim.x) {
    const int32_t r = rows[k];
    qpos[k] = (uint32_t)r < (uint32_t)n_rows ? __ldg(q + r) : make_int2(0, 0);
  }
}

// Block-wide inclusive scan of one int64 per thread (every thread calls it).
__device__ __forceinline__ int64_t block_incl_scan(int64_t v, int64_t *s_warp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) s_warp[w] = v;
  __syncthreads();
  if (w == 0) {
    int64_t x = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  const int64_t r = v + (w > 0 ? s_warp[w - 1] : 0);
  __syncthreads();
  return r;
}

// Level plan (one block). With T = target_items / n_fgroups chunks wanted,
// the base length L is the shortest of 16 candidates from ceil(R / T) to
// ceil(R / ceil(T / 2)) whose chunk count sum_n max(1, ceil(rows_n / L)) stays
// within T (the longest when none does; the longest keeps the count within T
// whenever T >= 2 x the nodes holding rows). L is at least CHUNK_MIN_ROWS and at
// most the int32 exactness bound rc = (2^31 - 1) / max|q| and the chunk cap.
// So no persistent CTA takes one item more than the others.
// A node's chunks have equal length ceil(rows_n / c_n) <= L, and its
// consecutive chunks form exactness groups of floor(rc / length) chunks, whose
// int32 sum cannot overflow either. Every work item (chunk, feature group) adds
// its shared-memory image into its group's image.
//
// Group images live in two regions. A node of one chunk ("store" node) owns
// group image r_cap + n, which its item overwrites with a bulk store. The
// groups of a node of several chunks ("reduce" nodes) are numbered from 0 in
// node order; their items bulk reduce-add into them. The reduce region is kept
// zero between calls (the host zeroes it once; every consumer zeroes the
// reduce images it reads), so nothing is zeroed here and one block plans the
// level. Offsets that do not start at 0, descend or leave [0, n_rows]
// invalidate the plan (no items; GBT_ERR_ROW_RANGE).
constexpr int PLAN_THREADS = 512;  // nodes per planning batch
constexpr int PLAN_CANDS = 16;     // chunk lengths the plan counts in one pass

// A node of rows_n rows in c equal chunks (ceil(rows_n / c) rows each, the
// last one shorter): consecutive chunks per exactness group.
// (32-bit arithmetic: rows_n, c and rc are below 2^31.)
__device__ __forceinline__ int64_t chunks_per_group(int64_t rows_n, int64_t c, int64_t rc) {
  const uint32_t len = ((uint32_t)rows_n + (uint32_t)c - 1) / (uint32_t)c;
  return len > 0 ? (int64_t)max(1u, min((uint32_t)rc / len, 0x3fffffffu)) : (int64_t)0x3fffffff;
}

__global__ void __launch_bounds__(PLAN_THREADS) k_level_plan(LevelParams p) {
  pdl_trigger();  // the histogram kernel may launch now; it waits for this grid to finish
  __shared__ int64_t s_warp[32];
  __shared__ int64_t s_a[PLAN_THREADS];         // first level position of each node of the batch
  __shared__ int32_t s_cpre[PLAN_THREADS + 1];  // chunk prefix within the batch
  __shared__ int32_t s_rows[PLAN_THREADS], s_len[PLAN_THREADS], s_cpg[PLAN_THREADS], s_img[PLAN_THREADS];
  __shared__ int32_t s_red[PLAN_THREADS];       // 1: a reduce node
  __shared__ int64_t s_tot[3];
  __shared__ uint32_t s_cnt[PLAN_CANDS];
  const int tid = threadIdx.x;
  // one read phase: the tree's max|q|, R and every node's offsets
  const uint32_t qm = max(p.qmax_plan ? p.qmax_plan : p.st->qmax, 1u);
  const int64_t R = p.offs[p.n_nodes];
  // PLAN_CANDS chunk lengths from ceil(R / T) to ceil(R / ceil(T / 2)) (32-bit:
  // R < 2^31), with T = target_items / n_fgroups chunks wanted
  const uint32_t T = (uint32_t)max(1, p.target_items / p.n_fgroups);
  const uint32_t R32 = (R > 0 && R <= p.n_rows) ? (uint32_t)R : 0u;
  const uint32_t lo = max(1u, (R32 + T - 1) / T), hi = max(lo, (R32 + (T + 1) / 2 - 1) / ((T + 1) / 2));
  uint32_t cand[PLAN_CANDS], cnt[PLAN_CANDS];
#pragma unroll
  for (int k = 0; k < PLAN_CANDS; ++k) {
    cand[k] = lo + (uint32_t)(((uint64_t)(hi - lo) * k + PLAN_CANDS - 2) / (PLAN_CANDS - 1));
    cnt[k] = 0;
  }
  if (tid < PLAN_CANDS) s_cnt[tid] = 0;
  bool bad = (tid == 0) && (p.offs[0] != 0);
  for (int n = tid; n < p.n_nodes; n += blockDim.x) {
    const int64_t a = p.offs[n], b = p.offs[n + 1];
    const bool ok = (a >= 0) && (b >= a) && (b <= p.n_rows);
    bad |= !ok;
    const uint32_t rows_n = ok ? (uint32_t)(b - a) : 0u;
#pragma unroll
    for (int k = 0; k < PLAN_CANDS; ++k) cnt[k] += max(1u, (rows_n + cand[k] - 1) / cand[k]);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) {
      p.st->plan_ok = 0;
      p.st->n_items = 0;
      raise_err(p.st, ERRBIT_ROW);
    }
    return;
  }
  // the shortest candidate whose chunk count sum_n max(1, ceil(rows_n / L))
  // stays within T (the longest when none does)
  if ((tid & ~31) < p.n_nodes) {  // warps holding nodes (warp-uniform)
#pragma unroll
    for (int k = 0; k < PLAN_CANDS; ++k) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt[k] += __shfl_xor_sync(0xffffffffu, cnt[k], o);
    }
    if ((tid & 31) == 0) {
#pragma unroll
      for (int k = 0; k < PLAN_CANDS; ++k) atomicAdd(&s_cnt[k], cnt[k]);
    }
  }
  __syncthreads();
  uint32_t len = cand[PLAN_CANDS - 1];
#pragma unroll
  for (int k = PLAN_CANDS - 1; k >= 0; --k)
    if (s_cnt[k] <= T) len = cand[k];
  const int64_t rc = (int64_t)(0x7fffffffu / qm);  // rows whose int32 partials cannot overflow
  int64_t chunk = max((int64_t)len, (int64_t)CHUNK_MIN_ROWS);
  chunk = max((int64_t)1, min(rc, chunk));
  if (p.chunk_cap > 0) chunk = min(chunk, (int64_t)p.chunk_cap);
  int64_t carry_c = 0, carry_g = 0, carry_r = 0;
  for (int base = 0; base < p.n_nodes; base += blockDim.x) {
    const int n = base + tid;
    int64_t c = 0, g = 0, cpg = 1, rows_n = 0, a = 0;
    bool red = false;
    if (n < p.n_nodes) {
      a = p.offs[n];
      rows_n = p.offs[n + 1] - a;
      c = max((int64_t)1, (int64_t)(((uint32_t)rows_n + (uint32_t)chunk - 1) / (uint32_t)chunk));
      cpg = chunks_per_group(rows_n, c, rc);
      g = (c + cpg - 1) / cpg;
      red = c >= 2;
    }
    const int64_t ic = block_incl_scan(c, s_warp);
    const int64_t ig = block_incl_scan(g, s_warp);
    const int64_t ir = block_incl_scan(red ? g : 0, s_warp);
    const int64_t img = red ? carry_r + ir - g : p.r_cap_groups + n;
    if (n < p.n_nodes) {
      p.group_prefix[n + 1] = (int32_t)(carry_g + ig);
      p.img_first[n] = (int32_t)img;
    }
    s_cpre[tid + 1] = (int32_t)ic;
    s_a[tid] = a;
    s_rows[tid] = (int32_t)rows_n;
    s_len[tid] = (int32_t)(((uint32_t)rows_n + (uint32_t)c - 1) / (uint32_t)max(c, (int64_t)1));
    s_cpg[tid] = (int32_t)cpg;
    s_img[tid] = (int32_t)img;
    s_red[tid] = red ? 1 : 0;
    if (tid == 0) s_cpre[0] = 0;
    if (tid == blockDim.x - 1) {
      s_tot[0] = ic;
      s_tot[1] = ig;
      s_tot[2] = ir;
    }
    __syncthreads();
    const int last = min(p.n_nodes - base, (int)blockDim.x) - 1;  // the batch's last node
    // the batch's work items
    const int64_t nfg = p.n_fgroups;
    const int64_t items = (int64_t)s_cpre[blockDim.x] * nfg;
    for (int64_t u = tid; u < items; u += blockDim.x) {
      const int32_t kc = (int32_t)(u / nfg);  // chunk within the batch
      const int32_t f = (int32_t)(u - (int64_t)kc * nfg);
      int lo2 = 0, hi2 = last;  // largest j with s_cpre[j] <= kc
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2 + 1) >> 1;
        if (s_cpre[mid] <= kc) lo2 = mid; else hi2 = mid - 1;
      }
      const int32_t cidx = kc - s_cpre[lo2], cpg_n = s_cpg[lo2];
      const int32_t gi = cidx / cpg_n;
      Item it;
      it.node = base + lo2;
      it.fgroup = f;
      it.k0 = s_a[lo2] + (int64_t)cidx * s_len[lo2];
      it.k1 = min(s_a[lo2] + s_rows[lo2], it.k0 + s_len[lo2]);
      it.image = (int64_t)(s_img[lo2] + gi) * nfg + f;
      it.multi = s_red[lo2];
      it.pad = 0;
      p.items[(carry_c * nfg) + u] = it;
    }
    carry_c += s_tot[0];
    carry_g += s_tot[1];
    carry_r += s_tot[2];
    __syncthreads();
  }
  if (tid == 0) {
    p.group_prefix[0] = 0;
    p.st->plan_ok = 1;
    p.st->n_items = (int32_t)(carry_c * p.n_fgroups);
  }
}

// ----------------------------------------------------------------------------
// The same plan, computed by every CTA of the histogram kernel itself for a
// level of at most FOLD_MAX_NODES nodes: no plan launch on the critical path.
// Each CTA keeps the chunk prefix and the first group image of every node in
// shared memory and decodes an item when it claims it (the node's offsets are
// read again, from L1 or L2). CTA 0 publishes group_prefix, img_first and
// plan_ok for the consumer kernels.
constexpr int FOLD_MAX_NODES = 256;

struct FoldPlan {
  int32_t cpre[FOLD_MAX_NODES + 1];  // chunk prefix over the nodes
  int32_t img[FOLD_MAX_NODES];       // first group image of each node
  int32_t wtot[3][FOLD_MAX_NODES / 32];
  uint32_t cnt[PLAN_CANDS], cand[PLAN_CANDS];
  int64_t chunk, rc;
  int64_t R;                         // level rows
  uint32_t qm;                       // max |q| bound of the plan
  int32_t n_items;
};

// Returns false (and, in CTA 0, reports GBT_ERR_ROW_RANGE) when the offsets are
// invalid. Called by every thread; blockDim.x >= FOLD_MAX_NODES and >= 32 *
// PLAN_CANDS. Warp k counts the chunks of candidate length k over all nodes
// (their offsets read again, from L1), so the sixteen counts take one pass.
// (The u8 kernels leave under 1 KB of shared memory for this record.)
__device__ __noinline__ bool plan_fold(const LevelParams &p, FoldPlan &fp) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bool has = tid < p.n_nodes;
  // every load of the plan in one round trip: the node's offsets, and R and
  // max|q| by one thread (152 CTAs x 32 warps reading one word would queue at its L2 slice)
  if (tid == 0) {
    fp.R = p.offs[p.n_nodes];
    fp.qm = max(p.qmax_plan ? p.qmax_plan : p.st->qmax, 1u);
  }
  bool ok = true;
  uint32_t rows_n = 0;
  if (has) {
    const int64_t a = __ldg(p.offs + tid), b = __ldg(p.offs + tid + 1);
    ok = (a >= 0) && (b >= a) && (b <= p.n_rows) && (tid > 0 || a == 0);
    rows_n = ok ? (uint32_t)(b - a) : 0u;
  }
  if (__syncthreads_or(!ok)) {
    if (blockIdx.x == 0 && tid == 0) {
      p.st->plan_ok = 0;
      raise_err(p.st, ERRBIT_ROW);
    }
    return false;
  }
  const int64_t R = fp.R;
  const uint32_t qm = fp.qm;
  const uint32_t T = (uint32_t)max(1, p.target_items / p.n_fgroups);
  const uint32_t R32 = (R > 0 && R <= p.n_rows) ? (uint32_t)R : 0u;
  const uint32_t lo = max(1u, (R32 + T - 1) / T), hi = max(lo, (R32 + (T + 1) / 2 - 1) / ((T + 1) / 2));
  if (w < PLAN_CANDS) {
    const uint32_t cand = lo + (uint32_t)(((uint64_t)(hi - lo) * w + PLAN_CANDS - 2) / (PLAN_CANDS - 1));
    uint32_t cnt = 0;
    for (int n = lane; n < p.n_nodes; n += 32) {
      const uint32_t r = (uint32_t)(__ldg(p.offs + n + 1) - __ldg(p.offs + n));  // valid: checked above
      cnt += max(1u, (r + cand - 1) / cand);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) {
      fp.cnt[w] = cnt;
      fp.cand[w] = cand;
    }
  }
  __syncthreads();
  // the shortest candidate whose chunk count stays within T (the longest when none does)
  int kb = PLAN_CANDS - 1;
#pragma unroll
  for (int k = PLAN_CANDS - 1; k >= 0; --k)
    if (fp.cnt[k] <= T) kb = k;
  uint32_t len = fp.cand[kb];
  if (kb > 0 && fp.cnt[kb] <= T && fp.cand[kb] > fp.cand[kb - 1] + 1) {
    // a second pass over the lengths between the last count above T and the first within it
    const uint32_t lo2 = fp.cand[kb - 1] + 1, hi2 = fp.cand[kb];
    __syncthreads();  // every thread has read the first pass
    if (w < PLAN_CANDS) {
      const uint32_t cand = lo2 + (uint32_t)(((uint64_t)(hi2 - lo2) * w + PLAN_CANDS - 2) / (PLAN_CANDS - 1));
      uint32_t cnt = 0;
      for (int n = lane; n < p.n_nodes; n += 32) {
        const uint32_t r = (uint32_t)(__ldg(p.offs + n + 1) - __ldg(p.offs + n));
        cnt += max(1u, (r + cand - 1) / cand);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (lane == 0) {
        fp.cnt[w] = cnt;
        fp.cand[w] = cand;
      }
    }
    __syncthreads();
    len = hi2;
#pragma unroll
    for (int k = PLAN_CANDS - 1; k >= 0; --k)
      if (fp.cnt[k] <= T) len = fp.cand[k];
  }
  const int64_t rc = (int64_t)(0x7fffffffu / qm);
  int64_t chunk = max((int64_t)len, (int64_t)CHUNK_MIN_ROWS);
  chunk = max((int64_t)1, min(rc, chunk));
  if (p.chunk_cap > 0) chunk = min(chunk, (int64_t)p.chunk_cap);
  // per node: chunks, groups, reduce flag; inclusive scans of (chunks, groups, reduce groups)
  int32_t c = 0, g = 0, rg = 0;
  if (has) {
    c = (int32_t)max((uint32_t)1, (rows_n + (uint32_t)chunk - 1) / (uint32_t)chunk);
    const int64_t cpg = chunks_per_group(rows_n, c, rc);
    g = (int32_t)((c + cpg - 1) / cpg);
    rg = c >= 2 ? g : 0;
  }
  int32_t ic = c, ig = g, ir = rg;
  if (w < FOLD_MAX_NODES / 32) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t yc = __shfl_up_sync(0xffffffffu, ic, o), yg = __shfl_up_sync(0xffffffffu, ig, o),
                    yr = __shfl_up_sync(0xffffffffu, ir, o);
      if (lane >= o) {
        ic += yc;
        ig += yg;
        ir += yr;
      }
    }
    if (lane == 31) {
      fp.wtot[0][w] = ic;
      fp.wtot[1][w] = ig;
      fp.wtot[2][w] = ir;
    }
  }
  __syncthreads();
  if (w < FOLD_MAX_NODES / 32) {
    for (int k = 0; k < w; ++k) {
      ic += fp.wtot[0][k];
      ig += fp.wtot[1][k];
      ir += fp.wtot[2][k];
    }
    if (has) {
      fp.cpre[tid + 1] = ic;
      const int32_t img = c >= 2 ? ir - rg : (int32_t)(p.r_cap_groups + tid);
      fp.img[tid] = img;
      if (blockIdx.x == 0) {
        p.group_prefix[tid + 1] = ig;
        p.img_first[tid] = img;
      }
    }
    if (tid == p.n_nodes - 1) fp.n_items = ic * p.n_fgroups;
  }
  if (tid == 0) {
    fp.cpre[0] = 0;
    fp.chunk = chunk;
    fp.rc = rc;
    if (blockIdx.x == 0) {
      p.group_prefix[0] = 0;
      p.st->plan_ok = 1;
    }
  }
  __syncthreads();
  return true;
}

// Work item `id` of a folded plan (one thread).
__device__ __forceinline__ Item fold_item(const LevelParams &p, const FoldPlan &fp, int32_t id) {
  const int32_t nfg = p.n_fgroups;
  const int32_t kc = id / nfg, f = id - kc * nfg;
  int lo = 0, hi = p.n_nodes - 1;  // largest node with cpre[node] <= kc
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (fp.cpre[mid] <= kc) lo = mid; else hi = mid - 1;
  }
  const int64_t a = __ldg(p.offs + lo), rows_n = __ldg(p.offs + lo + 1) - a;
  const int32_t c = fp.cpre[lo + 1] - fp.cpre[lo], cidx = kc - fp.cpre[lo];
  const int64_t len = ((uint32_t)rows_n + (uint32_t)c - 1) / (uint32_t)c;
  const int32_t gi = cidx / (int32_t)chunks_per_group(rows_n, c, fp.rc);
  Item it;
  it.node = lo;
  it.fgroup = f;
  it.k0 = a + (int64_t)cidx * len;
  it.k1 = min(a + rows_n, it.k0 + len);
  it.image = (int64_t)(fp.img[lo] + gi) * nfg + f;
  it.multi = c >= 2 ? 1 : 0;
  it.pad = 0;
  return it;
}

// The next item of a CTA (one thread): the first by block index, later ones from the launch's counter.
__device__ __forceinline__ int32_t claim_item(const LevelParams &p, bool first) {
  return first ? (int32_t)blockIdx.x : (int32_t)(gridDim.x + atomicAdd(&p.st->work_next, 1u));
}

// At the end of every CTA that claimed items: the last one resets the counters for the next launch
// (every other CTA has made its last claim before counting itself done).
__device__ __forceinline__ void claims_done(const LevelParams &p) {
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.st->work_done, 1u) == gridDim.x - 1) {
      p.st->work_next = 0;
      p.st->work_done = 0;
    }
  }
}


// ----------------------------------------------------------------------------
// Float cells [bonsai "10: CUDA histogram backend", "The kernel": shared
// accumulation in float with native shared-memory atomics, chunks of at most
// 32k rows, the cross-chunk merge in double]. The histogram kernels then hold
// (g, h) as float bit patterns and add them with red.shared.add.f32; the
// item's float image leaves as doubles, FL_PIECE cells at a time, through two
// alternating shared staging buffers: converted by the whole block, then
// stored (the node's only chunk) or reduce-added (cp.reduce.async.bulk .f64)
// into the node's double image.
constexpr int FL_PIECE = 4096;                     // floats per staged piece
constexpr int FL_STAGE_BYTES = 2 * FL_PIECE * 8;   // two double buffers
constexpr int FL_CHUNK_CAP = 32768;                // rows per float chunk

// nseg float segments of seg_floats floats each (segment i at src + i *
// seg_stride bytes) -> consecutive double segments at dst. Called by every
// thread of the block; returns with the staging buffers free again.
__device__ __forceinline__ void flush_float_image(const unsigned char *src, int nseg, int seg_stride,
                                                  uint32_t seg_floats, double *dst, bool multi, double *stage) {
  int idx = 0;
  for (int sg = 0; sg < nseg; ++sg) {
    const float *fs = reinterpret_cast<const float *>(src + (size_t)sg * seg_stride);
    for (uint32_t off = 0; off < seg_floats; off += FL_PIECE, ++idx) {
      const uint32_t n = min((uint32_t)FL_PIECE, seg_floats - off);
      double *buf = stage + (idx & 1) * FL_PIECE;
      if (idx >= 2) {  // the buffer's previous piece must have been read
        if (threadIdx.x == 0) bulk_wait_read_1();
        __syncthreads();
      }
      for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) buf[i] = (double)fs[off + i];
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        double *d = dst + (size_t)sg * seg_floats + off;
        if (multi) bulk_reduce_add_f64(d, buf, n * 8u);
        else bulk_store(d, buf, n * 8u);
        bulk_commit();
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait_read_all();
  __syncthreads();
}

// ----------------------------------------------------------------------------
// u8 kernel: items of one 64-feature mirror tile, 16-feature sub-blocks.
//
// Shared layout: sub-block sb (features 16 sb .. 16 sb + 15) is a [slot][16]
// array of (G, H) int32 pairs (128-byte slot rows) starting at byte
// sb * (32 KB + 32): consecutive sub-blocks are staggered by 8 banks.
//
// Lane l of a warp takes row rho = l/4 of an 8-row group and the 16-byte
// quarter w = l%4 of the row's strip, i.e. sub-block w, with one 128-bit load.
// In atomic instruction (e, j, c) the lane adds byte jj = (j + rho/2) & 3 of
// word e of its quarter (feature f = 4e + jj of sub-block w) for component
// c ^ (rho & 1) (0 = G, 1 = H). Its bank is (8w + 8e + 2jj + comp) mod 32:
// distinct over the 32 lanes, whatever the bin values. Per entry the lane
// spends one byte permute (slot), one multiply-add (cell address; 32e is an
// immediate offset), one xor (the other component) and two shared reductions.
//
// The gathers of the next U row groups (row ids one step further ahead) are
// in flight while the current groups' reductions issue. Rows past the chunk
// end or with an invalid id add zeros to slot 0, so the loop has no branches.
constexpr int H8_SB = 4;                                   // sub-blocks per tile
constexpr int H8_SB_BYTES = 256 * 16 * 8;                  // 32 KB of cells per sub-block
constexpr int H8_SB_STRIDE = H8_SB_BYTES + 32;             // shared bytes between sub-blocks
constexpr int H8_SMEM = H8_SB * H8_SB_STRIDE;
constexpr int H8_THREADS = 1024;
constexpr int H8_U = 2;                                    // 8-row groups per warp step
// Integer-cell instantiations stage the gathered strips in a shared ring of
// H8_RING steps per warp (cp.async), so that the gathers of the next
// H8_RING - 1 steps are in flight while a step's reductions issue; the
// float-cell instantiation keeps them in registers, one step ahead (its
// shared memory holds the double staging of the flush instead).
constexpr int H8_RING = 3;
constexpr int H8_RING_BYTES = H8_RING * (H8_THREADS / 32) * H8_U * 512;
constexpr int H8_SMEM_RING = H8_SMEM + H8_RING_BYTES;

struct Hist8Params {
  LevelParams lv;
  const uint8_t *mirror;  // tile pairs [ceil(n_tiles / 2)][N][128]
  int32_t n_features;
  int32_t n_slots;        // B
  int32_t n_targets;      // multi-output: k pairs per row in lv.q ([N][k]); 1 otherwise
};

// Gathered operands of U row groups of one lane.
template <int U>
struct H8Stage {
  uint4 bw[U];            // the lane's 16-byte quarter of each row's strip
  uint32_t v0[U], v1[U];  // (qg, qh) in the lane's component order
};

template <int U>
__device__ __forceinline__ void h8_rows(const LevelParams &p, bool ident, int64_t k, int64_t step, int64_t k1,
                                        int32_t (&rid)[U]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t kk = k + u * step;
    rid[u] = kk < k1 ? (ident ? (int32_t)kk : __ldg(p.rows + kk)) : -1;
  }
}

// q of row r: lv.q[r] (one target), or target tsel of lv.q[r][k] (multi-output;
// lanes of targets past k load nothing, lane_on false). Rows rid[u] sit at
// level positions kb + u * step; a position before k1 whose id is outside
// [0, n_rows) is a caller error (negative ids included), positions past k1
// are the loop's padding.
template <int U, bool MULTI>
__device__ __forceinline__ void h8_gather(const LevelParams &p, const unsigned char *strip, bool lane_on, int par,
                                          const int32_t (&rid)[U], int64_t kb, int64_t step, int64_t k1,
                                          H8Stage<U> &st, uint32_t &bad, int k, int tsel) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int32_t r = rid[u];
    const bool valid = (uint32_t)r < (uint32_t)p.n_rows;
    bad |= (kb + u * step < k1 && !valid) ? 1u : 0u;
    int2 qv = make_int2(0, 0);
    if (MULTI) {
      if (valid && lane_on) qv = __ldg(p.q + (int64_t)r * k + tsel);
    } else if (valid) {
      qv = __ldg(p.q + r);
    }
    st.bw[u] = (valid && lane_on) ? ldg_nc_v4(strip + (int64_t)r * MIRROR_ROW_BYTES) : make_uint4(0, 0, 0, 0);
    st.v0[u] = (uint32_t)(par ? qv.y : qv.x);
    st.v1[u] = (uint32_t)(par ? qv.x : qv.y);
  }
}

// Ring variant of h8_gather: the lane's 16-byte quarters go straight to its
// ring slots (ring_dst + 512 u) with cp.async (zero-filled for rows that are
// past the end, invalid or of an unused sub-block); only the (qg, qh) pairs
// come to registers, as loaded (the component order is chosen at use).
template <int U, bool MULTI>
__device__ __forceinline__ void h8_issue(const LevelParams &p, const unsigned char *strip, bool lane_on,
                                         const int32_t (&rid)[U], int64_t kb, int64_t step, int64_t k1,
                                         uint32_t ring_dst, int2 (&qv)[U], uint32_t &bad, int k, int tsel) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int32_t r = rid[u];
    const bool valid = (uint32_t)r < (uint32_t)p.n_rows;
    bad |= (kb + u * step < k1 && !valid) ? 1u : 0u;
    const bool ld = valid && lane_on;
    if (MULTI) {
      qv[u] = ld ? __ldg(p.q + (int64_t)r * k + tsel) : make_int2(0, 0);
    } else {
      qv[u] = valid ? __ldg(p.qpos ? p.qpos + kb + u * step : p.q + r) : make_int2(0, 0);
    }
    cp_async_16(ring_dst + (uint32_t)u * 512u, ld ? strip + (int64_t)r * MIRROR_ROW_BYTES : strip, ld ? 16u : 0u);
  }
}

template <int E, bool FLT>
__device__ __forceinline__ void h8_word(uint32_t word, const uint32_t (&sel)[4], const uint32_t (&cj)[4], uint32_t v0,
                                        uint32_t v1) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a = __byte_perm(word, 0u, sel[j]) * 128u + cj[j];
    if constexpr (FLT) {
      asm volatile("red.shared.add.f32 [%0+%2], %1;" ::"r"(a), "f"(__uint_as_float(v0)), "n"(32 * E) : "memory");
      asm volatile("red.shared.add.f32 [%0+%2], %1;" ::"r"(a ^ 4u), "f"(__uint_as_float(v1)), "n"(32 * E) : "memory");
    } else {
      asm volatile("red.shared.add.u32 [%0+%2], %1;" ::"r"(a), "r"(v0), "n"(32 * E) : "memory");
      asm volatile("red.shared.add.u32 [%0+%2], %1;" ::"r"(a ^ 4u), "r"(v1), "n"(32 * E) : "memory");
    }
  }
}

template <int U, bool FLT>
__device__ __forceinline__ void h8_scatter(const H8Stage<U> &st, const uint32_t (&sel)[4], const uint32_t (&cj)[4]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    h8_word<0, FLT>(st.bw[u].x, sel, cj, st.v0[u], st.v1[u]);
    h8_word<1, FLT>(st.bw[u].y, sel, cj, st.v0[u], st.v1[u]);
    h8_word<2, FLT>(st.bw[u].z, sel, cj, st.v0[u], st.v1[u]);
    h8_word<3, FLT>(st.bw[u].w, sel, cj, st.v0[u], st.v1[u]);
  }
}

// FLT: float cells (p.q holds the float (g, h) bit patterns; images are double).
// MULTI: multi-output (vector-leaf) histograms [hessboost PR #163 "Summary":
// a bin read serves every target's gradients]. An item is one 16-feature
// quarter of a mirror tile and up to four targets: sub-block w holds target
// 4 tg + w, lane quarter w loads that target's pair, and all four lanes of a
// row read the same 16-byte quarter. The bank map is the same (the sub-block
// is the target instead of the feature quarter).
// With the first gathers of an item in flight: the previous item's flush must
// have read the image before it is zeroed; zero the slot rows that will be
// read back, B rows of each used sub-block (lanes of unused sub-blocks add into
// their own, never read, sub-block).
__device__ __forceinline__ void h8_zero_image(unsigned char *smem, int nsb, int B) {
  if (threadIdx.x == 0) bulk_wait_read_all();
  __syncthreads();
  for (int sb = 0; sb < nsb; ++sb) {
    uint4 *h4 = reinterpret_cast<uint4 *>(smem + sb * H8_SB_STRIDE);
    for (int i = threadIdx.x; i < B * 8; i += blockDim.x) h4[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
}

// The mirror pads the features past the last one with bin 0, so the slot-0
// cells of those pad columns received the item's gradients; they are cleared
// before the flush, so that group images hold nothing but real features (the
// reduce region of the images must stay zero wherever no consumer reads).
// Columns valid .. 15 of sub-blocks sb0 .. sb1 - 1 (cells of 8 bytes).
__device__ __forceinline__ void h8_zero_pad(unsigned char *smem, int sb0, int sb1, int valid) {
  const int pad = 16 - valid;
  if (pad <= 0) return;
  for (int i = threadIdx.x; i < (sb1 - sb0) * pad; i += blockDim.x) {
    const int sb = sb0 + i / pad, col = valid + i % pad;
    *reinterpret_cast<uint2 *>(smem + sb * H8_SB_STRIDE + col * 8) = make_uint2(0u, 0u);
  }
}

template <bool FLT, bool MULTI = false>
__global__ void __launch_bounds__(H8_THREADS, 1) k_hist_u8(Hist8Params P) {
  constexpr int U = H8_U;
  constexpr bool RING = !FLT;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int32_t s_item;
  __shared__ Item s_it;  // the next item, claimed and decoded by thread 0 while the last one flushes
  __shared__ FoldPlan s_fp;

  const LevelParams &p = P.lv;
  pdl_wait();     // the level plan (or whatever produced the row lists)
  pdl_trigger();  // the consumer kernel may launch; it waits for this grid to finish
  int32_t n_items;
  if (p.fold) {
    if (!plan_fold(p, s_fp)) return;
    n_items = s_fp.n_items;
  } else {
    if (!p.st->plan_ok) return;
    n_items = p.st->n_items;
  }
  const int B = P.n_slots;
  const int64_t N = p.n_rows;
  const bool ident = (p.rows == nullptr);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rho = lane >> 2, w = lane & 3;
  const int pr = rho >> 1, par = rho & 1;
  const uint32_t hist_base = smem_addr(smem);
  uint32_t sel[4], cj[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = (j + pr) & 3;
    sel[j] = 0x4440u | (uint32_t)jj;  // byte jj, zero-extended
    cj[j] = hist_base + (uint32_t)(w * H8_SB_STRIDE) + (uint32_t)jj * 8u + (par ? 4u : 0u);
  }
  uint32_t bad = 0;
  // this lane's 16-byte slot of group 0 in ring slot 0 (ring after the image)
  const uint32_t ring_stage = (uint32_t)nwarps * U * 512u;
  const uint32_t ring_lane = hist_base + (uint32_t)H8_SMEM + (uint32_t)warp * U * 512u + (uint32_t)lane * 16u;

  if (threadIdx.x == 0) {  // the first item by block index, later ones from the counter
    s_item = claim_item(p, true);
    if (s_item < n_items) s_it = p.fold ? fold_item(p, s_fp, s_item) : p.items[s_item];
  }
  __syncthreads();
  for (;;) {
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = s_it;
    int nsb, tsel = 0;
    const unsigned char *strip;
    if (MULTI) {
      const int nfq = (P.n_features + 15) >> 4;  // feature quarters
      const int tg = it.fgroup / nfq, fq = it.fgroup - tg * nfq;
      nsb = min(H8_SB, P.n_targets - 4 * tg);  // targets of this item
      tsel = 4 * tg + w;
      strip = P.mirror + mirror_offset(fq >> 2, 0, N) + (fq & 3) * 16;
    } else {
      nsb = min(H8_SB, (P.n_features - it.fgroup * 64 + 15) >> 4);
      strip = P.mirror + mirror_offset(it.fgroup, 0, N) + w * 16;
    }
    const bool lane_on = w < nsb;
    const int64_t step = (int64_t)8 * nwarps;  // rows between a warp's consecutive groups
    const int64_t adv = step * U;              // rows per warp step
    int64_t g0 = it.k0 + 8 * warp + rho;
    int32_t rid[U];
    if constexpr (RING) {
      // Steps j, j + 1, j + 2 of the warp live in ring slots j % 3, ...; their
      // (qg, qh) in qa, qb, qc by the same rotation, and the row ids of steps
      // j + 2, j + 3, j + 4 in xa, xb, xc (step j + 2's set is reloaded with
      // step j + 5's, three steps ahead of its use). The loop is unrolled three
      // times so that no register is copied: a copy of a loaded register would
      // wait for the load.
      int2 qa[U], qb[U], qc[U];
      int32_t xa[U], xb[U], xc[U];
      h8_rows<U>(p, ident, g0, step, it.k1, xa);
      h8_rows<U>(p, ident, g0 + adv, step, it.k1, xb);
      h8_rows<U>(p, ident, g0 + 2 * adv, step, it.k1, xc);
      h8_issue<U, MULTI>(p, strip, lane_on, xa, g0, step, it.k1, ring_lane, qa, bad, P.n_targets, tsel);
      cp_async_commit();
      h8_issue<U, MULTI>(p, strip, lane_on, xb, g0 + adv, step, it.k1, ring_lane + ring_stage, qb, bad, P.n_targets,
                         tsel);
      cp_async_commit();
      h8_rows<U>(p, ident, g0 + 3 * adv, step, it.k1, xa);
      h8_rows<U>(p, ident, g0 + 4 * adv, step, it.k1, xb);
      h8_zero_image(smem, nsb, B);
      // one step: consume slot `use` (pairs qcur), issue step j + 2 (row ids
      // xnew) into slot `nxt2` (pairs qnew: the slot and pairs step j - 1 used)
      auto one_step = [&](uint32_t use, uint32_t nxt2, const int2(&qcur)[U], int2(&qnew)[U],
                          int32_t(&xnew)[U]) -> bool {
        if (!__any_sync(0xffffffffu, g0 < it.k1)) return false;
        if (__any_sync(0xffffffffu, g0 + 2 * adv < it.k1)) {
          h8_issue<U, MULTI>(p, strip, lane_on, xnew, g0 + 2 * adv, step, it.k1, ring_lane + nxt2 * ring_stage, qnew,
                             bad, P.n_targets, tsel);
          h8_rows<U>(p, ident, g0 + 5 * adv, step, it.k1, xnew);
        }
        cp_async_commit();   // possibly empty: one group per step keeps the count
        cp_async_wait<2>();  // this lane's copies of step j have landed
        H8Stage<U> cur;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          cur.bw[u] = lds_v4(ring_lane + use * ring_stage + (uint32_t)u * 512u);
          cur.v0[u] = (uint32_t)(par ? qcur[u].y : qcur[u].x);
          cur.v1[u] = (uint32_t)(par ? qcur[u].x : qcur[u].y);
        }
        h8_scatter<U, FLT>(cur, sel, cj);
        g0 += adv;
        return true;
      };
      for (;;) {
        if (!one_step(0, 2, qa, qc, xc)) break;
        if (!one_step(1, 0, qb, qa, xa)) break;
        if (!one_step(2, 1, qc, qb, xb)) break;
      }
      cp_async_wait<0>();  // the prologue's second step may be unused: no copy may land in the next item
    } else {
      H8Stage<U> cur, nxt;
      h8_rows<U>(p, ident, g0, step, it.k1, rid);
      h8_gather<U, MULTI>(p, strip, lane_on, par, rid, g0, step, it.k1, cur, bad, P.n_targets, tsel);
      h8_rows<U>(p, ident, g0 + adv, step, it.k1, rid);
      h8_zero_image(smem, nsb, B);
      // lanes of a warp run out of rows within one group of each other; any
      // lane with work keeps the warp going (the others add zeros)
      while (__any_sync(0xffffffffu, g0 < it.k1)) {
        if (__any_sync(0xffffffffu, g0 + adv < it.k1)) {
          h8_gather<U, MULTI>(p, strip, lane_on, par, rid, g0 + adv, step, it.k1, nxt, bad, P.n_targets, tsel);
          h8_rows<U>(p, ident, g0 + 2 * adv, step, it.k1, rid);
        }
        h8_scatter<U, FLT>(cur, sel, cj);
        cur = nxt;
        g0 += adv;
      }
    }
    __syncthreads();
    if (MULTI) {
      const int nfq = (P.n_features + 15) >> 4;
      const int fq = it.fgroup % nfq;
      h8_zero_pad(smem, 0, nsb, min(16, P.n_features - 16 * fq));
    } else {
      const int nf = P.n_features - it.fgroup * 64;
      if (nf < 64) h8_zero_pad(smem, nsb - 1, nsb, nf - 16 * (nsb - 1));
    }
    if constexpr (FLT) {
      __syncthreads();
      flush_float_image(smem, nsb, H8_SB_STRIDE, (uint32_t)B * 32u,
                        reinterpret_cast<double *>(p.partial) + it.image * p.image_int4s * 2, it.multi,
                        reinterpret_cast<double *>(smem + H8_SMEM));
    } else {
      // flush: the item's shared image (per sub-block [slot][16][G, H] int32)
      // leaves as is, one TMA bulk operation per sub-block: a store when the
      // item is its group's only chunk, else a reduce-add into the zeroed
      // group image (exact: the group's int32 sums cannot overflow). The
      // next item's claim, decode and first gathers overlap the copy-out.
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        int32_t *img_out = p.partial + it.image * p.image_int4s * 4;
        for (int sb = 0; sb < nsb; ++sb) {
          int32_t *dst = img_out + (int64_t)sb * B * 16 * 2;
          const unsigned char *src = smem + sb * H8_SB_STRIDE;
          if (it.multi) bulk_reduce_add_u32(dst, src, (uint32_t)B * 128u);
          else bulk_store(dst, src, (uint32_t)B * 128u);
        }
        bulk_commit();
      }
    }
    if (threadIdx.x == 0) {
      s_item = claim_item(p, false);
      if (s_item < n_items) s_it = p.fold ? fold_item(p, s_fp, s_item) : p.items[s_item];
    }
    __syncthreads();
  }
  if (bad) raise_err(p.st, ERRBIT_ROW);
  claims_done(p);
  if (threadIdx.x == 0) bulk_wait_all();
}

// ----------------------------------------------------------------------------
// u16 kernel: TS features per item (TS = 2..32), any B with TS * B * 8 within
// the shared budget. Missing-slot entries are summed in registers and added
// once per item (40% of entries can be missing; they would all hit one cell).
template <bool FLT>
__device__ __forceinline__ typename std::conditional<FLT, float, int32_t>::type h16_val(int32_t bits) {
  if constexpr (FLT) return __int_as_float(bits);
  else return bits;
}

// Adds (g, h) into the (G, H) cell pair c.
template <bool FLT, typename V>
__device__ __forceinline__ void h16_add(uint32_t *c, V g, V h) {
  if constexpr (FLT) {
    atomicAdd(reinterpret_cast<float *>(c), g);
    atomicAdd(reinterpret_cast<float *>(c) + 1, h);
  } else {
    atomicAdd(c, (uint32_t)g);
    atomicAdd(c + 1, (uint32_t)h);
  }
}

constexpr int H16_THREADS = 512;
constexpr int H16_HIST_MAX = 160 * 1024;
constexpr int H16_STAGE_SLOTS = 2048;
constexpr int H16_STAGE_BYTES = H16_STAGE_SLOTS * 8;

struct Hist16Params {
  LevelParams lv;
  const uint16_t *mirror;  // tile pairs [ceil(n_tiles / 2)][N][2 x 32]
  int32_t n_features;
  int32_t n_slots;         // B
  int32_t n_bins;
  int32_t ts;              // features per item
};

template <int TS, bool FLT>
__global__ void __launch_bounds__(H16_THREADS, 1) k_hist_u16(Hist16Params P) {
  using V = typename std::conditional<FLT, float, int32_t>::type;  // missing-slot partials
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int W = TS / 2;        // u32 words per row in an item
  constexpr int RPI = 32 / W;      // rows per warp instruction
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem);
  const int B = P.n_slots;
  const int hist_bytes = ((B * TS * 8) + 127) & ~127;
  unsigned char *stage = smem + hist_bytes;
  __shared__ int32_t s_item;
  __shared__ Item s_it;
  __shared__ FoldPlan s_fp;

  const LevelParams &p = P.lv;
  pdl_wait();     // the level plan (or whatever produced the row lists)
  pdl_trigger();  // the consumer kernel may launch; it waits for this grid to finish
  int32_t n_items;
  if (p.fold) {
    if (!plan_fold(p, s_fp)) return;
    n_items = s_fp.n_items;
  } else {
    if (!p.st->plan_ok) return;
    n_items = p.st->n_items;
  }
  const int64_t N = p.n_rows;
  const bool ident = (p.rows == nullptr);
  const uint32_t miss_slot = (uint32_t)P.n_bins;
  (void)stage;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rho = lane / W, wi = lane % W;
  constexpr int GROUPS_PER_TILE = 32 / TS;
  uint32_t bad = 0;
  bool first = true;  // the first item by block index, later ones from the counter

  for (;;) {
    if (threadIdx.x == 0) {
      s_item = claim_item(p, first);
      if (s_item < n_items) s_it = p.fold ? fold_item(p, s_fp, s_item) : p.items[s_item];
    }
    first = false;
    __syncthreads();
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = s_it;
    {
      uint4 *h4 = reinterpret_cast<uint4 *>(hist);
      const int n4 = (B * TS * 8) / 16;
      for (int i = threadIdx.x; i < n4; i += blockDim.x) h4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int tile = it.fgroup / GROUPS_PER_TILE;
    const int sub = it.fgroup % GROUPS_PER_TILE;
    const unsigned char *strip =
        reinterpret_cast<const unsigned char *>(P.mirror) + mirror_offset(tile, 0, N) + sub * TS * 2 + wi * 4;
    V mg0 = 0, mh0 = 0, mg1 = 0, mh1 = 0;  // missing-slot partials of features 2wi, 2wi+1
    const int64_t step = (int64_t)RPI * nwarps;
    const int64_t stride = step * 4;  // rows between a warp's consecutive iterations
    // Iteration j covers rows g0 + j stride + u step + rho (u < 4). Its row ids
    // are loaded two iterations ahead and its (qg, qh) and bins one iteration
    // ahead, while iteration j - 1 adds; the loop is unrolled twice so that no
    // loaded register is copied (a copy would wait for the load). Rows past
    // the item or invalid add zeros to slot 0, which is never the missing slot.
    auto rows4 = [&](int64_t gb, int32_t(&R)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = gb + u * step + rho;
        R[u] = k < it.k1 ? (ident ? (int32_t)k : __ldg(p.rows + k)) : -1;
      }
    };
    // rows R[u] sit at level positions gb + u * step + rho: an id outside [0, N)
    // at a position before the item's end is a caller error (negative ids
    // included); positions past the end are the loop's padding
    auto gather4 = [&](const int32_t(&R)[4], int64_t gb, int32_t(&vg)[4], int32_t(&vh)[4], uint32_t(&bw)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t r = R[u];
        const bool valid = (uint32_t)r < (uint32_t)N;
        bad |= (gb + u * step + rho < it.k1 && !valid) ? 1u : 0u;
        const int2 qv = valid ? __ldg(p.qpos ? p.qpos + gb + u * step + rho : p.q + r) : make_int2(0, 0);
        vg[u] = qv.x;
        vh[u] = qv.y;
        bw[u] = valid ? __ldg(reinterpret_cast<const uint32_t *>(strip + (int64_t)r * MIRROR_ROW_BYTES)) : 0u;
      }
    };
    auto scatter4 = [&](const int32_t(&vg)[4], const int32_t(&vh)[4], const uint32_t(&bw)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t s0 = bw[u] & 0xffffu, s1 = bw[u] >> 16;
        const V g = h16_val<FLT>(vg[u]), h = h16_val<FLT>(vh[u]);
        if (s0 == miss_slot) { mg0 += g; mh0 += h; }
        else h16_add<FLT>(hist + 2 * (s0 * TS + 2 * wi), g, h);
        if (s1 == miss_slot) { mg1 += g; mh1 += h; }
        else h16_add<FLT>(hist + 2 * (s1 * TS + 2 * wi + 1), g, h);
      }
    };
    int64_t g0 = it.k0 + RPI * warp;
    int32_t ra[4], rb[4], ga[4], ha[4], gb4[4], hb4[4];
    uint32_t ba[4], bb[4];
    rows4(g0, ra);
    rows4(g0 + stride, rb);
    gather4(ra, g0, ga, ha, ba);
    rows4(g0 + 2 * stride, ra);
    for (;;) {
      if (g0 >= it.k1) break;
      gather4(rb, g0 + stride, gb4, hb4, bb);  // iteration j + 1
      rows4(g0 + 3 * stride, rb);              // iteration j + 3
      scatter4(ga, ha, ba);                    // iteration j
      g0 += stride;
      if (g0 >= it.k1) break;
      gather4(ra, g0 + stride, ga, ha, ba);    // iteration j + 2
      rows4(g0 + 3 * stride, ra);     // iteration j + 4
      scatter4(gb4, hb4, bb);         // iteration j + 1
      g0 += stride;
    }
    // reduce missing partials over lanes sharing wi, add once
#pragma unroll
    for (int o = W; o < 32; o <<= 1) {
      mg0 += __shfl_xor_sync(0xffffffffu, mg0, o);
      mh0 += __shfl_xor_sync(0xffffffffu, mh0, o);
      mg1 += __shfl_xor_sync(0xffffffffu, mg1, o);
      mh1 += __shfl_xor_sync(0xffffffffu, mh1, o);
    }
    if (rho == 0) {
      h16_add<FLT>(hist + 2 * (miss_slot * TS + 2 * wi), mg0, mh0);
      h16_add<FLT>(hist + 2 * (miss_slot * TS + 2 * wi + 1), mg1, mh1);
    }
    __syncthreads();
    {
      // pad features past the last one (mirror bin 0): clear their slot-0 cells
      const int valid = P.n_features - it.fgroup * TS;
      if (valid < TS && (int)threadIdx.x < TS - valid)
        *reinterpret_cast<uint2 *>(hist + 2 * (valid + (int)threadIdx.x)) = make_uint2(0u, 0u);
      __syncthreads();
    }
    if constexpr (FLT) {
      flush_float_image(smem, 1, 0, (uint32_t)B * TS * 2u,
                        reinterpret_cast<double *>(p.partial) + it.image * p.image_int4s * 2, it.multi,
                        reinterpret_cast<double *>(stage));
      continue;
    }
    // flush: the item's shared image ([slot][TS][G, H] int32) in bulk stores
    // (or reduce-adds, for a group of several chunks) of <= 64 KB
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned char *img_out = reinterpret_cast<unsigned char *>(p.partial + it.image * p.image_int4s * 4);
      const unsigned char *src = reinterpret_cast<const unsigned char *>(hist);
      const uint32_t total = (uint32_t)B * TS * 8u;
      for (uint32_t off = 0; off < total; off += 65536u) {
        if (it.multi) bulk_reduce_add_u32(img_out + off, src + off, min(65536u, total - off));
        else bulk_store(img_out + off, src + off, min(65536u, total - off));
      }
      bulk_commit();
      bulk_wait_read_all();
    }
    __syncthreads();
  }
  if (bad) raise_err(p.st, ERRBIT_ROW);
  claims_done(p);
  if (threadIdx.x == 0) bulk_wait_all();
}

// ----------------------------------------------------------------------------
// Group images -> int64 histogram.
//
// Images are [image][sub-block][slot][sbw][G, H] int32 (nsb sub-blocks of sbw
// features): feature fl of an item's feature group is cell ((fl / sbw) * B +
// s) * sbw + fl % sbw. The images of node n are groups group_prefix[n] ..
// group_prefix[n+1]-1, image (group * n_fgroups + feature group).
struct PartialView {
  int32_t *partial;
  const int32_t *group_prefix;  // groups of node n: group_prefix[n + 1] - group_prefix[n]
  const int32_t *img_first;     // the first group image of node n (the node's images are consecutive)
  int64_t r_cap;                // images below r_cap (in groups) are in the reduce region: zeroed once read
  int64_t image_int4s;
  int32_t n_fgroups, sbw, nsb, B;
};

// Cell (slot s) of feature f of group image `group` (a node's first is
// img_first[n]); the next group's image is image_stride int2 further.
__device__ __forceinline__ int2 *image_cell(const PartialView &v, int32_t group, int f, int item_feats, int s) {
  const int fg = f / item_feats, fl = f - fg * item_feats;
  const int sb = fl / v.sbw, c = fl - sb * v.sbw;
  const int64_t image = (int64_t)group * v.n_fgroups + fg;
  return reinterpret_cast<int2 *>(v.partial) + image * v.image_int4s * 2 + ((int64_t)sb * v.B + s) * v.sbw + c;
}

// Finalize: the int64 histogram of every (node, feature, slot) is the sum of
// the node's group images (reduce-region images are zeroed as they are read).
// One thread per cell; four consecutive threads take four consecutive
// features of one slot (one 32-byte sector of an image row).
__global__ void __launch_bounds__(256) k_finalize(PartialView v, int32_t n_nodes, int32_t n_features,
                                                  int32_t item_feats, int64_t *__restrict__ hist_out,
                                                  const DevState *st) {
  pdl_wait();     // the histogram kernel
  pdl_trigger();  // the split find may launch; it waits for this grid to finish
  if (!st->plan_ok) return;
  const int nq = (n_features + 3) >> 2;
  const int64_t units = (int64_t)n_nodes * nq * v.B * 4;
  const int64_t image_stride = v.n_fgroups * v.image_int4s * 2;  // int2 between a node's group images
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int fi = (int)(u & 3);
    int64_t r = u >> 2;
    const int s = (int)(r % v.B);
    r /= v.B;
    const int qd = (int)(r % nq);
    const int n = (int)(r / nq);
    const int f = qd * 4 + fi;
    if (f >= n_features) continue;
    const int32_t g0 = v.group_prefix[n], g1 = v.group_prefix[n + 1], i0 = v.img_first[n];
    const bool zero = i0 < v.r_cap;
    int2 *cell = image_cell(v, i0, f, item_feats, s);
    int64_t g = 0, h = 0;
    // the loads first, then the zeroing stores (a store between two loads
    // would keep the next load from being issued before the store)
    int2 *c = cell;
    for (int32_t k = g0; k < g1; ++k, c += image_stride) {
      const int2 x = __ldcg(c);
      g += x.x;
      h += x.y;
    }
    if (zero)
      for (int32_t k = g0; k < g1; ++k, cell += image_stride) __stcg(cell, make_int2(0, 0));
    reinterpret_cast<longlong2 *>(hist_out)[((int64_t)n * n_features + f) * v.B + s] = make_longlong2(g, h);
  }
}

// Multi-output finalize: hist_out [k][n][F][B][2] int64, target-major, from the
// group images of the MULTI build (feature group = target group * nfq +
// feature quarter; sub-block = target within its group of four; column = the
// feature within its quarter). One thread per cell; four consecutive threads
// take four consecutive features of one slot (one 32-byte sector of an image
// row).
__global__ void __launch_bounds__(256) k_finalize_multi(PartialView v, int32_t n_targets, int32_t n_nodes,
                                                        int32_t n_features, int64_t *__restrict__ hist_out,
                                                        const DevState *st) {
  pdl_wait();  // the histogram kernel
  if (!st->plan_ok) return;
  const int nq = (n_features + 3) >> 2;
  const int nfq = (n_features + 15) >> 4;
  const int64_t units = (int64_t)n_targets * n_nodes * nq * v.B * 4;
  const int64_t image_stride = v.n_fgroups * v.image_int4s * 2;  // int2 between a node's group images
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int fi = (int)(u & 3);
    int64_t r = u >> 2;
    const int s = (int)(r % v.B);
    r /= v.B;
    const int qd = (int)(r % nq);
    r /= nq;
    const int n = (int)(r % n_nodes);
    const int t = (int)(r / n_nodes);
    const int f = qd * 4 + fi;
    if (f >= n_features) continue;
    const int fq = f >> 4, fl = f & 15, tg = t >> 2, tl = t & 3;
    const int32_t g0 = v.group_prefix[n], g1 = v.group_prefix[n + 1], i0 = v.img_first[n];
    const bool zero = i0 < v.r_cap;
    const int64_t image = (int64_t)i0 * v.n_fgroups + (int64_t)tg * nfq + fq;
    int2 *cell = reinterpret_cast<int2 *>(v.partial) + image * v.image_int4s * 2 + ((int64_t)tl * v.B + s) * 16 + fl;
    int64_t g = 0, h = 0;
    int2 *c = cell;
    for (int32_t k = g0; k < g1; ++k, c += image_stride) {  // loads first, then the zeroing stores
      const int2 x = __ldcg(c);
      g += x.x;
      h += x.y;
    }
    if (zero)
      for (int32_t k = g0; k < g1; ++k, cell += image_stride) __stcg(cell, make_int2(0, 0));
    reinterpret_cast<longlong2 *>(hist_out)[(((int64_t)t * n_nodes + n) * n_features + f) * v.B + s] =
        make_longlong2(g, h);
  }
}

}  // namespace gbt
