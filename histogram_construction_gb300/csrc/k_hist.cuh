// Level-batched histogram build: level prologue (plan, gather, zero) and the
// persistent shared-memory histogram kernels.
//
// What is computed [bonsai "10: CUDA histogram backend", "Level batching" and
// "The kernel"; "GBDT engine engineering deep-dive" (ybb.press), section 1
// per-row loop and section 7 shared-memory histograms]: for every node n of the
// batch, every feature f and slot s,
//   Hist[n][f][s] = sum over rows k of node n with slot(bins[f][row_k]) == s of (qg, qh).
//
// GB300 design (differs from the pages' (feature, node, row-chunk) grid with
// float shared cells):
//  * work items (node, 16-feature group, row chunk) handed out to a persistent
//    grid of several CTAs per SM by an atomic counter;
//  * a CTA holds a 16-feature x 256-slot histogram of int32 (G, H) pairs in
//    shared memory (32 KB); each lane adds (qg, qh) with two 32-bit shared
//    atomics, and lanes are assigned to (row, feature, component) so that the
//    32 lanes of every atomic instruction hit 32 different banks whatever the
//    bin values (no bank conflicts, no same-address conflicts);
//  * a chunk never holds more rows than keep every int32 partial exact
//    (rows * max|q| < 2^31), so the int64 result is exact;
//  * the flush transposes the cells to int64 through a small padded staging
//    buffer and writes each feature's slot range with one TMA bulk copy
//    (node built by one item) or one bulk reduce-add into the zeroed output
//    (node split into several chunks).
#pragma once

#include "common.cuh"

namespace gbt {

constexpr int CHUNK_MIN_ROWS = 2048;

struct LevelParams {
  const int32_t *rows;   // level row list or nullptr (identity)
  const int64_t *offs;   // [n_nodes + 1]
  int32_t n_nodes;
  int32_t n_fgroups;     // feature groups per node chunk (work items per chunk)
  int32_t target_items;  // load-balance target for the item count
  int32_t pad;
  int64_t n_rows;
  const int2 *q;         // quantised gpair [n_rows]
  int4 *rec;             // gathered level records {row, qg, qh, 0} [n_rows]
  int32_t *chunk_prefix; // [n_nodes + 1]
  int64_t *hist_out;     // [n_nodes][F][B][2]
  int64_t node_int64s;   // F * B * 2
  DevState *st;
};

__device__ __forceinline__ int64_t level_chunk_rows(const LevelParams &p) {
  const int64_t R = p.offs[p.n_nodes] - p.offs[0];
  const uint32_t qm = max(p.st->qmax, 1u);
  const int64_t rc = 2147483647LL / (int64_t)qm;  // rows whose int32 partials cannot overflow
  int64_t tgt = (max(R, (int64_t)0) * p.n_fgroups + p.target_items - 1) / max(p.target_items, 1);
  tgt = max(tgt, (int64_t)CHUNK_MIN_ROWS);
  return max((int64_t)1, min(rc, tgt));
}

// Level prologue: block 0 plans the work items; all blocks gather the level
// records (row id and its quantised pair, in level order) and zero the
// outputs of nodes that will be reduced from several chunks.
__global__ void __launch_bounds__(512) k_level_prologue(LevelParams p) {
  const int64_t chunk = level_chunk_rows(p);
  const int64_t R = p.offs[p.n_nodes] - p.offs[0];
  if (blockIdx.x == 0) {
    __shared__ int32_t s_carry;
    __shared__ int32_t s_bad;
    __shared__ int32_t s_warp[32];
    if (threadIdx.x == 0) {
      s_carry = 0;
      s_bad = (p.offs[0] != 0 || R > p.n_rows || R < 0) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < p.n_nodes; base += blockDim.x) {
      const int n = base + threadIdx.x;
      int32_t c = 0;
      if (n < p.n_nodes) {
        const int64_t a = p.offs[n], b = p.offs[n + 1];
        if (b < a) s_bad = 1;
        const int64_t rows_n = max(b - a, (int64_t)0);
        c = (int32_t)max((int64_t)1, (rows_n + chunk - 1) / chunk);
      }
      // block inclusive scan of c
      int32_t v = c;
      const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane == 31) s_warp[w] = v;
      __syncthreads();
      if (w == 0) {
        int32_t x = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        s_warp[lane] = x;
      }
      __syncthreads();
      const int32_t incl = v + (w > 0 ? s_warp[w - 1] : 0) + s_carry;
      if (n < p.n_nodes) p.chunk_prefix[n + 1] = incl;
      __syncthreads();
      if (threadIdx.x == blockDim.x - 1) s_carry = incl;
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      p.chunk_prefix[0] = 0;
      const int ok = !s_bad;
      p.st->plan_ok = ok;
      p.st->chunk_rows = chunk;
      p.st->n_items = ok ? s_carry * p.n_fgroups : 0;
      p.st->work_next = 0;
      if (!ok) raise_err(p.st, ERRBIT_ROW);
    }
  }
  // gather level records (bounded by n_rows whatever the offsets say)
  const int64_t Rg = min(max(R, (int64_t)0), p.n_rows);
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p.rows != nullptr) {
    uint32_t bad = 0;
    for (int64_t k0 = gtid; k0 < Rg; k0 += 4 * nthr) {
      int32_t r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = k0 + u * nthr;
        r[u] = k < Rg ? __ldg(p.rows + k) : -1;
      }
      int2 qq[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool ok = r[u] >= 0 && r[u] < p.n_rows;
        qq[u] = ok ? __ldg(p.q + r[u]) : make_int2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = k0 + u * nthr;
        if (k >= Rg) break;
        const bool ok = r[u] >= 0 && r[u] < p.n_rows;
        if (!ok) bad = 1;
        p.rec[k] = ok ? make_int4(r[u], qq[u].x, qq[u].y, 0) : make_int4(-1, 0, 0, 0);
      }
    }
    if (bad) raise_err(p.st, ERRBIT_ROW);
  }
  // zero the outputs of multi-chunk nodes (they are reduced into)
  const int64_t units = p.node_int64s / 2;
  for (int n = 0; n < p.n_nodes; ++n) {
    const int64_t rows_n = __ldg(p.offs + n + 1) - __ldg(p.offs + n);
    if (rows_n <= chunk) continue;
    int4 *dst = reinterpret_cast<int4 *>(p.hist_out + (int64_t)n * p.node_int64s);
    for (int64_t u = gtid; u < units; u += nthr) dst[u] = make_int4(0, 0, 0, 0);
  }
}

// Decode a work item id into node, feature group and row range.
struct Item {
  int32_t node, fgroup;
  int64_t k0, k1;
  int32_t multi;
};

__device__ __forceinline__ Item decode_item(int32_t id, const LevelParams &p, int64_t chunk) {
  Item it;
  const int32_t kc = id / p.n_fgroups;
  it.fgroup = id - kc * p.n_fgroups;
  int lo = 0, hi = p.n_nodes - 1;  // largest n with chunk_prefix[n] <= kc
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.chunk_prefix[mid] <= kc) lo = mid; else hi = mid - 1;
  }
  it.node = lo;
  const int32_t c = kc - p.chunk_prefix[lo];
  const int64_t a = p.offs[lo], b = p.offs[lo + 1];
  it.k0 = a + (int64_t)c * chunk;
  it.k1 = min(b, it.k0 + chunk);
  it.multi = (p.chunk_prefix[lo + 1] - p.chunk_prefix[lo]) > 1;
  return it;
}

// ----------------------------------------------------------------------------
// u8 kernel: 16 features per item (one quarter of a 64-byte mirror strip).
//
// Lane l of a warp takes row rho = l/4 of an 8-row group and byte word
// w = l%4 of the row's 16-byte quarter (one 32-bit load). In atomic
// instruction (j, c) the lane adds byte jj = (j + rho/2) & 3 of its word,
// i.e. feature f = 4w + jj, component (c ^ (rho & 1)) (0 = G, 1 = H). Cells
// are [slot][16 features][G, H]; a slot row is 128 bytes = 32 banks, so the
// bank of a lane is 2f + comp: distinct for the 32 lanes of every
// instruction (f covers 16 values over (w, rho/2), comp separates rho&1).
constexpr int H8_THREADS = 256;
constexpr int H8_TS = 16;                                  // features per item
constexpr int H8_HIST_BYTES = 256 * H8_TS * 8;             // 32 KB
constexpr int H8_STAGE_SLOTS = 64;                         // slots per flush round
constexpr int H8_STAGE_ROW = (H8_STAGE_SLOTS + 1) * 16;    // one feature's int64 pairs + pad
constexpr int H8_SMEM = H8_HIST_BYTES + H8_TS * H8_STAGE_ROW;
constexpr int H8_UNROLL = 8;

struct Hist8Params {
  LevelParams lv;
  const uint8_t *mirror;  // [n_tiles][N][64]
  int32_t n_features;
  int32_t n_slots;        // B
};

__global__ void __launch_bounds__(H8_THREADS, 4) k_hist_u8(Hist8Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem);
  unsigned char *stage = smem + H8_HIST_BYTES;
  __shared__ int32_t s_item;

  const LevelParams &p = P.lv;
  if (!p.st->plan_ok) return;
  const int64_t chunk = p.st->chunk_rows;
  const int32_t n_items = p.st->n_items;
  const int B = P.n_slots;
  const int64_t N = p.n_rows;
  const bool ident = (p.rows == nullptr);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rho = lane >> 2, w = lane & 3;
  const int pr = rho >> 1, par = rho & 1;
  // per-lane byte shift and column byte offset of instruction j
  uint32_t shift[4], colb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = (j + pr) & 3;
    shift[j] = 8u * jj;
    colb[j] = (uint32_t)(4 * w + jj) * 8u;
  }
  const uint32_t off0 = par ? 4u : 0u, off1 = par ? 0u : 4u;
  const uint32_t hist_base = smem_addr(hist);

  for (;;) {
    if (threadIdx.x == 0) s_item = (int32_t)atomicAdd(&p.st->work_next, 1u);
    __syncthreads();
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = decode_item(id, p, chunk);
    {
      uint4 *h4 = reinterpret_cast<uint4 *>(hist);
      const int n4 = B * H8_TS * 8 / 16;
      for (int i = threadIdx.x; i < n4; i += blockDim.x) h4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int tile = it.fgroup >> 2, sub = it.fgroup & 3;
    const unsigned char *strip = P.mirror + (int64_t)tile * N * MIRROR_STRIP_BYTES + sub * 16 + w * 4;
    const int64_t step = (int64_t)8 * nwarps;
    for (int64_t g0 = it.k0 + 8 * warp; g0 < it.k1; g0 += step * H8_UNROLL) {
      int32_t rr[H8_UNROLL], vg[H8_UNROLL], vh[H8_UNROLL];
#pragma unroll
      for (int u = 0; u < H8_UNROLL; ++u) {
        const int64_t k = g0 + u * step + rho;
        rr[u] = -1;
        vg[u] = 0;
        vh[u] = 0;
        if (k < it.k1) {
          if (ident) {
            const int2 qv = __ldg(&p.q[k]);
            rr[u] = (int32_t)k;
            vg[u] = qv.x;
            vh[u] = qv.y;
          } else {
            const int4 rc = __ldg(&p.rec[k]);
            rr[u] = rc.x;
            vg[u] = rc.y;
            vh[u] = rc.z;
          }
        }
      }
      uint32_t bw[H8_UNROLL];
#pragma unroll
      for (int u = 0; u < H8_UNROLL; ++u)
        bw[u] = rr[u] >= 0 ? __ldg(reinterpret_cast<const uint32_t *>(strip + (int64_t)rr[u] * MIRROR_STRIP_BYTES))
                           : 0u;
#pragma unroll
      for (int u = 0; u < H8_UNROLL; ++u) {
        if (rr[u] < 0) continue;
        const uint32_t v0 = par ? (uint32_t)vh[u] : (uint32_t)vg[u];
        const uint32_t v1 = par ? (uint32_t)vg[u] : (uint32_t)vh[u];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t slot = (bw[u] >> shift[j]) & 0xffu;
          const uint32_t a = hist_base + slot * (H8_TS * 8) + colb[j];
          asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a + off0), "r"(v0) : "memory");
          asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a + off1), "r"(v1) : "memory");
        }
      }
    }
    __syncthreads();
    // flush: rounds of 64 slots; lanes over features for conflict-free reads,
    // staging rows padded by 16 bytes for conflict-free 16-byte writes
    const int f0 = it.fgroup * H8_TS;
    int64_t *node_out = p.hist_out + (int64_t)it.node * p.node_int64s;
    for (int s0 = 0; s0 < B; s0 += H8_STAGE_SLOTS) {
      const int ns = min(H8_STAGE_SLOTS, B - s0);
      for (int idx = threadIdx.x; idx < H8_TS * H8_STAGE_SLOTS; idx += blockDim.x) {
        const int fl = idx & (H8_TS - 1), sl = idx >> 4;
        if (sl < ns) {
          const uint2 gh = *reinterpret_cast<const uint2 *>(hist + 2 * ((s0 + sl) * H8_TS + fl));
          longlong2 v;
          v.x = (long long)(int32_t)gh.x;
          v.y = (long long)(int32_t)gh.y;
          *reinterpret_cast<longlong2 *>(stage + fl * H8_STAGE_ROW + sl * 16) = v;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)ns * 16u;
        for (int k = 0; k < H8_TS; ++k) {
          const int f = f0 + k;
          if (f >= P.n_features) break;
          int64_t *dst = node_out + ((int64_t)f * B + s0) * 2;
          if (it.multi) bulk_reduce_add_u64(dst, stage + k * H8_STAGE_ROW, bytes);
          else bulk_store(dst, stage + k * H8_STAGE_ROW, bytes);
        }
        bulk_commit();
        bulk_wait_read_all();
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) bulk_wait_all();
}

// ----------------------------------------------------------------------------
// u16 kernel: TS features per item (TS = 2..32), any B with TS * B * 8 within
// the shared budget. Missing-slot entries are summed in registers and added
// once per item (40% of entries can be missing; they would all hit one cell).
constexpr int H16_THREADS = 512;
constexpr int H16_HIST_MAX = 160 * 1024;
constexpr int H16_STAGE_SLOTS = 2048;
constexpr int H16_STAGE_BYTES = H16_STAGE_SLOTS * 16;

struct Hist16Params {
  LevelParams lv;
  const uint16_t *mirror;  // [n_tiles][N][32]
  int32_t n_features;
  int32_t n_slots;         // B
  int32_t n_bins;
  int32_t ts;              // features per item
};

template <int TS>
__global__ void __launch_bounds__(H16_THREADS, 1) k_hist_u16(Hist16Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int W = TS / 2;        // u32 words per row in an item
  constexpr int RPI = 32 / W;      // rows per warp instruction
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem);
  const int B = P.n_slots;
  const int hist_bytes = ((B * TS * 8) + 127) & ~127;
  unsigned char *stage = smem + hist_bytes;
  __shared__ int32_t s_item;

  const LevelParams &p = P.lv;
  if (!p.st->plan_ok) return;
  const int64_t chunk = p.st->chunk_rows;
  const int32_t n_items = p.st->n_items;
  const int64_t N = p.n_rows;
  const bool ident = (p.rows == nullptr);
  const uint32_t miss_slot = (uint32_t)P.n_bins;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rho = lane / W, wi = lane % W;
  constexpr int GROUPS_PER_TILE = 32 / TS;

  for (;;) {
    if (threadIdx.x == 0) s_item = (int32_t)atomicAdd(&p.st->work_next, 1u);
    __syncthreads();
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = decode_item(id, p, chunk);
    {
      uint4 *h4 = reinterpret_cast<uint4 *>(hist);
      const int n4 = (B * TS * 8) / 16;
      for (int i = threadIdx.x; i < n4; i += blockDim.x) h4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int tile = it.fgroup / GROUPS_PER_TILE;
    const int sub = it.fgroup % GROUPS_PER_TILE;
    const unsigned char *strip =
        reinterpret_cast<const unsigned char *>(P.mirror) + (int64_t)tile * N * MIRROR_STRIP_BYTES + sub * TS * 2 + wi * 4;
    int32_t mg0 = 0, mh0 = 0, mg1 = 0, mh1 = 0;  // missing-slot partials of features 2wi, 2wi+1
    const int64_t step = (int64_t)RPI * nwarps;
    for (int64_t g0 = it.k0 + RPI * warp; g0 < it.k1; g0 += step * 4) {
      int32_t rr[4], vg[4], vh[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = g0 + u * step + rho;
        rr[u] = -1; vg[u] = 0; vh[u] = 0;
        if (k < it.k1) {
          if (ident) {
            const int2 qv = __ldg(&p.q[k]);
            rr[u] = (int32_t)k; vg[u] = qv.x; vh[u] = qv.y;
          } else {
            const int4 rc = __ldg(&p.rec[k]);
            rr[u] = rc.x; vg[u] = rc.y; vh[u] = rc.z;
          }
        }
      }
      uint32_t bw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        bw[u] = 0;
        if (rr[u] >= 0) bw[u] = __ldg(reinterpret_cast<const uint32_t *>(strip + (int64_t)rr[u] * MIRROR_STRIP_BYTES));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (rr[u] < 0) continue;
        const uint32_t s0 = bw[u] & 0xffffu, s1 = bw[u] >> 16;
        if (s0 == miss_slot) { mg0 += vg[u]; mh0 += vh[u]; }
        else {
          uint32_t *c = hist + 2 * (s0 * TS + 2 * wi);
          atomicAdd(c, (uint32_t)vg[u]);
          atomicAdd(c + 1, (uint32_t)vh[u]);
        }
        if (s1 == miss_slot) { mg1 += vg[u]; mh1 += vh[u]; }
        else {
          uint32_t *c = hist + 2 * (s1 * TS + 2 * wi + 1);
          atomicAdd(c, (uint32_t)vg[u]);
          atomicAdd(c + 1, (uint32_t)vh[u]);
        }
      }
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
      uint32_t *c0 = hist + 2 * (miss_slot * TS + 2 * wi);
      atomicAdd(c0, (uint32_t)mg0);
      atomicAdd(c0 + 1, (uint32_t)mh0);
      uint32_t *c1 = hist + 2 * (miss_slot * TS + 2 * wi + 1);
      atomicAdd(c1, (uint32_t)mg1);
      atomicAdd(c1 + 1, (uint32_t)mh1);
    }
    __syncthreads();
    // flush per feature in slot chunks
    const int f_item0 = it.fgroup * TS;
    int64_t *node_out = p.hist_out + (int64_t)it.node * p.node_int64s;
    for (int fl = 0; fl < TS; ++fl) {
      const int f = f_item0 + fl;
      if (f >= P.n_features) break;
      for (int s0 = 0; s0 < B; s0 += H16_STAGE_SLOTS) {
        const int ns = min(H16_STAGE_SLOTS, B - s0);
        for (int i = threadIdx.x; i < ns; i += blockDim.x) {
          const uint2 gh = *reinterpret_cast<const uint2 *>(hist + 2 * ((s0 + i) * TS + fl));
          longlong2 v;
          v.x = (long long)(int32_t)gh.x;
          v.y = (long long)(int32_t)gh.y;
          *reinterpret_cast<longlong2 *>(stage + i * 16) = v;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
          int64_t *dst = node_out + ((int64_t)f * B + s0) * 2;
          if (it.multi) bulk_reduce_add_u64(dst, stage, (uint32_t)ns * 16u);
          else bulk_store(dst, stage, (uint32_t)ns * 16u);
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncthreads();
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait_all();
}

}  // namespace gbt
