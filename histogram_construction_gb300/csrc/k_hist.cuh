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
//  * work items (node, feature group, row chunk) handed out to a persistent
//    grid by an atomic counter;
//  * one CTA holds a 64-feature x 256-slot histogram of int32 (G, H) pairs in
//    shared memory (128 KB); each lane adds (qg, qh) with two 32-bit shared
//    atomics, and the column order of the features is permuted so that the 32
//    lanes of every atomic instruction hit 32 different banks whatever the bin
//    values (no bank conflicts, no same-address conflicts);
//  * a chunk never holds more rows than keep every int32 partial exact
//    (rows * max|q| < 2^31), so the int64 result is exact;
//  * the flush converts to int64 in a padded staging buffer and writes each
//    feature's slot strip with one TMA bulk copy (single-chunk node) or one
//    bulk reduce-add into the zeroed output (multi-chunk node).
#pragma once

#include "common.cuh"

namespace gbt {

constexpr int CHUNK_MIN_ROWS = 4096;

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
__global__ void __launch_bounds__(1024) k_level_prologue(LevelParams p) {
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
  if (p.rows != nullptr) {
    uint32_t bad = 0;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < Rg; k += (int64_t)gridDim.x * blockDim.x) {
      const int32_t r = p.rows[k];
      int4 rec;
      if (r >= 0 && r < p.n_rows) {
        const int2 qq = p.q[r];
        rec = make_int4(r, qq.x, qq.y, 0);
      } else {
        rec = make_int4(-1, 0, 0, 0);
        bad = 1;
      }
      p.rec[k] = rec;
    }
    if (bad) raise_err(p.st, ERRBIT_ROW);
  }
  // zero the outputs of multi-chunk nodes (they are reduced into)
  for (int n = 0; n < p.n_nodes; ++n) {
    const int64_t rows_n = p.offs[n + 1] - p.offs[n];
    if (rows_n <= chunk) continue;
    int4 *dst = reinterpret_cast<int4 *>(p.hist_out + (int64_t)n * p.node_int64s);
    const int64_t units = p.node_int64s / 2;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x)
      dst[u] = make_int4(0, 0, 0, 0);
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
// u8 kernel: 64 features per item, conflict-free column permutation.
//
// Lane l of a warp takes row rho = l/4 of an 8-row group and the 16-byte
// quarter qq = l%4 of the row's 64-byte strip (words 4qq..4qq+3). For atomic
// instruction (e, j, c) the lane uses word w = 4qq + ((e + rho/2) & 3), byte j,
// and component (c ^ (rho & 1)) (0 = G, 1 = H). Feature f = 4w + j lives in
// column col(f) = 16 j + ((w + 4 j) & 15) of a 64-cell slot row; the word
// index of the component is 2 (slot * 64 + col) + comp, whose bank is
// 2 ((w + 4 j) & 15) + comp = 2 (4 ((qq + j) & 3) + ((e + rho/2) & 3)) + comp:
// distinct for the 32 lanes.
constexpr int H8_THREADS = 1024;
constexpr int H8_HIST_BYTES = 256 * 64 * 8;          // slots x columns x (G,H) int32
constexpr int H8_STAGE_ROW = 256 * 16 + 16;          // one feature's int64 strip + 16 B pad
constexpr int H8_STAGE_FEATS = 16;
constexpr int H8_SMEM = H8_HIST_BYTES + H8_STAGE_FEATS * H8_STAGE_ROW;
constexpr int H8_UNROLL = 4;

__device__ __forceinline__ int h8_col(int f) {
  const int w = f >> 2, j = f & 3;
  return 16 * j + ((w + 4 * j) & 15);
}

struct Hist8Params {
  LevelParams lv;
  const uint8_t *mirror;  // [n_tiles][N][64]
  int32_t n_features;
  int32_t n_slots;        // B
};

__global__ void __launch_bounds__(H8_THREADS, 1) k_hist_u8(Hist8Params P) {
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
  const int rho = lane >> 2, qq = lane & 3;
  const int pr = rho >> 1, par = rho & 1;
  // per-lane byte offsets of (e, j) columns, without the slot term
  int colbyte[4][4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int w = 4 * qq + ((e + pr) & 3);
      colbyte[e][j] = (16 * j + ((w + 4 * j) & 15)) * 8;
    }
  const int off0 = par ? 4 : 0;  // instruction c=0 component byte offset
  const int off1 = par ? 0 : 4;
  const uint32_t hist_base = smem_addr(hist);

  for (;;) {
    if (threadIdx.x == 0) s_item = (int32_t)atomicAdd(&p.st->work_next, 1u);
    __syncthreads();
    const int32_t id = s_item;
    if (id >= n_items) break;
    const Item it = decode_item(id, p, chunk);
    // zero the shared histogram (B slot rows)
    {
      uint4 *h4 = reinterpret_cast<uint4 *>(hist);
      const int n4 = B * 64 * 8 / 16;
      for (int i = threadIdx.x; i < n4; i += blockDim.x) h4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // accumulate
    const unsigned char *strip = P.mirror + (int64_t)it.fgroup * N * MIRROR_STRIP_BYTES + qq * 16;
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
      uint4 bv[H8_UNROLL];
#pragma unroll
      for (int u = 0; u < H8_UNROLL; ++u) {
        bv[u] = make_uint4(0, 0, 0, 0);
        if (rr[u] >= 0) bv[u] = ldg_nc_v4(strip + (int64_t)rr[u] * MIRROR_STRIP_BYTES);
      }
#pragma unroll
      for (int u = 0; u < H8_UNROLL; ++u) {
        if (rr[u] < 0) continue;
        const uint32_t v0 = par ? (uint32_t)vh[u] : (uint32_t)vg[u];
        const uint32_t v1 = par ? (uint32_t)vg[u] : (uint32_t)vh[u];
        // rotate the 4 words by pr so that word index e of the rotated set is (e + pr) & 3
        uint32_t wd[4];
        {
          const uint32_t a0 = bv[u].x, a1 = bv[u].y, a2 = bv[u].z, a3 = bv[u].w;
          wd[0] = pr == 0 ? a0 : pr == 1 ? a1 : pr == 2 ? a2 : a3;
          wd[1] = pr == 0 ? a1 : pr == 1 ? a2 : pr == 2 ? a3 : a0;
          wd[2] = pr == 0 ? a2 : pr == 1 ? a3 : pr == 2 ? a0 : a1;
          wd[3] = pr == 0 ? a3 : pr == 1 ? a0 : pr == 2 ? a1 : a2;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t slot = (wd[e] >> (8 * j)) & 0xffu;
            const uint32_t a = hist_base + slot * 512u + (uint32_t)colbyte[e][j];
            asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a + off0), "r"(v0) : "memory");
            asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a + off1), "r"(v1) : "memory");
          }
      }
    }
    __syncthreads();
    // flush: 4 rounds of 16 features
    const int f_tile0 = it.fgroup * 64;
    int64_t *node_out = p.hist_out + (int64_t)it.node * p.node_int64s;
    for (int r = 0; r < 4; ++r) {
      const int f_first = f_tile0 + 16 * r;
      if (f_first >= P.n_features) break;
      // convert: lane -> (fi = lane & 15, slot = 2*warp + (lane >> 4) + 2*nwarps*i)
      const int fi = lane & 15;
      const int col = h8_col(16 * r + fi);
      for (int s = 2 * warp + (lane >> 4); s < B; s += 2 * nwarps) {
        const uint2 gh = *reinterpret_cast<const uint2 *>(hist + 2 * (s * 64 + col));
        longlong2 v;
        v.x = (long long)(int32_t)gh.x;
        v.y = (long long)(int32_t)gh.y;
        *reinterpret_cast<longlong2 *>(stage + fi * H8_STAGE_ROW + s * 16) = v;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)B * 16u;
        for (int k = 0; k < 16; ++k) {
          const int f = f_first + k;
          if (f >= P.n_features) break;
          int64_t *dst = node_out + (int64_t)f * B * 2;
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
