// Level row partition [bonsai "10: CUDA histogram backend", "The device
// context lifecycle": each parent segment is routed into stable left and
// right child segments by a count / scan / scatter over the resident rows].
//
// Node n's rows (positions [offs[n], offs[n+1]) of the level list) go to child
// 2n when slot(bin[feature][row]) <= bin (or the slot is missing and
// default_left = 1) and to child 2n+1 otherwise, keeping their order. Left
// child 2n starts at offs[n]; right child 2n+1 starts at offs[n] + left_n.
//
// Three kernels over the flat level list in tiles of PART_TILE positions:
// per-tile left counts, one-block scan of the tile counts, then per-tile
// recompute + block scan + scatter.
//
// Optionally the scatter also writes every pair's smaller child (fewer rows;
// the left one on a tie) into a compact list: small_rows holds, in pair
// order, the rows of child 2n + small_side[n], in their order, with pair n's
// segment at [small_offs[n], small_offs[n+1]). This is the input of the next
// level's smaller-sibling build [bonsai "10: CUDA histogram backend", "The
// device context lifecycle": advance_level builds the smaller siblings in one
// pass].
#pragma once

#include "common.cuh"
#include "k_split.cuh"

namespace gbt {

constexpr int PART_THREADS = 512;
constexpr int PART_TILE = 4096;  // positions per tile (8 per thread)

struct PartParams {
  const int32_t *rows;  // nullptr = identity
  const int64_t *offs;  // [n_nodes + 1]
  int32_t n_nodes;
  int32_t tile_feats;   // features per mirror tile
  int32_t bin_bytes;
  int32_t n_bins;
  int32_t n_features;
  int32_t pad;
  int64_t n_rows;       // also the bound on the level length
  const unsigned char *mirror;
  const SplitOut *splits;
  int64_t *tile_counts;  // [n_tiles + 1]
  int32_t *out_rows;
  int64_t *out_offs;     // [2 n_nodes + 1]
  int32_t *small_rows;   // optional: rows of each pair's smaller child, pair order
  int64_t *small_offs;   // [n_nodes + 1] with small_rows
  uint8_t *small_side;   // [n_nodes] with small_rows: 0 = child 2n is the smaller, 1 = child 2n + 1
  DevState *st;
};

__device__ __forceinline__ int64_t part_len(const PartParams &p) {
  return min(max(p.offs[p.n_nodes], (int64_t)0), p.n_rows);
}

__device__ __forceinline__ int part_node_of(const PartParams &p, int64_t k) {
  int lo = 0, hi = p.n_nodes - 1;  // largest n with offs[n] <= k
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.offs[mid] <= k) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 1 = left, 0 = right; also returns the row id.
__device__ __forceinline__ int part_flag(const PartParams &p, int64_t k, int32_t &row) {
  const int n = part_node_of(p, k);
  const int32_t r = p.rows ? p.rows[k] : (int32_t)k;
  row = r;
  const SplitOut sp = p.splits[n];
  if (sp.feature < 0 || sp.feature >= p.n_features) return 1;  // no split (or an invalid one): all left
  if (r < 0 || r >= p.n_rows) return 1;
  const int64_t tile = sp.feature / p.tile_feats, fi = sp.feature % p.tile_feats;
  const unsigned char *strip = p.mirror + mirror_offset(tile, r, p.n_rows);
  const uint32_t slot = p.bin_bytes == 1 ? (uint32_t)strip[fi] : (uint32_t)reinterpret_cast<const uint16_t *>(strip)[fi];
  if (slot == (uint32_t)p.n_bins) return sp.default_left ? 1 : 0;
  return (int32_t)slot <= sp.bin ? 1 : 0;
}

__global__ void __launch_bounds__(PART_THREADS) k_part_count(PartParams p) {
  const int64_t R = part_len(p);
  if (blockIdx.x == 0) {
    // offsets must start at 0, ascend and stay within n_rows; otherwise the
    // later kernels do nothing (plan_ok = 0) and the error word says why
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = (p.offs[0] != 0 || p.offs[p.n_nodes] > p.n_rows) ? 1 : 0;
    __syncthreads();
    for (int n = threadIdx.x; n < p.n_nodes; n += blockDim.x)
      if (p.offs[n + 1] < p.offs[n]) s_bad = 1;
    __syncthreads();
    if (threadIdx.x == 0) {
      p.st->plan_ok = s_bad ? 0 : 1;
      if (s_bad) raise_err(p.st, ERRBIT_ROW);
    }
  }
  const int64_t base = (int64_t)blockIdx.x * PART_TILE;
  int c = 0;
  uint32_t bad = 0;
  for (int i = threadIdx.x; i < PART_TILE; i += blockDim.x) {
    const int64_t k = base + i;
    if (k < R) {
      int32_t r;
      c += part_flag(p, k, r);
      if (r < 0 || r >= p.n_rows) bad = 1;
    }
  }
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  __shared__ int s[PART_THREADS / 32];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < PART_THREADS / 32; ++w) t += s[w];
    p.tile_counts[blockIdx.x] = t;
  }
  if (bad) raise_err(p.st, ERRBIT_ROW);
}

// Exclusive scan of tile counts in place (tile_counts[n_tiles] = total); also
// writes the child offsets. One block.
__global__ void __launch_bounds__(1024) k_part_scan(PartParams p, int64_t n_tiles) {
  __shared__ long long s_carry;
  __shared__ long long s_w[32];
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int64_t base = 0; base < n_tiles; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    long long v = i < n_tiles ? p.tile_counts[i] : 0;
    long long x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_w[w] = x;
    __syncthreads();
    if (w == 0) {
      long long z = s_w[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      s_w[lane] = z;
    }
    __syncthreads();
    const long long incl = x + (w > 0 ? s_w[w - 1] : 0) + s_carry;
    if (i < n_tiles) p.tile_counts[i] = incl - v;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.tile_counts[n_tiles] = s_carry;
}

// Recompute flags, block exclusive scan, scatter. Needs the global left rank
// of the first position of every node: lrank(k) = number of left rows in
// [0, k). Node n: left child gets [offs[n], offs[n] + L_n) where
// L_n = lrank(offs[n+1]) - lrank(offs[n]).
// lrank at node boundaries is read from the scatter of the tile containing
// them, so node boundaries are resolved in a fourth tiny step (k_part_offsets).
__global__ void __launch_bounds__(PART_THREADS) k_part_rank(PartParams p, int64_t *lrank_at) {
  // lrank_at[k] for every k in this tile is not stored; instead each position
  // that starts a node (k == offs[n]) records its rank so offsets can be built.
  if (!p.st->plan_ok) return;
  const int64_t R = part_len(p);
  const int64_t base = (int64_t)blockIdx.x * PART_TILE;
  constexpr int PER = PART_TILE / PART_THREADS;  // 8 positions per thread, contiguous
  int flags[PER];
  int32_t rows[PER];
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int64_t k = base + (int64_t)threadIdx.x * PER + j;
    flags[j] = 0;
    rows[j] = -1;
    if (k < R) flags[j] = part_flag(p, k, rows[j]);
    cnt += flags[j];
  }
  // block exclusive scan of cnt
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __shared__ int s_w[PART_THREADS / 32];
  if (lane == 31) s_w[w] = x;
  __syncthreads();
  if (w == 0) {
    int z = lane < PART_THREADS / 32 ? s_w[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < PART_THREADS / 32) s_w[lane] = z;
  }
  __syncthreads();
  int64_t lr = p.tile_counts[blockIdx.x] + (x - cnt) + (w > 0 ? s_w[w - 1] : 0);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int64_t k = base + (int64_t)threadIdx.x * PER + j;
    if (k >= R) break;
    const int n = part_node_of(p, k);
    if (k == p.offs[n]) lrank_at[n] = lr;  // rank at the node's first position
    // node's left rank base is lrank(offs[n]); it is the same for all k in the node,
    // but it may live in another tile: scatter uses it via lrank_at after a
    // kernel boundary, so here only record; scatter happens in k_part_scatter.
    lr += flags[j];
  }
}

__global__ void __launch_bounds__(32) k_part_offsets(PartParams p, int64_t *lrank_at, int64_t n_tiles) {
  // lrank_at[n_nodes] = total left count; empty nodes: their rank equals the
  // next non-empty node's start rank, resolved by a backward pass.
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  if (!p.st->plan_ok) return;
  int64_t next = p.tile_counts[n_tiles];  // total left
  lrank_at[p.n_nodes] = next;
  for (int n = p.n_nodes - 1; n >= 0; --n) {
    if (p.offs[n + 1] == p.offs[n]) lrank_at[n] = next;
    next = lrank_at[n];
  }
  p.out_offs[0] = 0;
  int64_t small_total = 0;
  if (p.small_rows) p.small_offs[0] = 0;
  for (int n = 0; n < p.n_nodes; ++n) {
    const int64_t left = lrank_at[n + 1] - lrank_at[n];
    const int64_t right = (p.offs[n + 1] - p.offs[n]) - left;
    p.out_offs[2 * n + 1] = p.offs[n] + left;
    p.out_offs[2 * n + 2] = p.offs[n + 1];
    if (p.small_rows) {
      const bool right_smaller = right < left;  // ties go to the left child
      p.small_side[n] = right_smaller ? 1 : 0;
      small_total += right_smaller ? right : left;
      p.small_offs[n + 1] = small_total;
    }
  }
}

__global__ void __launch_bounds__(PART_THREADS) k_part_scatter(PartParams p, const int64_t *lrank_at) {
  if (!p.st->plan_ok) return;
  const int64_t R = part_len(p);
  const int64_t base = (int64_t)blockIdx.x * PART_TILE;
  constexpr int PER = PART_TILE / PART_THREADS;
  int flags[PER];
  int32_t rows[PER];
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int64_t k = base + (int64_t)threadIdx.x * PER + j;
    flags[j] = 0;
    rows[j] = -1;
    if (k < R) flags[j] = part_flag(p, k, rows[j]);
    cnt += flags[j];
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __shared__ int s_w[PART_THREADS / 32];
  if (lane == 31) s_w[w] = x;
  __syncthreads();
  if (w == 0) {
    int z = lane < PART_THREADS / 32 ? s_w[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < PART_THREADS / 32) s_w[lane] = z;
  }
  __syncthreads();
  int64_t lr = p.tile_counts[blockIdx.x] + (x - cnt) + (w > 0 ? s_w[w - 1] : 0);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int64_t k = base + (int64_t)threadIdx.x * PER + j;
    if (k >= R) break;
    const int n = part_node_of(p, k);
    const int64_t a = p.offs[n];
    const int64_t left_before = lr - lrank_at[n];  // left rows of node n before k
    const int64_t left_n = lrank_at[n + 1] - lrank_at[n];
    const int64_t rank = flags[j] ? left_before : (k - a) - left_before;  // position within its child
    const int64_t dst = flags[j] ? a + rank : a + left_n + rank;
    const int32_t row = (rows[j] >= 0 && rows[j] < p.n_rows) ? rows[j] : 0;
    if (dst >= 0 && dst < R) p.out_rows[dst] = row;
    if (p.small_rows && (flags[j] ? 0 : 1) == (int)p.small_side[n]) {
      const int64_t sd = p.small_offs[n] + rank;
      if (sd >= 0 && sd < p.small_offs[p.n_nodes]) p.small_rows[sd] = row;
    }
    lr += flags[j];
  }
}

}  // namespace gbt
