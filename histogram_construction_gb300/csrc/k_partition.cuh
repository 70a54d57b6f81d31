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
// k_part_flags gathers each position's bin of its node's split feature once
// and stores the left/right flags as a bit mask (and counts the left rows of
// each tile); k_part_scan (one block) scans the tile counts, derives every
// node's left count from the mask and writes the child offsets; k_part_scatter
// places every row from the mask.
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
  const unsigned char *cols;  // slots feature-major [n_features][n_rows], bin_bytes each
  const SplitOut *splits;
  int64_t *tile_counts;  // [n_tiles + 1] left rows per tile, then their exclusive prefix
  uint8_t *flags;        // [ceil(R / 8)] bit j of byte k / 8: position k (8-aligned k) goes left
  int64_t *lrank;        // [n_nodes + 1] left rows before each node's first position
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

// The fields of a node's split that route its rows.
struct NodeRoute {
  int32_t feature, bin, dleft;
};

__device__ __forceinline__ NodeRoute node_route(const PartParams &p, int n) {
  const SplitOut *s = p.splits + n;
  return NodeRoute{s->feature, s->bin, (int32_t)s->default_left};
}

// 1 = left, 0 = right for row `r` of a node with route `nr`.
__device__ __forceinline__ int route_left(const PartParams &p, const NodeRoute &nr, int32_t r) {
  if (nr.feature < 0 || nr.feature >= p.n_features) return 1;  // no split (or an invalid one): all left
  if (r < 0 || r >= p.n_rows) return 1;
  const int64_t at = (int64_t)nr.feature * p.n_rows + r;
  const uint32_t slot = p.bin_bytes == 1 ? (uint32_t)p.cols[at] : (uint32_t)reinterpret_cast<const uint16_t *>(p.cols)[at];
  if (slot == (uint32_t)p.n_bins) return nr.dleft ? 1 : 0;
  return (int32_t)slot <= nr.bin ? 1 : 0;
}

constexpr int PART_PER = PART_TILE / PART_THREADS;  // 8 consecutive positions per thread (one flag byte)

__global__ void __launch_bounds__(PART_THREADS) k_part_flags(PartParams p) {
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
  const int64_t k0 = (int64_t)blockIdx.x * PART_TILE + (int64_t)threadIdx.x * PART_PER;
  uint32_t bits = 0, bad = 0;
  if (k0 < R) {
    // all row ids and all bins of the thread's positions in flight together
    int n = part_node_of(p, k0);
    int64_t nend = p.offs[n + 1];
    NodeRoute nr = node_route(p, n);
    int32_t row[PART_PER];
    NodeRoute rt[PART_PER];
#pragma unroll
    for (int j = 0; j < PART_PER; ++j) {
      const int64_t k = k0 + j;
      row[j] = -1;
      rt[j] = nr;
      if (k < R) {
        while (k >= nend && n < p.n_nodes - 1) {  // the next non-empty node (bounded by the node count)
          ++n;
          nend = p.offs[n + 1];
          nr = node_route(p, n);
        }
        rt[j] = nr;
        row[j] = p.rows ? p.rows[k] : (int32_t)k;
      }
    }
#pragma unroll
    for (int j = 0; j < PART_PER; ++j) {
      if (k0 + j >= R) continue;
      if (row[j] < 0 || row[j] >= p.n_rows) bad = 1;
      bits |= (uint32_t)route_left(p, rt[j], row[j]) << j;
    }
    p.flags[k0 >> 3] = (uint8_t)bits;
  }
  int c = __popc(bits);
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

// One block: exclusive scan of the tile counts (tile_counts[n_tiles] = the
// total); each node's left rank lrank[n] = left rows before offs[n] (tile
// prefix + the mask bits of its tile before it); the child offsets; the
// smaller-child sides and offsets.
__global__ void __launch_bounds__(1024) k_part_scan(PartParams p, int64_t n_tiles) {
  if (!p.st->plan_ok) return;
  __shared__ long long s_carry;
  __shared__ long long s_w[32];
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  auto block_scan = [&](long long v) -> long long {  // inclusive, plus the carry of earlier batches
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
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = incl;
    __syncthreads();
    return incl;
  };
  for (int64_t base = 0; base < n_tiles; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    const long long v = i < n_tiles ? p.tile_counts[i] : 0;
    const long long incl = block_scan(v);
    if (i < n_tiles) p.tile_counts[i] = incl - v;
  }
  if (threadIdx.x == 0) p.tile_counts[n_tiles] = s_carry;
  __syncthreads();
  const int64_t R = part_len(p);
  // one warp per node boundary: the lanes count the mask words of its tile before it
  for (int n = w; n <= p.n_nodes; n += blockDim.x / 32) {
    const int64_t k = n < p.n_nodes ? min(p.offs[n], R) : R;
    const int64_t t = k / PART_TILE;
    const int64_t w0 = t * (PART_TILE / 32), w1 = k >> 5;  // whole 32-position words before k
    const uint32_t *fw = reinterpret_cast<const uint32_t *>(p.flags);
    int c = 0;
    for (int64_t q = w0 + lane; q < w1; q += 32) c += __popc(fw[q]);
    if (lane == 0 && (k & 31)) c += __popc(fw[w1] & ((1u << (k & 31)) - 1u));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) p.lrank[n] = p.tile_counts[t] + c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.out_offs[0] = 0;
    s_carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.n_nodes; base += blockDim.x) {
    const int n = base + threadIdx.x;
    long long small_n = 0;
    if (n < p.n_nodes) {
      const int64_t left = p.lrank[n + 1] - p.lrank[n];
      const int64_t right = (p.offs[n + 1] - p.offs[n]) - left;
      p.out_offs[2 * n + 1] = p.offs[n] + left;
      p.out_offs[2 * n + 2] = p.offs[n + 1];
      const bool right_smaller = right < left;  // ties go to the left child
      small_n = right_smaller ? right : left;
      if (p.small_rows) p.small_side[n] = right_smaller ? 1 : 0;
    }
    const long long incl = block_scan(small_n);
    if (p.small_rows && n < p.n_nodes) {
      p.small_offs[n + 1] = incl;
      if (n == 0) p.small_offs[0] = 0;
    }
  }
}

__global__ void __launch_bounds__(PART_THREADS) k_part_scatter(PartParams p) {
  if (!p.st->plan_ok) return;
  const int64_t R = part_len(p);
  const int64_t k0 = (int64_t)blockIdx.x * PART_TILE + (int64_t)threadIdx.x * PART_PER;
  const uint32_t bits = k0 < R ? (uint32_t)p.flags[k0 >> 3] : 0u;
  // block exclusive scan of the threads' left counts
  const int cnt = __popc(bits), lane = threadIdx.x & 31, w = threadIdx.x >> 5;
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
  if (k0 >= R) return;
  int64_t lr = p.tile_counts[blockIdx.x] + (x - cnt) + (w > 0 ? s_w[w - 1] : 0);  // left rows before k0
  int n = part_node_of(p, k0);
  int64_t a = p.offs[n], nend = p.offs[n + 1], lr_n = p.lrank[n], left_n = p.lrank[n + 1] - lr_n;
  const int64_t small_end = p.small_rows ? p.small_offs[p.n_nodes] : 0;
  int32_t rid[PART_PER];  // all row ids in flight before the stores
#pragma unroll
  for (int j = 0; j < PART_PER; ++j) rid[j] = k0 + j < R ? (p.rows ? p.rows[k0 + j] : (int32_t)(k0 + j)) : 0;
#pragma unroll
  for (int j = 0; j < PART_PER; ++j) {
    const int64_t k = k0 + j;
    if (k >= R) break;
    while (k >= nend && n < p.n_nodes - 1) {
      ++n;
      a = nend;
      nend = p.offs[n + 1];
      lr_n = p.lrank[n];
      left_n = p.lrank[n + 1] - lr_n;
    }
    const int flag = (bits >> j) & 1;
    const int32_t r0 = rid[j];
    const int32_t row = (r0 >= 0 && r0 < p.n_rows) ? r0 : 0;
    const int64_t left_before = lr - lr_n;                         // left rows of node n before k
    const int64_t rank = flag ? left_before : (k - a) - left_before;  // position within its child
    const int64_t dst = flag ? a + rank : a + left_n + rank;
    if (dst >= 0 && dst < R) p.out_rows[dst] = row;
    if (p.small_rows && (flag ? 0 : 1) == (int)p.small_side[n]) {
      const int64_t sd = p.small_offs[n] + rank;
      if (sd >= 0 && sd < small_end) p.small_rows[sd] = row;
    }
    lr += flag;
  }
}

}  // namespace gbt
