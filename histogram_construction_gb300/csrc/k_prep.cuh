// Dataset and tree preparation kernels: the tiled row-major bin mirror and the
// fixed-point quantisation of (g, h).
#pragma once

#include "common.cuh"

namespace gbt {

// Feature-major [F][N] bins -> tiled row-major mirror: 64-byte strips per
// (tile, row), tiles paired into 128-byte rows (see mirror_offset), holding
// histogram slots (bin, or n_bins for the missing sentinel).
// The mirror is the column tiling of bonsai "E6. The wide-data wall",
// "Epilogue": each row of a feature tile is one contiguous strip, so a node's
// gathered rows read whole 64-byte strips instead of one byte per feature.
// grid (ceil(rows/64), n_tiles), block 256. Validates every value. The slots
// are also written feature-major into cols [n_features][n_rows]: the row
// partition reads one feature of consecutive rows there (rows that are
// close share a sector) instead of one 32-byte sector of the mirror per row.
template <typename T>
__global__ void __launch_bounds__(256) k_mirror(const T *__restrict__ bins, int64_t n_rows, int64_t row0,
                                                int64_t rows_in_slab, int32_t f_base, int32_t n_features,
                                                int32_t n_bins, uint32_t sentinel, int64_t bins_stride,
                                                T *__restrict__ mirror, T *__restrict__ cols, DevState *st) {
  constexpr int TF = MIRROR_STRIP_BYTES / sizeof(T);  // features per tile
  __shared__ T sm[TF][64 + 2];
  const int tile = blockIdx.y;
  const int64_t rl0 = (int64_t)blockIdx.x * 64;  // row within slab
  const int f0 = tile * TF;                      // feature within slab
  uint32_t bad = 0;
  for (int i = threadIdx.x; i < TF * 64; i += blockDim.x) {
    const int fl = i >> 6, rl = i & 63;
    const int f = f0 + fl;
    const int64_t r = rl0 + rl;
    T v = 0;
    if (f_base + f < n_features && r < rows_in_slab) {
      const uint32_t b = bins[(int64_t)f * bins_stride + r];
      uint32_t slot;
      if (b == sentinel) {
        slot = (uint32_t)n_bins;
      } else if (b < (uint32_t)n_bins) {
        slot = b;
      } else {
        slot = (uint32_t)n_bins;
        bad = 1;
      }
      v = (T)slot;
      cols[(int64_t)(f_base + f) * n_rows + row0 + r] = v;
    }
    sm[fl][rl] = v;
  }
  __syncthreads();
  const int64_t gtile = (int64_t)(f_base / TF) + tile;
  for (int i = threadIdx.x; i < TF * 64; i += blockDim.x) {
    const int rl = i / TF, fl = i % TF;
    const int64_t r = rl0 + rl;
    if (r < rows_in_slab)
      reinterpret_cast<T *>(reinterpret_cast<unsigned char *>(mirror) + mirror_offset(gtile, row0 + r, n_rows))[fl] =
          sm[fl][rl];
  }
  if (bad) raise_err(st, ERRBIT_BIN);
}

// Largest admissible |q|: any 1024 rows then sum exactly in 32 bits.
constexpr int QMAX = (1 << 21) - 1;

// (g, h) float32 pairs -> int32 fixed-point pairs, q = round-half-even(fl32(x * s)),
// |q| <= QMAX (else the quantisation error bit).
// "GBDT engine engineering deep-dive" (ybb.press), section 7: gradients are
// quantised to fixed point before integer atomics; bonsai "9. Parallelism &
// determinism", "The idea": int64 cells are exact in any order.
// One (g, h) pair -> (qg, qh); accumulates max |q| and the overflow flag.
__device__ __forceinline__ int2 quantise_pair(float2 v, float sg, float sh, uint32_t &mx, uint32_t &bad) {
  const float pg = __fmul_rn(v.x, sg);
  const float ph = __fmul_rn(v.y, sh);
  int qg = 0, qh = 0;
  if (fabsf(pg) < 2097152.0f) {
    const int t = __float2int_rn(pg);
    if (t >= -QMAX && t <= QMAX) qg = t; else bad = 1;
  } else {
    bad = 1;
  }
  if (fabsf(ph) < 2097152.0f) {
    const int t = __float2int_rn(ph);
    if (t >= -QMAX && t <= QMAX) qh = t; else bad = 1;
  } else {
    bad = 1;
  }
  const uint32_t ag = qg < 0 ? (uint32_t)(-(int64_t)qg) : (uint32_t)qg;
  const uint32_t ah = qh < 0 ? (uint32_t)(-(int64_t)qh) : (uint32_t)qh;
  mx = max(mx, max(ag, ah));
  return make_int2(qg, qh);
}

// Block reduction of max |q| into *dst (one atomic per block: same-address
// atomics serialise in L2) and of the overflow flag into the error word.
__device__ __forceinline__ void block_qmax(uint32_t mx, uint32_t bad, uint32_t *dst, DevState *st) {
  __shared__ uint32_t s_mx[32];
  __shared__ uint32_t s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_mx[threadIdx.x >> 5] = mx;
  if (bad) s_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_mx[w]);
    if (m) atomicMax(dst, m);
    if (s_bad) raise_err(st, ERRBIT_QUANT);
  }
}

// Reduces max |q| into st->qmax (zeroed by the caller).
__global__ void __launch_bounds__(1024) k_quantise(const float2 *__restrict__ gp, int64_t n, float sg, float sh,
                                                  int2 *__restrict__ q, DevState *st) {
  uint32_t mx = 0, bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    q[i] = quantise_pair(gp[i], sg, sh, mx, bad);
  block_qmax(mx, bad, &st->qmax, st);
}

// Multi-output gradients [hessboost PR #163 "Change": vector-leaf nodes carry
// one (g, h) per target]: pairs [n_rows][k], target i % k of element i
// quantised with that target's scales; max |q| over all targets into
// st->qmax_multi.
constexpr int MULTI_MAX_TARGETS = 16;
struct MultiScales {
  float g[MULTI_MAX_TARGETS], h[MULTI_MAX_TARGETS];
  int32_t k;
};

__global__ void __launch_bounds__(1024) k_quantise_multi(const float2 *__restrict__ gp, int64_t n, MultiScales sc,
                                                        int2 *__restrict__ q, DevState *st) {
  uint32_t mx = 0, bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i % sc.k);
    q[i] = quantise_pair(gp[i], sc.g[t], sc.h[t], mx, bad);
  }
  block_qmax(mx, bad, &st->qmax_multi, st);
}

}  // namespace gbt
