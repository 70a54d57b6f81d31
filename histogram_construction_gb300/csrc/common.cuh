// Shared device-side definitions of the gbthist CUDA library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbt {

// Device error word bits (read and cleared by gbt_sync).
enum : uint32_t {
  ERRBIT_BIN = 1u << 0,
  ERRBIT_ROW = 1u << 1,
  ERRBIT_QUANT = 1u << 2,
  ERRBIT_TIMEOUT = 1u << 3,
  ERRBIT_INCONSISTENT = 1u << 4,
};

// Small device-resident state shared by the kernels of one context.
struct DevState {
  uint32_t err;        // error bits
  uint32_t qmax;       // max |q| over the current tree's rows, both components
  uint32_t work_next;  // dynamic work counter of the histogram kernel (0 between launches)
  uint32_t work_done;  // CTAs of the histogram kernel that have finished (0 between launches)
  uint32_t plan_ok;    // 1 when the level plan is valid
  int32_t n_items;     // work items of the level
  uint32_t qmax_multi; // max |q| over the multi-output tree's pairs, all targets
};

constexpr int MIRROR_STRIP_BYTES = 64;  // bytes per row per mirror tile of features
constexpr int MIRROR_ROW_BYTES = 128;   // a tile pair's row: tiles 2p and 2p + 1 side by side

// Byte offset of row `row` of tile `tile` in the mirror [ceil(n_tiles / 2)][N][128]:
// a gathered row of tile 2p and the same row of tile 2p + 1 share one 128-byte line,
// so the two items that read them take one line from memory between them.
__host__ __device__ __forceinline__ int64_t mirror_offset(int64_t tile, int64_t row, int64_t n_rows) {
  return ((tile >> 1) * n_rows + row) * MIRROR_ROW_BYTES + (tile & 1) * MIRROR_STRIP_BYTES;
}

__device__ __forceinline__ void raise_err(DevState *st, uint32_t bit) { atomicOr(&st->err, bit); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Make generic-proxy shared-memory writes visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy shared -> global (TMA engine, no tensor map): bytes % 16 == 0, both 16-B aligned.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
               "r"(bytes)
               : "memory");
}

// Bulk reduce-add shared -> global of 64-bit integers (two's complement add).
__device__ __forceinline__ void bulk_reduce_add_u64(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u64 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}

// Bulk reduce-add shared -> global of 32-bit integers (wraps modulo 2^32).
__device__ __forceinline__ void bulk_reduce_add_u32(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the committed bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until all but the most recent committed bulk group have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Bulk reduce-add of doubles from shared memory into global memory.
__device__ __forceinline__ void bulk_reduce_add_f64(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f64 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}

// Wait until the committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Named barrier over `threads` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor runs; pdl_wait() blocks until
// the predecessor grid has completed and its memory is visible (a no-op for
// an ordinary launch). pdl_trigger() lets the successor start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int4 ldg_v4s(const int4 *p) { return __ldg(p); }

// 16 bytes global -> shared without passing through registers (L2 only);
// src_bytes 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t sdst, const void *gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sdst), "l"(gsrc), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// this thread's copies of all but the newest N committed groups are complete
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
  return v;
}

}  // namespace gbt
