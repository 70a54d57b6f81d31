// gbthist C-ABI: context, uploads, level build, subtraction, split find and
// row partition on one GB300 (sm_103a). See include/gbthist.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/gbthist.h"
#include "common.cuh"
#include "k_f64.cuh"
#include "k_hist.cuh"
#include "k_level_split.cuh"
#include "k_partition.cuh"
#include "k_prep.cuh"
#include "k_split.cuh"

using namespace gbt;

static_assert(sizeof(gbt_split) == 56, "gbt_split layout");
static_assert(sizeof(SplitOut) == sizeof(gbt_split), "device split layout");
static_assert(sizeof(gbt_split_f64) == sizeof(gbt_split), "float-cell split layout");

namespace {

// ---------------------------------------------------------------------------- allocation with fault injection
// GBT_FAULT_ALLOC_AT="k[:tag]" makes the k-th device or pinned allocation
// counted from the moment the variable took its current value fail with
// GBT_ERR_OOM (host-side fault injection for tests; changing the value, e.g.
// its tag, restarts the count).
std::string g_fault_env;
long long g_alloc_count = 0;

bool alloc_should_fail() {
  const char *e = getenv("GBT_FAULT_ALLOC_AT");
  const std::string v = e ? e : "";
  if (v != g_fault_env) {
    g_fault_env = v;
    g_alloc_count = 0;
  }
  ++g_alloc_count;
  const long long at = v.empty() ? 0 : atoll(v.c_str());
  return at > 0 && g_alloc_count == at;
}

cudaError_t dev_alloc(void **p, size_t bytes, cudaStream_t s) {
  if (alloc_should_fail()) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMallocAsync(p, bytes, s);
}

}  // namespace

struct Buf {
  void *p = nullptr;
  size_t cap = 0;
};

struct gbt_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  int n_sm = 0;
  int smem_optin = 0;
  // dataset
  int bin_bytes = 0;
  int64_t n_rows = 0;
  int32_t n_features = 0;
  int32_t n_bins = 0;
  uint32_t sentinel = 0;
  int32_t n_tiles = 0;     // mirror tiles of 64-byte strips
  int32_t tile_feats = 0;  // features per mirror tile
  int32_t ts16 = 0;        // features per u16 work item
  Buf mirror;
  // tree
  bool tree_ready = false;
  float sg = 1.f, sh = 1.f;
  double inv_sg = 1.0, inv_sh = 1.0;
  Buf q;
  uint32_t qmax = 0;             // max |q| of the current tree, known on the host after ev_q
  bool qmax_known = false;
  cudaEvent_t ev_q = nullptr;
  // multi-output tree: k quantised pairs per row
  Buf qm;
  int32_t multi_k = 0;
  uint32_t qmax_multi = 0;       // known on the host after ev_qm
  bool qmax_multi_known = false;
  cudaEvent_t ev_qm = nullptr;
  // state + scratch
  DevState *st = nullptr;
  uint32_t *err_host = nullptr;  // pinned: [0] error word copy, [1] max |q| copy, [2] multi-output max |q| copy
  Buf gp_stage, chunk_prefix, partial, rows_in, offs_in, cand, splits_a, splits_b, parent_of_in, tile_counts, lrank,
      slab, counters, level_scratch, items, side_in, pflags, cols, qlev;
  std::string last_error;
  int64_t launches = 0;
  // tuning: work items the level plan aims for (default 1 per SM; GBT_TARGET_ITEMS overrides it for sweeps)
  int target_items = 0;
  bool plan_kernel = false;  // GBT_PLAN_KERNEL=1: always plan levels with the plan kernel (comparisons)
  // group images: bytes at the start of `partial` known to be zero (the reduce region must be, when a
  // level's histogram kernel starts); img_r_pending: this level's reduce region, zero again once the
  // level's consumer kernel (which zeroes what it reads) is launched
  size_t img_clean = 0, img_r_pending = 0;
  // diagnostics: per-launch event pairs
  bool prof = false;
  struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
  };
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> prof_pool;
  cudaEvent_t prof_open = nullptr;
};

namespace {

gbt_status fail(gbt_ctx *c, gbt_status s, const std::string &msg) {
  if (c) c->last_error = msg;
  return s;
}

gbt_status cuda_fail(gbt_ctx *c, cudaError_t e, const char *what) {
  std::string m = std::string(what) + ": " + cudaGetErrorString(e);
  if (e == cudaErrorMemoryAllocation) return fail(c, GBT_ERR_OOM, m);
  return fail(c, GBT_ERR_CUDA, m);
}

#define CUDA_TRY(c, expr, what)                 \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, what); \
  } while (0)

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel on the stream runs, and waits for it (pdl_wait) before
// touching its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(gbt_ctx *c, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaEvent_t prof_event(gbt_ctx *c) {
  if (!c->prof_pool.empty()) {
    cudaEvent_t e = c->prof_pool.back();
    c->prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Record the start event of a launch (diagnostics only).
void prof_begin(gbt_ctx *c) {
  if (!c->prof) return;
  c->prof_open = prof_event(c);
  cudaEventRecord(c->prof_open, c->stream);
}

void prof_end(gbt_ctx *c, const char *name) {
  if (!c->prof || !c->prof_open) return;
  cudaEvent_t b = prof_event(c);
  cudaEventRecord(b, c->stream);
  c->prof_pending.push_back({name, c->prof_open, b});
  c->prof_open = nullptr;
}

// After a kernel launch: count it, close its profiling record, check the launch.
#define LAUNCH_CHECK(c, what)                            \
  do {                                                   \
    ++(c)->launches;                                     \
    prof_end((c), what);                                 \
    cudaError_t e_ = cudaGetLastError();                 \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, what); \
  } while (0)

gbt_status ensure(gbt_ctx *c, Buf &b, size_t bytes, const char *what) {
  if (bytes == 0) bytes = 16;
  if (b.cap >= bytes) return GBT_OK;
  if (b.p) {
    cudaError_t e = cudaFreeAsync(b.p, c->stream);
    b.p = nullptr;
    b.cap = 0;
    if (e != cudaSuccess) return cuda_fail(c, e, what);
  }
  void *p = nullptr;
  cudaError_t e = dev_alloc(&p, bytes, c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, what);
  b.p = p;
  b.cap = bytes;
  return GBT_OK;
}

void release(gbt_ctx *c, Buf &b) {
  if (b.p) cudaFreeAsync(b.p, c->stream);
  b.p = nullptr;
  b.cap = 0;
}

// 1 device/managed, 0 host, -1 invalid
int ptr_kind(const void *p) {
  if (!p) return -1;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) ? 1 : 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device's address of pinned (page-locked) host memory, or nullptr for any other pointer. Kernels
// read and write such memory in place (over the host link), which for small buffers costs less than a
// copy's launch and completion.
void *pinned_device_ptr(const void *p) {
  if (!p) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
// pinned inputs up to this size are read in place (a row list is read once per feature tile, so a large
// one is copied once instead; measured on level5's 1.5 MB row list: e2e 5.2e11 -> 6.1e11 entries/s)
constexpr size_t ZERO_COPY_MAX_BYTES = 4 << 20;

// Return a device pointer holding `bytes` of `src` (copied into `stage` when src is host memory).
gbt_status device_view(gbt_ctx *c, const void *src, size_t bytes, Buf &stage, const void **out, const char *what) {
  const int k = ptr_kind(src);
  if (k < 0) return fail(c, GBT_ERR_INVALID_ARG, std::string(what) + ": NULL");
  if (k == 1) {
    *out = src;
    return GBT_OK;
  }
  if (bytes <= ZERO_COPY_MAX_BYTES) {
    if (void *d = pinned_device_ptr(src)) {
      *out = d;
      return GBT_OK;
    }
  }
  gbt_status s = ensure(c, stage, bytes, what);
  if (s != GBT_OK) return s;
  CUDA_TRY(c, cudaMemcpyAsync(stage.p, src, bytes, cudaMemcpyHostToDevice, c->stream), what);
  *out = stage.p;
  return GBT_OK;
}

gbt_status check_ctx(gbt_ctx *c) {
  if (!c) return GBT_ERR_INVALID_ARG;
  cudaError_t e = cudaSetDevice(c->device);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaSetDevice");
  c->last_error.clear();
  return GBT_OK;
}

int grid_for(gbt_ctx *c, int64_t work, int threads, int per_sm) {
  int64_t g = (work + threads - 1) / threads;
  g = std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)c->n_sm * per_sm));
  return (int)g;
}

int h16_ts_for(int B) {
  for (int ts = 32; ts >= 2; ts >>= 1)
    if ((int64_t)ts * B * 8 <= H16_HIST_MAX) return ts;
  return 0;
}

// Completion counters of the split kernels: zero when allocated, and every
// launch leaves them zero again (the last CTA of a group resets its counter).
gbt_status ensure_counters(gbt_ctx *c, size_t n) {
  const size_t bytes = std::max<size_t>(n, 1) * sizeof(uint32_t);
  if (c->counters.cap >= bytes) return GBT_OK;
  gbt_status s = ensure(c, c->counters, bytes, "split counters");
  if (s != GBT_OK) return s;
  CUDA_TRY(c, cudaMemsetAsync(c->counters.p, 0, c->counters.cap, c->stream), "zero split counters");
  return GBT_OK;
}

SplitParams make_sp(const gbt_ctx *c, const gbt_params *prm) {
  SplitParams sp;
  sp.lambda = prm->lambda;
  sp.gamma = prm->gamma;
  sp.inv_sg = c->inv_sg;
  sp.inv_sh = c->inv_sh;
  // smallest H >= 1 with (double)H * inv_sh >= min_child_weight; the map
  // H -> fl(fl(H) * inv_sh) is non-decreasing, so validity is H >= h_min
  const double mcw = prm->min_child_weight;
  auto ok = [&](int64_t h) { return (double)h * c->inv_sh >= mcw; };
  const int64_t top = (int64_t)1 << 62;
  if (!ok(top)) {
    sp.h_min = INT64_MAX;
  } else if (ok(1)) {
    sp.h_min = 1;
  } else {
    int64_t lo = 1, hi = top;  // ok(lo) false, ok(hi) true
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (ok(mid)) hi = mid; else lo = mid;
    }
    sp.h_min = hi;
  }
  sp.lambda_f = (float)prm->lambda;
  sp.gamma_f = (float)prm->gamma;
  sp.gamma_abs_f = fabsf((float)prm->gamma);
  sp.inv_sg_f = (float)c->inv_sg;
  sp.inv_sh_f = (float)c->inv_sh;
  sp.filter = (prm->lambda >= 0.0 && isfinite(prm->lambda) && isfinite(prm->gamma) && fabs(prm->gamma) < 1e30 &&
               prm->lambda < 1e30 && isfinite(sp.inv_sg_f) && isfinite(sp.inv_sh_f) && sp.inv_sg_f > 0.f &&
               sp.inv_sh_f > 0.f)
                  ? 1
                  : 0;
  return sp;
}

// Shared-memory limits of the histogram kernels (once per context).
bool set_hist_attributes() {
  const int u16_int = H16_HIST_MAX + H16_STAGE_BYTES + 128, u16_flt = H16_HIST_MAX + FL_STAGE_BYTES + 128;
  return cudaFuncSetAttribute(k_hist_u8<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, H8_SMEM_RING) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u8<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u8<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              H8_SMEM + FL_STAGE_BYTES) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u8<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u8<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, H8_SMEM_RING) ==
             cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u8<false, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100) ==
             cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_int) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_int) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_int) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_int) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_int) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_flt) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_flt) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_flt) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_flt) == cudaSuccess &&
         cudaFuncSetAttribute(k_hist_u16<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, u16_flt) == cudaSuccess;
}

}  // namespace

extern "C" {

gbt_status gbt_create(int device, void *cuda_stream, gbt_ctx **out) {
  if (!out) return GBT_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? GBT_ERR_OOM : GBT_ERR_CUDA;
  if (device < 0 || device >= ndev) return GBT_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return GBT_ERR_CUDA;
  gbt_ctx *c = new gbt_ctx();
  c->device = device;
  c->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (const char *e = getenv("GBT_TARGET_ITEMS")) c->target_items = std::max(0, atoi(e));
  if (const char *e = getenv("GBT_PLAN_KERNEL")) c->plan_kernel = atoi(e) != 0;
  void *st = nullptr;
  e = dev_alloc(&st, sizeof(DevState), c->stream);
  if (e != cudaSuccess) {
    delete c;
    return e == cudaErrorMemoryAllocation ? GBT_ERR_OOM : GBT_ERR_CUDA;
  }
  c->st = reinterpret_cast<DevState *>(st);
  cudaMemsetAsync(c->st, 0, sizeof(DevState), c->stream);
  if (alloc_should_fail() || cudaMallocHost(&c->err_host, 3 * sizeof(uint32_t)) != cudaSuccess) {
    cudaFreeAsync(c->st, c->stream);
    cudaStreamSynchronize(c->stream);
    delete c;
    return GBT_ERR_OOM;
  }
  c->err_host[0] = c->err_host[1] = c->err_host[2] = 0;
  if (cudaEventCreateWithFlags(&c->ev_q, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_qm, cudaEventDisableTiming) != cudaSuccess) {
    if (c->ev_q) cudaEventDestroy(c->ev_q);
    cudaFreeHost(c->err_host);
    cudaFreeAsync(c->st, c->stream);
    cudaStreamSynchronize(c->stream);
    delete c;
    return GBT_ERR_CUDA;
  }
  if (!set_hist_attributes()) {
    cudaGetLastError();
    cudaEventDestroy(c->ev_q);
    cudaEventDestroy(c->ev_qm);
    cudaFreeHost(c->err_host);
    cudaFreeAsync(c->st, c->stream);
    cudaStreamSynchronize(c->stream);
    delete c;
    return GBT_ERR_CUDA;
  }
  *out = c;
  return GBT_OK;
}

gbt_status gbt_destroy(gbt_ctx *c) {
  if (!c) return GBT_OK;
  cudaSetDevice(c->device);
  cudaStreamSynchronize(c->stream);
  Buf *bufs[] = {&c->mirror, &c->q, &c->gp_stage, &c->chunk_prefix, &c->partial, &c->rows_in, &c->offs_in,
                 &c->cand, &c->splits_a, &c->splits_b, &c->parent_of_in, &c->tile_counts, &c->lrank, &c->slab,
                 &c->counters, &c->level_scratch, &c->qm, &c->items, &c->side_in, &c->pflags, &c->cols, &c->qlev};
  for (Buf *b : bufs) release(c, *b);
  if (c->st) cudaFreeAsync(c->st, c->stream);
  cudaStreamSynchronize(c->stream);
  if (c->err_host) cudaFreeHost(c->err_host);
  if (c->ev_q) cudaEventDestroy(c->ev_q);
  if (c->ev_qm) cudaEventDestroy(c->ev_qm);
  for (auto &r : c->prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : c->prof_pool) cudaEventDestroy(e);
  delete c;
  return GBT_OK;
}

const char *gbt_last_error(const gbt_ctx *c) { return c ? c->last_error.c_str() : "NULL context"; }

gbt_status gbt_sync(gbt_ctx *c) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  CUDA_TRY(c, cudaMemcpyAsync(c->err_host, &c->st->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, c->stream),
           "read error word");
  CUDA_TRY(c, cudaMemsetAsync(&c->st->err, 0, sizeof(uint32_t), c->stream), "clear error word");
  CUDA_TRY(c, cudaStreamSynchronize(c->stream), "stream synchronize");
  const uint32_t e = *c->err_host;
  if (e & ERRBIT_BIN) return fail(c, GBT_ERR_BIN_RANGE, "device: bin value out of range");
  if (e & ERRBIT_ROW) return fail(c, GBT_ERR_ROW_RANGE, "device: row index or node offsets out of range");
  if (e & ERRBIT_QUANT) return fail(c, GBT_ERR_QUANT_OVERFLOW, "device: quantised value out of int32 range");
  if (e & ERRBIT_TIMEOUT) return fail(c, GBT_ERR_TIMEOUT, "device: bounded wait ran out");
  if (e & ERRBIT_INCONSISTENT) return fail(c, GBT_ERR_INCONSISTENT, "device: negative hessian after subtraction");
  return GBT_OK;
}

gbt_status gbt_upload_bins(gbt_ctx *c, const void *bins, int bin_bytes, int64_t n_rows, int32_t n_features,
                           int32_t n_bins, uint32_t sentinel) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!bins) return fail(c, GBT_ERR_INVALID_ARG, "bins is NULL");
  if (bin_bytes != 1 && bin_bytes != 2) return fail(c, GBT_ERR_INVALID_ARG, "bin_bytes must be 1 or 2");
  if (n_rows <= 0 || n_rows >= (1LL << 31)) return fail(c, GBT_ERR_UNSUPPORTED, "n_rows must be in [1, 2^31)");
  if (n_features <= 0 || n_features >= (1 << 24)) return fail(c, GBT_ERR_UNSUPPORTED, "n_features must be in [1, 2^24)");
  const uint32_t wmax = bin_bytes == 1 ? 0xFFu : 0xFFFFu;
  if (n_bins < 1 || (uint32_t)n_bins > wmax) return fail(c, GBT_ERR_INVALID_ARG, "n_bins must be in [1, width max]");
  if (sentinel > wmax || sentinel < (uint32_t)n_bins)
    return fail(c, GBT_ERR_INVALID_ARG, "missing_sentinel must fit the width and be >= n_bins");
  const int B = n_bins + 1;
  int ts16 = 0;
  if (bin_bytes == 2) {
    ts16 = h16_ts_for(B);
    if (ts16 == 0) return fail(c, GBT_ERR_UNSUPPORTED, "u16 n_bins too large for the shared-memory histogram");
  }
  const int tf = MIRROR_STRIP_BYTES / bin_bytes;
  const int n_tiles = (n_features + tf - 1) / tf;
  const size_t mbytes = (size_t)((n_tiles + 1) / 2) * (size_t)n_rows * MIRROR_ROW_BYTES;
  s = ensure(c, c->mirror, mbytes, "mirror allocation");
  if (s != GBT_OK) return s;
  s = ensure(c, c->cols, (size_t)n_features * (size_t)n_rows * bin_bytes, "slot columns");
  if (s != GBT_OK) return s;
  c->bin_bytes = bin_bytes;
  c->n_rows = n_rows;
  c->n_features = n_features;
  c->n_bins = n_bins;
  c->sentinel = sentinel;
  c->n_tiles = n_tiles;
  c->tile_feats = tf;
  c->ts16 = ts16;
  c->tree_ready = false;
  const int k = ptr_kind(bins);
  const dim3 block(256);
  if (k == 1) {
    const dim3 grid((unsigned)((n_rows + 63) / 64), (unsigned)n_tiles);
    prof_begin(c);
    if (bin_bytes == 1)
      k_mirror<uint8_t><<<grid, block, 0, c->stream>>>((const uint8_t *)bins, n_rows, 0, n_rows, 0, n_features,
                                                       n_bins, sentinel, n_rows, (uint8_t *)c->mirror.p,
                                                       (uint8_t *)c->cols.p, c->st);
    else
      k_mirror<uint16_t><<<grid, block, 0, c->stream>>>((const uint16_t *)bins, n_rows, 0, n_rows, 0, n_features,
                                                        n_bins, sentinel, n_rows, (uint16_t *)c->mirror.p,
                                                        (uint16_t *)c->cols.p, c->st);
    LAUNCH_CHECK(c, "k_mirror");
  } else {
    // host input: one feature tile (tf feature rows, contiguous) per copy + kernel
    const size_t slab_bytes = (size_t)tf * n_rows * bin_bytes;
    s = ensure(c, c->slab, slab_bytes, "upload slab");
    if (s != GBT_OK) return s;
    for (int t = 0; t < n_tiles; ++t) {
      const int f0 = t * tf;
      const int nf = std::min(tf, n_features - f0);
      const unsigned char *src = (const unsigned char *)bins + (size_t)f0 * n_rows * bin_bytes;
      CUDA_TRY(c, cudaMemcpyAsync(c->slab.p, src, (size_t)nf * n_rows * bin_bytes, cudaMemcpyHostToDevice, c->stream),
               "bins upload");
      const dim3 grid((unsigned)((n_rows + 63) / 64), 1u);
      prof_begin(c);
      if (bin_bytes == 1)
        k_mirror<uint8_t><<<grid, block, 0, c->stream>>>((const uint8_t *)c->slab.p, n_rows, 0, n_rows, f0,
                                                         n_features, n_bins, sentinel, n_rows,
                                                         (uint8_t *)c->mirror.p, (uint8_t *)c->cols.p, c->st);
      else
        k_mirror<uint16_t><<<grid, block, 0, c->stream>>>((const uint16_t *)c->slab.p, n_rows, 0, n_rows, f0,
                                                          n_features, n_bins, sentinel, n_rows,
                                                          (uint16_t *)c->mirror.p, (uint16_t *)c->cols.p,
                                                          c->st);
      LAUNCH_CHECK(c, "k_mirror");
    }
    // the slab is only needed during the upload
    release(c, c->slab);
  }
  return GBT_OK;
}

gbt_status gbt_begin_tree(gbt_ctx *c, const float *gpair, float scale_g, float scale_h) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (!(scale_g > 0.f) || !(scale_h > 0.f) || !isfinite(scale_g) || !isfinite(scale_h))
    return fail(c, GBT_ERR_INVALID_ARG, "scales must be finite and > 0");
  s = ensure(c, c->q, (size_t)c->n_rows * sizeof(int2), "quantised gpair");
  if (s != GBT_OK) return s;
  const void *gp = nullptr;
  s = device_view(c, gpair, (size_t)c->n_rows * 2 * sizeof(float), c->gp_stage, &gp, "gpair");
  if (s != GBT_OK) return s;
  if (!aligned16(gp) && ((reinterpret_cast<uintptr_t>(gp) & 7u) != 0))
    return fail(c, GBT_ERR_INVALID_ARG, "gpair must be 8-byte aligned");
  CUDA_TRY(c, cudaMemsetAsync(&c->st->qmax, 0, sizeof(uint32_t), c->stream), "reset qmax");
  const int grid = grid_for(c, c->n_rows, 1024, 2);
  prof_begin(c);
  k_quantise<<<grid, 1024, 0, c->stream>>>((const float2 *)gp, c->n_rows, scale_g, scale_h, (int2 *)c->q.p, c->st);
  LAUNCH_CHECK(c, "k_quantise");
  // bring max|q| home asynchronously: the build sizes its partial scratch from it
  CUDA_TRY(c, cudaMemcpyAsync(&c->err_host[1], &c->st->qmax, sizeof(uint32_t), cudaMemcpyDeviceToHost, c->stream),
           "read max|q|");
  CUDA_TRY(c, cudaEventRecord(c->ev_q, c->stream), "record max|q| event");
  c->qmax_known = false;
  c->sg = scale_g;
  c->sh = scale_h;
  c->inv_sg = 1.0 / (double)scale_g;
  c->inv_sh = 1.0 / (double)scale_h;
  c->tree_ready = true;
  return GBT_OK;
}

gbt_status gbt_begin_tree_multi(gbt_ctx *c, const float *gpair, int32_t n_targets, const float *scales_g,
                                const float *scales_h) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (n_targets < 1 || n_targets > MULTI_MAX_TARGETS)
    return fail(c, GBT_ERR_UNSUPPORTED, "n_targets must be in [1, 16]");
  if (!gpair || !scales_g || !scales_h) return fail(c, GBT_ERR_INVALID_ARG, "gpair and scales are required");
  MultiScales sc{};
  sc.k = n_targets;
  for (int t = 0; t < n_targets; ++t) {
    const float g = scales_g[t], h = scales_h[t];
    if (!(g > 0.f) || !(h > 0.f) || !isfinite(g) || !isfinite(h))
      return fail(c, GBT_ERR_INVALID_ARG, "scales must be finite and > 0");
    sc.g[t] = g;
    sc.h[t] = h;
  }
  const int64_t n = (int64_t)c->n_rows * n_targets;
  s = ensure(c, c->qm, (size_t)n * sizeof(int2), "quantised multi-output gpair");
  if (s != GBT_OK) return s;
  const void *gp = nullptr;
  s = device_view(c, gpair, (size_t)n * 2 * sizeof(float), c->gp_stage, &gp, "gpair");
  if (s != GBT_OK) return s;
  if ((reinterpret_cast<uintptr_t>(gp) & 7u) != 0) return fail(c, GBT_ERR_INVALID_ARG, "gpair must be 8-byte aligned");
  CUDA_TRY(c, cudaMemsetAsync(&c->st->qmax_multi, 0, sizeof(uint32_t), c->stream), "reset multi-output qmax");
  prof_begin(c);
  k_quantise_multi<<<grid_for(c, n, 1024, 2), 1024, 0, c->stream>>>((const float2 *)gp, n, sc, (int2 *)c->qm.p,
                                                                    c->st);
  LAUNCH_CHECK(c, "k_quantise_multi");
  CUDA_TRY(c, cudaMemcpyAsync(&c->err_host[2], &c->st->qmax_multi, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                              c->stream),
           "read multi-output max|q|");
  CUDA_TRY(c, cudaEventRecord(c->ev_qm, c->stream), "record multi-output max|q| event");
  c->qmax_multi_known = false;
  c->multi_k = n_targets;
  return GBT_OK;
}

gbt_status gbt_suggest_scales(int64_t rows_per_partial, float max_abs_g, float max_abs_h, float *sg, float *sh) {
  if (!sg || !sh) return GBT_ERR_INVALID_ARG;
  if (!(max_abs_g >= 0.f) || !(max_abs_h >= 0.f) || !isfinite(max_abs_g) || !isfinite(max_abs_h))
    return GBT_ERR_INVALID_ARG;
  if (rows_per_partial <= 0) rows_per_partial = 65536;
  rows_per_partial = std::max<int64_t>(rows_per_partial, 1024);
  const double lim = 2147483647.0 / (double)rows_per_partial;  // max |q| per row
  auto pick = [&](float m) -> float {
    if (m == 0.f) return 1.f;
    // largest power of two s with m * s <= lim
    int e = (int)floor(log2(lim / (double)m));
    e = std::max(-126, std::min(e, 126));
    double s = ldexp(1.0, e);
    while (s > ldexp(1.0, -126) && (double)m * s > lim) s *= 0.5;
    return (float)s;
  };
  *sg = pick(max_abs_g);
  *sh = pick(max_abs_h);
  return GBT_OK;
}

}  // extern "C"

namespace {


// Validate the level inputs, plan the work items on the device and run the
// histogram kernel, which leaves the group images in c->partial: exact int32
// sums of the quantised pairs, or, when gpair_f64 (device float (g, h) pairs)
// is given, double sums of those pairs.
gbt_status run_level_build(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                           LevelParams *out_lp, const float2 *gpair_f64 = nullptr, bool multi = false) {
  const int B = c->n_bins + 1;
  const void *offs_d = nullptr;
  int64_t R_host = -1;
  if (ptr_kind(node_offsets) == 0) {
    if (node_offsets[0] != 0) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets[0] must be 0");
    for (int32_t i = 0; i < n_nodes; ++i)
      if (node_offsets[i + 1] < node_offsets[i]) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets must ascend");
    R_host = node_offsets[n_nodes];
    if (R_host > c->n_rows) return fail(c, GBT_ERR_INVALID_ARG, "more level rows than dataset rows");
  }
  gbt_status s =
      device_view(c, node_offsets, (size_t)(n_nodes + 1) * sizeof(int64_t), c->offs_in, &offs_d, "node_offsets");
  if (s != GBT_OK) return s;
  const void *rows_d = nullptr;
  if (rows) {
    const int k = ptr_kind(rows);
    if (k == 0 && R_host < 0) return fail(c, GBT_ERR_INVALID_ARG, "host rows need host node_offsets");
    if (k == 0) {
      s = device_view(c, rows, (size_t)R_host * sizeof(int32_t), c->rows_in, &rows_d, "rows");
      if (s != GBT_OK) return s;
    } else {
      rows_d = rows;
    }
  }
  s = ensure(c, c->chunk_prefix, (size_t)(2 * n_nodes + 1) * sizeof(int32_t), "group prefixes and first images");
  if (s != GBT_OK) return s;
  const bool f64 = gpair_f64 != nullptr;
  if (multi) {
    if (!c->qmax_multi_known) {
      CUDA_TRY(c, cudaEventSynchronize(c->ev_qm), "wait for the multi-output max|q|");
      c->qmax_multi = c->err_host[2];
      c->qmax_multi_known = true;
    }
  } else if (!f64 && !c->qmax_known) {
    CUDA_TRY(c, cudaEventSynchronize(c->ev_q), "wait for max|q|");
    c->qmax = c->err_host[1];
    c->qmax_known = true;
  }
  const int K = multi ? c->multi_k : 1;

  LevelParams lp;
  lp.rows = (const int32_t *)rows_d;
  lp.offs = (const int64_t *)offs_d;
  lp.n_nodes = n_nodes;
  lp.item_feats = multi ? 16 : (c->bin_bytes == 1 ? 64 : c->ts16);
  // multi-output: an item is a 16-feature quarter and a group of up to four targets
  lp.n_fgroups = (c->n_features + lp.item_feats - 1) / lp.item_feats * (multi ? (K + 3) / 4 : 1);
  lp.target_items = c->target_items > 0 ? c->target_items : c->n_sm;
  lp.n_rows = c->n_rows;
  lp.q = f64 ? (const int2 *)gpair_f64 : (multi ? (const int2 *)c->qm.p : (const int2 *)c->q.p);
  lp.group_prefix = (int32_t *)c->chunk_prefix.p;
  lp.img_first = lp.group_prefix + (n_nodes + 1);
  lp.sbw = c->bin_bytes == 1 ? 16 : c->ts16;
  lp.nsb = c->bin_bytes == 1 ? H8_SB : 1;
  // nsb x B x sbw (G, H) pairs: int32 pairs (8 bytes), or double pairs (16 bytes) for float cells
  lp.image_int4s = f64 ? (int64_t)lp.nsb * lp.sbw * B : (int64_t)lp.nsb * lp.sbw * B / 2;
  // float cells: all chunks of a node merge into one double image; multi-output: the bound of its own pairs
  lp.qmax_plan = f64 ? 1u : (multi ? std::max(c->qmax_multi, 1u) : 0u);
  lp.chunk_cap = f64 ? FL_CHUNK_CAP : 0;    // ... and each chunk's float sums cover at most 32k rows
  lp.st = c->st;
  // image scratch for the largest item count the device plan can produce
  // (there are never more group images than items):
  // items <= n_fgroups * n_nodes + max(target_items, n_fgroups * n_rows / rows_per_chunk_min)
  // (a chunk holds at least min(rc, load-balance target) rows, and rc >= 1024 by the quantisation limit)
  int64_t rc = std::max<int64_t>(1, 2147483647LL / std::max<int64_t>(f64 ? 1 : (multi ? c->qmax_multi : c->qmax), 1));
  if (lp.chunk_cap > 0) rc = std::min<int64_t>(rc, lp.chunk_cap);  // the largest chunk the plan can form
  const int64_t items_max = (int64_t)lp.n_fgroups * (n_nodes + 1) +
                            std::max<int64_t>(lp.target_items, (int64_t)lp.n_fgroups * ((c->n_rows + rc - 1) / rc));
  if (items_max > INT32_MAX / 2) return fail(c, GBT_ERR_UNSUPPORTED, "level too large for the work-item plan");
  // group images: the reduce region (at most one group per chunk, chunks <= items_max / n_fgroups) and one
  // store image group per node after it
  const int64_t r_cap = (items_max + lp.n_fgroups - 1) / lp.n_fgroups;
  const size_t group_bytes = (size_t)lp.n_fgroups * lp.image_int4s * 16;
  const size_t r_bytes = (size_t)r_cap * group_bytes;
  const size_t old_cap = c->partial.cap;
  s = ensure(c, c->partial, r_bytes + (size_t)n_nodes * group_bytes, "level image scratch");
  if (s != GBT_OK) return s;
  if (c->partial.cap != old_cap) c->img_clean = 0;  // a new allocation holds anything
  if (r_bytes > c->img_clean)
    CUDA_TRY(c, cudaMemsetAsync((char *)c->partial.p + c->img_clean, 0, r_bytes - c->img_clean, c->stream),
             "zero the reduce images");
  c->img_clean = 0;  // in use until this level's consumer is launched
  c->img_r_pending = r_bytes;
  lp.r_cap_groups = r_cap;
  lp.partial = (int32_t *)c->partial.p;
  s = ensure(c, c->items, (size_t)items_max * sizeof(Item), "level work items");
  if (s != GBT_OK) return s;
  lp.items = (Item *)c->items.p;
  const int hist_ctas = c->n_sm;  // persistent: one resident CTA per SM
  // levels of few nodes are planned by the histogram kernel itself (GBT_PLAN_KERNEL=1 forces the plan kernel)
  lp.fold = (n_nodes <= FOLD_MAX_NODES && !c->plan_kernel) ? 1 : 0;
  lp.pad_ = 0;
  if (!lp.fold) {
    prof_begin(c);
    k_level_plan<<<1, PLAN_THREADS, 0, c->stream>>>(lp);
    LAUNCH_CHECK(c, "k_level_plan");
  }
  lp.qpos = nullptr;
  if (rows_d && !multi && !f64 && lp.n_fgroups >= 16) {
    // many feature tiles: the pairs in level order once, so that each tile's items load them by position
    // (measured: wide, 256 tiles, histogram 320 -> 309 us; u16miss, 16 groups, 193 -> 174 us; the dense
    // tree's 8 tiles gain about what the gather costs)
    s = ensure(c, c->qlev, (size_t)c->n_rows * sizeof(int2), "level gradient pairs");
    if (s != GBT_OK) return s;
    const int g = (int)std::min<int64_t>((c->n_rows + 255) / 256, (int64_t)c->n_sm * 8);
    prof_begin(c);
    launch_pdl(c, k_gather_q, dim3(g), dim3(256), 0, (const int32_t *)rows_d, (const int64_t *)offs_d, n_nodes,
               (int64_t)c->n_rows, (const int2 *)c->q.p, (int2 *)c->qlev.p);
    LAUNCH_CHECK(c, "k_gather_q");
    lp.qpos = (const int2 *)c->qlev.p;
  }
  if (c->bin_bytes == 1) {
    Hist8Params hp;
    hp.lv = lp;
    hp.mirror = (const uint8_t *)c->mirror.p;
    hp.n_features = c->n_features;
    hp.n_slots = B;
    hp.n_targets = K;
    prof_begin(c);
    if (multi) {
      launch_pdl(c, k_hist_u8<false, true>, dim3(hist_ctas), dim3(H8_THREADS), H8_SMEM_RING, hp);
      LAUNCH_CHECK(c, "k_hist_u8_multi");
    } else if (f64) {
      launch_pdl(c, k_hist_u8<true>, dim3(hist_ctas), dim3(H8_THREADS), H8_SMEM + FL_STAGE_BYTES, hp);
      LAUNCH_CHECK(c, "k_hist_u8_f32");
    } else {
      launch_pdl(c, k_hist_u8<false>, dim3(hist_ctas), dim3(H8_THREADS), H8_SMEM_RING, hp);
      LAUNCH_CHECK(c, "k_hist_u8");
    }
  } else {
    Hist16Params hp;
    hp.lv = lp;
    hp.mirror = (const uint16_t *)c->mirror.p;
    hp.n_features = c->n_features;
    hp.n_slots = B;
    hp.n_bins = c->n_bins;
    hp.ts = c->ts16;
    const int hist_bytes = ((B * c->ts16 * 8) + 127) & ~127;
    const int smem = hist_bytes + (f64 ? FL_STAGE_BYTES : H16_STAGE_BYTES);
    prof_begin(c);
    if (f64) {
      switch (c->ts16) {
        case 32: launch_pdl(c, k_hist_u16<32, true>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 16: launch_pdl(c, k_hist_u16<16, true>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 8: launch_pdl(c, k_hist_u16<8, true>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 4: launch_pdl(c, k_hist_u16<4, true>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        default: launch_pdl(c, k_hist_u16<2, true>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
      }
      LAUNCH_CHECK(c, "k_hist_u16_f32");
    } else {
      switch (c->ts16) {
        case 32: launch_pdl(c, k_hist_u16<32, false>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 16: launch_pdl(c, k_hist_u16<16, false>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 8: launch_pdl(c, k_hist_u16<8, false>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        case 4: launch_pdl(c, k_hist_u16<4, false>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
        default: launch_pdl(c, k_hist_u16<2, false>, dim3(hist_ctas), dim3(H16_THREADS), smem, hp); break;
      }
      LAUNCH_CHECK(c, "k_hist_u16");
    }
  }
  *out_lp = lp;
  return GBT_OK;
}

PartialView partial_view(const LevelParams &lp, int B) {
  PartialView v;
  v.partial = lp.partial;
  v.group_prefix = lp.group_prefix;
  v.img_first = lp.img_first;
  v.r_cap = lp.r_cap_groups;
  v.image_int4s = lp.image_int4s;
  v.n_fgroups = lp.n_fgroups;
  v.sbw = lp.sbw;
  v.nsb = lp.nsb;
  v.B = B;
  return v;
}

}  // namespace

extern "C" {

gbt_status gbt_build_level(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                           int64_t *hist_out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!c->tree_ready) return fail(c, GBT_ERR_STATE, "gbt_begin_tree first");
  if (n_nodes < 0 || n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be in [0, 65535]");
  if (!node_offsets || !hist_out) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets and hist_out are required");
  if (ptr_kind(hist_out) != 1 || !aligned16(hist_out))
    return fail(c, GBT_ERR_INVALID_ARG, "hist_out must be 16-byte aligned device memory");
  if (n_nodes == 0) return GBT_OK;
  LevelParams lp;
  s = run_level_build(c, rows, node_offsets, n_nodes, &lp);
  if (s != GBT_OK) return s;
  prof_begin(c);
  const int64_t cells = (int64_t)n_nodes * ((c->n_features + 3) / 4) * 4 * (c->n_bins + 1);
  launch_pdl(c, k_finalize, dim3(grid_for(c, cells, 256, 8)), dim3(256), 0, partial_view(lp, c->n_bins + 1), n_nodes,
             c->n_features, lp.item_feats, hist_out, (const DevState *)c->st);
  LAUNCH_CHECK(c, "k_finalize");
  c->img_clean = c->img_r_pending;
  return GBT_OK;
}

static gbt_status parent_of_view(gbt_ctx *c, const int32_t *parent_of, int32_t n_pairs, const int32_t **out) {
  *out = nullptr;
  if (!parent_of) return GBT_OK;
  const void *d = nullptr;
  gbt_status s = device_view(c, parent_of, (size_t)n_pairs * sizeof(int32_t), c->parent_of_in, &d, "parent_of");
  *out = (const int32_t *)d;
  return s;
}

gbt_status gbt_subtract_siblings(gbt_ctx *c, const int64_t *parent_hist, const int32_t *parent_of,
                                 const int64_t *small_hist, int64_t *large_hist, int32_t n_pairs) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (n_pairs < 0) return fail(c, GBT_ERR_INVALID_ARG, "n_pairs < 0");
  if (n_pairs == 0) return GBT_OK;
  for (const void *p : {(const void *)parent_hist, (const void *)small_hist, (const void *)large_hist})
    if (ptr_kind(p) != 1 || !aligned16(p)) return fail(c, GBT_ERR_INVALID_ARG, "histograms must be 16-byte aligned device memory");
  const int32_t *po = nullptr;
  s = parent_of_view(c, parent_of, n_pairs, &po);
  if (s != GBT_OK) return s;
  const int64_t upn = (int64_t)c->n_features * (c->n_bins + 1);
  const int grid = grid_for(c, (int64_t)n_pairs * upn, 256, 8);
  prof_begin(c);
  k_subtract<<<grid, 256, 0, c->stream>>>(parent_hist, po, small_hist, large_hist, n_pairs, upn, c->st);
  LAUNCH_CHECK(c, "k_subtract");
  return GBT_OK;
}

static gbt_status split_out_view(gbt_ctx *c, gbt_split *out, int32_t n, Buf &stage, SplitOut **dev, bool *host) {
  const int k = ptr_kind(out);
  if (k < 0) return fail(c, GBT_ERR_INVALID_ARG, "split output is NULL");
  *host = (k == 0);
  if (k == 1) {
    *dev = reinterpret_cast<SplitOut *>(out);
    return GBT_OK;
  }
  if (void *d = pinned_device_ptr(out)) {  // the kernels write the pinned host records in place
    *dev = reinterpret_cast<SplitOut *>(d);
    *host = false;
    return GBT_OK;
  }
  gbt_status s = ensure(c, stage, (size_t)n * sizeof(SplitOut), "split staging");
  if (s != GBT_OK) return s;
  *dev = reinterpret_cast<SplitOut *>(stage.p);
  return GBT_OK;
}

gbt_status gbt_find_splits(gbt_ctx *c, const int64_t *hist, int32_t n_nodes, const gbt_params *params,
                           gbt_split *out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!c->tree_ready) return fail(c, GBT_ERR_STATE, "gbt_begin_tree first (scales)");
  if (!params || n_nodes < 0) return fail(c, GBT_ERR_INVALID_ARG, "params NULL or n_nodes < 0");
  if (n_nodes == 0) return GBT_OK;
  if (n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be <= 65535");
  if (ptr_kind(hist) != 1 || !aligned16(hist)) return fail(c, GBT_ERR_INVALID_ARG, "hist must be 16-byte aligned device memory");
  SplitOut *dout = nullptr;
  bool host = false;
  s = split_out_view(c, out, n_nodes, c->splits_a, &dout, &host);
  if (s != GBT_OK) return s;
  const int nfb = (c->n_features + SCAN_WARPS - 1) / SCAN_WARPS;
  s = ensure(c, c->cand, (size_t)n_nodes * nfb * PUB_K * sizeof(Cand), "candidates");
  if (s != GBT_OK) return s;
  s = ensure_counters(c, (size_t)n_nodes);  // arrival counters
  if (s != GBT_OK) return s;
  const SplitParams sp = make_sp(c, params);
  prof_begin(c);
  launch_pdl(c, k_find, dim3(nfb, n_nodes), dim3(SCAN_THREADS), 0, hist, c->n_features, c->n_bins, sp,
             (Cand *)c->cand.p, (uint32_t *)c->counters.p, dout);
  LAUNCH_CHECK(c, "k_find");
  if (host)
    CUDA_TRY(c, cudaMemcpyAsync(out, dout, (size_t)n_nodes * sizeof(gbt_split), cudaMemcpyDeviceToHost, c->stream),
             "splits to host");
  return GBT_OK;
}

gbt_status gbt_build_level_multi(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                                 int64_t *hist_out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->multi_k == 0) return fail(c, GBT_ERR_STATE, "gbt_begin_tree_multi first");
  if (c->bin_bytes != 1) return fail(c, GBT_ERR_UNSUPPORTED, "multi-output histograms need u8 bins");
  if (n_nodes < 0 || n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be in [0, 65535]");
  if (!node_offsets || !hist_out) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets and hist_out are required");
  if (ptr_kind(hist_out) != 1 || !aligned16(hist_out))
    return fail(c, GBT_ERR_INVALID_ARG, "hist_out must be 16-byte aligned device memory");
  if (n_nodes == 0) return GBT_OK;
  LevelParams lp;
  s = run_level_build(c, rows, node_offsets, n_nodes, &lp, nullptr, true);
  if (s != GBT_OK) return s;
  const int B = c->n_bins + 1;
  const int64_t cells = (int64_t)c->multi_k * n_nodes * ((c->n_features + 3) / 4) * 4 * B;
  prof_begin(c);
  launch_pdl(c, k_finalize_multi, dim3(grid_for(c, cells, 256, 8)), dim3(256), 0, partial_view(lp, B), c->multi_k,
             n_nodes, c->n_features, hist_out, (const DevState *)c->st);
  LAUNCH_CHECK(c, "k_finalize_multi");
  c->img_clean = c->img_r_pending;
  return GBT_OK;
}

gbt_status gbt_build_level_f64(gbt_ctx *c, const float *gpair, const int32_t *rows, const int64_t *node_offsets,
                               int32_t n_nodes, double *hist_out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (n_nodes < 0 || n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be in [0, 65535]");
  if (!gpair || !node_offsets || !hist_out) return fail(c, GBT_ERR_INVALID_ARG, "gpair, node_offsets, hist_out required");
  if (ptr_kind(hist_out) != 1 || !aligned16(hist_out))
    return fail(c, GBT_ERR_INVALID_ARG, "hist_out must be 16-byte aligned device memory");
  if (n_nodes == 0) return GBT_OK;
  const void *gp = nullptr;
  s = device_view(c, gpair, (size_t)c->n_rows * 2 * sizeof(float), c->gp_stage, &gp, "gpair");
  if (s != GBT_OK) return s;
  if ((reinterpret_cast<uintptr_t>(gp) & 7u) != 0) return fail(c, GBT_ERR_INVALID_ARG, "gpair must be 8-byte aligned");
  LevelParams lp;
  s = run_level_build(c, rows, node_offsets, n_nodes, &lp, (const float2 *)gp);
  if (s != GBT_OK) return s;
  const int B = c->n_bins + 1;
  const int64_t cells = (int64_t)n_nodes * c->n_features * B;
  prof_begin(c);
  launch_pdl(c, k_finalize_f64, dim3(grid_for(c, cells, 256, 8)), dim3(256), 0, (double *)lp.partial,
             (const int32_t *)lp.group_prefix, (const int32_t *)lp.img_first, (int64_t)lp.r_cap_groups,
             (int64_t)lp.image_int4s * 2, lp.n_fgroups, lp.item_feats, lp.sbw, n_nodes, c->n_features, B, hist_out,
             (const DevState *)c->st);
  LAUNCH_CHECK(c, "k_finalize_f64");
  c->img_clean = c->img_r_pending;
  return GBT_OK;
}

gbt_status gbt_subtract_siblings_f64(gbt_ctx *c, const double *parent_hist, const int32_t *parent_of,
                                     const double *small_hist, double *large_hist, int32_t n_pairs) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (n_pairs < 0) return fail(c, GBT_ERR_INVALID_ARG, "n_pairs < 0");
  if (n_pairs == 0) return GBT_OK;
  for (const void *p : {(const void *)parent_hist, (const void *)small_hist, (const void *)large_hist})
    if (ptr_kind(p) != 1 || !aligned16(p)) return fail(c, GBT_ERR_INVALID_ARG, "histograms must be 16-byte aligned device memory");
  const int32_t *po = nullptr;
  s = parent_of_view(c, parent_of, n_pairs, &po);
  if (s != GBT_OK) return s;
  const int64_t cpn = (int64_t)c->n_features * (c->n_bins + 1);
  prof_begin(c);
  k_subtract_f64<<<grid_for(c, (int64_t)n_pairs * cpn, 256, 8), 256, 0, c->stream>>>(parent_hist, po, small_hist,
                                                                                       large_hist, n_pairs, cpn);
  LAUNCH_CHECK(c, "k_subtract_f64");
  return GBT_OK;
}

gbt_status gbt_find_splits_f64(gbt_ctx *c, const double *hist, int32_t n_nodes, const gbt_params *params,
                               gbt_split_f64 *out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (!params || n_nodes < 0) return fail(c, GBT_ERR_INVALID_ARG, "params NULL or n_nodes < 0");
  if (n_nodes == 0) return GBT_OK;
  if (n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be <= 65535");
  if (ptr_kind(hist) != 1 || !aligned16(hist)) return fail(c, GBT_ERR_INVALID_ARG, "hist must be 16-byte aligned device memory");
  if (c->n_bins > F64_MAX_CHUNKS * 32 * SCAN_SPL) return fail(c, GBT_ERR_UNSUPPORTED, "n_bins too large");
  SplitOut *dout = nullptr;
  bool host = false;
  s = split_out_view(c, reinterpret_cast<gbt_split *>(out), n_nodes, c->splits_a, &dout, &host);
  if (s != GBT_OK) return s;
  const int nfb = (c->n_features + SCAN_WARPS - 1) / SCAN_WARPS;
  s = ensure(c, c->cand, (size_t)n_nodes * nfb * sizeof(Cand), "candidates");
  if (s != GBT_OK) return s;
  s = ensure_counters(c, (size_t)n_nodes);
  if (s != GBT_OK) return s;
  prof_begin(c);
  SplitParams sp{};
  sp.lambda = params->lambda;
  sp.gamma = params->gamma;
  sp.inv_sg = sp.inv_sh = 1.0;
  sp.lambda_f = (float)params->lambda;
  sp.gamma_f = (float)params->gamma;
  sp.gamma_abs_f = fabsf(sp.gamma_f);
  sp.inv_sg_f = sp.inv_sh_f = 1.f;
  sp.filter = (params->lambda >= 0.0 && params->lambda < 1e30 && isfinite(params->gamma) && fabs(params->gamma) < 1e30)
                  ? 1
                  : 0;
  k_find_f64<<<dim3(nfb, n_nodes), SCAN_THREADS, 0, c->stream>>>(hist, c->n_features, c->n_bins, sp,
                                                                 params->min_child_weight, (Cand *)c->cand.p,
                                                                 (uint32_t *)c->counters.p, dout);
  LAUNCH_CHECK(c, "k_find_f64");
  if (host)
    CUDA_TRY(c, cudaMemcpyAsync(out, dout, (size_t)n_nodes * sizeof(gbt_split_f64), cudaMemcpyDeviceToHost, c->stream),
             "splits to host");
  return GBT_OK;
}

gbt_status gbt_find_level_split(gbt_ctx *c, const int64_t *hist, int32_t n_nodes, const gbt_params *params,
                                gbt_split *out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!c->tree_ready) return fail(c, GBT_ERR_STATE, "gbt_begin_tree first (scales)");
  if (!params || n_nodes < 1) return fail(c, GBT_ERR_INVALID_ARG, "params NULL or n_nodes < 1");
  if (n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be <= 65535");
  if (ptr_kind(hist) != 1 || !aligned16(hist)) return fail(c, GBT_ERR_INVALID_ARG, "hist must be 16-byte aligned device memory");
  SplitOut *dout = nullptr;
  bool host = false;
  s = split_out_view(c, out, 1, c->splits_a, &dout, &host);
  if (s != GBT_OK) return s;
  const int n_chunks = (c->n_bins + LS_CHUNK - 1) / LS_CHUNK;
  // warps per feature: enough to share the nodes, the rest of the CTA's 8 warps take more features
  int wpf = 1;
  while (wpf < SCAN_WARPS && wpf * 8 <= n_nodes) wpf *= 2;
  const int fpc = SCAN_WARPS / wpf;
  const int64_t ctas = (int64_t)((c->n_features + fpc - 1) / fpc) * n_chunks;
  if (n_chunks > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "too many bins for the level split grid");
  s = ensure(c, c->cand, (size_t)ctas * PUB_K * sizeof(Cand), "candidates");
  if (s != GBT_OK) return s;
  s = ensure_counters(c, 2);
  if (s != GBT_OK) return s;
  // [n_nodes][F] totals, [n_nodes][F][n_chunks] carries, [SCAN_WARPS + ctas][n_nodes] exact-gain buffers
  const size_t nf = (size_t)n_nodes * c->n_features;
  const size_t tot_bytes = nf * sizeof(LevelTot), carry_bytes = nf * n_chunks * sizeof(longlong2);
  s = ensure(c, c->level_scratch, tot_bytes + carry_bytes + (size_t)(SCAN_WARPS + ctas) * n_nodes * sizeof(double),
             "level split scratch");
  if (s != GBT_OK) return s;
  LevelTot *tot = (LevelTot *)c->level_scratch.p;
  longlong2 *carry = (longlong2 *)((char *)c->level_scratch.p + tot_bytes);
  double *gbuf = (double *)((char *)c->level_scratch.p + tot_bytes + carry_bytes);
  const SplitParams sp = make_sp(c, params);
  prof_begin(c);
  k_level_totals<<<(unsigned)((nf * 32 + 255) / 256), 256, 0, c->stream>>>(hist, n_nodes, c->n_features, c->n_bins,
                                                                          tot, carry);
  LAUNCH_CHECK(c, "k_level_totals");
  prof_begin(c);
  launch_pdl(c, k_level_split, dim3((c->n_features + fpc - 1) / fpc, n_chunks), dim3(SCAN_THREADS), 0, hist, n_nodes,
             c->n_features, c->n_bins, sp, (const LevelTot *)tot, (const longlong2 *)carry, (Cand *)c->cand.p,
             (uint32_t *)c->counters.p, gbuf, (int32_t)wpf, dout);
  LAUNCH_CHECK(c, "k_level_split");
  if (host)
    CUDA_TRY(c, cudaMemcpyAsync(out, dout, sizeof(gbt_split), cudaMemcpyDeviceToHost, c->stream), "split to host");
  return GBT_OK;
}

}  // extern "C"

namespace {

// Shared tail of gbt_subtract_and_find and gbt_level_step: one launch of the
// level-finish kernel (small strip from `src`, subtraction, split find).
template <bool FROM_PARTIALS>
gbt_status run_level_finish(gbt_ctx *c, const SmallSource &src, const int64_t *parent_hist, const int32_t *parent_of,
                            int64_t *large_hist, int32_t n_pairs, const gbt_params *params, gbt_split *small_out,
                            gbt_split *large_out, const uint8_t *side = nullptr) {
  const int32_t *po = nullptr;
  gbt_status s = parent_of_view(c, parent_of, n_pairs, &po);
  if (s != GBT_OK) return s;
  SplitOut *da = nullptr, *db = nullptr;
  bool ha = false, hb = false;
  // node order (side given): one array of 2 n_pairs splits, small and large interleaved by pair
  const int32_t n_out = side ? 2 * n_pairs : n_pairs;
  s = split_out_view(c, small_out, n_out, c->splits_a, &da, &ha);
  if (s != GBT_OK) return s;
  if (side) {
    db = da;
  } else {
    s = split_out_view(c, large_out, n_pairs, c->splits_b, &db, &hb);
    if (s != GBT_OK) return s;
  }
  const int nfb = (c->n_features + 3) / 4;
  // candidate records, then their bounds (lo, up) as float2 (16-byte aligned: the records are 64 bytes)
  const size_t n_ent = (size_t)2 * n_pairs * nfb * PUB_K;
  s = ensure(c, c->cand, n_ent * (sizeof(Cand) + sizeof(float2)), "candidates");
  if (s != GBT_OK) return s;
  float2 *cbounds = reinterpret_cast<float2 *>((Cand *)c->cand.p + n_ent);
  s = ensure_counters(c, (size_t)n_pairs);  // arrival counters
  if (s != GBT_OK) return s;
  const SplitParams sp = make_sp(c, params);
  prof_begin(c);
  // staged strips: when the grid is more than one wave of 3 CTAs per SM, the 4-CTA register budget
  // and FIN_PASSES groups of four features per CTA (its selection, publication and node-reduce
  // entries paid once for all); long strips: two CTAs per SM, whose register budget holds the long
  // scan without spills
  constexpr int FIN_PASSES = 4;  // measured on wide: 2 passes 341 us, 4 passes 314 us, 8 passes 313 us
  const bool many = c->n_bins + 1 <= STAGE_SLOTS && (int64_t)nfb * n_pairs > 3 * (int64_t)c->n_sm;
  // passes only while the grid of passes still fills three waves of four CTAs per SM (fewer, longer
  // chains would leave SMs idle)
  const bool passes = many && (int64_t)nfb * n_pairs / FIN_PASSES >= 3 * 4 * (int64_t)c->n_sm;
  const int nfb_launch = passes ? (c->n_features + 4 * FIN_PASSES - 1) / (4 * FIN_PASSES) : nfb;
  auto kern = c->n_bins + 1 > STAGE_SLOTS ? k_level_finish<FROM_PARTIALS, false, 2, 1>
               : passes                  ? k_level_finish<FROM_PARTIALS, true, 4, FIN_PASSES>
               : many                    ? k_level_finish<FROM_PARTIALS, true, 4, 1>
                                         : k_level_finish<FROM_PARTIALS, true, 3, 1>;
  launch_pdl(c, kern, dim3(nfb_launch, n_pairs), dim3(SCAN_THREADS), 0, src, parent_hist, po, large_hist,
             c->n_features, c->n_bins, sp, (Cand *)c->cand.p, cbounds, (uint32_t *)c->counters.p, da, db, c->st, side);
  LAUNCH_CHECK(c, FROM_PARTIALS ? "k_level_finish" : "k_subtract_find");
  if (FROM_PARTIALS) c->img_clean = c->img_r_pending;
  if (ha)
    CUDA_TRY(c, cudaMemcpyAsync(small_out, da, (size_t)n_out * sizeof(gbt_split), cudaMemcpyDeviceToHost, c->stream),
             "splits to host");
  if (hb)
    CUDA_TRY(c, cudaMemcpyAsync(large_out, db, (size_t)n_pairs * sizeof(gbt_split), cudaMemcpyDeviceToHost, c->stream),
             "splits to host");
  return GBT_OK;
}

gbt_status check_pair_args(gbt_ctx *c, const gbt_params *params, int32_t n_pairs,
                           std::initializer_list<const void *> hists) {
  if (!c->tree_ready) return fail(c, GBT_ERR_STATE, "gbt_begin_tree first (scales)");
  if (!params || n_pairs < 0) return fail(c, GBT_ERR_INVALID_ARG, "params NULL or n_pairs < 0");
  if (n_pairs > 32767) return fail(c, GBT_ERR_UNSUPPORTED, "n_pairs must be <= 32767");
  for (const void *p : hists)
    if (ptr_kind(p) != 1 || !aligned16(p))
      return fail(c, GBT_ERR_INVALID_ARG, "histograms must be 16-byte aligned device memory");
  return GBT_OK;
}

}  // namespace

extern "C" {

gbt_status gbt_subtract_and_find(gbt_ctx *c, const int64_t *parent_hist, const int32_t *parent_of,
                                 const int64_t *small_hist, int64_t *large_hist, int32_t n_pairs,
                                 const gbt_params *params, gbt_split *small_out, gbt_split *large_out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (n_pairs == 0 && params) return GBT_OK;
  s = check_pair_args(c, params, n_pairs, {parent_hist, small_hist, large_hist});
  if (s != GBT_OK) return s;
  SmallSource src{};
  src.hist = small_hist;
  return run_level_finish<false>(c, src, parent_hist, parent_of, large_hist, n_pairs, params, small_out, large_out);
}

gbt_status gbt_level_step(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_pairs,
                          const int64_t *parent_hist, const int32_t *parent_of, int64_t *small_hist,
                          int64_t *large_hist, const gbt_params *params, gbt_split *small_out,
                          gbt_split *large_out) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!node_offsets) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets is required");
  if (n_pairs == 0 && params) return GBT_OK;
  s = check_pair_args(c, params, n_pairs, {parent_hist, small_hist, large_hist});
  if (s != GBT_OK) return s;
  LevelParams lp;
  s = run_level_build(c, rows, node_offsets, n_pairs, &lp);
  if (s != GBT_OK) return s;
  SmallSource src{};
  src.view = partial_view(lp, c->n_bins + 1);
  src.item_feats = lp.item_feats;
  src.hist_out = small_hist;
  return run_level_finish<true>(c, src, parent_hist, parent_of, large_hist, n_pairs, params, small_out, large_out);
}

}  // extern "C"

namespace {

// Shared body of gbt_partition_level and gbt_partition_level_pairs (small_* NULL: no smaller-child list).
gbt_status partition_impl(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                          const gbt_split *splits, int32_t *out_rows, int64_t *out_offsets, int32_t *small_rows,
                          int64_t *small_offsets, uint8_t *small_side) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (c->n_rows == 0) return fail(c, GBT_ERR_STATE, "gbt_upload_bins first");
  if (n_nodes < 0 || n_nodes > 65535) return fail(c, GBT_ERR_UNSUPPORTED, "n_nodes must be in [0, 65535]");
  if (n_nodes == 0) return GBT_OK;
  if (!node_offsets || !splits || !out_rows || !out_offsets) return fail(c, GBT_ERR_INVALID_ARG, "NULL argument");
  if (ptr_kind(out_rows) != 1 || ptr_kind(out_offsets) != 1)
    return fail(c, GBT_ERR_INVALID_ARG, "out_rows and out_offsets must be device memory");
  const bool pairs = small_rows != nullptr || small_offsets != nullptr || small_side != nullptr;
  if (pairs && (ptr_kind(small_rows) != 1 || ptr_kind(small_offsets) != 1 || ptr_kind(small_side) != 1))
    return fail(c, GBT_ERR_INVALID_ARG, "small_rows, small_offsets and small_side must all be device memory");
  int64_t R_host = -1;
  if (ptr_kind(node_offsets) == 0) {
    if (node_offsets[0] != 0) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets[0] must be 0");
    for (int32_t i = 0; i < n_nodes; ++i)
      if (node_offsets[i + 1] < node_offsets[i]) return fail(c, GBT_ERR_INVALID_ARG, "node_offsets must ascend");
    R_host = node_offsets[n_nodes];
    if (R_host > c->n_rows) return fail(c, GBT_ERR_INVALID_ARG, "more level rows than dataset rows");
  }
  const void *offs_d = nullptr;
  s = device_view(c, node_offsets, (size_t)(n_nodes + 1) * sizeof(int64_t), c->offs_in, &offs_d, "node_offsets");
  if (s != GBT_OK) return s;
  const void *rows_d = nullptr;
  if (rows) {
    const int k = ptr_kind(rows);
    if (k == 0 && R_host < 0) return fail(c, GBT_ERR_INVALID_ARG, "host rows need host node_offsets");
    if (k == 0) {
      s = device_view(c, rows, (size_t)R_host * sizeof(int32_t), c->rows_in, &rows_d, "rows");
      if (s != GBT_OK) return s;
    } else {
      rows_d = rows;
    }
  }
  const void *sp_d = nullptr;
  s = device_view(c, splits, (size_t)n_nodes * sizeof(gbt_split), c->splits_b, &sp_d, "splits");
  if (s != GBT_OK) return s;
  const int64_t bound = R_host >= 0 ? R_host : c->n_rows;
  const int64_t n_tiles = std::max<int64_t>(1, (bound + PART_TILE - 1) / PART_TILE);
  s = ensure(c, c->tile_counts, (size_t)(n_tiles + 1) * sizeof(int64_t), "partition tile counts");
  if (s != GBT_OK) return s;
  s = ensure(c, c->lrank, (size_t)(n_nodes + 1) * sizeof(int64_t), "partition node ranks");
  if (s != GBT_OK) return s;
  s = ensure(c, c->pflags, (size_t)n_tiles * (PART_TILE / 8) + 16, "partition flags");
  if (s != GBT_OK) return s;
  PartParams pp;
  pp.rows = (const int32_t *)rows_d;
  pp.offs = (const int64_t *)offs_d;
  pp.n_nodes = n_nodes;
  pp.tile_feats = c->tile_feats;
  pp.bin_bytes = c->bin_bytes;
  pp.n_bins = c->n_bins;
  pp.n_features = c->n_features;
  pp.pad = 0;
  pp.n_rows = c->n_rows;
  pp.cols = (const unsigned char *)c->cols.p;
  pp.splits = (const SplitOut *)sp_d;
  pp.tile_counts = (int64_t *)c->tile_counts.p;
  pp.flags = (uint8_t *)c->pflags.p;
  pp.lrank = (int64_t *)c->lrank.p;
  pp.out_rows = out_rows;
  pp.out_offs = out_offsets;
  pp.small_rows = pairs ? small_rows : nullptr;
  pp.small_offs = pairs ? small_offsets : nullptr;
  pp.small_side = pairs ? small_side : nullptr;
  pp.st = c->st;
  prof_begin(c);
  k_part_flags<<<(unsigned)n_tiles, PART_THREADS, 0, c->stream>>>(pp);
  LAUNCH_CHECK(c, "k_part_flags");
  prof_begin(c);
  k_part_scan<<<1, 1024, 0, c->stream>>>(pp, n_tiles);
  LAUNCH_CHECK(c, "k_part_scan");
  prof_begin(c);
  k_part_scatter<<<(unsigned)n_tiles, PART_THREADS, 0, c->stream>>>(pp);
  LAUNCH_CHECK(c, "k_part_scatter");
  return GBT_OK;
}

}  // namespace

extern "C" {

gbt_status gbt_advance_level(gbt_ctx *c, const int32_t *small_rows, const int64_t *small_offsets,
                             const uint8_t *small_side, int32_t n_pairs, const int64_t *parent_hist,
                             int64_t *level_hist, const gbt_params *params, gbt_split *level_splits) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!small_offsets) return fail(c, GBT_ERR_INVALID_ARG, "small_offsets is required");
  if (n_pairs == 0 && params) return GBT_OK;
  s = check_pair_args(c, params, n_pairs, {parent_hist, level_hist});
  if (s != GBT_OK) return s;
  if (!level_splits) return fail(c, GBT_ERR_INVALID_ARG, "level_splits is required");
  const void *side_d = nullptr;
  if (small_side) {
    s = device_view(c, small_side, (size_t)n_pairs, c->side_in, &side_d, "small_side");
    if (s != GBT_OK) return s;
  } else {
    s = ensure(c, c->side_in, (size_t)n_pairs, "small_side zeros");
    if (s != GBT_OK) return s;
    CUDA_TRY(c, cudaMemsetAsync(c->side_in.p, 0, (size_t)n_pairs, c->stream), "small_side zeros");
    side_d = c->side_in.p;
  }
  LevelParams lp;
  s = run_level_build(c, small_rows, small_offsets, n_pairs, &lp);
  if (s != GBT_OK) return s;
  SmallSource src{};
  src.view = partial_view(lp, c->n_bins + 1);
  src.item_feats = lp.item_feats;
  src.hist_out = level_hist;
  return run_level_finish<true>(c, src, parent_hist, nullptr, level_hist, n_pairs, params, level_splits, level_splits,
                                (const uint8_t *)side_d);
}

gbt_status gbt_partition_level(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                               const gbt_split *splits, int32_t *out_rows, int64_t *out_offsets) {
  return partition_impl(c, rows, node_offsets, n_nodes, splits, out_rows, out_offsets, nullptr, nullptr, nullptr);
}

gbt_status gbt_partition_level_pairs(gbt_ctx *c, const int32_t *rows, const int64_t *node_offsets, int32_t n_nodes,
                                     const gbt_split *splits, int32_t *out_rows, int64_t *out_offsets,
                                     int32_t *small_rows, int64_t *small_offsets, uint8_t *small_side) {
  if (!small_rows || !small_offsets || !small_side) {
    if (c) c->last_error = "small_rows, small_offsets and small_side are required";
    return GBT_ERR_INVALID_ARG;
  }
  return partition_impl(c, rows, node_offsets, n_nodes, splits, out_rows, out_offsets, small_rows, small_offsets,
                        small_side);
}

gbt_status gbt_profile_enable(gbt_ctx *c, int on) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  c->prof = on != 0;
  return GBT_OK;
}

gbt_status gbt_profile_read(gbt_ctx *c, const char *kernel, double *total_ms, int64_t *launches) {
  gbt_status s = check_ctx(c);
  if (s != GBT_OK) return s;
  if (!total_ms || !launches) return fail(c, GBT_ERR_INVALID_ARG, "NULL output");
  CUDA_TRY(c, cudaStreamSynchronize(c->stream), "stream synchronize");
  double ms = 0.0;
  int64_t n = 0;
  std::vector<gbt_ctx::ProfRec> keep;
  for (const auto &r : c->prof_pending) {
    if (kernel && strcmp(kernel, r.name) != 0) {
      keep.push_back(r);
      continue;
    }
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      ms += t;
      ++n;
    } else {
      cudaGetLastError();
    }
    c->prof_pool.push_back(r.a);
    c->prof_pool.push_back(r.b);
  }
  c->prof_pending.swap(keep);
  *total_ms = ms;
  *launches = n;
  return GBT_OK;
}

int32_t gbt_slots_per_feature(const gbt_ctx *c) { return (c && c->n_rows > 0) ? c->n_bins + 1 : -1; }

int64_t gbt_kernel_launches(const gbt_ctx *c) { return c ? c->launches : 0; }

}  // extern "C"

// ---------------------------------------------------------------------------- split find without allocation
// For callers that may not allocate device memory at all: code running inside
// a host that owns every allocation (a pool or arena it hands out itself), or
// a stream-ordered pipeline where a cudaMalloc would synchronise the device
// and stall other work. The split find's scratch (per-CTA candidates and the
// per-node arrival counters) lives here in one fixed array that is part of the
// loaded module; every GPU that loads the library keeps it until exit.

namespace {
constexpr int NOALLOC_MAX_NODES = 4096;    // nodes per call
constexpr int NOALLOC_MAX_CANDS = 32768;   // nodes * ceil(n_features / 8) per call
constexpr size_t NOALLOC_COUNTER_BYTES = (size_t)2 * NOALLOC_MAX_NODES * sizeof(uint32_t);  // counters (two words per node reserved)
constexpr size_t NOALLOC_BYTES =
    NOALLOC_COUNTER_BYTES + (size_t)NOALLOC_MAX_CANDS * PUB_K * sizeof(Cand);  // 4 MiB + 32 KiB
static_assert(NOALLOC_COUNTER_BYTES % 256 == 0, "candidate area alignment");
constexpr int NOALLOC_MAX_DEVICES = 64;
}  // namespace

// Host code sees only a stand-in for this array; its device address comes from
// cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

namespace {
std::mutex g_noalloc_mu;
// Device address of g_noalloc_scratch per device, with the id of the context it was taken in: a context
// destroyed and created again (cudaDeviceReset, or the caller switching contexts) loads the module
// again, so the address is looked up again whenever the current context's id differs.
void *g_noalloc_addr[NOALLOC_MAX_DEVICES] = {};
unsigned long long g_noalloc_ctx[NOALLOC_MAX_DEVICES] = {};

// The calling thread's current context's process-unique id, or 0 when it cannot be read. The two
// driver entry points are looked up through the runtime, so the library links no driver library.
unsigned long long current_ctx_id() {
  static std::once_flag once;
  static CUresult (*get_current)(CUcontext *) = nullptr;
  static CUresult (*get_id)(CUcontext, unsigned long long *) = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CUresult (*)(CUcontext *)>(f);
    f = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long *)>(f);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace

extern "C" {

gbt_status gbt_find_splits_noalloc(const int64_t *hist, int32_t n_nodes, int32_t n_features, int32_t n_bins,
                                   float scale_g, float scale_h, const gbt_params *params, gbt_split *out,
                                   void *cuda_stream) {
  if (!hist || !params || !out) return GBT_ERR_INVALID_ARG;
  if (n_nodes < 0 || n_features < 1 || n_bins < 1 || n_bins > 65535) return GBT_ERR_INVALID_ARG;
  if (!(scale_g > 0.f) || !(scale_h > 0.f) || !isfinite(scale_g) || !isfinite(scale_h)) return GBT_ERR_INVALID_ARG;
  if (n_nodes == 0) return GBT_OK;
  const int64_t nfb = (n_features + SCAN_WARPS - 1) / SCAN_WARPS;
  if (n_nodes > NOALLOC_MAX_NODES || (int64_t)n_nodes * nfb > NOALLOC_MAX_CANDS) return GBT_ERR_UNSUPPORTED;
  if (ptr_kind(hist) != 1 || !aligned16(hist) || ptr_kind(out) != 1) return GBT_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GBT_ERR_CUDA;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return GBT_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const unsigned long long ctx_id = current_ctx_id();
    if (!g_noalloc_addr[dev] || ctx_id == 0 || ctx_id != g_noalloc_ctx[dev]) {
      void *p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return GBT_ERR_CUDA;
      }
      g_noalloc_addr[dev] = p;
      g_noalloc_ctx[dev] = current_ctx_id();  // the lookup may have made the primary context current
    }
    scratch = g_noalloc_addr[dev];
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  uint32_t *counters = static_cast<uint32_t *>(scratch);
  Cand *cand = reinterpret_cast<Cand *>(static_cast<unsigned char *>(scratch) + NOALLOC_COUNTER_BYTES);
  // the arrival counters must start at zero whatever an earlier call left
  if (cudaMemsetAsync(counters, 0, (size_t)2 * n_nodes * sizeof(uint32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    return GBT_ERR_CUDA;
  }
  // make_sp reads only the two inverse scales of the context
  gbt_ctx scales;
  scales.inv_sg = 1.0 / (double)scale_g;
  scales.inv_sh = 1.0 / (double)scale_h;
  const SplitParams sp = make_sp(&scales, params);
  k_find<<<dim3((unsigned)nfb, n_nodes), SCAN_THREADS, 0, stream>>>(hist, n_features, n_bins, sp, cand, counters,
                                                                     reinterpret_cast<SplitOut *>(out));
  if (cudaGetLastError() != cudaSuccess) return GBT_ERR_CUDA;
  return GBT_OK;
}

}  // extern "C"
