// moe_dispatch_layout_static: the dispatch layout for callers that cannot
// allocate device memory at all.
//
// Who needs it: a caller that is handed only its input and output buffers, with
// no device allocator to draw a workspace from -- for example a plugin inside a
// host runtime that owns every allocation and pre-budgets memory, or code on a
// latency-critical path where allocating (and the synchronisation cudaMalloc may
// imply) is not allowed.  moe_dispatch_layout needs a caller-provided workspace;
// this entry point takes its scratch from a fixed array compiled into the library
// instead and allocates nothing.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes (4 MiB).
// Every GPU that loads this library reserves it until the process exits.  All
// calls share it and it keeps whatever the previous call left there; the layout
// kernels overwrite every scratch entry before reading it, so nothing needs to be
// cleared.  Because of the sharing, two calls whose work overlaps on a GPU (on
// different streams, or from different host threads) race on the scratch and give
// wrong results: order them on one stream or synchronise between them.
//
// The device address of the array is looked up once per device, on the first call
// made while that device is current (cudaGetSymbolAddress), and again whenever the
// device's current context has changed since (after cudaDeviceReset the device gets
// a new context, and the array a new address).  Make the first call on a device, and
// the first call after a reset, before any stream capture begins.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace moe {

size_t dispatch_ws_bytes(int64_t T, int32_t k, int64_t P);
moe_status_t dispatch_shape_status(int64_t T, int32_t k, int64_t E, int32_t R, const moe_eplb_t *eplb);
moe_status_t dispatch_layout(const int32_t *, int64_t, int32_t, int64_t, int32_t, const moe_eplb_t *, int32_t *,
                             int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, moe_load_stats_t *,
                             void *, size_t, int32_t *, cudaStream_t);

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
static_assert(kStaticScratchBytes == MOE_DISPATCH_STATIC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddr {
  CUcontext ctx;  // the context the address was looked up in
  void *ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// The driver's cuCtxGetCurrent, reached through the runtime (the library links only cudart).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// Device address of the scratch array on the current device: looked up on the first
// use in the device's current context, and again when that context has changed.
moe_status_t scratch_on_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!ctx || !g_scratch[dev].ptr || g_scratch[dev].ctx != ctx) {
    // (no current context yet: the lookup makes the device's primary context current)
    void *p = nullptr;
    if (cuda_status(cudaGetSymbolAddress(&p, g_layout_scratch)) != MOE_OK || !p) return MOE_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return MOE_ERR_CUDA;
    g_scratch[dev] = {ctx, p};
  }
  *out = g_scratch[dev].ptr;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

MOE_API moe_status_t moe_dispatch_layout_static(const int32_t *topk_ids, int64_t T, int32_t k, int64_t E, int32_t R,
                                                const moe_eplb_t *eplb, int32_t *logical_counts, int32_t *phys_counts,
                                                int32_t *phys_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                                                int32_t *row_to_token, int32_t *slot_to_row, moe_load_stats_t *stats,
                                                int32_t *err, moe_stream_t stream) {
  using namespace moe;
  // the same answers as moe_dispatch_layout for bad sizes, before any size is computed
  const moe_status_t shape = dispatch_shape_status(T, k, E, R, eplb);
  if (shape != MOE_OK) return shape;
  const int64_t P = eplb ? eplb->P : E;
  const size_t need = dispatch_ws_bytes(T, k, P);
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // batch too large for the built-in scratch
  void *scratch = nullptr;
  moe_status_t s = scratch_on_current_device(&scratch);
  if (s != MOE_OK) return s;
  return dispatch_layout(topk_ids, T, k, E, R, eplb, logical_counts, phys_counts, phys_offsets, rank_counts,
                         rank_offsets, row_to_token, slot_to_row, stats, scratch, kStaticScratchBytes, err,
                         as_cuda(stream));
}
