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
// made while that device is current (cudaGetSymbolAddress).  Make that first call
// before any stream capture begins.
#include <mutex>

#include "common.cuh"

namespace moe {

size_t dispatch_ws_bytes(int64_t T, int32_t k, int64_t P);
moe_status_t dispatch_layout(const int32_t *, int64_t, int32_t, int64_t, int32_t, const moe_eplb_t *, int32_t *,
                             int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, moe_load_stats_t *,
                             void *, size_t, int32_t *, cudaStream_t);

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
static_assert(kStaticScratchBytes == MOE_DISPATCH_STATIC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).
moe_status_t scratch_on_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cuda_status(cudaGetSymbolAddress(&p, g_layout_scratch)) != MOE_OK || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  if (T < 0 || k < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  const int64_t P = eplb ? eplb->P : E;
  if (P < 1) return MOE_ERR_INVALID_ARG;
  const size_t need = dispatch_ws_bytes(T, k, P);
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // batch too large for the built-in scratch
  void *scratch = nullptr;
  moe_status_t s = scratch_on_current_device(&scratch);
  if (s != MOE_OK) return s;
  return dispatch_layout(topk_ids, T, k, E, R, eplb, logical_counts, phys_counts, phys_offsets, rank_counts,
                         rank_offsets, row_to_token, slot_to_row, stats, scratch, kStaticScratchBytes, err,
                         as_cuda(stream));
}
