// Router: softmax top-k per token ("6.4 Data parallelism and expert parallelism",
// section 3.1, step 1 "Route"): one warp per token, the step in route.cuh.
#include "route.cuh"

namespace moe {
namespace {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, const float *__restrict__ bias,
                                                     int64_t T, int E, int k, int32_t *__restrict__ ids,
                                                     float *__restrict__ w, int32_t *err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    int pick;
    float wt;
    rt::route_token<VPL>(logits + t * E, bias, E, k, err, pick, wt);
    if (lane < k) {
      ids[t * k + lane] = (int32_t)pick;
      w[t * k + lane] = wt;
    }
  }
}

template <int VPL>
void launch_route(const float *logits, const float *bias, int64_t T, int E, int k, int32_t *ids, float *w,
                  int32_t *err, cudaStream_t st) {
  const int64_t blocks_needed = (T + 7) / 8;
  const int blocks = (int)(blocks_needed < 148 * 16 ? blocks_needed : 148 * 16);
  route_kernel<VPL><<<blocks, 256, 0, st>>>(logits, bias, T, E, k, ids, w, err);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_route_biased(const float *logits, const float *selection_bias, int64_t T, int64_t E,
                                      int32_t k, int32_t *topk_ids, float *topk_w, int32_t *err,
                                      moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_cuda(stream);
  const int e = (int)E;
  const float *b = selection_bias;
  rt::with_vpl(e, [&](auto vpl) { launch_route<decltype(vpl)::value>(logits, b, T, e, k, topk_ids, topk_w, err, st); });
  return launch_status();
}

MOE_API moe_status_t moe_route(const float *logits, int64_t T, int64_t E, int32_t k, int32_t *topk_ids,
                               float *topk_w, int32_t *err, moe_stream_t stream) {
  return moe_route_biased(logits, nullptr, T, E, k, topk_ids, topk_w, err, stream);
}
