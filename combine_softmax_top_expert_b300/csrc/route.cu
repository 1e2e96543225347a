// Router: softmax top-k per token ("6.4 Data parallelism and expert parallelism",
// section 3.1, step 1 "Route").
//
// One warp per token.  Lane l holds experts l, l+32, ... as 64-bit keys
// (order-preserving bits of the selection score << 32 | ~index), so the warp
// maximum of the keys is the largest score with ties going to the lower index.  k
// rounds of a warp max pick the experts in order; lane j keeps the j-th pick and
// computes its renormalised weight exp(l_j - m) / sum_i exp(l_i - m) over the picked
// logits l (m their maximum).  The score is the logit, or with a selection bias
// (the bias-without-aux-loss balancing the page mentions, section 5.1) logit + b_e
// in fp32; the bias steers which experts are picked, never their weights.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 ties with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, const float *__restrict__ bias,
                                                     int64_t T, int E, int k, int32_t *__restrict__ ids,
                                                     float *__restrict__ w, int32_t *err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    const float *row = logits + t * E;
    uint64_t key[VPL];
    bool bad = false;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int e = lane + 32 * v;
      if (e < E) {
        const float f = __ldg(row + e);
        const float sc = bias ? f + __ldg(bias + e) : f;
        bad |= !isfinite(f) || !isfinite(sc);
        key[v] = ((uint64_t)ordered_key(sc) << 32) | (uint32_t)(0xffffffffu - (uint32_t)e);
      } else {
        key[v] = 0ull;
      }
    }
    if (__any_sync(kFull, bad) && lane == 0) raise_dev(err, MOE_DEV_NONFINITE_LOGIT);
    uint64_t best = 0ull;
#pragma unroll
    for (int v = 0; v < VPL; ++v) best = key[v] > best ? key[v] : best;
    uint64_t mine = 0ull;
    for (int r = 0; r < k; ++r) {
      const uint64_t m = warp_max_u64(best);
      if (lane == r) mine = m;
      if (best == m) {  // this lane owned the winner: drop it and refresh its best
        best = 0ull;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          if (key[v] == m) key[v] = 0ull;
          best = key[v] > best ? key[v] : best;
        }
      }
    }
    const int pick = (int)(0xffffffffu - (uint32_t)(mine & 0xffffffffull));
    // the picked expert's logit: the key's score without a bias, else reread
    float l = -INFINITY;
    if (lane < k) l = bias ? __ldg(row + pick) : key_value((uint32_t)(mine >> 32));
    float lmax = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(kFull, lmax, o));
    float ex = 0.f;
    if (lane < k) ex = expf(l - lmax);
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane < k) {
      ids[t * k + lane] = (int32_t)pick;
      w[t * k + lane] = ex / sum;
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
  if (e <= 32) launch_route<1>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  else if (e <= 64) launch_route<2>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  else if (e <= 128) launch_route<4>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  else if (e <= 256) launch_route<8>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  else if (e <= 512) launch_route<16>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  else launch_route<32>(logits, b, T, e, k, topk_ids, topk_w, err, st);
  return launch_status();
}

MOE_API moe_status_t moe_route(const float *logits, int64_t T, int64_t E, int32_t k, int32_t *topk_ids,
                               float *topk_w, int32_t *err, moe_stream_t stream) {
  return moe_route_biased(logits, nullptr, T, E, k, topk_ids, topk_w, err, stream);
}
