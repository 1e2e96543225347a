// Per-token router step shared by the route kernel and the fused small-batch
// route + layout kernel ("6.4 Data parallelism and expert parallelism", section
// 3.1, step 1 "Route").
//
// One warp per token.  Lane l holds experts l, l+32, ... as 64-bit keys
// (order-preserving bits of the selection score << 32 | ~index), so the warp
// maximum of the keys is the largest score with ties going to the lower index.  k
// rounds of a warp max pick the experts in order; lane j keeps the j-th pick and
// computes its renormalised weight exp(l_j - m) / sum_i exp(l_i - m) over the picked
// logits l (m their maximum).  The score is the logit, or with a selection bias
// (the bias-without-aux-loss balancing the page mentions, section 5.1) logit + b_e
// in fp32; the bias steers which experts are picked, never their weights.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace moe {
namespace rt {

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 ties with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

// Warp maximum of 64-bit keys, compared as (high word, low word): the largest high
// word, then the largest low word among the lanes holding it (two warp reductions).
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32);
  const uint32_t mhi = __reduce_max_sync(kFull, hi);
  const uint32_t mlo = __reduce_max_sync(kFull, hi == mhi ? static_cast<uint32_t>(v) : 0u);
  return (static_cast<uint64_t>(mhi) << 32) | mlo;
}

// Route the token whose logits start at `row` (E <= 32 * VPL).  Lane j < k gets the
// j-th pick and its weight; a non-finite logit or score raises MOE_DEV_NONFINITE_LOGIT.
template <int VPL>
__device__ __forceinline__ void route_token(const float *__restrict__ row, const float *__restrict__ bias, int E,
                                            int k, int32_t *err, int &pick, float &weight) {
  const int lane = threadIdx.x & 31;
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
  pick = (int)(0xffffffffu - (uint32_t)(mine & 0xffffffffull));
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
  weight = ex / sum;
}

// Call f(std::integral_constant<int, VPL>) with the smallest lanes-per-warp count
// that holds E experts.
template <typename F>
__host__ void with_vpl(int E, F &&f) {
  if (E <= 32) f(std::integral_constant<int, 1>{});
  else if (E <= 64) f(std::integral_constant<int, 2>{});
  else if (E <= 128) f(std::integral_constant<int, 4>{});
  else if (E <= 256) f(std::integral_constant<int, 8>{});
  else if (E <= 512) f(std::integral_constant<int, 16>{});
  else f(std::integral_constant<int, 32>{});
}

}  // namespace rt
}  // namespace moe
