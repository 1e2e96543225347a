// Internal interface of the expert-FFN implementations.
#pragma once

#include "common.cuh"

namespace moe {

struct FfnArgs {
  const void *x_perm;      // [N, d] in the expert input dtype
  const float *x_scales;   // e4m3: [N, d/128]
  const int32_t *offs;     // [P + 1] physical expert offsets
  const int32_t *p2l;      // [P] or null (identity)
  int64_t P, N;
  const moe_weights_t *w;
  const void *shared_x;    // [T_shared, d] or null
  int64_t T_shared;
  void *h;                 // [N + T_shared, I] workspace (+ e4m3 scales after it)
  float *h_scales;         // e4m3: [N + T_shared, I/128]
  void *y;                 // [N + T_shared, d]
  int32_t *err;
  // bf16 gate/up only: when set, the routed rows are gathered from x [T, d] by
  // row_to_token (gather_rows [N]) instead of read from x_perm
  const int32_t *gather_rows = nullptr;
  const void *gather_x = nullptr;
  int64_t gather_T = 0;
  // bf16 down only: when c_out is set, the combine runs in the down epilogue:
  // c_out [c_T, d] = sum_j topk_w[t, j] y[slot_to_row[t, j]] (+ y[N + t]); c_counts
  // [c_T, d / 128] is scratch
  const int32_t *c_row_to_token = nullptr;
  const int32_t *c_slot_to_row = nullptr;
  const float *c_topk_w = nullptr;
  int32_t *c_counts = nullptr;
  void *c_out = nullptr;
  int64_t c_T = 0;
  int32_t c_k = 0;
};

// Largest p in [0, P) with offs[p] <= row (callers guarantee row < offs[P]).
__device__ __forceinline__ int group_of_row(const int32_t *offs, int P, int row) {
  int lo = 0, hi = P - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// The two phases of the expert FFN: h = silu(x W_gate) * (x W_up), then y = h W_down.
moe_status_t gate_up_f32(const FfnArgs &a, cudaStream_t st);
moe_status_t down_f32(const FfnArgs &a, cudaStream_t st);
moe_status_t gate_up_bf16(const FfnArgs &a, cudaStream_t st);
moe_status_t down_bf16(const FfnArgs &a, cudaStream_t st);
moe_status_t gate_up_bf16_pair(const FfnArgs &a, cudaStream_t st);
moe_status_t down_bf16_pair(const FfnArgs &a, cudaStream_t st);
moe_status_t gate_up_e4m3(const FfnArgs &a, cudaStream_t st);
moe_status_t down_e4m3(const FfnArgs &a, cudaStream_t st);
moe_status_t gate_up_e4m3_pair(const FfnArgs &a, cudaStream_t st);
moe_status_t down_e4m3_pair(const FfnArgs &a, cudaStream_t st);

}  // namespace moe
