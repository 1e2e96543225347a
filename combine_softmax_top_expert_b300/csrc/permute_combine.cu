// Dispatch copy and combine ("6.4 Data parallelism and expert parallelism",
// section 3.1 steps 2 and 4; section 3.2: FP8 dispatch, BF16 combine).
//
// Both kernels are token-centric so that every token row is read from HBM once:
//   permute  reads x[t] once and writes it to its k rows x_perm[slot_to_row[t, j]]
//            (the e4m3 variant quantises the row once per 128-channel group first);
//   combine  reads the k rows y_perm[slot_to_row[t, j]] (+ the shared expert's row)
//            and writes out[t] once, accumulating in fp32 in j order.
// Loads and stores are 16 bytes wide (8 bf16 or 4 fp32 per access).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kTok = 128;  // threads per token block
constexpr int kMaxK = 32;

__global__ void __launch_bounds__(kTok) permute_copy_kernel(const uint4 *__restrict__ x, int64_t T, int64_t vecs,
                                                             int k, const int32_t *__restrict__ slot_to_row,
                                                             uint4 *__restrict__ xp) {
  __shared__ int32_t rows[kMaxK];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) rows[threadIdx.x] = slot_to_row[t * k + threadIdx.x];
    __syncthreads();
    for (int64_t v = threadIdx.x; v < vecs; v += kTok) {
      const uint4 val = __ldg(x + t * vecs + v);
      for (int j = 0; j < k; ++j) {
        const int r = rows[j];
        if (r >= 0) xp[(int64_t)r * vecs + v] = val;
      }
    }
  }
}

// bf16 -> e4m3 per token per 128-channel group: 16 threads x 8 channels per group.
__global__ void __launch_bounds__(kTok) permute_e4m3_kernel(const uint4 *__restrict__ x, int64_t T, int64_t d,
                                                             int k, const int32_t *__restrict__ slot_to_row,
                                                             uint2 *__restrict__ xq, float *__restrict__ scales) {
  __shared__ int32_t rows[kMaxK];
  const int64_t vecs = d / 8, groups = d / 128;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) rows[threadIdx.x] = slot_to_row[t * k + threadIdx.x];
    __syncthreads();
    // Every lane runs every step so the 16-lane shuffles see full groups; a
    // group is either wholly inside [0, vecs) or wholly outside (vecs % 16 == 0).
    for (int64_t v0 = 0; v0 < vecs; v0 += kTok) {
      const int64_t v = v0 + threadIdx.x;
      const bool active = v < vecs;
      const uint4 raw = active ? __ldg(x + t * vecs + v) : make_uint4(0u, 0u, 0u, 0u);
      float f[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                    bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      uint2 q;
      q.x = e4m3x2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale)) |
            (e4m3x2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale)) << 16);
      q.y = e4m3x2(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale)) |
            (e4m3x2(__fdiv_rn(f[6], scale), __fdiv_rn(f[7], scale)) << 16);
      const int64_t g = v / 16;
      if (!active) continue;
      for (int j = 0; j < k; ++j) {
        const int r = rows[j];
        if (r < 0) continue;
        xq[(int64_t)r * vecs + v] = q;
        if ((v & 15) == 0) scales[(int64_t)r * groups + g] = scale;
      }
    }
  }
}

template <bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(kTok) combine_kernel(const void *__restrict__ y, const int32_t *__restrict__ s2r,
                                                        const float *__restrict__ tw, int64_t T, int k, int64_t d,
                                                        const void *__restrict__ shared_y, void *__restrict__ out) {
  __shared__ int32_t rows[kMaxK];
  __shared__ float wts[kMaxK];
  const int64_t vecs = d / 8;  // 8 values per step
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      rows[threadIdx.x] = s2r[t * k + threadIdx.x];
      wts[threadIdx.x] = tw[t * k + threadIdx.x];
    }
    __syncthreads();
    for (int64_t v = threadIdx.x; v < vecs; v += kTok) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      auto add_row = [&](const void *base, int64_t row, float w) {
        float f[8];
        if (kBf16In) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(base) + row * vecs + v);
          f[0] = bf16_lo(raw.x); f[1] = bf16_hi(raw.x); f[2] = bf16_lo(raw.y); f[3] = bf16_hi(raw.y);
          f[4] = bf16_lo(raw.z); f[5] = bf16_hi(raw.z); f[6] = bf16_lo(raw.w); f[7] = bf16_hi(raw.w);
        } else {
          const float4 *p = reinterpret_cast<const float4 *>(base) + (row * vecs + v) * 2;
          const float4 a = __ldg(p), b = __ldg(p + 1);
          f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
      };
      for (int j = 0; j < k; ++j) {
        const int r = rows[j];
        if (r >= 0) add_row(y, r, wts[j]);
      }
      if (shared_y) add_row(shared_y, t, 1.0f);
      if (kBf16Out) {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4 *>(out)[t * vecs + v] = o;
      } else {
        float4 *p = reinterpret_cast<float4 *>(out) + (t * vecs + v) * 2;
        p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
}

inline int token_grid(int64_t T) { return (int)(T < 148 * 64 ? T : 148 * 64); }

}  // namespace

moe_status_t permute(const void *x, moe_dtype_t x_dt, int64_t T, int64_t d, int32_t k, const int32_t *slot_to_row,
                     void *x_perm, moe_dtype_t perm_dt, float *perm_scales, cudaStream_t st) {
  if (T < 0 || d <= 0 || k < 1 || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !slot_to_row || !x_perm || !aligned(x, 16) || !aligned(x_perm, 16)) return MOE_ERR_INVALID_ARG;
  if (x_dt == perm_dt && (x_dt == MOE_F32 || x_dt == MOE_BF16)) {
    const int64_t bytes = d * (x_dt == MOE_F32 ? 4 : 2);
    if (bytes % 16) return MOE_ERR_INVALID_ARG;
    permute_copy_kernel<<<token_grid(T), kTok, 0, st>>>(static_cast<const uint4 *>(x), T, bytes / 16, k,
                                                         slot_to_row, static_cast<uint4 *>(x_perm));
    return launch_status();
  }
  if (x_dt == MOE_BF16 && perm_dt == MOE_E4M3) {
    if (d % 128 || !perm_scales) return MOE_ERR_INVALID_ARG;
    permute_e4m3_kernel<<<token_grid(T), kTok, 0, st>>>(static_cast<const uint4 *>(x), T, d, k, slot_to_row,
                                                         static_cast<uint2 *>(x_perm), perm_scales);
    return launch_status();
  }
  return MOE_ERR_UNSUPPORTED;
}

moe_status_t combine(const void *y, moe_dtype_t y_dt, const int32_t *s2r, const float *tw, int64_t T, int32_t k,
                     int64_t d, const void *shared_y, void *out, moe_dtype_t out_dt, cudaStream_t st) {
  if (T < 0 || d <= 0 || d % 8 || k < 1 || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !s2r || !tw || !out || !aligned(y, 16) || !aligned(out, 16) || (shared_y && !aligned(shared_y, 16)))
    return MOE_ERR_INVALID_ARG;
  const int g = token_grid(T);
  if (y_dt == MOE_BF16 && out_dt == MOE_BF16)
    combine_kernel<true, true><<<g, kTok, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_BF16 && out_dt == MOE_F32)
    combine_kernel<true, false><<<g, kTok, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_F32 && out_dt == MOE_F32)
    combine_kernel<false, false><<<g, kTok, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_F32 && out_dt == MOE_BF16)
    combine_kernel<false, true><<<g, kTok, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else
    return MOE_ERR_UNSUPPORTED;
  return launch_status();
}

}  // namespace moe

MOE_API moe_status_t moe_permute(const void *x, moe_dtype_t x_dt, int64_t T, int64_t d, int32_t k,
                                 const int32_t *slot_to_row, void *x_perm, moe_dtype_t perm_dt, float *perm_scales,
                                 moe_stream_t stream) {
  return moe::permute(x, x_dt, T, d, k, slot_to_row, x_perm, perm_dt, perm_scales, moe::as_cuda(stream));
}

MOE_API moe_status_t moe_combine(const void *y_perm, moe_dtype_t y_dt, const int32_t *slot_to_row,
                                 const float *topk_w, int64_t T, int32_t k, int64_t d, const void *shared_y,
                                 void *out, moe_dtype_t out_dt, moe_stream_t stream) {
  return moe::combine(y_perm, y_dt, slot_to_row, topk_w, T, k, d, shared_y, out, out_dt, moe::as_cuda(stream));
}
