// Dispatch copy and combine ("6.4 Data parallelism and expert parallelism",
// section 3.1 steps 2 and 4; section 3.2: FP8 dispatch, BF16 combine).
//
// Both are token-centric so that every token row is read from HBM once:
//   permute  reads x[t] once and writes it to its k rows x_perm[slot_to_row[t, j]]
//            (the e4m3 variant quantises the row once per 128-channel group first);
//   combine  reads the k rows y_perm[slot_to_row[t, j]] (+ the shared expert's row)
//            and writes out[t] once, accumulating in fp32 in j order.
// A unit of work is one chunk of at most 256 16-byte vectors of one token row (the
// block's threads; the host sizes blocks so a row's chunks are equal, e.g. four
// 224-vector chunks for d = 7168 rather than three of 256 and a half-empty one),
// so even a decode batch of 128 tokens spreads over hundreds of blocks; the token's k rows are
// staged in shared memory and combine keeps eight row loads in flight per thread.
// Accesses are 16 bytes wide.
//
// FP8 dispatch for bf16 experts (section 3.2: tokens travel in FP8, experts and
// the combine stay in BF16) is the e4m3 permute followed by the receive side,
// dequant_e4m3_kernel: codes and their group scales back to bf16 rows.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kTok = 256;      // most threads per block = 16-byte vectors per chunk
constexpr int kMaxK = 32;
constexpr int kRowsAhead = 8;  // combine: row loads in flight per thread

// The token's k destination rows (and weights), staged once per work item.
__device__ __forceinline__ void stage_rows(const int32_t *s2r, const float *tw, int64_t t, int k, int32_t *rows,
                                           float *wts) {
  __syncthreads();
  if (threadIdx.x < k) {
    rows[threadIdx.x] = __ldg(s2r + t * k + threadIdx.x);
    if (wts) wts[threadIdx.x] = __ldg(tw + t * k + threadIdx.x);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTok) permute_copy_kernel(const uint4 *__restrict__ x, int64_t T, int64_t vecs,
                                                             int k, const int32_t *__restrict__ slot_to_row,
                                                             uint4 *__restrict__ xp) {
  __shared__ int32_t rows[kMaxK];
  const int64_t chunks = (vecs + blockDim.x - 1) / blockDim.x;
  for (int64_t w = blockIdx.x; w < T * chunks; w += gridDim.x) {
    const int64_t t = w / chunks, v = (w % chunks) * blockDim.x + threadIdx.x;
    stage_rows(slot_to_row, nullptr, t, k, rows, nullptr);
    if (v >= vecs) continue;
    const uint4 val = __ldg(x + t * vecs + v);
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) xp[(int64_t)r * vecs + v] = val;
    }
  }
}

// bf16 -> e4m3 per token per 128-channel group: 16 threads x 8 channels per group.
// Each thread reads the token's destination rows itself rather than through the
// shared-memory staging of the other kernels: with the divisions to overlap, that
// measured faster here (114.7 against 120.8 us on 8192 x 7168 tokens, top-8), and
// slower in the copy and the combine.
// Chunks are 256 vectors = 16 whole groups; every lane runs so the 16-lane
// shuffles see full groups (a group lies wholly inside or outside the row).
__global__ void __launch_bounds__(kTok) permute_e4m3_kernel(const uint4 *__restrict__ x, int64_t T, int64_t d,
                                                             int k, const int32_t *__restrict__ slot_to_row,
                                                             uint2 *__restrict__ xq, float *__restrict__ scales) {
  const int64_t vecs = d / 8, groups = d / 128;
  const int64_t chunks = (vecs + blockDim.x - 1) / blockDim.x;
  for (int64_t w = blockIdx.x; w < T * chunks; w += gridDim.x) {
    const int64_t t = w / chunks, v = (w % chunks) * blockDim.x + threadIdx.x;
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
    if (!active) continue;
    const int64_t g = v / 16;
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(slot_to_row + t * k + j);  // the same address in every thread: one cached line
      if (r < 0) continue;
      xq[(int64_t)r * vecs + v] = q;
      if ((v & 15) == 0) scales[(int64_t)r * groups + g] = scale;
    }
  }
}

// 8 consecutive values of row `row` (bf16 or fp32 storage) as floats.
template <bool kBf16>
__device__ __forceinline__ void load8(const void *base, int64_t row, int64_t vecs, int64_t v, float (&f)[8]) {
  if (kBf16) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(base) + row * vecs + v);
    f[0] = bf16_lo(raw.x); f[1] = bf16_hi(raw.x); f[2] = bf16_lo(raw.y); f[3] = bf16_hi(raw.y);
    f[4] = bf16_lo(raw.z); f[5] = bf16_hi(raw.z); f[6] = bf16_lo(raw.w); f[7] = bf16_hi(raw.w);
  } else {
    const float4 *p = reinterpret_cast<const float4 *>(base) + (row * vecs + v) * 2;
    const float4 a = __ldg(p), b = __ldg(p + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

template <bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(kTok) combine_kernel(const void *__restrict__ y, const int32_t *__restrict__ s2r,
                                                        const float *__restrict__ tw, int64_t T, int k, int64_t d,
                                                        const void *__restrict__ shared_y, void *__restrict__ out) {
  __shared__ int32_t rows[kMaxK];
  __shared__ float wts[kMaxK];
  const int64_t vecs = d / 8;  // 8 values per vector
  const int64_t chunks = (vecs + blockDim.x - 1) / blockDim.x;
  for (int64_t w = blockIdx.x; w < T * chunks; w += gridDim.x) {
    const int64_t t = w / chunks, v = (w % chunks) * blockDim.x + threadIdx.x;
    stage_rows(s2r, tw, t, k, rows, wts);
    if (v >= vecs) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += kRowsAhead) {
      // all of the group's row loads go out before any is used
      uint4 raw[kRowsAhead][kBf16In ? 1 : 2];
#pragma unroll
      for (int jj = 0; jj < kRowsAhead; ++jj) {
        const int r = j0 + jj < k ? rows[j0 + jj] : -1;
        if (r < 0) continue;
        if (kBf16In) {
          raw[jj][0] = __ldg(reinterpret_cast<const uint4 *>(y) + (int64_t)r * vecs + v);
        } else {
          const uint4 *p = reinterpret_cast<const uint4 *>(y) + ((int64_t)r * vecs + v) * 2;
          raw[jj][0] = __ldg(p);
          raw[jj][kBf16In ? 0 : 1] = __ldg(p + 1);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kRowsAhead; ++jj) {  // j order, as the definition reads
        if (j0 + jj >= k || rows[j0 + jj] < 0) continue;
        const float wt = wts[j0 + jj];
        float f[8];
        if (kBf16In) {
          const uint4 q = raw[jj][0];
          f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x); f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
          f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z); f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
        } else {
          const uint4 a = raw[jj][0], b = raw[jj][kBf16In ? 0 : 1];
          f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y); f[2] = __uint_as_float(a.z);
          f[3] = __uint_as_float(a.w); f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
          f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt, f[i], acc[i]);
      }
    }
    if (shared_y) {
      float f[8];
      load8<kBf16In>(shared_y, t, vecs, v, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(1.0f, f[i], acc[i]);
    }
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

// Two OCP e4m3 codes (bits 0-7 and 8-15) -> f16x2 by the hardware conversion (exact:
// every e4m3 value is an f16 value), then each times the scale as one IEEE fp32
// multiply, rounded to bf16 to nearest even.
__device__ __forceinline__ uint32_t dequant2(uint32_t codes, float s) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
  const float lo = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 >> 16)));
  return pack_bf16x2(__fmul_rn(lo, s), __fmul_rn(hi, s));
}

// Receive side of the FP8 dispatch: out = bf16_rn(code * scale), the product an
// IEEE fp32 multiply.  Item i is 8 codes (an 8-byte load, a 16-byte store, so a
// warp's accesses are contiguous); codes [rows, d] and scales [rows, d/128] are
// both dense, so item i's scale is scales[i / 16] with no row arithmetic.  Loads
// are a third of the traffic here, so each thread keeps four items' loads in
// flight before it converts and stores them.
__device__ __forceinline__ uint4 dequant8(uint2 c, float s) {
  return make_uint4(dequant2(c.x, s), dequant2(c.x >> 16, s), dequant2(c.y, s), dequant2(c.y >> 16, s));
}

constexpr int kDequantUnroll = 4;

__global__ void __launch_bounds__(kTok) dequant_e4m3_kernel(const uint2 *__restrict__ q,
                                                             const float *__restrict__ scales, int64_t items,
                                                             uint4 *__restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * kTok;
  int64_t i = (int64_t)blockIdx.x * kTok + threadIdx.x;
  for (; i + (kDequantUnroll - 1) * stride < items; i += kDequantUnroll * stride) {
    uint2 c[kDequantUnroll];
    float s[kDequantUnroll];
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u) {
      c[u] = __ldg(q + i + u * stride);
      s[u] = __ldg(scales + ((i + u * stride) >> 4));
    }
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u) out[i + u * stride] = dequant8(c[u], s[u]);
  }
  for (; i < items; i += stride) out[i] = dequant8(__ldg(q + i), __ldg(scales + (i >> 4)));
}

// One block per (token, chunk) work item: blocks that finish make room for new
// ones, so no block waits on another item's stragglers.  (The loops stride only
// past the grid-size limit.)
// Threads per block for rows of `vecs` 16-byte vectors: split the row into the
// fewest chunks of at most kTok vectors, each as even as whole warps allow.  A
// multiple of 32, so 16-lane groups never straddle a chunk.
inline int chunk_threads(int64_t vecs) {
  const int64_t chunks = (vecs + kTok - 1) / kTok;
  const int64_t per = (vecs + chunks - 1) / chunks;
  return (int)((per + 31) / 32 * 32);
}

inline int work_grid(int64_t T, int64_t vecs) {
  const int nt = chunk_threads(vecs);
  const int64_t items = T * ((vecs + nt - 1) / nt);
  return (int)(items < INT32_MAX ? items : INT32_MAX);
}

}  // namespace

moe_status_t permute(const void *x, moe_dtype_t x_dt, int64_t T, int64_t d, int32_t k, const int32_t *slot_to_row,
                     void *x_perm, moe_dtype_t perm_dt, float *perm_scales, cudaStream_t st) {
  if (T < 0 || d <= 0 || k < 1 || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !slot_to_row || !x_perm || !aligned(x, 16) || !aligned(x_perm, 16)) return MOE_ERR_INVALID_ARG;
  if (x_dt == perm_dt && (x_dt == MOE_F32 || x_dt == MOE_BF16)) {
    const int64_t bytes = d * (x_dt == MOE_F32 ? 4 : 2);
    if (bytes % 16) return MOE_ERR_INVALID_ARG;
    permute_copy_kernel<<<work_grid(T, bytes / 16), chunk_threads(bytes / 16), 0, st>>>(static_cast<const uint4 *>(x), T, bytes / 16, k,
                                                                    slot_to_row, static_cast<uint4 *>(x_perm));
    return launch_status();
  }
  if (x_dt == MOE_BF16 && perm_dt == MOE_E4M3) {
    if (d % 128 || !perm_scales) return MOE_ERR_INVALID_ARG;
    permute_e4m3_kernel<<<work_grid(T, d / 8), chunk_threads(d / 8), 0, st>>>(static_cast<const uint4 *>(x), T, d, k, slot_to_row,
                                                               static_cast<uint2 *>(x_perm), perm_scales);
    return launch_status();
  }
  return MOE_ERR_UNSUPPORTED;
}

moe_status_t dequantize_e4m3(const void *codes, const float *scales, int64_t rows, int64_t d, void *out,
                             cudaStream_t st) {
  if (rows < 0 || d <= 0 || d % 128) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!codes || !scales || !out || !aligned(codes, 16) || !aligned(out, 16) || !aligned(scales, 4))
    return MOE_ERR_INVALID_ARG;
  const int64_t items = rows * (d / 8);
  const int64_t blocks = (items + kTok - 1) / kTok;
  const int grid = (int)(blocks < 148 * 8 ? blocks : 148 * 8);  // 8 resident blocks per SM, grid-stride past that
  dequant_e4m3_kernel<<<grid, kTok, 0, st>>>(static_cast<const uint2 *>(codes), scales, items,
                                             static_cast<uint4 *>(out));
  return launch_status();
}

moe_status_t combine(const void *y, moe_dtype_t y_dt, const int32_t *s2r, const float *tw, int64_t T, int32_t k,
                     int64_t d, const void *shared_y, void *out, moe_dtype_t out_dt, cudaStream_t st) {
  if (T < 0 || d <= 0 || d % 8 || k < 1 || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !s2r || !tw || !out || !aligned(y, 16) || !aligned(out, 16) || (shared_y && !aligned(shared_y, 16)))
    return MOE_ERR_INVALID_ARG;
  const int g = work_grid(T, d / 8), nt = chunk_threads(d / 8);
  if (y_dt == MOE_BF16 && out_dt == MOE_BF16)
    combine_kernel<true, true><<<g, nt, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_BF16 && out_dt == MOE_F32)
    combine_kernel<true, false><<<g, nt, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_F32 && out_dt == MOE_F32)
    combine_kernel<false, false><<<g, nt, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
  else if (y_dt == MOE_F32 && out_dt == MOE_BF16)
    combine_kernel<false, true><<<g, nt, 0, st>>>(y, s2r, tw, T, k, d, shared_y, out);
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

MOE_API moe_status_t moe_dequantize_e4m3(const void *codes, const float *scales, int64_t rows, int64_t d, void *out,
                                         moe_stream_t stream) {
  return moe::dequantize_e4m3(codes, scales, rows, d, out, moe::as_cuda(stream));
}

MOE_API moe_status_t moe_combine(const void *y_perm, moe_dtype_t y_dt, const int32_t *slot_to_row,
                                 const float *topk_w, int64_t T, int32_t k, int64_t d, const void *shared_y,
                                 void *out, moe_dtype_t out_dt, moe_stream_t stream) {
  return moe::combine(y_perm, y_dt, slot_to_row, topk_w, T, k, d, shared_y, out, out_dt, moe::as_cuda(stream));
}
