// One-time weight packing: the logical per-expert matrices W_gate, W_up [d, I]
// and W_down [I, d] become the K-major layouts the kernels stream,
//   w13 [2I, d] = [W_gate^T ; W_up^T]   and   w2 [d, I] = W_down^T,
// optionally quantised to e4m3 per 128x128 block of the logical matrix with
// scale = amax / 448 (fp32) and code = e4m3(w / scale), round to nearest even,
// saturating.  Not part of the timed forward.
#include "common.cuh"

namespace moe {
namespace {

template <typename S>
__device__ __forceinline__ float load_f(const S *p);
template <>
__device__ __forceinline__ float load_f<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f<uint16_t>(const uint16_t *p) {
  return __uint_as_float((uint32_t)__ldg(p) << 16);
}

// scale[cb][rb] for the 128x128 block (rb, cb) of src [R, C] (stored transposed
// to match the transposed weight layout).
template <typename S>
__global__ void __launch_bounds__(256) block_scale_kernel(const S *__restrict__ src, int64_t R, int64_t C,
                                                          float *__restrict__ scale) {
  const int64_t rb = blockIdx.y, cb = blockIdx.x;
  float amax = 0.f;
  for (int i = threadIdx.x; i < 128 * 128; i += 256) {
    const int64_t r = rb * 128 + i / 128, c = cb * 128 + i % 128;
    amax = fmaxf(amax, fabsf(load_f(src + r * C + c)));
  }
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < 8; ++w) m = fmaxf(m, red[w]);
    scale[cb * (R / 128) + rb] = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
  }
}

// Element offset of (row, k) in the tiled layout of a K-major matrix whose rows
// are K elements of E bytes.  Rows go in groups of 128; group g of this matrix
// fills rows half*128 .. half*128+127 of the tile_rows-row blocks of tile g (so
// two matrices can share blocks, W_gate^T in the first half and W_up^T in the
// second).  Blocks hold 128 bytes of every row, are ordered tile major then K
// block, keep rows 128 bytes apart, and store the 16-byte chunk j of block row r
// at chunk j ^ (r % 8) (the 128-byte swizzle of the tensor-core operand tiles).
template <int E>
__device__ __forceinline__ int64_t tiled_offset(int64_t row, int64_t k, int64_t K, int tile_rows, int half) {
  const int64_t byte = k * E, kb = byte / 128, within = byte % 128;
  const int64_t r = half * 128 + row % 128, chunk = (within / 16) ^ (r % 8);
  const int64_t off = (((row / 128) * (K * E / 128) + kb) * tile_rows + r) * 128 + chunk * 16 + within % 16;
  return off / E;
}

// dst[c][r] = src[r][c], 32x32 tiles through shared memory.  D is float (plain
// K-major rows), uint16_t (bf16, tiled) or uint8_t (e4m3 with the block scales,
// tiled).
template <typename S, typename D>
__global__ void __launch_bounds__(256) transpose_kernel(const S *__restrict__ src, int64_t R, int64_t C,
                                                        D *__restrict__ dst, const float *__restrict__ scale,
                                                        int tile_rows, int half) {
  __shared__ float tile[32][33];
  const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < R && c < C) ? load_f(src + r * C + c) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (c >= C || r >= R) continue;
    const float v = tile[threadIdx.x][i];
    if constexpr (sizeof(D) == 4) {
      dst[c * R + r] = v;
    } else if constexpr (sizeof(D) == 2) {
      dst[tiled_offset<2>(c, r, R, tile_rows, half)] = (uint16_t)f2bf(v);
    } else {
      const float s = scale[(c / 128) * (R / 128) + r / 128];
      dst[tiled_offset<1>(c, r, R, tile_rows, half)] = (uint8_t)(e4m3x2(__fdiv_rn(v, s), 0.f) & 0xff);
    }
  }
}

template <typename S, typename D>
moe_status_t pack_one(const S *src, int64_t R, int64_t C, D *dst, float *scale, int tile_rows, int half,
                      cudaStream_t st) {
  if (scale) block_scale_kernel<S><<<dim3((unsigned)(C / 128), (unsigned)(R / 128)), 256, 0, st>>>(src, R, C, scale);
  transpose_kernel<S, D><<<dim3((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32)), dim3(32, 8), 0, st>>>(
      src, R, C, dst, scale, tile_rows, half);
  return launch_status();
}

// Tiled layouts: W_gate^T and W_up^T share 256-row blocks (gate rows, then up
// rows of the same 128 features), so one contiguous 32 KB copy brings both
// operand tiles of a K block; W_down^T uses 128-row blocks.
template <typename S>
moe_status_t pack_src(const S *wg, const S *wu, const S *wd, int64_t d, int64_t I, moe_dtype_t dst_dt, void *w13,
                      void *w2, float *s13, float *s2, cudaStream_t st) {
  moe_status_t s;
  if (dst_dt == MOE_E4M3) {
    uint8_t *a = static_cast<uint8_t *>(w13), *b = static_cast<uint8_t *>(w2);
    if ((s = pack_one<S, uint8_t>(wg, d, I, a, s13, 256, 0, st)) != MOE_OK) return s;
    if ((s = pack_one<S, uint8_t>(wu, d, I, a, s13 + (I / 128) * (d / 128), 256, 1, st)) != MOE_OK) return s;
    return pack_one<S, uint8_t>(wd, I, d, b, s2, 128, 0, st);
  }
  if (dst_dt == MOE_BF16) {
    if (sizeof(S) != 2) return MOE_ERR_UNSUPPORTED;
    uint16_t *a = static_cast<uint16_t *>(w13), *b = static_cast<uint16_t *>(w2);
    if ((s = pack_one<S, uint16_t>(wg, d, I, a, nullptr, 256, 0, st)) != MOE_OK) return s;
    if ((s = pack_one<S, uint16_t>(wu, d, I, a, nullptr, 256, 1, st)) != MOE_OK) return s;
    return pack_one<S, uint16_t>(wd, I, d, b, nullptr, 128, 0, st);
  }
  if (dst_dt == MOE_F32) {
    if (sizeof(S) != 4) return MOE_ERR_UNSUPPORTED;
    float *a = static_cast<float *>(w13), *b = static_cast<float *>(w2);
    if ((s = pack_one<S, float>(wg, d, I, a, nullptr, 0, 0, st)) != MOE_OK) return s;
    if ((s = pack_one<S, float>(wu, d, I, a + I * d, nullptr, 0, 0, st)) != MOE_OK) return s;
    return pack_one<S, float>(wd, I, d, b, nullptr, 0, 0, st);
  }
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace moe

MOE_API moe_status_t moe_pack_weights(const void *w_gate, const void *w_up, const void *w_down, moe_dtype_t src_dt,
                                      int64_t d, int64_t I, moe_dtype_t dst_dt, void *w13_e, void *w2_e,
                                      float *s13_e, float *s2_e, moe_stream_t stream) {
  using namespace moe;
  if (!w_gate || !w_up || !w_down || !w13_e || !w2_e || d <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (dst_dt == MOE_E4M3 && (!s13_e || !s2_e)) return MOE_ERR_INVALID_ARG;
  if (dst_dt != MOE_F32 && (d % 128 || I % 128)) return MOE_ERR_INVALID_ARG;  // whole 128-row tiles
  if (dst_dt != MOE_F32 && (!aligned(w13_e, 16) || !aligned(w2_e, 16))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_cuda(stream);
  if (src_dt == MOE_F32)
    return pack_src<float>(static_cast<const float *>(w_gate), static_cast<const float *>(w_up),
                           static_cast<const float *>(w_down), d, I, dst_dt, w13_e, w2_e, s13_e, s2_e, st);
  if (src_dt == MOE_BF16)
    return pack_src<uint16_t>(static_cast<const uint16_t *>(w_gate), static_cast<const uint16_t *>(w_up),
                              static_cast<const uint16_t *>(w_down), d, I, dst_dt, w13_e, w2_e, s13_e, s2_e, st);
  return MOE_ERR_UNSUPPORTED;
}
