// Shared helpers for the sm_103a MoE kernels and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

inline cudaStream_t as_cuda(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// The last CUDA error a call of this library saw on the calling thread.
cudaError_t &last_cuda_error();

inline moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  last_cuda_error() = e;
  return MOE_ERR_CUDA;
}

inline moe_status_t launch_status() { return cuda_status(cudaGetLastError()); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

__device__ __forceinline__ void raise_dev(int32_t *err, int bits) {
  if (err) atomicOr(err, bits);
}

// A strong (relaxed, GPU-scope) load: reads what other threads' atomics left in L2.
__device__ __forceinline__ int32_t ld_relaxed_gpu(const int32_t *p) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// float -> bf16 bits, round to nearest even (the cuda_bf16 intrinsic).
__device__ __forceinline__ uint32_t f2bf(float f) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}
// Two floats -> two bf16 (round to nearest even) in one conversion: lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> two OCP e4m3 codes (round to nearest even, saturate to +-448).
// Returns lo's code in bits 0..7 and hi's code in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// acc[i] = fma(v[i], f, acc[i]) for i < n (n even), two lanes per instruction
// (fma.rn.f32x2: each element rounded once, as fmaf).
template <int n>
__device__ __forceinline__ void fma2_scaled(float *acc, const float *v, float f) {
#pragma unroll
  for (int i = 0; i < n; i += 2)
    asm("{\n\t.reg .b64 a, x, s;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 s, {%4, %4};\n\t"
        "fma.rn.f32x2 a, x, s, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(acc[i]), "+f"(acc[i + 1])
        : "f"(v[i]), "f"(v[i + 1]), "f"(f));
}

// acc[i] = fma(acc[i], f, +0) for even n, two lanes per instruction: the first fold
// of a block sequence with the block already in acc, rounded as fma2_scaled into zeros.
template <int n>
__device__ __forceinline__ void scale2_inplace(float *acc, float f) {
#pragma unroll
  for (int i = 0; i < n; i += 2)
    asm("{\n\t.reg .b64 a, s, z;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 s, {%2, %2};\n\t"
        "mov.b64 z, 0;\n\t"
        "fma.rn.f32x2 a, a, s, z;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(acc[i]), "+f"(acc[i + 1])
        : "f"(f));
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Reciprocal by the hardware approximation (rcp.approx.ftz.f32: about 1 ulp;
// 1/inf = 0).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// silu for the e4m3 epilogue, whose result is rounded to e4m3 (3 mantissa bits):
// silu(z) = z * sigmoid(z) = z/2 + (z/2) * tanh(z/2), with the hardware tanh
// approximation (tanh.approx.f32, relative error about 2^-11) -- one special-function
// operation per value where exp + reciprocal take two.  Large |z| saturate tanh to
// +-1 and give z or 0 exactly.
__device__ __forceinline__ float silu_fast(float z) {
  const float hz = 0.5f * z;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hz));
  return fmaf(hz, t, hz);
}

}  // namespace moe
