// Expert FFN in fp32 on the CUDA cores, for fp32 workloads whose tolerance
// (1e-5 relative) rules out TF32 tensor cores.  ("6.4 Data parallelism and expert
// parallelism", section 2.1: one expert is the three matrices gate, up, down.)
//
// Two launches: h[row, i] = silu(x W_gate)_i * (x W_up)_i with one thread per
// (row, i), then y[row, c] = (h W_down)_c with one thread per (row, c).  Each
// row finds its physical expert by binary search over the expert offsets; rows at
// and after N belong to the shared expert (weight set E_w - 1, input shared_x).
#include "common.cuh"
#include "ffn.cuh"

namespace moe {
namespace {

struct SimtArgs {
  const float *x_perm;
  const float *shared_x;
  const int32_t *offs;
  const int32_t *p2l;
  int P;
  int64_t N, rows, d, I, E_w;
  const float *w13;
  const float *w2;
  float *h;
  float *y;
  int32_t *err;
};

__device__ __forceinline__ bool row_expert(const SimtArgs &a, int64_t row, int64_t *e, const float **xr) {
  if (row < a.N) {
    if (row >= a.offs[a.P]) return false;
    const int p = group_of_row(a.offs, a.P, (int)row);
    *e = a.p2l ? a.p2l[p] : p;
    if (*e < 0 || *e >= a.E_w) {
      raise_dev(a.err, MOE_DEV_LAYOUT);
      return false;
    }
    if (xr) *xr = a.x_perm + row * a.d;
  } else {
    *e = a.E_w - 1;
    if (xr) *xr = a.shared_x + (row - a.N) * a.d;
  }
  return true;
}

__global__ void __launch_bounds__(256) gateup_f32_kernel(SimtArgs a) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.rows * a.I) return;
  const int64_t row = idx / a.I, i = idx % a.I;
  int64_t e;
  const float *xr;
  if (!row_expert(a, row, &e, &xr)) return;
  const float *wg = a.w13 + (e * 2 * a.I + i) * a.d;
  const float *wu = wg + a.I * a.d;
  float g = 0.f, u = 0.f;
  for (int64_t c = 0; c < a.d; ++c) {
    const float xv = xr[c];
    g = fmaf(xv, __ldg(wg + c), g);
    u = fmaf(xv, __ldg(wu + c), u);
  }
  a.h[row * a.I + i] = silu(g) * u;
}

__global__ void __launch_bounds__(256) down_f32_kernel(SimtArgs a) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.rows * a.d) return;
  const int64_t row = idx / a.d, c = idx % a.d;
  int64_t e;
  if (!row_expert(a, row, &e, nullptr)) return;
  const float *hr = a.h + row * a.I;
  const float *wd = a.w2 + (e * a.d + c) * a.I;
  float acc = 0.f;
  for (int64_t i = 0; i < a.I; ++i) acc = fmaf(hr[i], __ldg(wd + i), acc);
  a.y[row * a.d + c] = acc;
}

}  // namespace

static SimtArgs simt_args(const FfnArgs &f) {
  SimtArgs a;
  a.x_perm = static_cast<const float *>(f.x_perm);
  a.shared_x = static_cast<const float *>(f.shared_x);
  a.offs = f.offs;
  a.p2l = f.p2l;
  a.P = (int)f.P;
  a.N = f.N;
  a.rows = f.N + f.T_shared;
  a.d = f.w->d;
  a.I = f.w->I;
  a.E_w = f.w->E_w;
  a.w13 = static_cast<const float *>(f.w->w13);
  a.w2 = static_cast<const float *>(f.w->w2);
  a.h = static_cast<float *>(f.h);
  a.y = static_cast<float *>(f.y);
  a.err = f.err;
  return a;
}

moe_status_t gate_up_f32(const FfnArgs &f, cudaStream_t st) {
  const SimtArgs a = simt_args(f);
  if (a.rows == 0) return MOE_OK;
  const int64_t n = a.rows * a.I;
  gateup_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return launch_status();
}

moe_status_t down_f32(const FfnArgs &f, cudaStream_t st) {
  const SimtArgs a = simt_args(f);
  if (a.rows == 0) return MOE_OK;
  const int64_t n = a.rows * a.d;
  down_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return launch_status();
}

}  // namespace moe
