// Grouped SwiGLU expert FFN on the tcgen05 tensor cores ("6.4 Data parallelism
// and expert parallelism", section 2.1: gate, up, down; section 7: the shared
// expert is one more always-on group).
//
// Two launches per forward, each a persistent grouped GEMM over all experts:
//   gate/up   h = silu(X W_gate) * (X W_up)   (SwiGLU fused in the epilogue, bf16 h)
//   down      y = h W_down                    (bf16 y)
// One CTA per SM, 6 warps: warp 0 issues TMA loads into a ring of shared-memory
// stages, warp 1 issues tcgen05.mma into a double-buffered TMEM accumulator,
// warps 2-5 drain the accumulator (tcgen05.ld), apply the epilogue and store.
// Tiles are enumerated per group (physical expert, then the shared expert) from
// the expert offsets on the device, so nothing returns to the host.
//
// Tile orientations (both K-major operands, 128-byte swizzled, K blocks of 64):
//   wide  A = 128 token rows, B = weight rows (gate 128 + up 128, or 256 of
//         W_down): one 128x256xK tile per feature block.  For many rows per expert.
//   swap  A = 128 weight rows (gate and up as two MMAs), B = up to 32 token rows:
//         D is features x tokens, so a group of a few tokens streams its weights
//         at HBM speed without padding tokens to 128.  For decode-sized batches.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "ffn.cuh"
#include "tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kThreads = 192;
constexpr int kMaxGroups = 2048 + 1;

template <bool kGated, bool kSwap, int kBW>
struct Cfg {
  static constexpr int kABytes = 128 * 128 * ((kSwap && kGated) ? 2 : 1);
  static constexpr int kBRows = kSwap ? 32 : (kGated ? 256 : kBW);
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kStages = kSwap ? (kGated ? 5 : 8) : 4;
  static constexpr int kAccCols = kSwap ? (kGated ? 64 : 32) : (kGated ? 256 : kBW);
  static constexpr int kTmemCols = kSwap ? (kGated ? 128 : 64) : (2 * kAccCols >= 512 ? 512 : 256);
  static constexpr int kTokTile = kSwap ? 32 : 128;
  static constexpr int kFeatTile = kSwap ? 128 : (kGated ? 128 : kBW);
  static constexpr int kBars = 2 * kStages + 5;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kBars * 8 + 16 + (kMaxGroups + 1) * 4;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct GemmParams {
  const int32_t *offs;  // [P + 1]
  const int32_t *p2l;   // [P] or null
  int P, N, T_shared, E_w;
  int feat;             // output features: I (gate/up) or d (down)
  int K;                // reduction length: d (gate/up) or I (down)
  int w_rows;           // weight rows per expert: 2I (gate/up) or d (down)
  int shared_row0;      // row of the shared group's first token in its token map
  uint16_t *out;        // h [rows, I] or y [rows, d], bf16
  int64_t ld;
  int32_t *err;
};

struct Tile {
  int e, tok_row, out_row, valid, nt;
  bool shared;
};

__device__ __forceinline__ void group_span(const GemmParams &p, int g, int *r0, int *n) {
  if (g < p.P) {
    const int a = min(max(p.offs[g], 0), p.N);
    const int b = min(max(p.offs[g + 1], 0), p.N);
    *r0 = a;
    *n = max(b - a, 0);
  } else {
    *r0 = 0;
    *n = p.T_shared;
  }
}

// In-place inclusive scan of a[0..n) by the whole block.
__device__ void block_scan(int *a, int n) {
  __shared__ int wsum[kThreads / 32];
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += a[i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  int off = v - s;
  for (int w = 0; w < warp; ++w) off += wsum[w];
  for (int i = lo; i < hi; ++i) {
    off += a[i];
    a[i] = off;
  }
  __syncthreads();
}

template <class C>
__device__ __forceinline__ Tile decode(const GemmParams &p, const int *tile_start, int G, int NT, int tile) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo, local = tile - tile_start[g];
  int r0, n;
  group_span(p, g, &r0, &n);
  const int MT = (n + C::kTokTile - 1) / C::kTokTile;
  int mt, nt;
  if (C::kTokTile == 32) {  // swap: token tiles of one feature block run back to back
    nt = local / MT;
    mt = local % MT;
  } else {                  // wide: feature blocks of one token tile run back to back
    mt = local / NT;
    nt = local % NT;
  }
  Tile t;
  t.shared = g >= p.P;
  int e = t.shared ? p.E_w - 1 : (p.p2l ? p.p2l[g] : g);
  if (e < 0 || e >= p.E_w) e = -1;
  t.e = e;
  t.nt = nt;
  t.valid = min(C::kTokTile, n - mt * C::kTokTile);
  t.tok_row = (t.shared ? p.shared_row0 : r0) + mt * C::kTokTile;
  t.out_row = (t.shared ? p.N : r0) + mt * C::kTokTile;
  return t;
}

template <bool kGated, bool kSwap, int kBW>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16(const GemmParams p, const __grid_constant__ CUtensorMap tm_tok,
                      const __grid_constant__ CUtensorMap tm_sh, const __grid_constant__ CUtensorMap tm_w) {
  using C = Cfg<kGated, kSwap, kBW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)C::kStages * C::kStage);
  int *misc = reinterpret_cast<int *>(bars + C::kBars);  // [0] TMEM base, [1] abort flag
  int *tile_start = misc + 4;
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[C::kStages + s]); };
  auto tfull = [&](int b) { return smem_u32(&bars[2 * C::kStages + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[2 * C::kStages + 2 + b]); };
  const uint32_t drain = smem_u32(&bars[2 * C::kStages + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.P + (p.T_shared > 0 ? 1 : 0);
  const int NT = p.feat / C::kFeatTile;
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 128);
    }
    mbar_init(drain, 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
    tma_prefetch(&tm_sh);
    tma_prefetch(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), C::kTmemCols);
    tmem_relinquish();
  }
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int r0, n;
    group_span(p, g, &r0, &n);
    tile_start[g + 1] = n > 0 ? ((n + C::kTokTile - 1) / C::kTokTile) * NT : 0;
  }
  if (threadIdx.x == 0) tile_start[0] = 0;
  __syncthreads();
  block_scan(tile_start + 1, G);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[1]);
  const int total = tile_start[G];

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode<C>(p, tile_start, G, NT, tile);
      const CUtensorMap *tmt = (kGated && t.shared) ? &tm_sh : &tm_tok;
      const int nb = kSwap ? (t.valid + 15) / 16 : 0;
      const uint32_t bytes = C::kABytes + (kSwap ? nb * 2048 : C::kBBytes);
      const int wrow = max(t.e, 0) * p.w_rows + t.nt * C::kFeatTile;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t st = stage0 + s * C::kStage, bar = full(s);
        mbar_expect_tx(bar, bytes);
        const int kx = kb * 64;
        if (kSwap) {
          tma_load_2d(st, &tm_w, bar, kx, wrow);
          if (kGated) tma_load_2d(st + 16384, &tm_w, bar, kx, wrow + p.feat);
          for (int i = 0; i < nb; ++i) tma_load_2d(st + C::kABytes + i * 2048, tmt, bar, kx, t.tok_row + 16 * i);
        } else {
          tma_load_2d(st, tmt, bar, kx, t.tok_row);
          tma_load_2d(st + C::kABytes, &tm_w, bar, kx, wrow);
          if (kGated) tma_load_2d(st + C::kABytes + 16384, &tm_w, bar, kx, wrow + p.feat);
        }
        ++issued;
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
    }
    if (*abort_flag) {  // let every copy still in flight land before the CTA exits
      for (int j = issued - 1; j >= 0 && j >= issued - C::kStages; --j)
        mbar_wait_drain(full(j % C::kStages), (uint32_t)((j / C::kStages) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    int s = 0, it = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = decode<C>(p, tile_start, G, NT, tile);
      const int b = it & 1;
      if (!mbar_wait(tempty(b), ((it >> 1) & 1) ^ 1, abort_flag, p.err)) break;
      fence_after();
      const uint32_t d = tmem + b * C::kAccCols;
      const int nb = kSwap ? (t.valid + 15) / 16 : 0;
      const uint32_t id = kSwap ? idesc(128, 16 * nb, 1) : idesc(128, C::kBRows, 1);
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(full(s), ph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t a = stage0 + s * C::kStage, bb = a + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (kb | kk) != 0;
          mma_bf16(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id, acc);
          if (kSwap && kGated) mma_bf16(d + 32, sdesc_sw128(a + 16384 + kk * 32), sdesc_sw128(bb + kk * 32), id, acc);
        }
        commit(empty(s));
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      commit(tfull(b));
    }
    if (*abort_flag) {  // no MMA may still write TMEM when it is freed
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;  // TMEM lane: token row (wide) or feature (swap)
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = decode<C>(p, tile_start, G, NT, tile);
      const int b = it & 1;
      if (!mbar_wait(tfull(b), (it >> 1) & 1, abort_flag, p.err)) break;
      fence_after();
      if (t.e < 0 && r == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * C::kAccCols;
      if (!kSwap) {
        const bool ok = r < t.valid && t.e >= 0;
        uint16_t *orow = p.out + (int64_t)(t.out_row + (ok ? r : 0)) * p.ld + (int64_t)t.nt * C::kFeatTile;
        constexpr int kChunks = kGated ? 4 : kBW / 32;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          float v[32], u[32];
          tmem_ld32(tb + 32 * c, v);
          if (kGated) tmem_ld32(tb + 128 + 32 * c, u);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0 = v[2 * i], a1 = v[2 * i + 1];
            if (kGated) {
              a0 = silu(a0) * u[2 * i];
              a1 = silu(a1) * u[2 * i + 1];
            }
            pk[i] = pack_bf16x2(a0, a1);
          }
          if (ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
        float v[32], u[32];
        tmem_ld32(tb, v);
        if (kGated) tmem_ld32(tb + 32, u);
        tmem_wait_ld();
        if (t.e >= 0) {
          uint16_t *col = p.out + (int64_t)t.out_row * p.ld + (int64_t)t.nt * 128 + r;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < t.valid) {
              const float a = kGated ? silu(v[c]) * u[c] : v[c];
              col[(int64_t)c * p.ld] = (uint16_t)f2bf(a);
            }
          }
        }
      }
      fence_before();
      mbar_arrive(tempty(b));
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 2-D map over a row-major [rows, cols] matrix of `esize`-byte elements; boxes of
// box_rows x (128 / esize) elements, 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, int esize, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || rows == 0 || !aligned(base, 16) || (cols * esize) % 16) return false;
  const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esize), box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 0;
  return n;
}

template <bool kGated, bool kSwap, int kBW>
moe_status_t launch(const GemmParams &p, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c,
                    cudaStream_t st) {
  using Cf = Cfg<kGated, kSwap, kBW>;
  auto k = grouped_gemm_bf16<kGated, kSwap, kBW>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::kSmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = sm_count();
  if (grid <= 0) return MOE_ERR_CUDA;
  k<<<grid, kThreads, Cf::kSmem, st>>>(p, a, b, c);
  return launch_status();
}

// Tile orientation: "swap" for few rows per expert, "wide" otherwise; the
// environment variable MOE_B300_FFN_TILES=swap|wide overrides the choice.
bool use_swap(int64_t N, int64_t P) {
  const char *env = std::getenv("MOE_B300_FFN_TILES");
  if (env && !std::strcmp(env, "swap")) return true;
  if (env && !std::strcmp(env, "wide")) return false;
  return N < 64 * P;
}

// Maps and parameters shared by both phases.
struct Plan {
  GemmParams p;
  bool swap;
  int kbw;
  uint32_t tok_box;
};

moe_status_t plan_bf16(const FfnArgs &f, Plan *pl) {
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I;
  if (d % 128 || I % 128 || f.P > 2048) return MOE_ERR_UNSUPPORTED;
  if (w.E_w * 2 * I > INT32_MAX || w.E_w * d > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  pl->swap = use_swap(f.N + f.T_shared, f.P);
  pl->tok_box = pl->swap ? 16 : 128;
  pl->kbw = (d % 256 == 0) ? 256 : 128;
  GemmParams &p = pl->p;
  p = GemmParams{};
  p.offs = f.offs;
  p.p2l = f.p2l;
  p.P = (int)f.P;
  p.N = (int)f.N;
  p.T_shared = (int)f.T_shared;
  p.E_w = (int)w.E_w;
  p.err = f.err;
  return MOE_OK;
}

}  // namespace

moe_status_t gate_up_bf16(const FfnArgs &f, cudaStream_t st) {
  Plan pl;
  moe_status_t s = plan_bf16(f, &pl);
  if (s != MOE_OK) return s;
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I;
  if (f.N + f.T_shared == 0) return MOE_OK;
  CUtensorMap m_x, m_sh, m_w13;
  const void *xsrc = f.N > 0 ? f.x_perm : f.shared_x;
  const int64_t xrows = f.N > 0 ? f.N : f.T_shared;
  if (!make_map(&m_x, xsrc, xrows, d, 2, pl.tok_box)) return MOE_ERR_INVALID_ARG;
  if (f.T_shared > 0) {
    if (!make_map(&m_sh, f.shared_x, f.T_shared, d, 2, pl.tok_box)) return MOE_ERR_INVALID_ARG;
  } else {
    m_sh = m_x;
  }
  if (!make_map(&m_w13, w.w13, (uint64_t)w.E_w * 2 * I, d, 2, 128)) return MOE_ERR_INVALID_ARG;
  GemmParams p = pl.p;
  p.feat = (int)I;
  p.K = (int)d;
  p.w_rows = (int)(2 * I);
  p.shared_row0 = 0;
  p.out = static_cast<uint16_t *>(f.h);
  p.ld = I;
  return pl.swap ? launch<true, true, 128>(p, m_x, m_sh, m_w13, st) : launch<true, false, 128>(p, m_x, m_sh, m_w13, st);
}

moe_status_t down_bf16(const FfnArgs &f, cudaStream_t st) {
  Plan pl;
  moe_status_t s = plan_bf16(f, &pl);
  if (s != MOE_OK) return s;
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I, rows = f.N + f.T_shared;
  if (rows == 0) return MOE_OK;
  CUtensorMap m_h, m_w2;
  if (!make_map(&m_h, f.h, rows, I, 2, pl.tok_box)) return MOE_ERR_INVALID_ARG;
  if (!make_map(&m_w2, w.w2, (uint64_t)w.E_w * d, I, 2, pl.swap ? 128 : pl.kbw)) return MOE_ERR_INVALID_ARG;
  GemmParams p = pl.p;
  p.feat = (int)d;
  p.K = (int)I;
  p.w_rows = (int)d;
  p.shared_row0 = (int)f.N;
  p.out = static_cast<uint16_t *>(f.y);
  p.ld = d;
  if (pl.swap) return launch<false, true, 128>(p, m_h, m_h, m_w2, st);
  return pl.kbw == 256 ? launch<false, false, 256>(p, m_h, m_h, m_w2, st) : launch<false, false, 128>(p, m_h, m_h, m_w2, st);
}

moe_status_t gate_up_e4m3(const FfnArgs &, cudaStream_t) { return MOE_ERR_UNSUPPORTED; }
moe_status_t down_e4m3(const FfnArgs &, cudaStream_t) { return MOE_ERR_UNSUPPORTED; }


}  // namespace moe
