// Grouped SwiGLU expert FFN with e4m3 operands and fp32 block scales ("6.4 Data
// parallelism and expert parallelism", section 2.1 gate/up/down; section 3.2 FP8).
//
// Weights carry one fp32 scale per 128x128 block, activations one per row per 128
// channels.  Those scales are not powers of two, so they cannot ride in the
// hardware's block-scaled MMA; instead each 128-deep K block is one group of four
// tcgen05.mma.kind::f8f6f4 (K = 32 each) into a fresh TMEM accumulator, and the
// epilogue warps fold it into fp32 registers:
//     acc += D_kb * (s_row[kb] * s_weight_block[kb]).
// Two TMEM accumulators alternate so the tensor cores work on block kb+1 while the
// epilogue folds block kb.
//
// This is the one-SM form, for few rows per expert (and MOE_B300_FFN_TILES=swap or
// wide); ffn_fp8_pair.cu holds the SM-pair form used for many.  Tiles: A = 128 token rows, B = 256 weight rows (gate 128 + up 128 of
// one 128-feature block, or 256 output features of W_down), K blocks of 128 bytes.
// 12 warps: warp 0 TMA, warp 1 MMA, warps 4-11 epilogue; epilogue warps w and w+4
// share TMEM lanes (token rows) and split the 256 columns.
//   gate/up  h = silu(g) * u for the tile's 128 features, quantised per row over
//            exactly those 128 channels (the two halves exchange their amax through
//            shared memory): scale = amax / 448, code = e4m3(h * (1 / scale)).
//   down     y = acc, stored as bf16.
#include "grouped.cuh"

namespace moe {
namespace {

using namespace tc;
using grouped::Params;
using grouped::Tile;

// Three warpgroups.  The register file is split four ways by SM sub-partition,
// so a 384-thread block gets 168 registers per thread at launch; setmaxnreg then
// moves them to where the fp32 accumulators are:
//   warpgroup 0 (TMA warp, MMA warp, two idle warps): 168 -> 56
//   warpgroups 1-2 (epilogue, 8 warps):                168 -> 224
// 128 x 56 + 256 x 224 = 64512 = 384 x 168, the registers the block launched with.
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168, kRegsIssue = 56, kRegsEpilogue = 224;
static_assert(128 * kRegsIssue + 256 * kRegsEpilogue == kThreads * kRegsLaunch, "register split");
constexpr int kStages = 4;
constexpr int kABytes = 128 * 128;
constexpr int kBBytes = 256 * 128;
constexpr int kStage = kABytes + kBBytes;
constexpr int kAccCols = 256;
constexpr int kBars = 2 * kStages + 6;
constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kBars * 8 + 16 + 2 * 256 * 4 +
                         (grouped::kMaxGroups + 1) * 4;
static_assert(kSmem <= 227 * 1024, "shared memory budget");

template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_e4m3(const Params p, const __grid_constant__ CUtensorMap tm_tok) {
  constexpr int kFeatTile = kGated ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * kStage);
  int *misc = reinterpret_cast<int *>(bars + kBars);  // [0] TMEM base, [1] abort flag
  float *amax_x = reinterpret_cast<float *>(misc + 4);  // [2 tiles][2 halves][128 rows]
  int *tile_start = reinterpret_cast<int *>(amax_x + 512);
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto dfull = [&](int b) { return smem_u32(&bars[2 * kStages + b]); };
  auto dempty = [&](int b) { return smem_u32(&bars[2 * kStages + 2 + b]); };
  const uint32_t drain = smem_u32(&bars[2 * kStages + 4]);
  const uint32_t xbar = smem_u32(&bars[2 * kStages + 5]);  // amax exchange between halves

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.P;
  const int NT = p.feat / kFeatTile;
  const int KB = p.K / 128;
  const int wblocks = p.w_rows / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(dfull(b), 1);
      mbar_init(dempty(b), 256);
    }
    mbar_init(drain, 1);
    mbar_init(xbar, 256);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  }
  grouped::build_tile_table<128>(p, tile_start, G, NT);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[1]);
  const int total = tile_start[G];

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = grouped::decode<128>(p, tile_start, G, NT, tile);
      const int e = max(t.e, 0);
      // gated: the gate+up block of this 128-feature block; down: the two tiles of
      // these 256 output features
      const int rt0 = kGated ? t.nt : 2 * t.nt;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t st = stage0 + s * kStage, bar = full(s);
        mbar_expect_tx(bar, kStage);
        tma_load_2d(st, &tm_tok, bar, kb * 128, t.tok_row);
        if (kGated) {
          bulk_load(st + kABytes, grouped::weight_block(p, e, rt0, kb, KB, grouped::kPairBytes), grouped::kPairBytes,
                    bar);
        } else {
          bulk_load(st + kABytes, grouped::weight_block(p, e, rt0, kb, KB, grouped::kTileBytes), grouped::kTileBytes,
                    bar);
          bulk_load(st + kABytes + grouped::kTileBytes, grouped::weight_block(p, e, rt0 + 1, kb, KB, grouped::kTileBytes),
                    grouped::kTileBytes, bar);
        }
        ++issued;
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j)
        mbar_wait_drain(full(j % kStages), (uint32_t)((j / kStages) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer: one accumulator per K block
    int s = 0, gk = 0;
    uint32_t ph = 0;
    const uint32_t id = idesc(128, 256, 0);
    bool ok = true;
    // the next block's barriers are tested before this block's commits (as in the
    // pair kernel), so the tests' latency hides behind them
    bool pre_full = false, pre_empty = false;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        const int b = gk & 1;
        if (!(pre_full || mbar_wait(full(s), ph, abort_flag, p.err)) ||
            !(pre_empty || mbar_wait(dempty(b), ((gk >> 1) & 1) ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t a = stage0 + s * kStage, bb = a + kABytes, d = tmem + b * kAccCols;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id, kk != 0);
        const int s1 = s + 1 == kStages ? 0 : s + 1;
        const uint32_t ph1 = s + 1 == kStages ? ph ^ 1 : ph;
        pre_full = mbar_test(full(s1), ph1);
        pre_empty = mbar_test(dempty((gk + 1) & 1), (((gk + 1) >> 1) & 1) ^ 1);
        commit(empty(s));
        commit(dfull(b));
        s = s1;
        ph = ph1;
      }
    }
    if (*abort_flag) {
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
    // ------------------------------------------------ epilogue: promotion and output
    const int q = warp & 3, half = (warp - 4) >> 2;
    const int r = q * 32 + lane;  // token row of the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    int gk = 0, it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = grouped::decode<128>(p, tile_start, G, NT, tile);
      const bool row_ok = r < t.valid && t.e >= 0;
      const int grow = t.out_row + (row_ok ? r : 0);  // also the row of the token operand's scales
      const int e = max(t.e, 0);
      // weight-scale rows: gated -> gate block nt and up block I/128 + nt; down -> 2nt + half
      const float *sw0 = p.w_scales + ((int64_t)e * wblocks + (kGated ? t.nt : 2 * t.nt + half)) * KB;
      const float *sw1 = p.w_scales + ((int64_t)e * wblocks + (kGated ? p.feat / 128 + t.nt : 0)) * KB;
      const float *sa = p.a_scales + (int64_t)grow * KB;
      float acc0[64], acc1[64];  // gated: gate, up halves; down: columns 0-63, 64-127 of this half
#pragma unroll
      for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0.f;
      bool ok = true;
      // scales of the next K block are loaded one block ahead
      float xs_n = row_ok ? __ldg(sa) : 0.f, s0_n = __ldg(sw0), s1_n = kGated ? __ldg(sw1) : 0.f;
      // gated: gate columns [64*half, +64) and up columns [128 + 64*half, +64)
      // down:  columns [128*half, +128)
      const uint32_t c0 = kGated ? 64 * half : 128 * half;
      const uint32_t c1 = kGated ? 128 + 64 * half : 128 * half + 64;
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        const int b = gk & 1;
        const float f0 = xs_n * s0_n;
        const float f1 = kGated ? xs_n * s1_n : f0;
        if (kb + 1 < KB) {
          xs_n = row_ok ? __ldg(sa + kb + 1) : 0.f;
          s0_n = __ldg(sw0 + kb + 1);
          if (kGated) s1_n = __ldg(sw1 + kb + 1);
        }
        if (!mbar_wait(dfull(b), (gk >> 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t d = lane_base + b * kAccCols;
        float v[64];
        tmem_ld32(d + c0, v);
        tmem_ld32(d + c0 + 32, v + 32);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 64; ++i) acc0[i] = fmaf(v[i], f0, acc0[i]);
        tmem_ld32(d + c1, v);
        tmem_ld32(d + c1 + 32, v + 32);
        tmem_wait_ld();
        fence_before();
        mbar_arrive_relaxed(dempty(b));  // the accumulator is in registers: let the next K block in
#pragma unroll
        for (int i = 0; i < 64; ++i) acc1[i] = fmaf(v[i], f1, acc1[i]);
      }
      if (!ok) break;
      if (t.e < 0 && r == 0 && half == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      if (kGated) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc0[i] = silu_fast(acc0[i]) * acc1[i];
          amax = fmaxf(amax, fabsf(acc0[i]));
        }
        // the row's two halves meet through shared memory; the slot alternates by tile
        // so a fast thread cannot overwrite a value its partner has yet to read
        float *slot = amax_x + (it & 1) * 256;
        slot[half * 128 + r] = amax;
        mbar_arrive(xbar);
        if (!mbar_wait(xbar, it & 1, abort_flag, p.err)) break;
        amax = fmaxf(slot[r], slot[128 + r]);
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        // h is an intermediate: multiplying by 1/scale instead of dividing moves the
        // value before rounding by at most an fp32 ulp
        const float inv = __frcp_rn(scale);
        if (row_ok) {
          uint8_t *orow = static_cast<uint8_t *>(p.out) + (int64_t)grow * p.ld + t.nt * 128 + 64 * half;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 16 * c + 4 * i;
              w[i] = e4m3x2(acc0[j] * inv, acc0[j + 1] * inv) | (e4m3x2(acc0[j + 2] * inv, acc0[j + 3] * inv) << 16);
            }
            reinterpret_cast<uint4 *>(orow)[c] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (half == 0) p.out_scales[(int64_t)grow * (p.feat / 128) + t.nt] = scale;
        }
      } else if (row_ok) {
        uint16_t *orow = static_cast<uint16_t *>(p.out) + (int64_t)grow * p.ld + t.nt * 256 + 128 * half;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 8 * c + 2 * i;
            w[i] = pack_bf16x2(acc0[j], acc0[j + 1]);
          }
          reinterpret_cast<uint4 *>(orow)[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 8 * c + 2 * i;
            w[i] = pack_bf16x2(acc1[j], acc1[j + 1]);
          }
          reinterpret_cast<uint4 *>(orow + 64)[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kGated>
moe_status_t launch(const Params &p, const CUtensorMap &a, cudaStream_t st) {
  auto k = grouped_gemm_e4m3<kGated>;
  if (cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem)) != MOE_OK)
    return MOE_ERR_CUDA;
  const int grid = grouped::sm_count();
  if (grid <= 0) return MOE_ERR_CUDA;
  k<<<grid, kThreads, kSmem, st>>>(p, a);
  return launch_status();
}

moe_status_t check_e4m3(const FfnArgs &f) {
  const moe_weights_t &w = *f.w;
  if (w.d % 256 || w.I % 128 || f.P > 2048 || f.T_shared > 0) return MOE_ERR_UNSUPPORTED;
  if (w.E_w * 2 * w.I > INT32_MAX || w.E_w * w.d > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (!w.s13 || !w.s2) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

moe_status_t gate_up_e4m3(const FfnArgs &f, cudaStream_t st) {
  moe_status_t s = check_e4m3(f);
  if (s != MOE_OK) return s;
  if (f.N == 0) return MOE_OK;
  if (!f.x_scales || !f.h_scales) return MOE_ERR_INVALID_ARG;
  const moe_weights_t &w = *f.w;
  if (!aligned(w.w13, 16)) return MOE_ERR_INVALID_ARG;
  if (grouped::tile_kind(f.N, f.P) == grouped::Tiles::kPair) return gate_up_e4m3_pair(f, st);
  CUtensorMap m_x;
  if (!grouped::make_map(&m_x, f.x_perm, f.N, w.d, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!aligned(w.w13, 16)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)w.I;
  p.K = (int)w.d;
  p.w_rows = (int)(2 * w.I);
  p.w = static_cast<const uint8_t *>(w.w13);
  p.w_tiles = (int)(w.I / 128);  // gate+up blocks of 128 features
  p.out = f.h;
  p.ld = w.I;
  p.a_scales = f.x_scales;
  p.w_scales = w.s13;
  p.out_scales = f.h_scales;
  return launch<true>(p, m_x, st);
}

moe_status_t down_e4m3(const FfnArgs &f, cudaStream_t st) {
  moe_status_t s = check_e4m3(f);
  if (s != MOE_OK) return s;
  if (f.N == 0) return MOE_OK;
  if (!f.h_scales) return MOE_ERR_INVALID_ARG;
  const moe_weights_t &w = *f.w;
  if (!aligned(w.w2, 16)) return MOE_ERR_INVALID_ARG;
  if (grouped::tile_kind(f.N, f.P) == grouped::Tiles::kPair) return down_e4m3_pair(f, st);
  CUtensorMap m_h;
  if (!grouped::make_map(&m_h, f.h, f.N, w.I, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!aligned(w.w2, 16)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)w.d;
  p.K = (int)w.I;
  p.w_rows = (int)w.d;
  p.w = static_cast<const uint8_t *>(w.w2);
  p.w_tiles = (int)(w.d / 128);
  p.out = f.y;
  p.ld = w.d;
  p.a_scales = f.h_scales;
  p.w_scales = w.s2;
  return launch<false>(p, m_h, st);
}

}  // namespace moe
