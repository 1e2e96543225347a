// Grouped SwiGLU expert FFN with e4m3 operands and fp32 block scales on pairs of
// SMs ("6.4 Data parallelism and expert parallelism", section 2.1 gate/up/down;
// section 3.2 FP8).  The tile orientation for many rows per expert.
//
// As in the one-SM kernel (ffn_fp8.cu), every 128-deep K block gets a fresh TMEM
// accumulator that the epilogue warps fold into fp32 registers with the block's
// scales, acc += D_kb * (s_row[kb] * s_weight_block[kb]).  That fold is a chain
// (MMA, commit, TMEM load, release) that TMEM's two 256-column buffers must
// cover.  Here a cluster of two CTAs owns a 256-token tile (128 rows per CTA) and
// each K block is two independent groups of tcgen05.mma.cta_group::2 with
// M = 256, N = 128, each committed and released on its own.  With four
// 128-column half buffers in flight the chain is cut into shorter links, and
// each SM loads only half of the weight rows, so a stage is 32 KB and six fit.
//
// Group h of a K block (columns [128h, 128h+128) of its buffer):
//   gate/up  the even CTA holds W_gate^T rows of the tile's 128 features, the
//            odd CTA the W_up^T rows; group h reads rows [64h, 64h+64) of both,
//            so its columns are gate then up of features [64h, 64h+64).
//   down     the tile has 256 output features; CTA r holds rows [64r, 64r+64)
//            of the two 128-feature weight tiles; group h reads tile h's rows
//            of both CTAs, so column c is output feature c.
// Epilogue warp w (w = 4..11) reads TMEM lanes 32*(w % 4).. of its own CTA and
// group (w - 4) / 4: the same per-thread work as the one-SM kernel.
//   gate/up  h = silu(g) * u for the tile's 128 features, quantised per row over
//            those 128 channels (the two groups exchange their amax):
//            scale = amax / 448, code = e4m3(h * (1 / scale)).
//   down     y = acc, bf16.
#include "grouped.cuh"

namespace moe {
namespace {

using namespace tc;
using grouped::Params;
using grouped::Tile;

constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168, kRegsIssue = 56, kRegsEpilogue = 224;
static_assert(128 * kRegsIssue + 256 * kRegsEpilogue == kThreads * kRegsLaunch, "register split");
constexpr int kStages = 6;
constexpr int kTokTile = 256;
constexpr int kABytes = 128 * 128;  // this CTA's 128 token rows x 128 K bytes
constexpr int kBBytes = 128 * 128;  // this CTA's 128 weight rows
constexpr int kStage = kABytes + kBBytes;
constexpr int kAccCols = 256;  // one K block = two 128-column groups
constexpr int kGroupWarps = 4;  // epilogue warps per group per CTA
// full[s], empty[s], dfull[b][h], dempty[b][h], drain, xbar
constexpr int kBars = 2 * kStages + 4 + 4 + 2;
constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kBars * 8 + 16 + 2 * 256 * 4 +
                         (grouped::kMaxGroups + 1) * 4;
static_assert(kSmem <= 227 * 1024, "shared memory budget");
constexpr uint64_t kAbortSettleNs = 100000;

template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_e4m3_pair(const Params p, const __grid_constant__ CUtensorMap tm_tok,
                           const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * kStage);
  int *misc = reinterpret_cast<int *>(bars + kBars);  // [0] TMEM base, [1] abort flag
  float *amax_x = reinterpret_cast<float *>(misc + 4);  // [2 tiles][2 groups][128 rows]
  int *tile_start = reinterpret_cast<int *>(amax_x + 512);
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };  // used in the even CTA
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto dfull = [&](int b, int h) { return smem_u32(&bars[2 * kStages + 2 * b + h]); };
  auto dempty = [&](int b, int h) { return smem_u32(&bars[2 * kStages + 4 + 2 * b + h]); };  // even CTA
  const uint32_t drain = smem_u32(&bars[2 * kStages + 8]);
  const uint32_t xbar = smem_u32(&bars[2 * kStages + 9]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();
  const int G = p.P;
  const int NT = p.feat / (kGated ? 128 : 256);
  const int KB = p.K / 128;
  const int wblocks = p.w_rows / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b)
      for (int h = 0; h < 2; ++h) {
        mbar_init(dfull(b, h), 1);
        mbar_init(dempty(b, h), 2 * kGroupWarps);
      }
    mbar_init(drain, 1);
    mbar_init(xbar, 256);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
    tma_prefetch(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(&misc[0]), 2 * kAccCols);
    tmem_relinquish2();
  }
  grouped::build_tile_table<kTokTile>(p, tile_start, G, NT);
  fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other's
  fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[1]);
  const int total = tile_start[G];

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int tile = pair; tile < total; tile += npairs) {
        const Tile t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile);
        const int e = max(t.e, 0);
        // gated: rows [128r, +128) of the 256-row gate+up block; down: rows [64r, +64)
        // of the two 128-row blocks of output features 256nt ..
        // (the map holds fewer than 2^31 rows)
        int w0 = kGated ? ((e * p.w_tiles + t.nt) * KB * 256 + 128 * (int)rank)
                        : ((e * p.w_tiles + 2 * t.nt) * KB * 128 + 64 * (int)rank);
        const int w1 = KB * 128;  // down: the second tile's block, relative to the first
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t st = stage0 + s * kStage, bar = peer_addr(full(s), 0);
          if (rank == 0) mbar_expect_tx(full(s), 2 * kStage);
          tma_load_2d_pair(st, &tm_tok, bar, kb * 128, t.tok_row + 128 * (int)rank);
          tma_load_2d_pair(st + kABytes, &tm_w, bar, 0, w0);
          if (!kGated) tma_load_2d_pair(st + kABytes + kBBytes / 2, &tm_w, bar, 0, w0 + w1);
          w0 += kGated ? 256 : 128;
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        if (rank == 0) {
          for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j)
            mbar_wait_drain(full(j % kStages), (uint32_t)((j / kStages) & 1));
        }
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < kAbortSettleNs) __nanosleep(1000);
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (even CTA)
      int s = 0, gk = 0;
      uint32_t ph = 0;
      const uint32_t id = idesc(256, 128, 0);
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const int b = gk & 1;
          if (!mbar_wait(full(s), ph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t a = stage0 + s * kStage, bb = a + kABytes;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait(dempty(b, h), ((gk >> 1) & 1) ^ 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            fence_after();
            const uint32_t d = tmem + b * kAccCols + h * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_2(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + h * (kBBytes / 2) + kk * 32), id, kk != 0);
            commit2_both(dfull(b, h));
          }
          if (!ok) break;
          commit2_both(empty(s));
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort_flag) {  // no MMA may still run when TMEM is freed or the odd CTA leaves
        commit2(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3, half = (warp - 4) >> 2;
    const int r = q * 32 + lane;  // TMEM lane = this CTA's token row
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    int gk = 0, it = 0;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      const Tile t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile);
      const int row = 128 * (int)rank + r;
      const bool row_ok = row < t.valid && t.e >= 0;
      const int grow = t.out_row + (row_ok ? row : 0);  // also the row of the token operand's scales
      const int e = max(t.e, 0);
      // weight-scale rows: gated -> gate block nt and up block I/128 + nt; down -> 2nt + half
      const int sw0 = (e * wblocks + (kGated ? t.nt : 2 * t.nt + half)) * KB;
      const int sw1 = kGated ? (e * wblocks + p.feat / 128 + t.nt) * KB : sw0;
      const int sa = grow * KB;
      float acc0[64], acc1[64];  // gated: gate, up of 64 features; down: 128 output features
#pragma unroll
      for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0.f;
      bool ok = true;
      // the scales of the next K block load one block ahead
      float xs_n = row_ok ? __ldg(p.a_scales + sa) : 0.f, s0_n = __ldg(p.w_scales + sw0);
      float s1_n = kGated ? __ldg(p.w_scales + sw1) : 0.f;
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        const int b = gk & 1;
        const float f0 = xs_n * s0_n;
        const float f1 = kGated ? xs_n * s1_n : f0;
        if (kb + 1 < KB) {
          xs_n = row_ok ? __ldg(p.a_scales + sa + kb + 1) : 0.f;
          s0_n = __ldg(p.w_scales + sw0 + kb + 1);
          if (kGated) s1_n = __ldg(p.w_scales + sw1 + kb + 1);
        }
        if (!mbar_wait(dfull(b, half), (gk >> 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t d = lane_base + b * kAccCols;
        float v[64];
        tmem_ld32(d + 128 * half, v);
        tmem_ld32(d + 128 * half + 32, v + 32);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 64; ++i) acc0[i] = fmaf(v[i], f0, acc0[i]);
        tmem_ld32(d + 128 * half + 64, v);
        tmem_ld32(d + 128 * half + 96, v + 32);
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        // the group's columns are in registers: release them to the even CTA's MMA
        if (lane == 0) {
          if (rank == 0) mbar_arrive(dempty(b, half));
          else mbar_arrive_cluster_relaxed(peer_addr(dempty(b, half), 0));
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) acc1[i] = fmaf(v[i], f1, acc1[i]);
      }
      if (!ok) break;
      if (t.e < 0 && r == 0 && half == 0 && rank == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      if (kGated) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc0[i] = silu_fast(acc0[i]) * acc1[i];
          amax = fmaxf(amax, fabsf(acc0[i]));
        }
        // the row's two groups meet through shared memory; the slot alternates by
        // tile so a fast thread cannot overwrite a value its partner has yet to read
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
  cluster_sync();  // the even CTA's MMAs read the odd CTA's shared memory until here
  fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc2(tmem, 2 * kAccCols);
  }
}

template <bool kGated>
moe_status_t launch(const Params &p, const CUtensorMap &a, const CUtensorMap &w, cudaStream_t st) {
  static int pairs = 0;
  return grouped::launch_pairs(grouped_gemm_e4m3_pair<kGated>, kThreads, kSmem, &pairs, st, p, a, w);
}

}  // namespace

// The pair orientation of gate_up_e4m3 / down_e4m3, which have checked the shapes
// (d % 256 == 0, I % 128 == 0, no shared expert) and the scale pointers.
moe_status_t gate_up_e4m3_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  CUtensorMap m_x, m_w;
  if (!grouped::make_map(&m_x, f.x_perm, f.N, w.d, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_map_tiled(&m_w, w.w13, (uint64_t)w.E_w * 2 * w.I * (w.d / 128), 128))
    return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)w.I;
  p.K = (int)w.d;
  p.w_rows = (int)(2 * w.I);
  p.w = static_cast<const uint8_t *>(w.w13);
  p.w_tiles = (int)(w.I / 128);
  p.out = f.h;
  p.ld = w.I;
  p.a_scales = f.x_scales;
  p.w_scales = w.s13;
  p.out_scales = f.h_scales;
  return launch<true>(p, m_x, m_w, st);
}

moe_status_t down_e4m3_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  CUtensorMap m_h, m_w;
  if (!grouped::make_map(&m_h, f.h, f.N, w.I, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_map_tiled(&m_w, w.w2, (uint64_t)w.E_w * w.d * (w.I / 128), 64)) return MOE_ERR_INVALID_ARG;
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
  return launch<false>(p, m_h, m_w, st);
}

}  // namespace moe
