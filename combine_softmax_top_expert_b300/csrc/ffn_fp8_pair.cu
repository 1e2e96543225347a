// Grouped SwiGLU expert FFN with e4m3 operands and fp32 block scales on pairs of
// SMs ("6.4 Data parallelism and expert parallelism", section 2.1 gate/up/down;
// section 3.2 FP8).  The tile orientation for many rows per expert.
//
// As in the one-SM kernel (ffn_fp8.cu), every 128-deep K block gets a fresh TMEM
// accumulator that the epilogue warps fold into fp32 registers with the block's
// scales, acc += D_kb * (s_row[kb] * s_weight_block[kb]), and two 256-column
// accumulators alternate.  Here a cluster of two CTAs owns a 256-token tile (128
// rows per CTA): each K block is four tcgen05.mma.cta_group::2 (M = 256, N = 256,
// K = 32) issued by the even CTA, and each SM loads only half of the weight rows,
// so a stage is 32 KB and six fit.  (Splitting a K block into two separately
// committed N = 128 groups was measured and is slower: every commit-and-wait hand-off
// costs a few hundred cycles of issue time.)
//
// Weight rows of a tile, as in the bf16 pair kernel:
//   gate/up  the even CTA holds W_gate^T rows of the tile's 128 features, the odd
//            CTA the W_up^T rows: D columns 0-127 gate, 128-255 up.
//   down     256 output features: the even CTA's 128 then the odd CTA's.
// Epilogue warp w (w = 4..11) reads TMEM lanes 32*(w % 4).. of its own CTA; warps w
// and w+4 split the columns (gate/up: features [64h, 64h+64) of gate and of up;
// down: columns [128h, 128h+128)):
//   gate/up  h = silu(g) * u for the tile's 128 features, quantised per row over
//            those 128 channels (the two halves exchange their amax):
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
constexpr int kAccCols = 256;
constexpr int kEpiWarps = 8;  // per CTA
// full[s], empty[s], dfull[b], dempty[b], drain, xbar
constexpr int kBars = 2 * kStages + 2 + 2 + 2;
constexpr int kOutBox = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes staged for a TMA store
constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kEpiWarps * kOutBox + kBars * 8 + 16 + 2 * 256 * 4 +
                         (grouped::kMaxGroups + 1) * 4;
static_assert(kSmem <= 227 * 1024, "shared memory budget");
constexpr uint64_t kAbortSettleNs = 100000;

template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_e4m3_pair(const Params p, const __grid_constant__ CUtensorMap tm_tok,
                           const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *out_box = smem + (size_t)kStages * kStage;  // [kEpiWarps][32 rows][64 bytes]
  uint64_t *bars = reinterpret_cast<uint64_t *>(out_box + kEpiWarps * kOutBox);
  int *misc = reinterpret_cast<int *>(bars + kBars);  // [0] TMEM base, [1] abort flag
  float *amax_x = reinterpret_cast<float *>(misc + 4);  // [2 tiles][2 groups][128 rows]
  int *tile_start = reinterpret_cast<int *>(amax_x + 512);
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };  // used in the even CTA
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto dfull = [&](int b) { return smem_u32(&bars[2 * kStages + b]); };
  auto dempty = [&](int b) { return smem_u32(&bars[2 * kStages + 2 + b]); };  // used in the even CTA
  const uint32_t drain = smem_u32(&bars[2 * kStages + 4]);
  const uint32_t xbar = smem_u32(&bars[2 * kStages + 5]);

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
    for (int b = 0; b < 2; ++b) {
      mbar_init(dfull(b), 1);
      mbar_init(dempty(b), 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(xbar, 256);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
    tma_prefetch(&tm_w);
    tma_prefetch(&tm_out);
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
        // gated: rows [128r, +128) of the 256-row gate+up block; down: the 128-row
        // block of tile 2nt + r (the map holds fewer than 2^31 rows)
        int w0 = kGated ? ((e * p.w_tiles + t.nt) * KB * 256 + 128 * (int)rank)
                        : ((e * p.w_tiles + 2 * t.nt + (int)rank) * KB * 128);
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
      const uint32_t id = idesc(256, 256, 0);
      bool ok = true;
      // the next block's two barriers are tested right after this block's MMAs, and
      // the answers read after its commits, so the tests' latency hides behind the
      // commits (a phase found complete stays complete: the next phase of either
      // barrier needs a commit this thread has not issued yet)
      bool pre_full = false, pre_empty = false;
      for (int tile = pair; tile < total && ok; tile += npairs) {
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
          for (int kk = 0; kk < 4; ++kk) mma_f8_2(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id, kk != 0);
          const int s1 = s + 1 == kStages ? 0 : s + 1;
          const uint32_t ph1 = s + 1 == kStages ? ph ^ 1 : ph;
          pre_full = mbar_test(full(s1), ph1);
          pre_empty = mbar_test(dempty((gk + 1) & 1), (((gk + 1) >> 1) & 1) ^ 1);
          commit2_both(dfull(b));
          commit2_both(empty(s));
          s = s1;
          ph = ph1;
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
    // 64 bytes of output per row (w = 16 words) of this warp's 32 rows.  When all 32
    // rows belong to the tile they go through this warp's staging box and one TMA
    // store at column x (elements) of rows grow - lane ..; otherwise each row is
    // written directly to `dst`.
    uint8_t *box = out_box + (warp - 4) * kOutBox;
    auto store_rows = [&](const uint32_t *w, int x, bool ok, int grow, uint8_t *dst) {
      if (__all_sync(kFull, ok)) {
        if (lane == 0) bulk_wait_read();  // the previous store has read the box
        __syncwarp();
        warp_store_box(&tm_out, box, w, x, grow, lane);
      } else if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          reinterpret_cast<uint4 *>(dst)[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    };
    // gated: gate columns [64h, +64) and up columns [128 + 64h, +64); down: [128h, +128)
    const uint32_t c0 = kGated ? 64 * half : 128 * half;
    const uint32_t c1 = kGated ? 128 + 64 * half : 128 * half + 64;
    // A tile's coordinates and the scales of its first K block.  In the down
    // projection the next tile's are fetched before this tile's outputs are stored, so
    // the latency of the decode's loads and of the scale loads hides behind the stores
    // (+3.5 % there; the gate/up epilogue, with more live registers at that point,
    // measured 1.5 % slower with it and fetches them at the top of the tile).
    struct TileCtx {
      Tile t;
      bool row_ok;
      int grow, sw0, sw1, sa;
      float xs, s0, s1;
    };
    grouped::GroupCache gcache;
    auto prep = [&](int tile) {
      TileCtx c;
      c.t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile, &gcache);
      const int row = 128 * (int)rank + r;
      c.row_ok = row < c.t.valid && c.t.e >= 0;
      c.grow = c.t.out_row + (c.row_ok ? row : 0);  // also the row of the token operand's scales
      const int e = max(c.t.e, 0);
      // weight-scale rows: gated -> gate block nt and up block I/128 + nt; down -> 2nt + half
      c.sw0 = (e * wblocks + (kGated ? c.t.nt : 2 * c.t.nt + half)) * KB;
      c.sw1 = kGated ? (e * wblocks + p.feat / 128 + c.t.nt) * KB : c.sw0;
      c.sa = c.grow * KB;
      c.xs = c.row_ok ? __ldg(p.a_scales + c.sa) : 0.f;
      c.s0 = __ldg(p.w_scales + c.sw0);
      c.s1 = kGated ? __ldg(p.w_scales + c.sw1) : 0.f;
      return c;
    };
    // down: the second half of a finished tile's outputs (this thread's columns
    // c1..c1+63 of its row, packed to bf16) waits in pk until the next tile's first
    // accumulator is read and released, so the MMA runs on while it is stored
    uint32_t pk[32];
    bool pend = false, pend_ok = false;
    int pend_x = 0, pend_grow = 0;
    uint8_t *pend_dst = nullptr;
    auto store_pend = [&]() {
      if (pend) {
        store_rows(pk, pend_x, pend_ok, pend_grow, pend_dst);
        store_rows(pk + 16, pend_x + 32, pend_ok, pend_grow, pend_dst + 64);
        pend = false;
      }
    };
    int gk = 0, it = 0;
    TileCtx cur;
    if (!kGated && pair < total) cur = prep(pair);
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      if (kGated) cur = prep(tile);
      const Tile t = cur.t;
      const bool row_ok = cur.row_ok;
      const int grow = cur.grow, sw0 = cur.sw0, sw1 = cur.sw1, sa = cur.sa;
      float acc0[64], acc1[64];  // gated: gate, up of 64 features; down: columns c0.., c1..
      if (kGated) {
#pragma unroll
        for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0.f;
      }
      bool ok = true;
      // the scales of the next K block load one block ahead
      float xs_n = cur.xs, s0_n = cur.s0, s1_n = cur.s1;
      int kb0 = 0;
      if (!kGated) {
        // block 0 goes straight into the sums; once its accumulator is released, the
        // previous tile's deferred half is stored
        const int b = gk & 1;
        const float f0 = xs_n * s0_n;
        if (KB > 1) {
          xs_n = row_ok ? __ldg(p.a_scales + sa + 1) : 0.f;
          s0_n = __ldg(p.w_scales + sw0 + 1);
        }
        if (!mbar_wait(dfull(b), (gk >> 1) & 1, abort_flag, p.err)) break;
        fence_after();
        const uint32_t d = lane_base + b * kAccCols;
        tmem_ld32(d + c0, acc0);
        tmem_ld32(d + c0 + 32, acc0 + 32);
        tmem_ld32(d + c1, acc1);
        tmem_ld32(d + c1 + 32, acc1 + 32);
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive_relaxed(dempty(b));
          else mbar_arrive_cluster_relaxed(peer_addr(dempty(b), 0));
        }
        store_pend();
        scale2_inplace<64>(acc0, f0);
        scale2_inplace<64>(acc1, f0);
        ++gk;
        kb0 = 1;
      }
      for (int kb = kb0; kb < KB; ++kb, ++gk) {
        const int b = gk & 1;
        const float f0 = xs_n * s0_n;
        const float f1 = kGated ? xs_n * s1_n : f0;
        if (kb + 1 < KB) {
          xs_n = row_ok ? __ldg(p.a_scales + sa + kb + 1) : 0.f;
          s0_n = __ldg(p.w_scales + sw0 + kb + 1);
          if (kGated) s1_n = __ldg(p.w_scales + sw1 + kb + 1);
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
        fma2_scaled<64>(acc0, v, f0);
        tmem_ld32(d + c1, v);
        tmem_ld32(d + c1 + 32, v + 32);
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        // this warp's columns are in registers: release them to the even CTA's MMA
        if (lane == 0) {
          if (rank == 0) mbar_arrive_relaxed(dempty(b));
          else mbar_arrive_cluster_relaxed(peer_addr(dempty(b), 0));
        }
        fma2_scaled<64>(acc1, v, f1);
      }
      if (!ok) break;
      if (t.e < 0 && r == 0 && half == 0 && rank == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      if (!kGated && tile + npairs < total) cur = prep(tile + npairs);
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
        uint32_t w[16];  // this row's 64 codes
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = e4m3x2(acc0[4 * i] * inv, acc0[4 * i + 1] * inv) |
                 (e4m3x2(acc0[4 * i + 2] * inv, acc0[4 * i + 3] * inv) << 16);
        store_rows(w, t.nt * 128 + 64 * half, row_ok, grow, static_cast<uint8_t *>(p.out) + (int64_t)grow * p.ld +
                                                            t.nt * 128 + 64 * half);
        if (row_ok && half == 0) p.out_scales[(int64_t)grow * (p.feat / 128) + t.nt] = scale;
      } else {
        // four 32-column pieces of this thread's 128 output features: the first two now,
        // the last two after the next tile's first block (at once on the last tile)
        uint8_t *dst = static_cast<uint8_t *>(p.out) + ((int64_t)grow * p.ld + t.nt * 256 + 128 * half) * 2;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(acc0[32 * c + 2 * i], acc0[32 * c + 2 * i + 1]);
          store_rows(w, t.nt * 256 + 128 * half + 32 * c, row_ok, grow, dst + 64 * c);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(acc1[2 * i], acc1[2 * i + 1]);
        pend = true;
        pend_ok = row_ok;
        pend_grow = grow;
        pend_x = t.nt * 256 + 128 * half + 64;
        pend_dst = dst + 128;
        if (tile + npairs >= total) store_pend();  // this CTA's last tile
      }
    }
    if (lane == 0) bulk_wait();
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
moe_status_t launch(const Params &p, const CUtensorMap &a, const CUtensorMap &w, const CUtensorMap &o,
                    cudaStream_t st) {
  static int pairs = 0;
  return grouped::launch_pairs(grouped_gemm_e4m3_pair<kGated>, kThreads, kSmem, &pairs, st, p, a, w, o);
}

}  // namespace

// The pair orientation of gate_up_e4m3 / down_e4m3, which have checked the shapes
// (d % 256 == 0, I % 128 == 0, no shared expert) and the scale pointers.
moe_status_t gate_up_e4m3_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  CUtensorMap m_x, m_w, m_h;
  if (!grouped::make_map(&m_x, f.x_perm, f.N, w.d, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_store_map(&m_h, f.h, f.N, w.I, 1, 32)) return MOE_ERR_INVALID_ARG;
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
  return launch<true>(p, m_x, m_w, m_h, st);
}

moe_status_t down_e4m3_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  CUtensorMap m_h, m_w, m_y;
  if (!grouped::make_map(&m_h, f.h, f.N, w.I, 1, 128)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_store_map(&m_y, f.y, f.N, w.d, 2, 32)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_map_tiled(&m_w, w.w2, (uint64_t)w.E_w * w.d * (w.I / 128), 128)) return MOE_ERR_INVALID_ARG;
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
  return launch<false>(p, m_h, m_w, m_y, st);
}

}  // namespace moe
