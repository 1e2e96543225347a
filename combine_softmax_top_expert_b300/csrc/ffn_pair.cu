// Grouped SwiGLU expert FFN, bf16, on pairs of SMs ("6.4 Data parallelism and
// expert parallelism", section 2.1: gate, up, down; section 7: the shared expert
// is one more always-on group).  The tile orientation for many rows per expert.
//
// A cluster of two CTAs owns one 256-token x 256-weight-row tile: CTA r loads
// token rows [128r, 128r+128) and 128 of the weight rows of every K block into its
// own shared memory, and the even CTA issues tcgen05.mma.cta_group::2 (M = 256,
// N = 256) that reads both CTAs' operands and leaves D rows [128r, +128) in CTA r's
// TMEM (columns 0-127 from the even CTA's weight rows, 128-255 from the odd CTA's).
// Per SM that is the MMA rate of a 128 x 256 tile with half of the weight traffic
// into shared memory, so a 32 KB stage feeds as many tensor cycles as a 48 KB stage
// of a one-SM tile and six stages fit.
// A group's last tile, when it holds at most 128 rows, is a half tile: M = 128, CTA
// r supplies token rows [64r, 64r+64) (the first 64 rows of its A stage) and its TMEM
// lanes 0-63 get those rows x columns 0-127, lanes 64-127 the same rows x columns
// 128-255 -- half the MMA work instead of padding to 256 rows.
//   gate/up   CTA r holds W_gate^T then W_up^T rows of features [64r, 64r+64) of
//             the tile's 128, so a 128-column half of D is gate then up of 64
//             features; h = silu(gate) * up, bf16.
//   down      CTA r holds the 128 weight rows of output features [128r, +128); y bf16.
// Roles per CTA: warp 0 TMA (both CTAs; all copies complete on the even CTA's
// stage barrier), warp 1 MMA (even CTA; TMEM allocation in both), warps 2-5
// epilogue (both CTAs, each its own 128 rows).
#include "grouped.cuh"

namespace moe {
namespace {

using namespace tc;
using grouped::Params;
using grouped::Tile;

constexpr int kThreads = 192;
constexpr int kStages = 6;
constexpr int kTokTile = 256;
constexpr int kABytes = 128 * 128;  // this CTA's 128 token rows x 128 bytes of K
constexpr int kBBytes = 128 * 128;  // this CTA's 128 of the tile's 256 weight rows
constexpr int kStage = kABytes + kBBytes;
constexpr int kAccCols = 256;
constexpr int kEpiWarps = 4;
constexpr int kBars = 2 * kStages + 5;
constexpr int kOutBox = 32 * 64;  // 32 rows x 64 bytes staged for a TMA store; two per epilogue warp
constexpr size_t kSmem =
    1024 + (size_t)kStages * kStage + 2 * kEpiWarps * kOutBox + kBars * 8 + 16 + (grouped::kMaxGroups + 1) * 4;
static_assert(kSmem <= 227 * 1024, "shared memory budget");

// After an abort a CTA cannot see its own copies land (they complete on the even
// CTA's barrier), so it waits this long before leaving.
constexpr uint64_t kAbortSettleNs = 100000;

template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_pair(const Params p, const __grid_constant__ CUtensorMap tm_tok,
                           const __grid_constant__ CUtensorMap tm_sh, const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *out_box = smem + (size_t)kStages * kStage;  // [kEpiWarps][2][32 rows][64 bytes]
  uint64_t *bars = reinterpret_cast<uint64_t *>(out_box + 2 * kEpiWarps * kOutBox);
  int *misc = reinterpret_cast<int *>(bars + kBars);  // [0] TMEM base, [1] abort flag
  int *tile_start = misc + 4;
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };  // used in the even CTA
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  auto tfull = [&](int b) { return smem_u32(&bars[2 * kStages + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[2 * kStages + 2 + b]); };  // used in the even CTA
  const uint32_t drain = smem_u32(&bars[2 * kStages + 4]);
  uint16_t *out = static_cast<uint16_t *>(p.out);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();
  const int G = p.P + (p.T_shared > 0 ? 1 : 0);
  const int NT = p.feat / (kGated ? 128 : 256);
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
    tma_prefetch(&tm_sh);
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int tile = pair; tile < total; tile += npairs) {
      const Tile t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile);
      const CUtensorMap *tmt = (kGated && t.shared) ? &tm_sh : &tm_tok;
      const int e = max(t.e, 0);
      // first weight row of this CTA in the K-block-0 block: gated, the gate rows of
      // features [64r, +64) (the up rows follow 128 rows later); down, tile 2nt + r
      const int wt = kGated ? t.nt : 2 * t.nt + (int)rank;
      const int wrows = kGated ? 256 : 128;
      const int64_t w0 = ((int64_t)e * p.w_tiles + wt) * KB * wrows + (kGated ? 64 * rank : 0);
      const int a_row = t.tok_row + (t.half ? 64 : 128) * (int)rank;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(empty(s), ph ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t st = stage0 + s * kStage, bar = peer_addr(full(s), 0);
        if (rank == 0) mbar_expect_tx(full(s), 2 * kStage);
        tma_load_2d_pair(st, tmt, bar, kb * 64, a_row);
        const int wr = (int)(w0 + (int64_t)kb * wrows);
        if (kGated) {
          tma_load_2d_pair(st + kABytes, &tm_w, bar, 0, wr);
          tma_load_2d_pair(st + kABytes + kBBytes / 2, &tm_w, bar, 0, wr + 128);
        } else {
          tma_load_2d_pair(st + kABytes, &tm_w, bar, 0, wr);
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
      if (rank == 0) {
        for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j)
          mbar_wait_drain(full(j % kStages), (uint32_t)((j / kStages) & 1));
      }
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < kAbortSettleNs) __nanosleep(1000);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------ MMA issuer (even CTA)
    int s = 0, it = 0;
    uint32_t ph = 0;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      const Tile t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile);
      const uint32_t id = idesc(t.half ? 128 : 256, 256, 1);
      const int b = it & 1;
      if (!mbar_wait(tempty(b), ((it >> 1) & 1) ^ 1, abort_flag, p.err)) break;
      fence_after();
      const uint32_t d = tmem + b * kAccCols;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(full(s), ph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t a = stage0 + s * kStage, bb = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_2(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id, (kb | kk) != 0);
        commit2_both(empty(s));
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      commit2_both(tfull(b));
    }
    if (*abort_flag) {  // no MMA may still run when TMEM is freed or the odd CTA leaves
      commit2(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int r = q * 32 + lane;  // TMEM lane = this CTA's token row
    const uint32_t tempty_even0 = peer_addr(tempty(0), 0), tempty_even1 = peer_addr(tempty(1), 0);
    uint8_t *boxes = out_box + (warp - 2) * 2 * kOutBox;
    int nbox = 0;  // TMA stores this warp has issued; they alternate between its two boxes
    int it = 0;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      const Tile t = grouped::decode<kTokTile>(p, tile_start, G, NT, tile);
      const int b = it & 1;
      if (!mbar_wait(tfull(b), (it >> 1) & 1, abort_flag, p.err)) break;
      fence_after();
      if (t.e < 0 && r == 0 && rank == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * kAccCols;
      // full tile: lane r is token row 128*rank + r and holds all 256 columns.
      // half tile: lane r is token row 64*rank + r % 64 and holds the 128 columns of
      // feature half r / 64 (in TMEM columns 0-127).
      const bool hv = t.half;
      const int row = hv ? 64 * (int)rank + (r & 63) : 128 * (int)rank + r;
      const bool ok = row < t.valid && t.e >= 0;
      const int fbase = hv ? (r >> 6) * (kGated ? 64 : 128) : 0;  // first output feature
      uint16_t *orow =
          out + (int64_t)(t.out_row + (ok ? row : 0)) * p.ld + (int64_t)t.nt * (kGated ? 128 : 256) + fbase;
      // all 32 rows of this warp belong to the tile: stage each 32-column piece and
      // store it with TMA (two boxes in flight); otherwise store row by row
      const bool whole = __all_sync(kFull, ok);
      const int nchunks = (kGated ? 4 : 8) >> (hv ? 1 : 0);
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        // gated: gate columns of features fbase + 32c .. (the up columns are 64 later)
        const int col = kGated ? ((hv || c < 2) ? 32 * c : 128 + 32 * (c - 2)) : 32 * c;
        float v[32], u[32];
        tmem_ld32(tb + col, v);
        if (kGated) tmem_ld32(tb + col + 64, u);
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
        if (whole) {
          if (lane == 0) bulk_wait_read_1();  // the store that last used this box has read it
          __syncwarp();
          warp_store_box(&tm_out, boxes + (nbox & 1) * kOutBox, pk, t.nt * (kGated ? 128 : 256) + fbase + 32 * c,
                         t.out_row + row, lane);
          ++nbox;
        } else if (ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive_relaxed(tempty(b));
        else mbar_arrive_cluster_relaxed(b ? tempty_even1 : tempty_even0);
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
moe_status_t launch(const Params &p, const CUtensorMap &a, const CUtensorMap &sh, const CUtensorMap &w,
                    const CUtensorMap &o, cudaStream_t st) {
  static int pairs = 0;
  return grouped::launch_pairs(grouped_gemm_bf16_pair<kGated>, kThreads, kSmem, &pairs, st, p, a, sh, w, o);
}

}  // namespace

// The pair orientation of gate_up_bf16 / down_bf16, which have checked the shapes.
moe_status_t gate_up_bf16_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I;
  CUtensorMap m_x, m_sh, m_w, m_h;
  const void *xsrc = f.N > 0 ? f.x_perm : f.shared_x;
  const int64_t xrows = f.N > 0 ? f.N : f.T_shared;
  if (!grouped::make_map(&m_x, xsrc, xrows, d, 2, 128)) return MOE_ERR_INVALID_ARG;
  if (f.T_shared > 0) {
    if (!grouped::make_map(&m_sh, f.shared_x, f.T_shared, d, 2, 128)) return MOE_ERR_INVALID_ARG;
  } else {
    m_sh = m_x;
  }
  if (!grouped::make_store_map(&m_h, f.h, f.N + f.T_shared, I, 2, 32)) return MOE_ERR_INVALID_ARG;
  // the packed W_gate^T/W_up^T as 128-byte rows
  if (!grouped::make_map_tiled(&m_w, w.w13, (uint64_t)w.E_w * 2 * I * (d / 64), 64)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)I;
  p.K = (int)d;
  p.w_rows = (int)(2 * I);
  p.w = static_cast<const uint8_t *>(w.w13);
  p.w_tiles = (int)(I / 128);
  p.shared_row0 = 0;
  p.out = f.h;
  p.ld = I;
  return launch<true>(p, m_x, m_sh, m_w, m_h, st);
}

// Needs d % 256 == 0 (256 output features per pair tile).
moe_status_t down_bf16_pair(const FfnArgs &f, cudaStream_t st) {
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I, rows = f.N + f.T_shared;
  if (d % 256) return MOE_ERR_UNSUPPORTED;
  CUtensorMap m_h, m_w, m_y;
  if (!grouped::make_map(&m_h, f.h, rows, I, 2, 128)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_store_map(&m_y, f.y, rows, d, 2, 32)) return MOE_ERR_INVALID_ARG;
  if (!grouped::make_map_tiled(&m_w, w.w2, (uint64_t)w.E_w * d * (I / 64), 128)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)d;
  p.K = (int)I;
  p.w_rows = (int)d;
  p.w = static_cast<const uint8_t *>(w.w2);
  p.w_tiles = (int)(d / 128);
  p.shared_row0 = (int)f.N;
  p.out = f.y;
  p.ld = d;
  return launch<false>(p, m_h, m_h, m_w, m_y, st);
}

}  // namespace moe
