// Grouped SwiGLU expert FFN on the tcgen05 tensor cores, bf16 ("6.4 Data
// parallelism and expert parallelism", section 2.1: gate, up, down; section 7:
// the shared expert is one more always-on group).
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
//         W_down): one 128x256xK tile per feature block.  The one-SM form of the
//         pair tiles (ffn_pair.cu) used for many rows per expert.
//   swap  A = 128 weight rows, B = up to 32 token rows: D is features x tokens, so a
//         group of a few tokens streams its weights at HBM speed without padding
//         tokens to 128.  For decode-sized batches.  Gate/up tiles hold 64 features:
//         A rows 0-63 are W_gate^T, 64-127 W_up^T of the same features (two 8 KB
//         copies of the packed block), so one MMA per K step gives gate in TMEM lanes
//         0-63 and up in lanes 64-127; the up lanes' warps hand their values to the
//         gate lanes' warps through shared memory (a bounded mbarrier each way).
#include "grouped.cuh"

namespace moe {
namespace {

using namespace tc;
using grouped::Params;
using grouped::Tile;

constexpr int kThreads = 192;

template <bool kGated, bool kSwap, int kBW>
struct Cfg {
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBRows = kSwap ? 32 : (kGated ? 256 : kBW);
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kStages = kSwap ? 8 : 4;
  static constexpr int kAccCols = kSwap ? 32 : (kGated ? 256 : kBW);
  static constexpr int kTmemCols = kSwap ? 64 : (2 * kAccCols >= 512 ? 512 : 256);
  static constexpr int kTokTile = kSwap ? 32 : 128;
  static constexpr int kFeatTile = kSwap ? (kGated ? 64 : 128) : (kGated ? 128 : kBW);
  static constexpr bool kXchg = kSwap && kGated;  // up -> gate hand-off through shared memory
  static constexpr int kXchgFloats = kXchg ? 2 * 64 * 33 : 0;  // [2 tiles][64 features][32 tokens + 1 pad]
  static constexpr int kBars = 2 * kStages + 5 + (kXchg ? 4 : 0);
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kBars * 8 + 16 + (size_t)kXchgFloats * 4 +
                                  (grouped::kMaxGroups + 1) * 4;
  static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// ---------------------------------------------------------------- fused combine
// out[t] for one block of kFeat features, by one warp (lane: 8 features): the k rows
// y[slot_to_row[t, j]] weighted in j order with fp32 fused multiply-adds, then the
// shared expert's row y[N + t] added, then rounded to bf16 -- the same operations,
// in the same order, as the separate combine kernel, so the result is identical.
// The rows are read from L2 (other CTAs wrote them).
template <int kFeat>
__device__ __forceinline__ void combine_block(const Params &p, int tok, int nt, int lane) {
  const uint16_t *y = static_cast<const uint16_t *>(p.out);
  const int k = p.c_k;
  const int64_t col = (int64_t)nt * kFeat;
  const int32_t *s2r = p.c_slot_to_row + (int64_t)tok * k;
  const float *tw = p.c_topk_w + (int64_t)tok * k;
  for (int v = lane; v < kFeat / 8; v += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 raw[8];
      int rr[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {  // all of the group's row loads go out first
        int r = j0 + jj < k ? __ldg(s2r + j0 + jj) : -1;
        if (r >= p.N) {
          raise_dev(p.err, MOE_DEV_LAYOUT);
          r = -1;
        }
        rr[jj] = r;
        if (r >= 0) raw[jj] = __ldcg(reinterpret_cast<const uint4 *>(y + (int64_t)r * p.ld + col) + v);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (rr[jj] < 0) continue;
        const float wt = __ldg(tw + j0 + jj);
        const uint4 q = raw[jj];
        const float f[8] = {bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y),
                            bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt, f[i], acc[i]);
      }
    }
    if (p.T_shared > 0) {
      const uint4 q = __ldcg(reinterpret_cast<const uint4 *>(y + (int64_t)(p.N + tok) * p.ld + col) + v);
      const float f[8] = {bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y),
                          bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(1.0f, f[i], acc[i]);
    }
    reinterpret_cast<uint4 *>(p.c_out + (int64_t)tok * p.ld + col)[v] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

// After a tile's rows of y are stored (every lane of an epilogue warp calls this for
// its row r): count the row against its token's block, and let the warp sum the
// blocks whose last row this was.  Counting is release (fence, then the atomic);
// summing is acquire (a strong read of the count, then a fence).  No CTA waits for
// another: whichever CTA completes a block does its sum.
template <int kFeat>
__device__ __forceinline__ void combine_after_rows(const Params &p, const Tile &t, int r, int lane, int NT) {
  int tok = -1;
  bool last = false;
  if (t.e >= 0 && r < t.valid) {
    const int row = t.out_row + r;
    tok = t.shared ? row - p.N : __ldg(p.c_row_to_token + row);
    if (tok >= 0 && tok < p.c_T) {
      __threadfence();
      last = atomicAdd(p.c_counts + (int64_t)tok * NT + t.nt, 1) == -1;
    } else {
      raise_dev(p.err, MOE_DEV_LAYOUT);
    }
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  while (m) {
    const int src = __ffs(m) - 1;
    m &= m - 1;
    const int tk = __shfl_sync(0xffffffffu, tok, src);
    (void)ld_relaxed_gpu(p.c_counts + (int64_t)tk * NT + t.nt);
    __threadfence();
    combine_block<kFeat>(p, tk, t.nt, lane);
  }
}

// kGather (gate/up, wide tiles only): the dispatch permute fused into the A-load.  The
// routed token rows are gathered straight from x through row_to_token by the producer
// warp: the 8 lanes of quarter g = lane / 8 copy the 8 16-byte chunks (c = lane % 8)
// of tile rows 4i + g, i < 32, with cp.async, so each copy instruction reads 4 whole
// 128-byte lines; chunk c of tile row r lands at chunk c ^ (r % 8) of its 128-byte
// row, the layout a 128-row TMA box with 128-byte swizzle gives.  Each lane's copies
// count as one arrival on the stage's barrier.  The weights still come by bulk copy;
// the shared expert's rows are x itself and keep their tile load.
// kCombine (down, wide tiles only): the combine fused into the epilogue
// (combine_after_rows); the shared expert's group is tiled first, so that the blocks'
// last rows, and with them the sums, spread over the routed tiles.
template <bool kGated, bool kSwap, int kBW, bool kGather = false, bool kCombine = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16(const Params p, const __grid_constant__ CUtensorMap tm_tok,
                      const __grid_constant__ CUtensorMap tm_sh) {
  static_assert(!kGather || (kGated && !kSwap), "the gathered A-load is a wide gate/up tile");
  static_assert(!kCombine || (!kGated && !kSwap), "the fused combine is a wide down tile");
  using C = Cfg<kGated, kSwap, kBW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)C::kStages * C::kStage);
  int *misc = reinterpret_cast<int *>(bars + C::kBars);  // [0] TMEM base, [1] abort flag
  float *xchg = reinterpret_cast<float *>(misc + 4);      // up values on their way to the gate lanes
  int *tile_start = reinterpret_cast<int *>(xchg + C::kXchgFloats);
  const uint32_t stage0 = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[C::kStages + s]); };
  auto tfull = [&](int b) { return smem_u32(&bars[2 * C::kStages + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[2 * C::kStages + 2 + b]); };
  const uint32_t drain = smem_u32(&bars[2 * C::kStages + 4]);
  auto xfull = [&](int b) { return smem_u32(&bars[2 * C::kStages + 5 + b]); };  // kXchg only
  auto xfree = [&](int b) { return smem_u32(&bars[2 * C::kStages + 7 + b]); };
  uint16_t *out = static_cast<uint16_t *>(p.out);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.P + (p.T_shared > 0 ? 1 : 0);
  const int NT = p.feat / C::kFeatTile;
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full(s), kGather ? 1 + 32 : 1);  // + one arrival per copying lane
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 128);
    }
    mbar_init(drain, 1);
    if (C::kXchg)
      for (int b = 0; b < 2; ++b) {
        mbar_init(xfull(b), 64);
        mbar_init(xfree(b), 64);
      }
    misc[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch(&tm_tok);
    tma_prefetch(&tm_sh);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), C::kTmemCols);
    tmem_relinquish();
  }
  grouped::build_tile_table<C::kTokTile>(p, tile_start, G, NT);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(&misc[1]);
  const int total = tile_start[G];

  if (warp == 0 && (kGather || lane == 0)) {
    // ------------------------------------------------ TMA producer (the whole warp with kGather)
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = grouped::decode<C::kTokTile>(p, tile_start, G, NT, tile);
      const CUtensorMap *tmt = (kGated && t.shared) ? &tm_sh : &tm_tok;
      const int nb = kSwap ? (t.valid + 15) / 16 : 0;
      const bool gathered = kGather && !t.shared;
      // gathered rows past the group's end, or naming a token outside x (reported),
      // are not loaded: they keep older data, and those outputs are never stored
      const uint32_t bytes = (gathered ? 0 : C::kABytes) + (kSwap ? nb * 2048 : C::kBBytes);
      const int g4 = lane >> 3, c8 = lane & 7;
      int tok[kGather ? 32 : 1];
#pragma unroll
      for (int i = 0; i < (kGather ? 32 : 0); ++i) {
        const int row = 4 * i + g4;
        tok[i] = -1;
        if (gathered && row < t.valid) {
          const int v = p.gather_rows[t.tok_row + row];
          if (v >= 0 && v < p.gather_T) tok[i] = v;
          else raise_dev(p.err, MOE_DEV_LAYOUT);
        }
      }
      const int e = max(t.e, 0);
      // gated: the gate+up block of this tile's 128-feature block (swap tiles take
      // 64 of its features); down: the tile(s) of this block of output features
      const int rt0 = kGated ? (kSwap ? t.nt >> 1 : t.nt) : t.nt * (C::kFeatTile / 128);
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        bool waited = mbar_wait(empty(s), ph ^ 1, abort_flag, p.err);
        // the gathering lanes give up together, so each stage they issue gets all its arrivals
        if (kGather) waited = __all_sync(0xffffffffu, waited);
        if (!waited) {
          ok = false;
          break;
        }
        const uint32_t st = stage0 + s * C::kStage, bar = full(s);
        if (kGather) {
          if (gathered) {
            const uint8_t *col = p.gather_x + kb * 128 + c8 * 16;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int r = 4 * i + g4;
              if (tok[i] >= 0) cp_async16(st + r * 128 + ((c8 ^ (r & 7)) << 4), col + (int64_t)tok[i] * p.gather_ld);
            }
          }
          cp_async_arrive(bar);
          if (lane != 0) {
            ++issued;
            if (++s == C::kStages) {
              s = 0;
              ph ^= 1;
            }
            continue;
          }
        }
        mbar_expect_tx(bar, bytes);
        const int kx = kb * 64;
        const uint32_t wdst = kSwap ? st : st + C::kABytes;
        auto wload = [&](uint32_t dst, const uint8_t *src, uint32_t n) { bulk_load(dst, src, n, bar); };
        if (kGated && kSwap) {
          // gate rows [64h, +64) and up rows [128 + 64h, +64) of the 256-row block
          const uint8_t *blk = grouped::weight_block(p, e, rt0, kb, KB, grouped::kPairBytes);
          const int h = t.nt & 1;
          wload(wdst, blk + 8192 * h, 8192);
          wload(wdst + 8192, blk + 16384 + 8192 * h, 8192);
        } else if (kGated) {
          wload(wdst, grouped::weight_block(p, e, rt0, kb, KB, grouped::kPairBytes), grouped::kPairBytes);
        } else {
          wload(wdst, grouped::weight_block(p, e, rt0, kb, KB, grouped::kTileBytes), grouped::kTileBytes);
          if (!kSwap && kBW == 256)
            wload(wdst + grouped::kTileBytes, grouped::weight_block(p, e, rt0 + 1, kb, KB, grouped::kTileBytes),
                  grouped::kTileBytes);
        }
        if (kSwap) {
          for (int i = 0; i < nb; ++i) tma_load_2d(st + C::kABytes + i * 2048, tmt, bar, kx, t.tok_row + 16 * i);
        } else if (!gathered) {
          tma_load_2d(st, tmt, bar, kx, t.tok_row);
        }
        ++issued;
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
    }
    if (kGather) cp_async_wait_all();  // this lane's row copies have landed
    if (*abort_flag) {  // let every copy still in flight land before the CTA exits
      for (int j = issued - 1; j >= 0 && j >= issued - C::kStages; --j)
        mbar_wait_drain(full(j % C::kStages), (uint32_t)((j / C::kStages) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    int s = 0, it = 0;
    uint32_t ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = grouped::decode<C::kTokTile>(p, tile_start, G, NT, tile);
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
        if (kGather) fence_proxy_async();  // rows written by cp.async, read by the MMA
        const uint32_t a = stage0 + s * C::kStage, bb = a + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (kb | kk) != 0;
          mma_bf16(d, sdesc_sw128(a + kk * 32), sdesc_sw128(bb + kk * 32), id, acc);
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
      const Tile t = grouped::decode<C::kTokTile>(p, tile_start, G, NT, tile);
      const int b = it & 1;
      bool waited = mbar_wait(tfull(b), (it >> 1) & 1, abort_flag, p.err);
      if (kCombine) waited = __all_sync(0xffffffffu, waited);  // the warp's lanes stay together
      if (!waited) break;
      fence_after();
      if (t.e < 0 && r == 0) raise_dev(p.err, MOE_DEV_LAYOUT);
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + b * C::kAccCols;
      if (!kSwap) {
        const bool ok = r < t.valid && t.e >= 0;
        uint16_t *orow = out + (int64_t)(t.out_row + (ok ? r : 0)) * p.ld + (int64_t)t.nt * C::kFeatTile;
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
      } else if (!kGated) {
        float v[32];
        tmem_ld32(tb, v);
        tmem_wait_ld();
        if (t.e >= 0) {
          uint16_t *col = out + (int64_t)t.out_row * p.ld + (int64_t)t.nt * C::kFeatTile + r;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < t.valid) col[(int64_t)c * p.ld] = (uint16_t)f2bf(v[c]);
        }
      } else {
        // lanes 0-63: gate of feature r; lanes 64-127: up of feature r - 64
        float v[32];
        tmem_ld32(tb, v);
        tmem_wait_ld();
        fence_before();
        mbar_arrive_relaxed(tempty(b));  // the accumulator is in registers
        const int xb = it & 1, use = it >> 1;
        float *xs = xchg + xb * 64 * 33;
        if (q >= 2) {
          // up lanes: pass the values on once the gate lanes have read the previous use
          if (use > 0 && !mbar_wait(xfree(xb), (use - 1) & 1, abort_flag, p.err)) break;
#pragma unroll
          for (int c = 0; c < 32; ++c) xs[(r - 64) * 33 + c] = v[c];
          mbar_arrive(xfull(xb));
        } else {
          if (!mbar_wait(xfull(xb), use & 1, abort_flag, p.err)) break;
          if (t.e >= 0) {
            uint16_t *col = out + (int64_t)t.out_row * p.ld + (int64_t)t.nt * C::kFeatTile + r;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < t.valid) col[(int64_t)c * p.ld] = (uint16_t)f2bf(silu(v[c]) * xs[r * 33 + c]);
          }
          mbar_arrive(xfree(xb));
        }
        continue;
      }
      fence_before();
      mbar_arrive_relaxed(tempty(b));
      if (kCombine) combine_after_rows<C::kFeatTile>(p, t, r, lane, NT);
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

// The fused combine's counts: each (token, feature block) starts at minus the rows
// the token has (its slots with a row, plus its shared row).  A token with none gets
// out = 0 here, as the separate combine gives it.
__global__ void combine_counts_init(const int32_t *__restrict__ s2r, int T, int k, int N, int with_shared, int NT,
                                    int32_t *__restrict__ counts, uint16_t *__restrict__ out, int64_t d) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    int need = with_shared;
    for (int j = 0; j < k; ++j) {
      const int r = s2r[(int64_t)t * k + j];
      need += (r >= 0 && r < N) ? 1 : 0;
    }
    for (int nt = 0; nt < NT; ++nt) counts[(int64_t)t * NT + nt] = -need;
    if (need == 0)
      for (int64_t c = 0; c < d; c += 8) *reinterpret_cast<uint4 *>(out + (int64_t)t * d + c) = make_uint4(0, 0, 0, 0);
  }
}

template <bool kGated, bool kSwap, int kBW, bool kGather = false, bool kCombine = false>
moe_status_t launch(const Params &p, const CUtensorMap &a, const CUtensorMap &b, cudaStream_t st) {
  using Cf = Cfg<kGated, kSwap, kBW>;
  auto k = grouped_gemm_bf16<kGated, kSwap, kBW, kGather, kCombine>;
  if (cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::kSmem)) != MOE_OK)
    return MOE_ERR_CUDA;
  const int grid = grouped::sm_count();
  if (grid <= 0) return MOE_ERR_CUDA;
  k<<<grid, kThreads, Cf::kSmem, st>>>(p, a, b);
  return launch_status();
}

moe_status_t check_bf16(const FfnArgs &f) {
  const moe_weights_t &w = *f.w;
  if (w.d % 128 || w.I % 128 || f.P > 2048) return MOE_ERR_UNSUPPORTED;
  if (w.E_w * 2 * w.I > INT32_MAX || w.E_w * w.d > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

moe_status_t gate_up_bf16(const FfnArgs &f, cudaStream_t st) {
  moe_status_t s = check_bf16(f);
  if (s != MOE_OK) return s;
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I;
  if (f.N + f.T_shared == 0) return MOE_OK;
  const bool gather = f.gather_rows != nullptr;
  if (gather && (!f.gather_x || f.gather_T < 1 || f.gather_T > INT32_MAX || !aligned(f.gather_x, 16)))
    return MOE_ERR_INVALID_ARG;
  const grouped::Tiles kind = gather ? grouped::Tiles::kWide : grouped::tile_kind(f.N + f.T_shared, f.P);
  if (kind == grouped::Tiles::kPair) return gate_up_bf16_pair(f, st);
  const bool swap = kind == grouped::Tiles::kSwap;
  const uint32_t tok_box = swap ? 16 : 128;
  CUtensorMap m_x, m_sh;
  // gathered: the routed tiles read x by rows and need no map (one over x stands in)
  const void *xsrc = gather ? f.gather_x : f.N > 0 ? f.x_perm : f.shared_x;
  const int64_t xrows = gather ? f.gather_T : f.N > 0 ? f.N : f.T_shared;
  if (!grouped::make_map(&m_x, xsrc, xrows, d, 2, tok_box)) return MOE_ERR_INVALID_ARG;
  if (f.T_shared > 0) {
    if (!grouped::make_map(&m_sh, f.shared_x, f.T_shared, d, 2, tok_box)) return MOE_ERR_INVALID_ARG;
  } else {
    m_sh = m_x;
  }
  if (!aligned(w.w13, 16)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)I;
  p.K = (int)d;
  p.w_rows = (int)(2 * I);
  p.w = static_cast<const uint8_t *>(w.w13);
  p.w_tiles = (int)(I / 128);  // gate+up blocks of 128 features
  p.shared_row0 = 0;
  p.out = f.h;
  p.ld = I;
  if (gather) {
    p.gather_rows = f.gather_rows;
    p.gather_x = static_cast<const uint8_t *>(f.gather_x);
    p.gather_ld = d * 2;
    p.gather_T = (int)f.gather_T;
    return launch<true, false, 128, true>(p, m_x, m_sh, st);
  }
  return swap ? launch<true, true, 128>(p, m_x, m_sh, st) : launch<true, false, 128>(p, m_x, m_sh, st);
}

moe_status_t down_bf16(const FfnArgs &f, cudaStream_t st) {
  moe_status_t s = check_bf16(f);
  if (s != MOE_OK) return s;
  const moe_weights_t &w = *f.w;
  const int64_t d = w.d, I = w.I, rows = f.N + f.T_shared;
  if (rows == 0) return MOE_OK;
  const bool fused = f.c_out != nullptr;
  if (fused && (!f.c_row_to_token || !f.c_slot_to_row || !f.c_topk_w || !f.c_counts || f.c_T < 1 ||
                f.c_T > INT32_MAX / 32 || f.c_k < 1 || f.c_k > 32 || (f.T_shared != 0 && f.T_shared != f.c_T) ||
                !aligned(f.c_out, 16) || !aligned(f.y, 16)))
    return MOE_ERR_INVALID_ARG;
  const grouped::Tiles kind = fused ? grouped::Tiles::kWide : grouped::tile_kind(rows, f.P);
  const int kbw = (d % 256 == 0) ? 256 : 128;
  if (kind == grouped::Tiles::kPair && kbw == 256) return down_bf16_pair(f, st);
  const bool swap = kind == grouped::Tiles::kSwap;
  CUtensorMap m_h;
  if (!grouped::make_map(&m_h, f.h, rows, I, 2, swap ? 16 : 128)) return MOE_ERR_INVALID_ARG;
  if (!aligned(w.w2, 16)) return MOE_ERR_INVALID_ARG;
  Params p = grouped::base_params(f);
  p.feat = (int)d;
  p.K = (int)I;
  p.w_rows = (int)d;
  p.w = static_cast<const uint8_t *>(w.w2);
  p.w_tiles = (int)(d / 128);
  p.shared_row0 = (int)f.N;
  p.out = f.y;
  p.ld = d;
  if (fused) {
    p.c_row_to_token = f.c_row_to_token;
    p.c_slot_to_row = f.c_slot_to_row;
    p.c_topk_w = f.c_topk_w;
    p.c_counts = f.c_counts;
    p.c_out = static_cast<uint16_t *>(f.c_out);
    p.c_k = f.c_k;
    p.c_T = (int)f.c_T;
    p.shared_first = 1;
    const int NTc = (int)(d / kbw);
    const int blocks = (int)((f.c_T + 255) / 256);
    combine_counts_init<<<blocks < 1184 ? blocks : 1184, 256, 0, st>>>(
        f.c_slot_to_row, (int)f.c_T, f.c_k, (int)f.N, f.T_shared > 0 ? 1 : 0, NTc, f.c_counts, p.c_out, d);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    return kbw == 256 ? launch<false, false, 256, false, true>(p, m_h, m_h, st)
                      : launch<false, false, 128, false, true>(p, m_h, m_h, st);
  }
  if (swap) return launch<false, true, 128>(p, m_h, m_h, st);
  return kbw == 256 ? launch<false, false, 256>(p, m_h, m_h, st) : launch<false, false, 128>(p, m_h, m_h, st);
}

}  // namespace moe
