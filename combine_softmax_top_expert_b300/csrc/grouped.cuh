// Tile scheduling and TMA descriptors shared by the grouped expert GEMMs.
//
// A grouped GEMM runs over groups: the P physical experts (rows offs[g] ..
// offs[g+1]-1 of the permuted activations) and, when present, the shared expert
// (T_shared rows).  Each group is cut into token tiles x feature tiles; a table
// of cumulative tile counts, built in shared memory by every CTA from the expert
// offsets, maps a global tile index back to its group.  Persistent CTAs take tiles
// blockIdx.x, blockIdx.x + gridDim.x, ...
#pragma once

#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <utility>

#include "ffn.cuh"
#include "tc.cuh"

namespace moe {
namespace grouped {

constexpr int kMaxGroups = 2048 + 1;

struct Params {
  const int32_t *offs;  // [P + 1]
  const int32_t *p2l;   // [P] or null
  int P, N, T_shared, E_w;
  int feat;             // output features: I (gate/up) or d (down)
  int K;                // reduction length: d (gate/up) or I (down)
  int w_rows;           // weight rows per expert: 2I (gate/up) or d (down)
  int shared_row0;      // row of the shared group's first token in its token map
  void *out;            // h or y
  int64_t ld;           // elements per output row
  int32_t *err;
  // packed weights (see weight_block)
  const uint8_t *w;
  int w_tiles;            // tiles per expert
  // block-scaled e4m3 only
  const float *a_scales;  // [rows, K/128] scales of the token operand
  const float *w_scales;  // [E_w, w_rows/128, K/128]
  float *out_scales;      // gate/up: [rows, I/128] scales of the quantised h
  // gathered token operand (the dispatch permute fused into the bf16 gate/up A-load):
  // routed row r is row gather_rows[r] of gather_x, gather_ld bytes apart
  const int32_t *gather_rows;
  const uint8_t *gather_x;
  int64_t gather_ld;
  int gather_T;  // rows of gather_x
  // the combine fused into the bf16 down epilogue: out[t] = sum_j topk_w[t, j] *
  // y[slot_to_row[t, j]] (+ y[N + t]) for the c_T tokens, each 128/256-feature block
  // summed by the tile that writes its last row (c_counts [c_T, feat / tile
  // features] starts at minus the rows each token has)
  const int32_t *c_row_to_token;
  const int32_t *c_slot_to_row;
  const float *c_topk_w;
  int32_t *c_counts;
  uint16_t *c_out;
  int c_k, c_T;
  int shared_first;  // 1: the shared expert's group is tiled first
};

// Group at position g of the tile order: the routed groups 0..P-1, then the shared
// expert's (P), or with shared_first the shared expert's first.
__device__ __forceinline__ int group_at(const Params &p, int g) {
  if (!p.shared_first || p.T_shared == 0) return g;
  return g == 0 ? p.P : g - 1;
}

struct Tile {
  int e, tok_row, out_row, valid, nt;
  bool shared;
  bool half;  // SM-pair tiles (256 tokens): the group's last tile holds at most 128 rows
};

// The packed weights are tiled: for expert e, tile t and K block kb (128 bytes
// of every row), one contiguous block whose rows are 128 bytes apart with the
// 16-byte chunks of row r permuted by chunk ^ (r % 8) -- the arrangement the
// 128-byte swizzle gives in shared memory -- so one bulk copy moves it straight
// into MMA operand tiles.  W_down^T: 128-row tiles (16 KB blocks).  W_gate^T and
// W_up^T: 256-row tiles holding the gate rows then the up rows of the same 128
// features (32 KB blocks).
constexpr int kTileBytes = 128 * 128;
constexpr int kPairBytes = 2 * kTileBytes;

__device__ __forceinline__ const uint8_t *weight_block(const Params &p, int e, int t, int kb, int KB, int bytes) {
  return p.w + (((int64_t)e * p.w_tiles + t) * KB + kb) * bytes;
}

__device__ __forceinline__ void group_span(const Params &p, int g, int *r0, int *n) {
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

// In-place inclusive scan of a[0..n) by the whole block (blockDim.x <= 1024).
__device__ __forceinline__ void block_scan(int *a, int n) {
  __shared__ int wsum[32];
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

// tile_start[0..G]: cumulative tile counts per group.  Call with all threads.
template <int kTokTile>
__device__ __forceinline__ void build_tile_table(const Params &p, int *tile_start, int G, int NT) {
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int r0, n;
    group_span(p, group_at(p, g), &r0, &n);
    tile_start[g + 1] = n > 0 ? ((n + kTokTile - 1) / kTokTile) * NT : 0;
  }
  if (threadIdx.x == 0) tile_start[0] = 0;
  __syncthreads();
  block_scan(tile_start + 1, G);
}

// The group a thread decoded last: its tile range and what decode reads from global
// memory for it, so the next tile of the same group is decoded from registers.
struct GroupCache {
  int lo = 0, hi = 0;  // tiles [lo, hi); empty until the first decode
  int g, r0, n, e;
};

// kTokTile == 32 (swap): token tiles of one feature block run back to back.
// Otherwise (wide): feature blocks of one token tile run back to back.
template <int kTokTile>
__device__ __forceinline__ Tile decode(const Params &p, const int *tile_start, int G, int NT, int tile,
                                       GroupCache *cache = nullptr) {
  int g, r0, n, e, local;
  if (cache && tile >= cache->lo && tile < cache->hi) {
    g = cache->g, r0 = cache->r0, n = cache->n, e = cache->e;
    local = tile - cache->lo;
  } else {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    g = group_at(p, lo);
    local = tile - tile_start[lo];
    group_span(p, g, &r0, &n);
    e = g >= p.P ? p.E_w - 1 : (p.p2l ? p.p2l[g] : g);
    if (e < 0 || e >= p.E_w) e = -1;
    if (cache) *cache = GroupCache{tile_start[lo], tile_start[lo + 1], g, r0, n, e};
  }
  const int MT = (n + kTokTile - 1) / kTokTile;
  int mt, nt;
  if (kTokTile == 32) {
    nt = local / MT;
    mt = local % MT;
  } else {
    mt = local / NT;
    nt = local % NT;
  }
  Tile t;
  t.shared = g >= p.P;
  t.e = e;
  t.nt = nt;
  t.valid = min(kTokTile, n - mt * kTokTile);
  t.half = kTokTile == 256 && t.valid <= 128;
  t.tok_row = (t.shared ? p.shared_row0 : r0) + mt * kTokTile;
  t.out_row = (t.shared ? p.N : r0) + mt * kTokTile;
  return t;
}

// ------------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
// box_rows x (128 / esize) elements (128 bytes), 128-byte swizzle, zero fill outside.
inline bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, int esize, uint32_t box_rows) {
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

// 2-D map for TMA stores of a row-major [rows, cols] output: boxes of box_rows rows
// x 64 bytes, 64-byte swizzle (16-byte chunk c of box row r at c ^ ((r / 2) % 4)).
inline bool make_store_map(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, int esize, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || rows == 0 || !aligned(base, 16) || (cols * esize) % 16) return false;
  const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {(cuuint32_t)(64 / esize), box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over packed (tiled, already swizzled) weights seen as `rows` rows of 128
// bytes; boxes of box_rows rows copied as they are (no swizzle).  Row
// ((e * w_tiles + t) * KB + kb) * tile_rows + i is row i of weight_block(e, t, kb).
inline bool make_map_tiled(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || rows == 0 || rows > (1ull << 31) || !aligned(base, 16)) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// Launch `kernel` as clusters of two CTAs (the SM-pair tiles), as many pairs as
// the GPU holds at once with `threads` threads and `smem` bytes of dynamic shared
// memory per CTA; *pairs caches that count between calls.
template <typename... KArgs, typename... Args>
moe_status_t launch_pairs(void (*kernel)(KArgs...), int threads, size_t smem, int *pairs, cudaStream_t st,
                          Args &&...args) {
  if (cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != MOE_OK)
    return MOE_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (*pairs <= 0) {
    const int sms = sm_count();
    cfg.gridDim = dim3(2 * (sms > 1 ? sms / 2 : 1));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    *pairs = n;
  }
  cfg.gridDim = dim3(2 * *pairs);
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// Tile orientation: "swap" for few rows per expert, "pair" (two SMs per tile)
// otherwise; "wide" is the one-SM form of pair.  The environment variable
// MOE_B300_FFN_TILES=swap|wide|pair overrides the choice.
enum class Tiles { kSwap, kWide, kPair };
inline Tiles tile_kind(int64_t N, int64_t P) {
  const char *env = std::getenv("MOE_B300_FFN_TILES");
  if (env && !std::strcmp(env, "swap")) return Tiles::kSwap;
  if (env && !std::strcmp(env, "wide")) return Tiles::kWide;
  if (env && !std::strcmp(env, "pair")) return Tiles::kPair;
  return N < 64 * P ? Tiles::kSwap : Tiles::kPair;
}

inline Params base_params(const FfnArgs &f) {
  Params p{};
  p.offs = f.offs;
  p.p2l = f.p2l;
  p.P = (int)f.P;
  p.N = (int)f.N;
  p.T_shared = (int)f.T_shared;
  p.E_w = (int)f.w->E_w;
  p.err = f.err;
  return p;
}

}  // namespace grouped
}  // namespace moe
