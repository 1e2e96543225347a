// Dispatch layout and EPLB map.
//
// Layout ("6.4 Data parallelism and expert parallelism", section 3.1 step 2 and
// its figure; section 5.1 busiest card / average): a stable, atomic-free counting
// sort of the N = T*k slots by physical expert, in three launches (one, by
// route_layout_small_kernel below, when the slots fit a single count chunk).
//
//   count   one CTA per chunk of 2048 consecutive slots (slot s = t*k + j); each
//           warp takes 256 slots in batches of 32.  __match_any_sync groups the
//           lanes of a batch that share an expert; a lane's rank is the number of
//           lower lanes in its group plus the warp's running count, so ranks follow
//           slot order.  Slots of one expert come from distinct tokens, so slot
//           order is token order.  A scan over the 8 warps turns warp ranks into
//           chunk ranks; the chunk histogram goes to hist[chunk][P].
//   scan    one CTA: column scans of hist give each chunk's base per expert and
//           the expert counts; a block scan gives the expert offsets; rank counts,
//           rank offsets and the load statistics follow.
//   scatter row = offset[p] + chunk base[p] + chunk rank; slot_to_row, row_to_token.
//
// EPLB map ("6.4 ...", section 5.3; "How Expert Parallelism Works for
// Mixture-of-Experts Models in vLLM", "MoE Layer Construction"): one CTA ranks the
// experts by (count desc, index asc) and writes the physical tables.  The base
// slots follow the placement strategy ("How Expert Parallelism Works ...",
// "Configuring Expert Parallelism", linear or round_robin): linear puts logical
// expert e on rank e / (E/R), round-robin on rank e % R, in local slot e % (E/R)
// or e / R.
#include "route.cuh"

namespace moe {
namespace {

constexpr int kChunk = 2048;        // slots per CTA in the count pass
constexpr int kCountWarps = 8;      // 8 warps x 256 slots
constexpr int kSlotsPerWarp = kChunk / kCountWarps;
constexpr int kMaxP = 2048;

struct PhysMap {
  int E;
  int k;
  const int32_t *replica_count;    // null: identity map
  const int32_t *logical_to_phys;  // [E, stride]
  int stride;
};

__device__ __forceinline__ int phys_of(const int32_t *ids, int64_t s, const PhysMap &m, int32_t *err) {
  const int e = ids[s];
  if (e < 0 || e >= m.E) {
    raise_dev(err, MOE_DEV_ID_RANGE);
    return -1;
  }
  if (!m.replica_count) return e;
  const int64_t t = s / m.k;
  const int rc = m.replica_count[e];
  return m.logical_to_phys[m.stride * e + (int)(t % rc)];
}

// One warp's pass over its slots base .. base + kSlotsPerWarp - 1 (in batches of 32):
// phys[b] is the physical expert of the lane's slot in batch b (-1 outside [0, N) or
// for a bad id) and rank[b] its rank among this warp's earlier slots of that expert;
// wc[P] holds the warp's running counts.
__device__ __forceinline__ void count_warp(const int32_t *ids, int64_t N, int64_t base, const PhysMap &m,
                                           int32_t *wc, int32_t *err, int (&rank)[kSlotsPerWarp / 32],
                                           int (&phys)[kSlotsPerWarp / 32]) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int b = 0; b < kSlotsPerWarp / 32; ++b) {
    const int64_t s = base + b * 32 + lane;
    const int p = s < N ? phys_of(ids, s, m, err) : -1;
    const unsigned peers = __match_any_sync(kFull, p);
    int r = -1;
    if (p >= 0) r = wc[p] + __popc(peers & lt);
    __syncwarp();
    if (p >= 0 && lane == __ffs(peers) - 1) wc[p] += __popc(peers);
    __syncwarp();
    rank[b] = r;
    phys[b] = p;
  }
}

__global__ void __launch_bounds__(256) layout_count_kernel(const int32_t *__restrict__ ids, int64_t N, int P,
                                                           PhysMap m, int32_t *__restrict__ hist,
                                                           int32_t *__restrict__ chunk_rank, int32_t *err) {
  extern __shared__ int32_t cnt[];  // [kCountWarps][P]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kCountWarps * P; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kChunk + warp * kSlotsPerWarp;
  int32_t *wc = cnt + warp * P;
  int rank[kSlotsPerWarp / 32];
  int phys[kSlotsPerWarp / 32];
  count_warp(ids, N, base, m, wc, err, rank, phys);
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kCountWarps; ++w) {
      const int v = cnt[w * P + p];
      cnt[w * P + p] = run;
      run += v;
    }
    hist[(int64_t)blockIdx.x * P + p] = run;
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < kSlotsPerWarp / 32; ++b) {
    const int64_t s = base + b * 32 + lane;
    if (s < N) chunk_rank[s] = phys[b] >= 0 ? wc[phys[b]] + rank[b] : -1;
  }
}

struct StatsOut {
  moe_load_stats_t *stats;  // [2]
};

// Warp-level statistics of `counts` [n] grouped into R ranks of n/R entries: rank r
// holds entries r*(n/R) .. (linear) or r, r + R, r + 2R, .. (round-robin).
__device__ void warp_stats(const int32_t *counts, int n, int R, int64_t total, bool round_robin,
                           moe_load_stats_t *out) {
  const int lane = threadIdx.x & 31;
  const int per = n / R;
  int max_rank = 0, max_exp = 0, active = 0;
  for (int r = lane; r < R; r += 32) {
    int s = 0;
    for (int i = 0; i < per; ++i) s += counts[round_robin ? r + i * R : r * per + i];
    max_rank = max(max_rank, s);
  }
  for (int i = lane; i < n; i += 32) {
    max_exp = max(max_exp, counts[i]);
    active += counts[i] > 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    max_rank = max(max_rank, __shfl_xor_sync(kFull, max_rank, o));
    max_exp = max(max_exp, __shfl_xor_sync(kFull, max_exp, o));
    active += __shfl_xor_sync(kFull, active, o);
  }
  if (lane == 0) {
    moe_load_stats_t st;
    st.max_rank = max_rank;
    st.max_expert = max_exp;
    st.n_active_experts = active;
    st.pad_ = 0;
    st.mean_rank = (float)((double)total / (double)R);
    st.max_over_mean = st.mean_rank > 0.f ? (float)((double)max_rank * R / (double)total) : 0.f;
    st.balancedness = max_rank > 0 ? (float)((double)total / ((double)R * max_rank)) : 0.f;
    st.pad2_ = 0.f;
    *out = st;
  }
}

// The rest of the layout statistics from the physical counts cnt[P] (shared
// memory; a block of 1024 threads): logical counts through p2l, the exclusive scan
// into phys_offsets, rank counts and offsets (P/R physical experts per rank), and
// the before/after load statistics.  lcnt [E], warp_sums [32] and rcnt [R] are
// shared scratch.
__device__ void scan_finish(const int32_t *cnt, int32_t *lcnt, int32_t *warp_sums, int32_t *rcnt, int P, int E,
                            int R, int64_t N, const int32_t *p2l, bool base_rr, int32_t *logical_counts,
                            int32_t *phys_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                            moe_load_stats_t *stats) {
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) lcnt[e] = 0;
  __syncthreads();
  // logical counts: physical counts folded through phys_to_logical (integer adds)
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = p2l ? p2l[p] : p;
    if (e >= 0 && e < E) atomicAdd(&lcnt[e], cnt[p]);
  }
  // exclusive scan of cnt[0..P) -> offsets; each thread owns two consecutive entries
  const int a = 2 * tid < P ? cnt[2 * tid] : 0;
  const int b = 2 * tid + 1 < P ? cnt[2 * tid + 1] : 0;
  int v = a + b;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, ws, o);
      if (lane >= o) ws += n;
    }
    warp_sums[lane] = ws;
  }
  __syncthreads();
  const int excl = v - (a + b) + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (2 * tid < P) phys_offsets[2 * tid] = excl;
  if (2 * tid + 1 < P) phys_offsets[2 * tid + 1] = excl + a;
  if (tid == 0) phys_offsets[P] = warp_sums[31];
  // rank counts / offsets (linear placement, P/R physical experts per rank)
  const int per = P / R;
  for (int r = tid; r < R; r += blockDim.x) {
    int s = 0;
    for (int i = 0; i < per; ++i) s += cnt[r * per + i];
    rcnt[r] = s;
    rank_counts[r] = s;
  }
  for (int e = tid; e < E; e += blockDim.x) logical_counts[e] = lcnt[e];
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int r0 = 0; r0 < R; r0 += 32) {
      const int r = r0 + lane;
      int x = r < R ? rcnt[r] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += n;
      }
      if (r < R) rank_offsets[r] = run + x - rcnt[r];
      run += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) rank_offsets[R] = run;
  }
  if (stats) {
    // before: the logical experts in their base placement; after: the physical ones
    if (warp == 1) warp_stats(lcnt, E, R, N, base_rr, &stats[0]);
    if (warp == 2) warp_stats(cnt, P, R, N, false, &stats[1]);
  }
}

__global__ void __launch_bounds__(1024) layout_scan_kernel(int32_t *__restrict__ hist, int chunks, int P, int E,
                                                           int R, int64_t N, const int32_t *p2l, bool base_rr,
                                                           int32_t *logical_counts, int32_t *phys_counts,
                                                           int32_t *phys_offsets, int32_t *rank_counts,
                                                           int32_t *rank_offsets, moe_load_stats_t *stats) {
  __shared__ int32_t cnt[kMaxP];
  __shared__ int32_t lcnt[1024];
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t rcnt[kMaxP];
  const int tid = threadIdx.x;
  for (int p = tid; p < P; p += blockDim.x) {
    int run = 0;
    for (int c = 0; c < chunks; ++c) {
      const int v = hist[(int64_t)c * P + p];
      hist[(int64_t)c * P + p] = run;
      run += v;
    }
    cnt[p] = run;
    phys_counts[p] = run;
  }
  scan_finish(cnt, lcnt, warp_sums, rcnt, P, E, R, N, p2l, base_rr, logical_counts, phys_offsets, rank_counts,
              rank_offsets, stats);
}

__global__ void __launch_bounds__(256) layout_scatter_kernel(const int32_t *__restrict__ ids, int64_t N, int P,
                                                             PhysMap m, const int32_t *__restrict__ hist,
                                                             const int32_t *__restrict__ chunk_rank,
                                                             const int32_t *__restrict__ phys_offsets,
                                                             int32_t *__restrict__ row_to_token,
                                                             int32_t *__restrict__ slot_to_row) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= N) return;
  const int r = chunk_rank[s];
  if (r < 0) {
    slot_to_row[s] = -1;
    return;
  }
  const int p = phys_of(ids, s, m, nullptr);
  const int row = phys_offsets[p] + hist[(s / kChunk) * P + p] + r;
  slot_to_row[s] = row;
  row_to_token[row] = (int32_t)(s / m.k);
}

// counts may be null when n_red == 0 (no hot list to rank).
// Route + layout of a small batch (N = T*k <= kChunk slots, P <= kSmallP) in one
// CTA of 1024 threads: each warp routes tokens warp, warp + 32, ... (route.cuh) and
// keeps the ids in shared memory; warps 0-7 rank the slots as the count kernel
// does for its one chunk; scan_finish writes the offsets and statistics; warps 0-7
// scatter.  The results are those of route_kernel followed by the three layout
// kernels, for a batch that would occupy one count chunk anyway, in one launch.
// Each warp routes its tokens one after another, so the launch saved only pays
// while that chain is short: it is used when ceil(T/32) * k * ceil(E/32) <= 16
// (measured on the B300: a 64-token, 8-expert, top-2 batch went from 89 to 76 us
// per layer; the decode batch, 128 tokens over 256 experts, top-8, took 47 us in
// this kernel against 26 us in the four separate ones).
constexpr int kSmallP = 512;
constexpr int kSmallRouteWork = 16;

// kRoute false: the layout alone, from ids already in global memory (a batch of one
// count chunk laid out in one launch instead of three).
template <int VPL, bool kRoute>
__global__ void __launch_bounds__(1024) route_layout_small_kernel(
    const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k, int R, int P, PhysMap m,
    const int32_t *p2l, bool base_rr, int32_t *__restrict__ ids, float *__restrict__ w, int32_t *logical_counts,
    int32_t *phys_counts, int32_t *phys_offsets, int32_t *rank_counts, int32_t *rank_offsets,
    int32_t *__restrict__ row_to_token, int32_t *__restrict__ slot_to_row, moe_load_stats_t *stats, int32_t *err) {
  __shared__ int32_t sids[kChunk];
  __shared__ int32_t cnt[kCountWarps * kSmallP];  // per-warp counts, then per-warp bases
  __shared__ int32_t tot[kSmallP];
  __shared__ int32_t lcnt[1024];
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t rcnt[kSmallP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t N = (int64_t)T * k;
  if (kRoute) {
    for (int t = warp; t < T; t += 32) {
      int pick;
      float wt;
      rt::route_token<VPL>(logits + (int64_t)t * E, bias, E, k, err, pick, wt);
      if (lane < k) {
        ids[t * k + lane] = pick;
        w[t * k + lane] = wt;
        sids[t * k + lane] = pick;
      }
    }
  } else {
    for (int s = threadIdx.x; s < N; s += blockDim.x) sids[s] = ids[s];
  }
  for (int i = threadIdx.x; i < kCountWarps * P; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  int rank[kSlotsPerWarp / 32];
  int phys[kSlotsPerWarp / 32];
  if (warp < kCountWarps) count_warp(sids, N, (int64_t)warp * kSlotsPerWarp, m, cnt + warp * P, err, rank, phys);
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w2 = 0; w2 < kCountWarps; ++w2) {
      const int v = cnt[w2 * P + p];
      cnt[w2 * P + p] = run;
      run += v;
    }
    tot[p] = run;
    phys_counts[p] = run;
  }
  scan_finish(tot, lcnt, warp_sums, rcnt, P, E, R, N, p2l, base_rr, logical_counts, phys_offsets, rank_counts,
              rank_offsets, stats);
  __syncthreads();  // phys_offsets (global, this block's writes) and the warp bases are visible
  if (warp < kCountWarps) {
#pragma unroll
    for (int b = 0; b < kSlotsPerWarp / 32; ++b) {
      const int64_t s = (int64_t)warp * kSlotsPerWarp + b * 32 + lane;
      if (s >= N) continue;
      if (phys[b] < 0) {
        slot_to_row[s] = -1;
        continue;
      }
      const int row = phys_offsets[phys[b]] + cnt[warp * P + phys[b]] + rank[b];
      slot_to_row[s] = row;
      row_to_token[row] = (int32_t)(s / k);
    }
  }
}

__global__ void __launch_bounds__(1024) eplb_map_kernel(const int32_t *__restrict__ counts, int E, int R, int n_red,
                                                        bool round_robin, int32_t *phys_to_logical,
                                                        int32_t *phys_rank, int32_t *replica_count,
                                                        int32_t *logical_to_phys) {
  __shared__ int32_t c[1024];
  if (n_red > 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) c[e] = counts[e];
  __syncthreads();
  const int base = E / R, S = (E + n_red) / R;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int rank = n_red;  // position in the hot list; n_red = not hot
    if (n_red > 0) {
      const int ce = c[e];
      rank = 0;
      for (int f = 0; f < E; ++f) rank += (c[f] > ce) || (c[f] == ce && f < e);
    }
    const int home = round_robin ? e % R : e / base, slot0 = round_robin ? e / R : e % base;
    const int pr = home * S + slot0;
    phys_to_logical[pr] = e;
    phys_rank[pr] = home;
    logical_to_phys[2 * e] = pr;
    if (rank < n_red) {
      const int r = rank % R, slot = base + rank / R;
      const int pp = r * S + slot;
      phys_to_logical[pp] = e;
      phys_rank[pp] = r;
      logical_to_phys[2 * e + 1] = pp;
      replica_count[e] = 2;
    } else {
      logical_to_phys[2 * e + 1] = -1;
      replica_count[e] = 1;
    }
  }
}

// The page's load-aware placement ("6.4 ...", section 5.2) as a physical-expert map.
// One CTA of 1024 threads; E <= 1024, P = E + n_red <= 2048, R <= 1024.
// Loads per replica are count / replicas, the correctly rounded fp64 quotients the
// page's procedure compares; the redundant slots are handed out by comparing them.
// Ordering the replicas uses exact cross-multiplication, a/b > c/d <=> a*d > c*b:
// with counts below 2^31 and at most 1025 replicas two different quotients differ
// by at least 1/1025^2, more than an fp64 ulp of any of them, so the fp64 quotients
// are ordered the same way (and equal only when exactly equal).  The per-rank loads
// are summed in fp64 in the procedure's order, so the map and the loads are exactly
// the ones it gives.
__device__ __forceinline__ bool heavier(int64_t ca, int ra, int ia, int64_t cb, int rb, int ib) {
  const int64_t l = ca * rb, r = cb * ra;
  return l > r || (l == r && ia < ib);
}

// Warp-wide argmin of 64-bit keys held one per lane, the lowest `id` on ties; lanes
// without a candidate pass key = ~0.  Three 32-bit warp reductions.
__device__ __forceinline__ int warp_argmin64(uint64_t key, int id) {
  const uint32_t hi = (uint32_t)(key >> 32), lo = (uint32_t)key;
  const uint32_t mh = __reduce_min_sync(kFull, hi);
  const uint32_t ml = __reduce_min_sync(kFull, hi == mh ? lo : ~0u);
  return (int)__reduce_min_sync(kFull, hi == mh && lo == ml ? (uint32_t)id : ~0u);
}

__global__ void __launch_bounds__(1024) eplb_balanced_kernel(const int32_t *__restrict__ counts, int E, int R,
                                                             int n_red, int32_t *phys_to_logical, int32_t *phys_rank,
                                                             int32_t *replica_count, int32_t *logical_to_phys,
                                                             int stride, double *rank_load) {
  __shared__ int32_t cnt[1024], rep[1024];
  __shared__ double per[1024];              // load of one replica of expert e
  __shared__ int16_t oe[kMaxP], oj[kMaxP];  // replicas in placement order: expert, replica index
  __shared__ double load[1024];             // per rank
  __shared__ int32_t used[1024];            // slots taken per rank
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = E + n_red, S = P / R;
  for (int e = tid; e < E; e += blockDim.x) {
    cnt[e] = counts[e];
    rep[e] = 1;
    per[e] = (double)counts[e];
  }
  for (int r = tid; r < R; r += blockDim.x) {
    load[r] = 0.0;
    used[r] = 0;
  }
  for (int i = tid; i < E * stride; i += blockDim.x) logical_to_phys[i] = -1;
  __syncthreads();
  // 1. each redundant slot to the expert with the highest load per replica (lowest
  // index on a tie).  One warp: lane l keeps the best of experts l, l + 32, ... (the
  // float64 loads count / replicas, whose bit patterns order as the values do), a
  // warp reduction picks the winner, and only the winner's lane looks again.
  if (warp == 0) {
    auto lane_best = [&](uint64_t *key, int *id) {
      *key = ~0ull;
      *id = -1;
      for (int e = lane; e < E; e += 32) {
        const uint64_t k = ~(uint64_t)__double_as_longlong(per[e]);  // larger load -> smaller key
        if (*id < 0 || k < *key) {
          *key = k;
          *id = e;
        }
      }
    };
    uint64_t key;
    int id;
    lane_best(&key, &id);
    for (int it = 0; it < n_red; ++it) {
      const int bi = warp_argmin64(key, id < 0 ? 0x7fffffff : id);
      if ((bi & 31) == lane) {
        rep[bi] += 1;
        per[bi] = (double)cnt[bi] / (double)rep[bi];
        lane_best(&key, &id);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // 2. replicas heaviest first; equal loads keep expert order, then replica order.
  // per[e] now holds count / replicas of every expert; G consecutive threads count the
  // replicas heavier than expert e's over interleaved parts of the experts.
  {
    const int G = E <= 256 ? 4 : (E <= 512 ? 2 : 1);  // threads per expert (1024 threads)
    const int e = tid / G, part = tid % G;
    int pos = 0;
    int64_t ce = 0;
    int re = 0;
    if (e < E) {
      ce = cnt[e];
      re = rep[e];
      for (int f = part; f < E; f += G) pos += heavier(cnt[f], rep[f], f, ce, re, e) ? rep[f] : 0;
    }
    for (int o = 1; o < G; o <<= 1) pos += __shfl_xor_sync(kFull, pos, o);
    if (e < E && part == 0) {
      for (int j = 0; j < re; ++j) {
        oe[pos + j] = (int16_t)e;
        oj[pos + j] = (int16_t)j;
      }
      replica_count[e] = re;
    }
  }
  __syncthreads();
  // 3. each replica onto the lightest rank with a free slot (lowest rank on a tie).
  // One warp.  With R <= 32 lane r holds rank r's load and used slots in registers; a
  // warp reduction over the loads' bit patterns (non-negative doubles order like their
  // bits) picks the rank and its lane adds the replica's load.
  if (warp == 0 && R <= 32) {
    double my_load = 0.0;
    int my_used = 0;
    int e_n = oe[0], j_n = oj[0];
    double q_n = per[e_n];
    for (int p = 0; p < P; ++p) {
      const int e = e_n, j = j_n;
      const double q = q_n;
      if (p + 1 < P) {  // the next replica's expert, index and load, read ahead
        e_n = oe[p + 1];
        j_n = oj[p + 1];
        q_n = per[e_n];
      }
      const uint64_t key = lane < R && my_used < S ? (uint64_t)__double_as_longlong(my_load) : ~0ull;
      const int g = warp_argmin64(key, lane);
      if (g == lane) {
        const int pid = g * S + my_used;
        my_load += q;
        my_used += 1;
        phys_to_logical[pid] = e;
        phys_rank[pid] = g;
        logical_to_phys[stride * e + j] = pid;
      }
      __syncwarp();
    }
    if (lane < R) load[lane] = my_load;
  } else if (warp == 0) {
    // more ranks than lanes: lane l keeps the lightest of ranks l, l + 32, ... with a
    // free slot, and only the winning rank's lane updates it and looks again
    auto lane_best = [&](uint64_t *key, int *id) {
      *key = ~0ull;
      *id = -1;
      for (int r = lane; r < R; r += 32) {
        const uint64_t k = (uint64_t)__double_as_longlong(load[r]);
        if (used[r] < S && (*id < 0 || k < *key)) {
          *key = k;
          *id = r;
        }
      }
    };
    uint64_t key;
    int id;
    lane_best(&key, &id);
    int e_next = oe[0], j_next = oj[0];
    for (int p = 0; p < P; ++p) {
      const int e = e_next, j = j_next;
      if (p + 1 < P) {
        e_next = oe[p + 1];
        j_next = oj[p + 1];
      }
      const int g = warp_argmin64(key, id < 0 ? 0x7fffffff : id);
      if ((g & 31) == lane) {
        const int pid = g * S + used[g];
        load[g] += per[e];
        used[g] += 1;
        phys_to_logical[pid] = e;
        phys_rank[pid] = g;
        logical_to_phys[stride * e + j] = pid;
        lane_best(&key, &id);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (rank_load)
    for (int r = tid; r < R; r += blockDim.x) rank_load[r] = load[r];
}

// Sliding window of per-step logical expert counts ("6.4 ...", section 5.3: load
// is averaged over window_size recent steps).  Thread e owns column e of the ring.
__global__ void __launch_bounds__(256) eplb_window_kernel(const int32_t *__restrict__ counts, int32_t *ring,
                                                          int64_t W, int E, int64_t step, int32_t *window_sum) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  ring[(step % W) * E + e] = counts[e];
  int64_t sum = 0;
  for (int64_t w = 0; w < W; ++w) sum += ring[w * E + e];
  window_sum[e] = (int32_t)min(sum, (int64_t)INT32_MAX);
}

}  // namespace

size_t dispatch_ws_bytes(int64_t T, int32_t k, int64_t P) {
  const int64_t N = T * k;
  const int64_t chunks = (N + kChunk - 1) / kChunk;
  return align_up((size_t)(chunks * P) * 4, 256) + align_up((size_t)N * 4, 256);
}

// The size checks of a dispatch layout, before anything is computed from the sizes
// (T * k is formed only once it cannot overflow).
moe_status_t dispatch_shape_status(int64_t T, int32_t k, int64_t E, int32_t R, const moe_eplb_t *eplb) {
  const int64_t P = eplb ? eplb->P : E;
  if (T < 0 || k < 1 || E < 1 || E > 1024 || R < 1 || P < E || P > kMaxP || P % R || E % R)
    return MOE_ERR_INVALID_ARG;
  if (eplb && eplb->base_placement != 0 && eplb->base_placement != 1) return MOE_ERR_INVALID_ARG;
  if (T > (INT32_MAX / 2) / k) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t dispatch_layout(const int32_t *topk_ids, int64_t T, int32_t k, int64_t E, int32_t R,
                             const moe_eplb_t *eplb, int32_t *logical_counts, int32_t *phys_counts,
                             int32_t *phys_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                             int32_t *row_to_token, int32_t *slot_to_row, moe_load_stats_t *stats, void *ws,
                             size_t ws_bytes, int32_t *err, cudaStream_t st) {
  const moe_status_t shape = dispatch_shape_status(T, k, E, R, eplb);
  if (shape != MOE_OK) return shape;
  const int64_t P = eplb ? eplb->P : E;
  if (!logical_counts || !phys_counts || !phys_offsets || !rank_counts || !rank_offsets)
    return MOE_ERR_INVALID_ARG;
  if (eplb && (!eplb->phys_to_logical || !eplb->replica_count || !eplb->logical_to_phys))
    return MOE_ERR_INVALID_ARG;
  const int64_t N = T * k;
  if (N > 0 && (!topk_ids || !row_to_token || !slot_to_row)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < dispatch_ws_bytes(T, k, P) || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  const int chunks = (int)((N + kChunk - 1) / kChunk);
  int32_t *hist = static_cast<int32_t *>(ws);
  int32_t *chunk_rank = reinterpret_cast<int32_t *>(static_cast<char *>(ws) +
                                                    align_up((size_t)chunks * P * 4, 256));
  PhysMap m{(int)E, k, eplb ? eplb->replica_count : nullptr, eplb ? eplb->logical_to_phys : nullptr,
            eplb && eplb->max_replicas > 0 ? eplb->max_replicas : 2};
  if (N > 0 && N <= kChunk && P <= kSmallP) {  // one chunk: count, scan and scatter in one launch
    route_layout_small_kernel<1, false><<<1, 1024, 0, st>>>(
        nullptr, nullptr, (int)T, (int)E, k, R, (int)P, m, eplb ? eplb->phys_to_logical : nullptr,
        eplb != nullptr && eplb->base_placement == 1, const_cast<int32_t *>(topk_ids), nullptr, logical_counts,
        phys_counts, phys_offsets, rank_counts, rank_offsets, row_to_token, slot_to_row, stats, err);
    return launch_status();
  }
  if (chunks > 0) {
    const size_t smem = (size_t)kCountWarps * P * 4;
    if (smem > 48 * 1024) {
      if (cuda_status(cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
          MOE_OK)
        return MOE_ERR_CUDA;
    }
    layout_count_kernel<<<chunks, 256, smem, st>>>(topk_ids, N, (int)P, m, hist, chunk_rank, err);
  }
  layout_scan_kernel<<<1, 1024, 0, st>>>(hist, chunks, (int)P, (int)E, R, N,
                                         eplb ? eplb->phys_to_logical : nullptr,
                                         eplb != nullptr && eplb->base_placement == 1, logical_counts, phys_counts,
                                         phys_offsets, rank_counts, rank_offsets, stats);
  if (N > 0)
    layout_scatter_kernel<<<(unsigned)((N + 255) / 256), 256, 0, st>>>(topk_ids, N, (int)P, m, hist, chunk_rank,
                                                                       phys_offsets, row_to_token, slot_to_row);
  return launch_status();
}

// Route and layout in one launch for a small batch (see route_layout_small_kernel;
// returns MOE_ERR_UNSUPPORTED otherwise: the caller runs the separate steps).
moe_status_t route_layout_small(const float *logits, const float *bias, int64_t T, int64_t E, int32_t k, int32_t R,
                                const moe_eplb_t *eplb, int32_t *ids, float *w, int32_t *logical_counts,
                                int32_t *phys_counts, int32_t *phys_offsets, int32_t *rank_counts,
                                int32_t *rank_offsets, int32_t *row_to_token, int32_t *slot_to_row,
                                moe_load_stats_t *stats, int32_t *err, cudaStream_t st) {
  const int64_t P = eplb ? eplb->P : E;
  if (T < 1 || k < 1 || k > 32 || E < 1 || E > 1024 || k > E || R < 1 || P < E || P % R || E % R)
    return MOE_ERR_INVALID_ARG;
  if (T * k > kChunk || P > kSmallP || (T + 31) / 32 * k * ((E + 31) / 32) > kSmallRouteWork)
    return MOE_ERR_UNSUPPORTED;
  if (!logits || !ids || !w || !logical_counts || !phys_counts || !phys_offsets || !rank_counts || !rank_offsets ||
      !row_to_token || !slot_to_row)
    return MOE_ERR_INVALID_ARG;
  if (eplb && (!eplb->phys_to_logical || !eplb->replica_count || !eplb->logical_to_phys)) return MOE_ERR_INVALID_ARG;
  if (eplb && eplb->base_placement != 0 && eplb->base_placement != 1) return MOE_ERR_INVALID_ARG;
  PhysMap m{(int)E, k, eplb ? eplb->replica_count : nullptr, eplb ? eplb->logical_to_phys : nullptr,
            eplb && eplb->max_replicas > 0 ? eplb->max_replicas : 2};
  const int32_t *p2l = eplb ? eplb->phys_to_logical : nullptr;
  const bool rr = eplb != nullptr && eplb->base_placement == 1;
  rt::with_vpl((int)E, [&](auto vpl) {
    route_layout_small_kernel<decltype(vpl)::value, true><<<1, 1024, 0, st>>>(
        logits, bias, (int)T, (int)E, k, R, (int)P, m, p2l, rr, ids, w, logical_counts, phys_counts, phys_offsets,
        rank_counts, rank_offsets, row_to_token, slot_to_row, stats, err);
  });
  return launch_status();
}

moe_status_t placement_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_red, int32_t placement,
                           int32_t *phys_to_logical, int32_t *phys_rank, int32_t *replica_count,
                           int32_t *logical_to_phys, cudaStream_t st) {
  if (E < 1 || E > 1024 || R < 1 || E % R || n_red < 0 || n_red % R || n_red > E) return MOE_ERR_INVALID_ARG;
  if (placement != 0 && placement != 1) return MOE_ERR_INVALID_ARG;
  if ((n_red > 0 && !logical_counts) || !phys_to_logical || !phys_rank || !replica_count || !logical_to_phys)
    return MOE_ERR_INVALID_ARG;
  eplb_map_kernel<<<1, 1024, 0, st>>>(logical_counts, (int)E, R, n_red, placement == 1, phys_to_logical, phys_rank,
                                      replica_count, logical_to_phys);
  return launch_status();
}

moe_status_t eplb_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_red, int32_t *phys_to_logical,
                      int32_t *phys_rank, int32_t *replica_count, int32_t *logical_to_phys, cudaStream_t st) {
  if (!logical_counts) return MOE_ERR_INVALID_ARG;
  return placement_map(logical_counts, E, R, n_red, 0, phys_to_logical, phys_rank, replica_count, logical_to_phys,
                       st);
}

moe_status_t eplb_balanced_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_red,
                               int32_t *phys_to_logical, int32_t *phys_rank, int32_t *replica_count,
                               int32_t *logical_to_phys, double *rank_load, cudaStream_t st) {
  if (E < 1 || E > 1024 || R < 1 || R > 1024 || n_red < 0 || E + n_red > kMaxP || (E + n_red) % R)
    return MOE_ERR_INVALID_ARG;
  if (!logical_counts || !phys_to_logical || !phys_rank || !replica_count || !logical_to_phys)
    return MOE_ERR_INVALID_ARG;
  eplb_balanced_kernel<<<1, 1024, 0, st>>>(logical_counts, (int)E, R, n_red, phys_to_logical, phys_rank,
                                           replica_count, logical_to_phys, 1 + n_red, rank_load);
  return launch_status();
}

}  // namespace moe

MOE_API size_t moe_dispatch_workspace_size(int64_t T, int32_t k, int64_t P) {
  if (T < 0 || k < 1 || P < 1 || T > (INT32_MAX / 2) / k) return 0;
  return moe::dispatch_ws_bytes(T, k, P);
}

MOE_API moe_status_t moe_dispatch_layout(const int32_t *topk_ids, int64_t T, int32_t k, int64_t E, int32_t R,
                                         const moe_eplb_t *eplb, int32_t *logical_counts, int32_t *phys_counts,
                                         int32_t *phys_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                                         int32_t *row_to_token, int32_t *slot_to_row, moe_load_stats_t *stats,
                                         void *ws, size_t ws_bytes, int32_t *err, moe_stream_t stream) {
  return moe::dispatch_layout(topk_ids, T, k, E, R, eplb, logical_counts, phys_counts, phys_offsets, rank_counts,
                              rank_offsets, row_to_token, slot_to_row, stats, ws, ws_bytes, err,
                              moe::as_cuda(stream));
}

MOE_API moe_status_t moe_eplb_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_redundant,
                                  int32_t *phys_to_logical, int32_t *phys_rank, int32_t *replica_count,
                                  int32_t *logical_to_phys, moe_stream_t stream) {
  return moe::eplb_map(logical_counts, E, R, n_redundant, phys_to_logical, phys_rank, replica_count,
                       logical_to_phys, moe::as_cuda(stream));
}

MOE_API moe_status_t moe_placement_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_redundant,
                                       int32_t placement, int32_t *phys_to_logical, int32_t *phys_rank,
                                       int32_t *replica_count, int32_t *logical_to_phys, moe_stream_t stream) {
  return moe::placement_map(logical_counts, E, R, n_redundant, placement, phys_to_logical, phys_rank, replica_count,
                            logical_to_phys, moe::as_cuda(stream));
}

MOE_API moe_status_t moe_eplb_balanced_map(const int32_t *logical_counts, int64_t E, int32_t R, int32_t n_redundant,
                                           int32_t *phys_to_logical, int32_t *phys_rank, int32_t *replica_count,
                                           int32_t *logical_to_phys, double *rank_load, moe_stream_t stream) {
  return moe::eplb_balanced_map(logical_counts, E, R, n_redundant, phys_to_logical, phys_rank, replica_count,
                                logical_to_phys, rank_load, moe::as_cuda(stream));
}

MOE_API moe_status_t moe_eplb_window_update(const int32_t *logical_counts, int32_t *window, int64_t W, int64_t E,
                                            int64_t step, int32_t *window_sum, moe_stream_t stream) {
  if (W < 1 || W > (1 << 20) || E < 1 || E > 1024 || step < 0) return MOE_ERR_INVALID_ARG;
  if (!logical_counts || !window || !window_sum) return MOE_ERR_INVALID_ARG;
  moe::eplb_window_kernel<<<(unsigned)((E + 255) / 256), 256, 0, moe::as_cuda(stream)>>>(
      logical_counts, window, W, (int)E, step, window_sum);
  return moe::launch_status();
}
