// CPU oracle for the routed MoE layer forward, in C++ with float64 accumulation.
//
// Test infrastructure only: the tests, the package's smoke check and the benchmark's
// CPU legs load it (through oracle/cpp_oracle.py).  It shares no code with the CUDA
// library, is never linked into it, and takes nothing from it: its only inputs are
// host arrays from the seeded generator.  Plain loops, the reduction of every sum in
// index order, no blocking of a sum; work is split over std::thread workers by
// (row block, column block), which changes no result.
//
// Sources (page title, then the section each step follows):
//   "6.4 Data parallelism and expert parallelism"
//     section 3.1 "Dataflow inside one MoE layer": Route -> Dispatch -> Expert
//       compute -> Combine, and the dispatch figure (copies per card);
//     section 2.1: an expert is the three matrices gate, up, down;
//     section 3.2: FP8 dispatch, BF16 combine;
//     sections 5.1-5.3: load per card, busiest / average, balancedness, the
//       rebalanced placement with redundant slots, (E + redundant) / EP per card;
//     section 7: the shared expert every token picks ("picks 9").
//   "How Expert Parallelism Works for Mixture-of-Experts Models in vLLM",
//     "MoE Layer Construction" (physical = logical + redundant experts) and
//     "Configuring Expert Parallelism" (linear or round-robin placement).
//   "Your expert-parallel deployment is slower than the tensor-parallel one. Find
//     out why.", "The three causes": max rank load against mean rank load.
//
// Readings where the pages are silent (the same as the float64 numpy oracle's):
// selection on the fp32 logits (plus the selection bias, summed in fp32), ties to the
// lower expert index, -0 == +0; weights = softmax over E renormalised over the k, from
// the unbiased logits; rows ordered by physical expert, then token; hot list = the
// n_red largest counts (lower index on ties), replica j on rank j mod R, token t uses
// replica t mod replica_count; round-robin puts expert e on rank e mod R, slot e div R;
// SwiGLU = silu(x W_gate) * (x W_up), then W_down; shared expert weight 1; bf16
// workloads round h and y to bf16; fp8 workloads quantise x and h per row per 128
// channels and the weights per 128x128 block: scale = amax / 448 in fp32 (1 when amax
// is 0), code = e4m3(v / scale) in fp32, nearest with ties to the even code, saturating.
//
// Planted mistakes for the tests: compiling with -DORC_PLANT=n changes one step
// (see the `plant` switches below); the default build has none.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

namespace {

constexpr int kPlant = ORC_PLANT;

// ============================================================== work split
template <class F>
void parallel_for(int64_t units, int threads, F fn) {
  if (units <= 0) return;
  int n = (int)std::min<int64_t>(std::max(threads, 1), units);
  std::atomic<int64_t> next{0};
  auto worker = [&] {
    for (int64_t u = next.fetch_add(1); u < units; u = next.fetch_add(1)) fn(u);
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < n; ++i) pool.emplace_back(worker);
  worker();
  for (auto &t : pool) t.join();
}

double seconds_since(std::chrono::steady_clock::time_point t0) {
  return std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
}

// ============================================================== number formats
float f32_of_bits(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
uint32_t bits_of_f32(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// bfloat16 keeps the top 16 bits of a float32.  Round a float32 to the nearer of the
// two bfloat16 values around it (truncated, and one bfloat16 step further from zero);
// on a tie keep the one whose last kept bit is 0.
float round_to_bf16(float f) {
  const uint32_t u = bits_of_f32(f);
  if ((u & 0xFFFFu) == 0) return f;
  const uint32_t lo = u & 0xFFFF0000u;
  const uint32_t hi = lo + 0x10000u;  // one step further from zero (may reach inf)
  const double dlo = std::fabs((double)f - (double)f32_of_bits(lo));
  const double dhi = std::fabs((double)f32_of_bits(hi) - (double)f);
  if (dlo < dhi) return f32_of_bits(lo);
  if (dhi < dlo) return f32_of_bits(hi);
  return ((lo >> 16) & 1u) ? f32_of_bits(hi) : f32_of_bits(lo);
}
double bf16_value(double v) { return (double)round_to_bf16((float)v); }
double bf16_bits_value(uint16_t b) { return (double)f32_of_bits((uint32_t)b << 16); }

// The bfloat16 value next above r (r itself a bfloat16 value).
double bf16_next_up(float r) {
  if (r == 0.f) return (double)f32_of_bits(0x00010000u);
  const uint32_t u = bits_of_f32(r);
  return (double)f32_of_bits(r > 0.f ? u + 0x10000u : u - 0x10000u);
}

// The two bfloat16 values around v: lo <= v <= hi (equal when v is one).  Either is
// a correct rounding of v by a computation whose own value of v may lie on the other
// side of the midpoint between them.
void bf16_bracket(double v, double *lo, double *hi) {
  const double r = bf16_value(v);
  if (r == v) {
    *lo = *hi = r;
  } else if (r < v) {
    *lo = r;
    *hi = bf16_next_up((float)r);
  } else {
    *hi = r;
    *lo = -bf16_next_up(-(float)r);
  }
}

// OCP FP8 E4M3 ("fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
// field 0 holds the subnormals m/8 * 2^-6; 0x7F and 0xFF are NaN; no infinities.
double e4m3_value(int code) {
  const double s = (code & 0x80) ? -1.0 : 1.0;
  const int ex = (code >> 3) & 0xF, m = code & 7;
  if (ex == 15 && m == 7) return NAN;
  if (ex == 0) return s * std::ldexp(m / 8.0, -6);
  return s * std::ldexp(1.0 + m / 8.0, ex - 7);
}

struct E4m3Table {
  double pos[127];  // codes 0 .. 126 (0 .. 448), ascending
  E4m3Table() {
    for (int c = 0; c < 127; ++c) pos[c] = e4m3_value(c);
  }
};
const E4m3Table &e4m3_table() {
  static const E4m3Table t;
  return t;
}

// Nearest e4m3 value to a finite float32, ties to the even code, saturating at 448.
uint8_t e4m3_encode(float v) {
  const double a = std::fabs((double)v);
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double *p = e4m3_table().pos;
  int code;
  if (a >= p[126]) {
    code = 126;
  } else {
    const int lo = (int)(std::upper_bound(p, p + 127, a) - p) - 1;  // largest code whose value is <= a
    if (p[lo] == a) {
      code = lo;
    } else {
      const double dlo = a - p[lo], dhi = p[lo + 1] - a;
      code = dlo < dhi ? lo : dhi < dlo ? lo + 1 : ((lo & 1) ? lo + 1 : lo);
    }
  }
  return (uint8_t)(code | sign);
}

// One group (or block) of float32 values: scale = amax / 448 (fp32), 1 if amax is 0.
float group_scale(float amax) { return amax > 0.f ? amax / 448.0f : 1.0f; }

// Per-row, per-`group`-channel quantisation of float32 values [rows, n].
void quantize_groups(const float *v, int64_t rows, int64_t n, int64_t group, uint8_t *codes, float *scales) {
  const int64_t G = n / group;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < G; ++g) {
      const float *src = v + r * n + g * group;
      float amax = 0.f;
      for (int64_t c = 0; c < group; ++c) amax = std::max(amax, std::fabs(src[c]));
      const float s = group_scale(amax);
      scales[r * G + g] = s;
      for (int64_t c = 0; c < group; ++c) codes[r * n + g * group + c] = e4m3_encode(src[c] / s);
    }
}

// Per-`block` x `block` quantisation of a float32 matrix [R, C] (the weight rule).
void quantize_blocks(const float *w, int64_t R, int64_t C, int64_t block, uint8_t *codes, float *scales) {
  const int64_t BR = R / block, BC = C / block;
  for (int64_t bi = 0; bi < BR; ++bi)
    for (int64_t bj = 0; bj < BC; ++bj) {
      float amax = 0.f;
      for (int64_t i = 0; i < block; ++i)
        for (int64_t j = 0; j < block; ++j) amax = std::max(amax, std::fabs(w[(bi * block + i) * C + bj * block + j]));
      const float s = group_scale(amax);
      scales[bi * BC + bj] = s;
      for (int64_t i = 0; i < block; ++i)
        for (int64_t j = 0; j < block; ++j) {
          const int64_t at = (bi * block + i) * C + bj * block + j;
          codes[at] = e4m3_encode(w[at] / s);
        }
    }
}

// ============================================================== route
// For each token: experts ordered by (score descending, index ascending), the first k
// kept; score = logit (+ bias, summed in fp32).  Weights from the unbiased logits:
// w_j = exp(l_j - m) / sum_i exp(l_i - m), m the largest chosen logit, float64.  With
// no bias this is the softmax over all E renormalised over the k (the full
// denominator cancels, and the largest chosen logit is the largest logit).
int route(const float *logits, int64_t T, int64_t E, int k, const float *bias, int32_t *ids, double *w) {
  if (k < 1 || k > E) return 2;
  std::vector<float> score(E);
  std::vector<int> order(E);
  for (int64_t t = 0; t < T; ++t) {
    const float *l = logits + t * E;
    for (int64_t e = 0; e < E; ++e) {
      score[e] = bias ? l[e] + bias[e] : l[e];
      if (!std::isfinite(l[e]) || !std::isfinite(score[e])) return 1;
    }
    std::iota(order.begin(), order.end(), 0);
    if (kPlant == 1)  // planted: ties to the higher index
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        return score[a] > score[b] || (score[a] == score[b] && a > b);
      });
    else
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return score[a] > score[b]; });
    double m = -INFINITY;
    for (int j = 0; j < k; ++j) m = std::max(m, (double)l[order[j]]);
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += std::exp((double)l[order[j]] - m);
    for (int j = 0; j < k; ++j) {
      ids[t * k + j] = order[j];
      w[t * k + j] = kPlant == 2 ? std::exp((double)l[order[j]] - m)  // planted: no renormalisation
                                 : std::exp((double)l[order[j]] - m) / sum;
    }
  }
  return 0;
}

// The weights the long way: softmax over all E, the chosen k picked, divided by their sum.
int route_softmax_then_renorm(const float *logits, int64_t T, int64_t E, int k, int32_t *ids, double *w) {
  int rc = route(logits, T, E, k, nullptr, ids, w);
  if (rc) return rc;
  std::vector<double> p(E);
  for (int64_t t = 0; t < T; ++t) {
    const float *l = logits + t * E;
    double mx = -INFINITY, z = 0.0;
    for (int64_t e = 0; e < E; ++e) mx = std::max(mx, (double)l[e]);
    for (int64_t e = 0; e < E; ++e) z += (p[e] = std::exp((double)l[e] - mx));
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += p[ids[t * k + j]] / z;
    for (int j = 0; j < k; ++j) w[t * k + j] = (p[ids[t * k + j]] / z) / s;
  }
  return 0;
}

// ============================================================== load statistics
// stats[6] = max rank load, mean rank load, max / mean, mean / max (balancedness),
// largest expert count, active experts.  Loads count token-copies (t, j).
void rank_stats(const int64_t *rank_counts, int R, int64_t total, const int64_t *expert_counts, int64_t n_exp,
                double *stats) {
  int64_t mx = 0;
  for (int r = 0; r < R; ++r) mx = std::max(mx, rank_counts[r]);
  const double mean = (double)total / R;
  int64_t me = 0, act = 0;
  for (int64_t e = 0; e < n_exp; ++e) {
    me = std::max(me, expert_counts[e]);
    act += expert_counts[e] > 0;
  }
  stats[0] = (double)mx;
  stats[1] = mean;
  stats[2] = mean > 0 ? (double)mx / mean : 0.0;
  stats[3] = mx > 0 ? mean / (double)mx : 0.0;
  stats[4] = (double)me;
  stats[5] = (double)act;
}

// Rank of each of n experts placed on R ranks: linear (blocks of n / R) or round-robin.
int base_rank(int64_t e, int64_t n, int R, int placement) {
  return placement == 1 ? (int)(e % R) : (int)(e / (n / R));
}

// ============================================================== EPLB maps
// Hottest-experts map: P = E + n_red, S = P / R per rank; rank r's slots 0 .. E/R-1
// hold its base experts (linear: r*E/R + s; round-robin: r + s*R), then replicas: the
// j-th hottest expert (count desc, index asc) on rank j mod R, slot E/R + j div R.
int eplb_map(const int64_t *counts, int64_t E, int R, int n_red, int placement, int32_t *p2l, int32_t *prank,
             int32_t *repc, int32_t *l2p /*[E,2]*/, int32_t *hot) {
  if (R < 1 || E % R || n_red % R || n_red > E || n_red < 0) return 2;
  const int64_t P = E + n_red, S = P / R, base = E / R;
  std::vector<int> order(E);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
  for (int64_t e = 0; e < E; ++e) {
    repc[e] = 1;
    l2p[2 * e] = l2p[2 * e + 1] = -1;
  }
  for (int r = 0; r < R; ++r)
    for (int64_t s = 0; s < base; ++s) {
      const int64_t e = placement == 1 ? r + s * R : r * base + s;
      const int64_t p = r * S + s;
      p2l[p] = (int32_t)e;
      prank[p] = r;
      l2p[2 * e] = (int32_t)p;
    }
  for (int j = 0; j < n_red; ++j) {
    const int e = order[j];
    const int r = j % R;
    const int64_t p = r * S + base + j / R;
    hot[j] = e;
    p2l[p] = e;
    prank[p] = r;
    l2p[2 * e + 1] = (int32_t)p;
    repc[e] = 2;
  }
  return 0;
}

// Load-aware map ("6.4 ...", section 5.2): each redundant slot to the expert with the
// most load per replica (lower id on ties); an expert's load split evenly over its
// replicas; replicas placed heaviest first (ties: expert id, then replica index) on the
// least loaded rank with a free slot (lower rank on ties), S = P / R slots per rank
// filled in arrival order.  Written as plain scans.
int eplb_balanced_map(const int64_t *counts, int64_t E, int R, int n_red, int32_t *p2l, int32_t *prank,
                      int32_t *repc, int32_t *l2p /*[E, 1+n_red]*/, double *rank_load) {
  const int64_t P = E + n_red;
  if (R < 1 || P % R || n_red < 0) return 2;
  const int64_t S = P / R, cols = 1 + n_red;
  std::vector<int64_t> rep(E, 1);
  for (int i = 0; i < n_red; ++i) {
    int64_t best = 0;
    for (int64_t e = 1; e < E; ++e)
      if ((double)counts[e] / rep[e] > (double)counts[best] / rep[best]) best = e;
    ++rep[best];
  }
  struct Piece {
    double load;
    int64_t e, j;
  };
  std::vector<Piece> pieces;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t j = 0; j < rep[e]; ++j) pieces.push_back({(double)counts[e] / rep[e], e, j});
  // heaviest first; equal loads stay in (expert, replica) order
  std::stable_sort(pieces.begin(), pieces.end(), [](const Piece &a, const Piece &b) { return a.load > b.load; });
  std::vector<double> load(R, 0.0);
  std::vector<int64_t> used(R, 0);
  for (int64_t e = 0; e < E; ++e) {
    repc[e] = (int32_t)rep[e];
    for (int64_t c = 0; c < cols; ++c) l2p[e * cols + c] = -1;
  }
  for (const Piece &pc : pieces) {
    int g = -1;
    for (int r = 0; r < R; ++r)
      if (used[r] < S && (g < 0 || load[r] < load[g])) g = r;
    const int64_t p = g * S + used[g]++;
    load[g] += pc.load;
    p2l[p] = (int32_t)pc.e;
    prank[p] = g;
    l2p[pc.e * cols + pc.j] = (int32_t)p;
  }
  for (int r = 0; r < R; ++r) rank_load[r] = load[r];
  return 0;
}

// ============================================================== dispatch layout
// Physical id of slot (t, j): e, or with a map l2p[e][t mod replica_count[e]].  Rows
// are a counting sort of the slots by physical id (stable: slot order within an
// expert, i.e. ascending token).  Physical ids are rank-major, so rank of p = p / (P/R).
struct Layout {
  int64_t *logical_counts, *phys_counts, *phys_offsets, *rank_counts, *rank_offsets;
  int32_t *row_to_token, *slot_to_row, *phys_ids;
  double *stats;  // [2][6]: before (logical counts on the base placement), after
};

int dispatch_layout(const int32_t *ids, int64_t T, int k, int64_t E, int R, int64_t P, const int32_t *l2p,
                    int l2p_cols, const int32_t *repc, int placement, const Layout &L) {
  if (R < 1 || P % R || E % R) return 2;
  const int64_t N = T * k;
  std::fill(L.logical_counts, L.logical_counts + E, 0);
  std::fill(L.phys_counts, L.phys_counts + P, 0);
  for (int64_t s = 0; s < N; ++s) {
    const int64_t t = s / k, e = ids[s];
    if (e < 0 || e >= E) return 3;
    const int64_t p = l2p ? l2p[e * l2p_cols + (t % repc[e])] : e;
    L.phys_ids[s] = (int32_t)p;
    ++L.logical_counts[e];
    ++L.phys_counts[p];
  }
  L.phys_offsets[0] = 0;
  for (int64_t p = 0; p < P; ++p) L.phys_offsets[p + 1] = L.phys_offsets[p] + L.phys_counts[p];
  std::vector<int64_t> fill(P, 0);
  for (int64_t s = 0; s < N; ++s) {
    const int64_t p = L.phys_ids[s];
    const int64_t row = L.phys_offsets[p] + fill[p]++;
    L.row_to_token[row] = (int32_t)(s / k);
    L.slot_to_row[s] = (int32_t)row;
  }
  std::fill(L.rank_counts, L.rank_counts + R, 0);
  for (int64_t p = 0; p < P; ++p) L.rank_counts[p / (P / R)] += L.phys_counts[p];
  L.rank_offsets[0] = 0;
  for (int r = 0; r < R; ++r) L.rank_offsets[r + 1] = L.rank_offsets[r] + L.rank_counts[r];
  std::vector<int64_t> before(R, 0);
  for (int64_t e = 0; e < E; ++e) before[base_rank(e, E, R, placement)] += L.logical_counts[e];
  rank_stats(before.data(), R, N, L.logical_counts, E, L.stats);
  rank_stats(L.rank_counts, R, N, L.phys_counts, P, L.stats + 6);
  return 0;
}

// ============================================================== expert FFN
double silu(double z) { return kPlant == 3 ? z / (1.0 + std::exp(z)) : z / (1.0 + std::exp(-z)); }

// The intermediate h as the down projection takes it: mode 1 rounds to bf16, mode 2
// quantises each row per 128 channels to e4m3 and dequantises, mode 0 keeps it.
void stored_h(double *h, int64_t n, int64_t I, int mode) {
  if (mode == 1 && kPlant != 4) {
    for (int64_t i = 0; i < n * I; ++i) h[i] = bf16_value(h[i]);
  } else if (mode == 2 && kPlant != 6) {
    const int64_t group = kPlant == 5 ? 256 : 128;  // planted 5: one group of 256 channels
    std::vector<float> f(I);
    std::vector<uint8_t> q(I);
    std::vector<float> s(I / group);
    for (int64_t r = 0; r < n; ++r) {
      for (int64_t i = 0; i < I; ++i) f[i] = (float)h[r * I + i];
      quantize_groups(f.data(), 1, I, group, q.data(), s.data());
      for (int64_t i = 0; i < I; ++i) h[r * I + i] = e4m3_value(q[i]) * (double)s[i / group];
    }
  }
}

// An expert's output row as the combine reads it: bf16 for modes 1 and 2.
void stored_y(double *y, int64_t n, int64_t d, int mode) {
  if ((mode == 1 || mode == 2) && kPlant != 7)
    for (int64_t i = 0; i < n * d; ++i) y[i] = bf16_value(y[i]);
}

// y[n, d] for the rows x[n, d] of one expert: g = x W_gate, u = x W_up (d x I),
// h = silu(g) * u, y = stored_h(h) W_down (I x d), then stored_y.  Every dot product
// sums in index order in float64; threads take (4-row block, 256-column block) units.
void expert_rows(const double *x, int64_t n, int64_t d, int64_t I, const double *wg, const double *wu,
                 const double *wd, int mode, double *y, int threads, double *y_exact = nullptr) {
  constexpr int64_t RB = 4, CB = 256;
  std::vector<double> h(n * I);
  const int64_t nrb = (n + RB - 1) / RB, ncb_i = (I + CB - 1) / CB, ncb_d = (d + CB - 1) / CB;
  if (kPlant == 8) std::swap(wg, wu);  // planted: gate and up exchanged
  parallel_for(nrb * ncb_i, threads, [&](int64_t u) {
    const int64_t r0 = (u / ncb_i) * RB, r1 = std::min(n, r0 + RB);
    const int64_t c0 = (u % ncb_i) * CB, c1 = std::min(I, c0 + CB);
    double g[RB][CB], up[RB][CB];
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t i = c0; i < c1; ++i) g[r - r0][i - c0] = up[r - r0][i - c0] = 0.0;
    for (int64_t c = 0; c < d; ++c)
      for (int64_t r = r0; r < r1; ++r) {
        const double xv = x[r * d + c];
        const double *a = wg + c * I, *b = wu + c * I;
        for (int64_t i = c0; i < c1; ++i) {
          g[r - r0][i - c0] += xv * a[i];
          up[r - r0][i - c0] += xv * b[i];
        }
      }
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t i = c0; i < c1; ++i) h[r * I + i] = silu(g[r - r0][i - c0]) * up[r - r0][i - c0];
  });
  stored_h(h.data(), n, I, mode);
  parallel_for(nrb * ncb_d, threads, [&](int64_t u) {
    const int64_t r0 = (u / ncb_d) * RB, r1 = std::min(n, r0 + RB);
    const int64_t c0 = (u % ncb_d) * CB, c1 = std::min(d, c0 + CB);
    double acc[RB][CB];
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t i = c0; i < c1; ++i) acc[r - r0][i - c0] = 0.0;
    for (int64_t c = 0; c < I; ++c)
      for (int64_t r = r0; r < r1; ++r) {
        const double hv = h[r * I + c];
        const double *a = wd + c * d;
        for (int64_t i = c0; i < c1; ++i) acc[r - r0][i - c0] += hv * a[i];
      }
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t i = c0; i < c1; ++i) y[r * d + i] = acc[r - r0][i - c0];
  });
  if (y_exact) std::copy(y, y + n * d, y_exact);
  stored_y(y, n, d, mode);
}

// Element i of a stored matrix: fp32 (is_f32) or bf16 bits.
double stored_value(const void *src, bool is_f32, int64_t i) {
  return is_f32 ? (double)((const float *)src)[i] : bf16_bits_value(((const uint16_t *)src)[i]);
}

// A logical weight matrix [R, C] as float64 values: as stored (modes 0, 1), or for
// mode 2 quantised per 128x128 block and dequantised.
void weight_values(const void *src, bool is_f32, int64_t R, int64_t C, int mode, double *dst, int threads) {
  if (mode == 2) {
    std::vector<float> f(R * C);
    parallel_for(R, threads, [&](int64_t r) {
      for (int64_t c = 0; c < C; ++c) f[r * C + c] = (float)stored_value(src, is_f32, r * C + c);
    });
    std::vector<uint8_t> q(R * C);
    std::vector<float> s((R / 128) * (C / 128));
    // each band of 128 rows is its own set of blocks
    parallel_for(R / 128, threads, [&](int64_t b) {
      quantize_blocks(f.data() + b * 128 * C, 128, C, 128, q.data() + b * 128 * C, s.data() + b * (C / 128));
    });
    parallel_for(R, threads, [&](int64_t r) {
      for (int64_t c = 0; c < C; ++c) dst[r * C + c] = e4m3_value(q[r * C + c]) * (double)s[(r / 128) * (C / 128) + c / 128];
    });
    return;
  }
  parallel_for(R, threads, [&](int64_t r) {
    for (int64_t c = 0; c < C; ++c) dst[r * C + c] = stored_value(src, is_f32, r * C + c);
  });
}

}  // namespace

// ============================================================== C ABI
extern "C" {

// A logical weight matrix: which = 0, 1, 2 for the routed expert e's gate [d, I], up
// [d, I], down [I, d]; 3, 4, 5 for the shared expert's.  *is_f32 = 1 for fp32 values,
// 0 for bf16 bits.  NULL if it is missing.
typedef const void *(*orc_weight_fn)(int32_t which, int32_t e, int32_t *is_f32);

struct orc_layer_cfg {
  int64_t T, d, E, I;
  int32_t k, R, shared, n_red;
  int32_t mode;              // 0 fp32, 1 bf16, 2 fp8 experts (bf16 x and out)
  int32_t eplb;              // build the replica map (n_red > 0)
  int32_t eplb_placement;    // 0 hottest experts, 1 load-aware
  int32_t expert_placement;  // 0 linear, 1 round-robin
  int32_t fp8_dispatch;      // bf16 experts fed e4m3-dispatched rows
  int32_t threads;
};

struct orc_layer_out {
  int32_t *topk_ids;
  double *topk_w;
  int64_t *logical_counts, *phys_counts, *phys_offsets, *rank_counts, *rank_offsets;
  int32_t *row_to_token, *slot_to_row, *phys_ids;
  double *stats;  // [12]
  int32_t *phys_to_logical, *phys_rank, *replica_count, *logical_to_phys;  // map (when one is built)
  int32_t l2p_cols;
  int32_t *hot;         // [n_red], hottest-experts map
  double *rank_load;    // [R], load-aware map
  uint8_t *x_q;         // [n_tok, d] (fp8 experts or fp8 dispatch)
  float *x_scales;      // [n_tok, d/128]
  double *out;          // [n_tok, d], before the output rounding
  double *out_rounded;  // [n_tok, d]
  double *out_lo;       // [n_tok, d] or NULL: out with every bf16-stored y at the bf16
  double *out_hi;       //   value just below / above its exact value (bf16 and fp8 modes)
  double *seconds;      // [7]: route, layout (with the map), permute, expert FFN rows, combine,
                        //      weight fetch (the caller's callback), weight preparation (to float64,
                        //      with the block quantisation of the fp8 workload)
};

int orc_threads_default(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}
int orc_plant(void) { return kPlant; }

int orc_route(const float *logits, int64_t T, int64_t E, int32_t k, const float *bias, int32_t *ids, double *w) {
  return route(logits, T, E, k, bias, ids, w);
}
int orc_route_softmax_then_renorm(const float *logits, int64_t T, int64_t E, int32_t k, int32_t *ids, double *w) {
  return route_softmax_then_renorm(logits, T, E, k, ids, w);
}
void orc_rank_stats(const int64_t *rank_counts, int32_t R, int64_t total, double *stats4) {
  double st[6];
  rank_stats(rank_counts, R, total, rank_counts, 0, st);
  std::memcpy(stats4, st, 4 * sizeof(double));
}
int orc_base_rank_counts(const int64_t *counts, int64_t E, int32_t R, int32_t placement, int64_t *out) {
  if (R < 1 || E % R) return 2;
  for (int r = 0; r < R; ++r) out[r] = 0;
  for (int64_t e = 0; e < E; ++e) out[base_rank(e, E, R, placement)] += counts[e];
  return 0;
}
int orc_eplb_map(const int64_t *counts, int64_t E, int32_t R, int32_t n_red, int32_t placement, int32_t *p2l,
                 int32_t *prank, int32_t *repc, int32_t *l2p, int32_t *hot) {
  return eplb_map(counts, E, R, n_red, placement, p2l, prank, repc, l2p, hot);
}
int orc_eplb_balanced_map(const int64_t *counts, int64_t E, int32_t R, int32_t n_red, int32_t *p2l, int32_t *prank,
                          int32_t *repc, int32_t *l2p, double *rank_load) {
  return eplb_balanced_map(counts, E, R, n_red, p2l, prank, repc, l2p, rank_load);
}
// EPLB's load window ("6.4 ...", section 5.3): per-expert sum of the last W of the
// `steps` count vectors [steps, E] (all of them while fewer than W).
int orc_eplb_window_sum(const int64_t *history, int64_t steps, int64_t E, int64_t W, int64_t *out) {
  if (W < 1 || steps < 1) return 2;
  for (int64_t e = 0; e < E; ++e) out[e] = 0;
  for (int64_t s = std::max<int64_t>(0, steps - W); s < steps; ++s)
    for (int64_t e = 0; e < E; ++e) out[e] += history[s * E + e];
  return 0;
}
int orc_dispatch_layout(const int32_t *ids, int64_t T, int32_t k, int64_t E, int32_t R, int64_t P,
                        const int32_t *l2p, int32_t l2p_cols, const int32_t *repc, int32_t placement,
                        int32_t *phys_ids, int64_t *logical_counts, int64_t *phys_counts, int64_t *phys_offsets,
                        int64_t *rank_counts, int64_t *rank_offsets, int32_t *row_to_token, int32_t *slot_to_row,
                        double *stats) {
  Layout L{logical_counts, phys_counts, phys_offsets, rank_counts, rank_offsets, row_to_token, slot_to_row, phys_ids,
           stats};
  return dispatch_layout(ids, T, k, E, R, P, l2p, l2p_cols, repc, placement, L);
}
void orc_bf16_bracket(const double *v, int64_t n, double *lo, double *hi) {
  for (int64_t i = 0; i < n; ++i) bf16_bracket(v[i], lo + i, hi + i);
}
void orc_round_bf16(const double *v, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(v[i]);
}
double orc_e4m3_value(int32_t code) { return e4m3_value(code & 0xFF); }
void orc_e4m3_encode(const float *v, int64_t n, uint8_t *codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_encode(v[i]);
}
void orc_quantize_groups(const float *v, int64_t rows, int64_t n, int64_t group, uint8_t *codes, float *scales) {
  quantize_groups(v, rows, n, group, codes, scales);
}
void orc_quantize_blocks(const float *w, int64_t R, int64_t C, int64_t block, uint8_t *codes, float *scales) {
  quantize_blocks(w, R, C, block, codes, scales);
}
// FP8 dispatch receive side ("6.4 ...", section 3.2): code * scale as one fp32
// multiply, then rounded to bf16.
void orc_dequantize_groups_bf16(const uint8_t *codes, const float *scales, int64_t rows, int64_t n, int64_t group,
                                double *out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < n; ++c)
      out[r * n + c] = (double)round_to_bf16((float)e4m3_value(codes[r * n + c]) * scales[r * (n / group) + c / group]);
}
void orc_dequantize_groups(const uint8_t *codes, const float *scales, int64_t rows, int64_t n, int64_t group,
                           double *out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < n; ++c) out[r * n + c] = e4m3_value(codes[r * n + c]) * (double)scales[r * (n / group) + c / group];
}
void orc_dequantize_blocks(const uint8_t *codes, const float *scales, int64_t R, int64_t C, int64_t block,
                           double *out) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c)
      out[r * C + c] = e4m3_value(codes[r * C + c]) * (double)scales[(r / block) * (C / block) + c / block];
}
// Dispatch copy ("6.4 ...", section 3.1 step 2): x_perm[r] = x[row_to_token[r]], rows
// of `row_bytes` bytes copied as they are (whatever the element type).
void orc_permute(const uint8_t *x, int64_t row_bytes, const int32_t *row_to_token, int64_t N, uint8_t *x_perm) {
  for (int64_t r = 0; r < N; ++r)
    for (int64_t b = 0; b < row_bytes; ++b) x_perm[r * row_bytes + b] = x[(int64_t)row_to_token[r] * row_bytes + b];
}
// Combine ("6.4 ...", section 3.1 step 4): out[t] = sum_j w[t,j] y[slot_to_row[t,j]]
// (+ shared[t] with weight 1, section 7), j in order, float64.
void orc_combine(const double *y, int64_t d, const int32_t *slot_to_row, const double *w, int64_t T, int32_t k,
                 const double *shared, double *out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[t * k + j] * y[(int64_t)slot_to_row[t * k + j] * d + c];
      out[t * d + c] = shared ? acc + shared[t * d + c] : acc;
    }
}
void orc_stored_h(double *h, int64_t n, int64_t I, int32_t mode) { stored_h(h, n, I, mode); }
void orc_stored_y(double *y, int64_t n, int64_t d, int32_t mode) { stored_y(y, n, d, mode); }
void orc_expert_rows(const double *x, int64_t n, int64_t d, int64_t I, const double *wg, const double *wu,
                     const double *wd, int32_t mode, double *y, int32_t threads) {
  expert_rows(x, n, d, I, wg, wu, wd, mode, y, threads);
}

// The whole layer for the tokens `tokens[0 .. n_tok)` (ascending; NULL = all T):
// routing and layout over all T tokens, then the dispatch permute of those tokens'
// rows (in layout row order), each expert's FFN over its rows, and the combine.
// x: fp32 [T, d] (mode 0) or bf16 bits (modes 1, 2).  Returns 0, or 1 (non-finite
// logit), 2 (bad shape), 3 (expert id out of range), 4 (missing weight).
int orc_layer_forward(const orc_layer_cfg *cfg, const float *logits, const void *x, int32_t x_is_f32,
                      const float *selection_bias,
                      orc_weight_fn weight, const int64_t *tokens, int64_t n_tok, const orc_layer_out *o) {
  using clock = std::chrono::steady_clock;
  const int64_t T = cfg->T, d = cfg->d, E = cfg->E, I = cfg->I;
  const int k = cfg->k, R = cfg->R, mode = cfg->mode;
  const int threads = cfg->threads > 0 ? cfg->threads : orc_threads_default();
  const int64_t N = T * k;
  for (int i = 0; i < 7; ++i) o->seconds[i] = 0.0;
  if (d % 128 && (mode == 2 || cfg->fp8_dispatch)) return 2;

  // -------- route
  auto t0 = clock::now();
  int rc = route(logits, T, E, k, selection_bias, o->topk_ids, o->topk_w);
  o->seconds[0] = seconds_since(t0);
  if (rc) return rc;

  // -------- EPLB map and dispatch layout
  t0 = clock::now();
  const int placement = cfg->expert_placement == 1 ? 1 : 0;
  int64_t P = E;
  const int32_t *l2p = nullptr;
  const int32_t *repc = nullptr;
  int l2p_cols = 0;
  std::vector<int64_t> counts(E, 0);
  for (int64_t s = 0; s < N; ++s) {
    if (o->topk_ids[s] < 0 || o->topk_ids[s] >= E) return 3;
    ++counts[o->topk_ids[s]];
  }
  if (cfg->eplb && cfg->eplb_placement == 1) {
    P = E + cfg->n_red;
    rc = eplb_balanced_map(counts.data(), E, R, cfg->n_red, o->phys_to_logical, o->phys_rank, o->replica_count,
                           o->logical_to_phys, o->rank_load);
    l2p_cols = 1 + cfg->n_red;
  } else if (cfg->eplb || placement == 1) {
    const int nr = cfg->eplb ? cfg->n_red : 0;
    P = E + nr;
    rc = eplb_map(counts.data(), E, R, nr, placement, o->phys_to_logical, o->phys_rank, o->replica_count,
                  o->logical_to_phys, o->hot);
    l2p_cols = 2;
  }
  if (rc) return rc;
  if (l2p_cols) {
    l2p = o->logical_to_phys;
    repc = o->replica_count;
  }
  Layout L{o->logical_counts, o->phys_counts, o->phys_offsets, o->rank_counts, o->rank_offsets,
           o->row_to_token,   o->slot_to_row, o->phys_ids,     o->stats};
  rc = dispatch_layout(o->topk_ids, T, k, E, R, P, l2p, l2p_cols, repc, placement, L);
  o->seconds[1] = seconds_since(t0);
  if (rc) return rc;

  // -------- dispatch permute: the needed tokens' x rows as the experts take them
  t0 = clock::now();
  std::vector<int64_t> tok(n_tok);
  std::vector<int64_t> tok_index(T, -1);  // token -> position in `tokens`
  for (int64_t i = 0; i < n_tok; ++i) {
    tok[i] = tokens ? tokens[i] : i;
    tok_index[tok[i]] = i;
  }
  // x of each needed token: as the routed experts take it (xs) and as the shared
  // expert takes it (x_local: never dispatched)
  std::vector<double> xs(n_tok * d), x_local(n_tok * d);
  parallel_for(n_tok, threads, [&](int64_t i) {
    const int64_t t = tok[i];
    for (int64_t c = 0; c < d; ++c)
      x_local[i * d + c] = stored_value(x, x_is_f32 != 0, t * d + c);
    const bool quant = mode == 2 || (mode == 1 && cfg->fp8_dispatch);
    if (!quant) {
      std::copy(&x_local[i * d], &x_local[i * d] + d, &xs[i * d]);
      return;
    }
    std::vector<float> f(d);
    for (int64_t c = 0; c < d; ++c) f[c] = (float)x_local[i * d + c];
    quantize_groups(f.data(), 1, d, 128, o->x_q + i * d, o->x_scales + i * (d / 128));
    for (int64_t c = 0; c < d; ++c) {
      const float s = o->x_scales[i * (d / 128) + c / 128];
      const double v = e4m3_value(o->x_q[i * d + c]);
      xs[i * d + c] = mode == 2 ? v * (double)s : (double)round_to_bf16((float)v * s);
    }
    if (mode == 2) std::copy(&xs[i * d], &xs[i * d] + d, &x_local[i * d]);
  });
  // rows of the layout that belong to a needed token, in row order: x_perm
  std::vector<int64_t> rows;  // layout row ids
  std::vector<int64_t> compact(N, -1);
  for (int64_t r = 0; r < N; ++r)
    if (tok_index[o->row_to_token[r]] >= 0) {
      compact[r] = (int64_t)rows.size();
      rows.push_back(r);
    }
  const int64_t M = (int64_t)rows.size();
  std::vector<double> x_perm(M * d);
  parallel_for(M, threads, [&](int64_t m) {
    const int64_t i = tok_index[o->row_to_token[rows[m]]];
    std::copy(&xs[i * d], &xs[i * d] + d, &x_perm[m * d]);
  });
  o->seconds[2] = seconds_since(t0);

  // -------- expert FFN: each logical expert over the rows of all its physical replicas
  const bool bracket = o->out_lo && o->out_hi;
  std::vector<double> y_perm(M * d), y_perm_exact(bracket ? M * d : 0);
  std::vector<std::vector<int64_t>> rows_of(E);
  {
    // physical id of each layout row, from the offsets
    int64_t p = 0;
    for (int64_t m = 0; m < M; ++m) {
      const int64_t r = rows[m];
      while (o->phys_offsets[p + 1] <= r) ++p;
      const int64_t e = l2p_cols ? o->phys_to_logical[p] : p;
      rows_of[e].push_back(m);
    }
  }
  std::vector<double> wg(d * I), wu(d * I), wd(I * d);
  double fetch = 0.0, prep = 0.0, ffn = 0.0;
  auto run_expert = [&](int which0, int64_t e, const std::vector<int64_t> &idx, const double *src_rows,
                        bool gathered, std::vector<double> &dst, std::vector<double> &dst_exact) -> bool {
    auto tf = clock::now();
    int32_t fg = 0, fu = 0, fd = 0;
    const void *pg = weight(which0, (int32_t)e, &fg);
    const void *pu = weight(which0 + 1, (int32_t)e, &fu);
    const void *pd = weight(which0 + 2, (int32_t)e, &fd);
    fetch += seconds_since(tf);
    if (!pg || !pu || !pd) return false;
    auto tp = clock::now();
    weight_values(pg, fg != 0, d, I, mode, wg.data(), threads);
    weight_values(pu, fu != 0, d, I, mode, wu.data(), threads);
    weight_values(pd, fd != 0, I, d, mode, wd.data(), threads);
    prep += seconds_since(tp);
    auto tc = clock::now();
    const int64_t n = (int64_t)idx.size();
    std::vector<double> xin(n * d), yout(n * d), yexact(bracket ? n * d : 0);
    for (int64_t a = 0; a < n; ++a)
      std::copy(src_rows + (gathered ? idx[a] : a) * d, src_rows + (gathered ? idx[a] : a) * d + d, &xin[a * d]);
    expert_rows(xin.data(), n, d, I, wg.data(), wu.data(), wd.data(), mode, yout.data(), threads,
                bracket ? yexact.data() : nullptr);
    for (int64_t a = 0; a < n; ++a) {
      std::copy(&yout[a * d], &yout[a * d] + d, &dst[(gathered ? idx[a] : a) * d]);
      if (bracket) std::copy(&yexact[a * d], &yexact[a * d] + d, &dst_exact[(gathered ? idx[a] : a) * d]);
    }
    ffn += seconds_since(tc);
    return true;
  };
  for (int64_t e = 0; e < E; ++e) {
    if (rows_of[e].empty()) continue;
    if (!run_expert(0, e, rows_of[e], x_perm.data(), true, y_perm, y_perm_exact)) return 4;
  }
  std::vector<double> shared_y, shared_y_exact;
  if (cfg->shared && n_tok > 0) {
    shared_y.assign(n_tok * d, 0.0);
    shared_y_exact.assign(bracket ? n_tok * d : 0, 0.0);
    std::vector<int64_t> all(n_tok);
    std::iota(all.begin(), all.end(), 0);
    if (!run_expert(3, 0, all, x_local.data(), false, shared_y, shared_y_exact)) return 4;
  }
  o->seconds[3] = ffn;
  o->seconds[5] = fetch;
  o->seconds[6] = prep;

  // -------- combine: out[t] = sum_j w[t,j] y[slot_to_row[t,j]] (+ shared), j in order
  t0 = clock::now();
  parallel_for(n_tok, threads, [&](int64_t i) {
    const int64_t t = tok[i];
    for (int64_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += o->topk_w[t * k + j] * y_perm[compact[o->slot_to_row[t * k + j]] * d + c];
      if (cfg->shared) acc += shared_y[i * d + c];
      o->out[i * d + c] = acc;
      o->out_rounded[i * d + c] = mode == 0 ? acc : bf16_value(acc);
      if (!bracket) continue;
      // the same sum with each stored y at the bf16 value below / above its exact
      // value (the weights are positive)
      double lo = 0.0, hi = 0.0, a, b;
      for (int j = 0; j < k; ++j) {
        const double v = y_perm_exact[compact[o->slot_to_row[t * k + j]] * d + c];
        if (mode == 0) a = b = v;
        else bf16_bracket(v, &a, &b);
        lo += o->topk_w[t * k + j] * a;
        hi += o->topk_w[t * k + j] * b;
      }
      if (cfg->shared) {
        const double v = shared_y_exact[i * d + c];
        if (mode == 0) a = b = v;
        else bf16_bracket(v, &a, &b);
        lo += a;
        hi += b;
      }
      o->out_lo[i * d + c] = lo;
      o->out_hi[i * d + c] = hi;
    }
  });
  o->seconds[4] = seconds_since(t0);
  return 0;
}

}  // extern "C"
