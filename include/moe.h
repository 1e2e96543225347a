/*
 * moe.h -- C ABI of the B300 (sm_103a) routed mixture-of-experts layer forward.
 *
 * The layer, as "6.4 Data parallelism and expert parallelism" (section 3.1,
 * "Dataflow inside one MoE layer") describes it, run on one GPU:
 *
 *   route    -> softmax over E experts, top-k experts and weights per token
 *   dispatch -> count tokens per expert, scan, lay the k copies of every token out
 *               expert-contiguously in expert-parallel rank order (the buffer an
 *               all-to-all dispatch would send), per-rank load statistics
 *   experts  -> grouped SwiGLU FFN (gate, up, down) per expert
 *   combine  -> weighted sum of each token's k expert outputs (+ shared expert)
 *
 * Notation: T tokens, d hidden size, E routed (logical) experts, k experts per
 * token, I expert intermediate size, R logical expert-parallel ranks,
 * P = E + n_redundant physical experts, N = T*k routed rows.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; they must stay
 *     valid until the work queued on `stream` has finished.  The library never
 *     allocates or frees device memory, and keeps none between calls, with one
 *     exception: the scratch array built into the library for
 *     moe_dispatch_layout_static (MOE_DISPATCH_STATIC_SCRATCH_BYTES on every GPU
 *     that loads it, until the process exits).  Struct arguments
 *     (moe_shape_t, moe_weights_t, moe_eplb_t, moe_layer_aux_t) are HOST structs
 *     read during the call; the pointers inside them are device pointers.
 *   - Tensors are dense and row-major.  bf16 is stored as uint16 bit patterns,
 *     e4m3 as one byte (OCP FP8 E4M3, "fn": no infinities, max 448).
 *   - Work is queued on `stream` and the call returns at once.  The returned
 *     status reports host-side validation and launch errors only.
 *   - Problems found on the device (a non-finite logit, an expert id out of
 *     range, a pipeline wait that ran out) are OR-ed as MOE_DEV_* bits into the
 *     caller's device word `err` (int32, may be NULL to ignore them); the caller
 *     reads it after synchronising.  Kernels never trap.
 *   - Apart from that array (and its device address, looked up once per device
 *     and context), the library holds no global state: calls on different streams
 *     may run concurrently when they share no output buffer.  Calls of
 *     moe_dispatch_layout_static share the array, so they must not overlap.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned tensor          */
  MOE_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement  */
  MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than *_workspace_size */
  MOE_ERR_CUDA = 4         /* a CUDA runtime/driver call failed (launch, attrs)  */
} moe_status_t;

/* Bits OR-ed into the caller's device error word. */
enum {
  MOE_DEV_NONFINITE_LOGIT = 1, /* a router logit was NaN or +-Inf: ids/weights undefined */
  MOE_DEV_ID_RANGE = 2,        /* an expert id outside [0, E): the slot was skipped      */
  MOE_DEV_TIMEOUT = 4,         /* a pipeline wait gave up: outputs of that launch undefined */
  MOE_DEV_LAYOUT = 8           /* expert offsets inconsistent with the rows: tile skipped */
};

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2 } moe_dtype_t;

/* Per-rank load statistics ("Your expert-parallel deployment is slower than the
 * tensor-parallel one", "The three causes": max rank load against mean rank
 * load; "6.4 ...", section 5.3: balancedness = average / max).  Loads count
 * token-copies (t, j).  Written on the device. */
typedef struct {
  int32_t max_rank;         /* busiest rank's load                         */
  int32_t max_expert;       /* busiest (physical or logical) expert's load */
  int32_t n_active_experts; /* experts with at least one row               */
  int32_t pad_;
  float mean_rank;          /* T*k / R                                     */
  float max_over_mean;      /* max_rank / mean_rank                        */
  float balancedness;       /* mean_rank / max_rank                        */
  float pad2_;
} moe_load_stats_t;

/* EPLB replica map (device arrays), as written by moe_eplb_map or
 * moe_eplb_balanced_map. */
typedef struct {
  int32_t P;                      /* physical experts, E + n_redundant                  */
  const int32_t *phys_to_logical; /* [P]                                                 */
  const int32_t *replica_count;   /* [E], >= 1                                           */
  const int32_t *logical_to_phys; /* [E, max_replicas]: replica j of expert e (-1 unused) */
  int32_t max_replicas;           /* row length of logical_to_phys: 2 for moe_eplb_map and
                                     moe_placement_map, 1 + n_redundant for
                                     moe_eplb_balanced_map; 0 reads as 2 */
  int32_t base_placement;         /* placement of the logical experts before replication,
                                     for stats[0] of moe_dispatch_layout: 0 = linear
                                     (rank e / (E/R)), 1 = round-robin (rank e % R) */
} moe_eplb_t;

/* Packed expert weights (produced by moe_pack_weights), one set per logical
 * expert; with has_shared the set at index E is the always-on shared expert.
 *   w13: [E_w, 2I, d]  rows 0..I-1 = W_gate^T, rows I..2I-1 = W_up^T (d per row)
 *   w2 : [E_w, d, I]   W_down^T (I per row)
 *   MOE_F32 rows are stored plainly.  MOE_BF16 and MOE_E4M3 rows are tiled: per
 *   expert, tiles cut into 128-byte column blocks (tile major, then column
 *   block); inside a block the rows are 128 bytes apart and the 16-byte chunk j
 *   of block row r sits at chunk j ^ (r % 8), the arrangement the tensor cores
 *   read from shared memory, so each block is one contiguous copy.  w2 tiles are
 *   128 rows (16 KB blocks); w13 tiles are 256 rows: the W_gate^T rows, then the
 *   W_up^T rows, of the same 128 features (32 KB blocks).
 *   (Requires d % 128 == 0 and I % 128 == 0; base pointers 16-byte aligned.)
 *   e4m3 only: s13 [E_w, 2I/128, d/128], s2 [E_w, d/128, I/128] fp32 block scales,
 *   dequantised weight = code * scale of its 128x128 block. */
typedef struct {
  moe_dtype_t dtype; /* MOE_F32, MOE_BF16 or MOE_E4M3 */
  int32_t has_shared;
  int64_t E_w, d, I;
  const void *w13;
  const void *w2;
  const float *s13;
  const float *s2;
  const float *selection_bias; /* [E] fp32 or NULL: moe_layer_forward routes with
                                  moe_route_biased (experts picked by logit + bias,
                                  weighted by the unbiased logits); NULL = moe_route */
} moe_weights_t;

/* Whole-layer shape and precision. */
typedef struct {
  int64_t T, d, E, I;
  int32_t k, R;
  int32_t n_redundant;      /* EPLB replicas, 0 = off; with eplb_placement 0 a multiple
                               of R and <= E                                           */
  int32_t shared;           /* 1 = always-on shared expert (weight set E, weight 1)     */
  moe_dtype_t act_dtype;    /* x and out: MOE_F32 (with f32 experts) or MOE_BF16        */
  moe_dtype_t expert_dtype; /* MOE_F32, MOE_BF16 or MOE_E4M3                            */
  int32_t eplb_placement;   /* with n_redundant > 0: 0 = one replica for each of the
                               n_redundant hottest experts (moe_placement_map); 1 = the
                               load-aware placement (moe_eplb_balanced_map, needs only
                               (E + n_redundant) % R == 0)                              */
  int32_t expert_placement; /* base placement of the logical experts over the R ranks:
                               0 = linear (rank e / (E/R)), 1 = round-robin (rank e % R).
                               Sets the base slots of moe_placement_map and the "before"
                               statistics; the load-aware map places every expert
                               itself, so with eplb_placement 1 only the statistics
                               change                                                   */
  int32_t fp8_dispatch;     /* 1 with bf16 experts: tokens are dispatched as e4m3 with
                               per-128-channel scales (moe_permute to MOE_E4M3) and
                               turned back into bf16 rows (moe_dequantize_e4m3) for
                               the experts; needs d % 128 == 0.  e4m3 experts always
                               take e4m3 rows, so there it changes nothing           */
} moe_shape_t;

/* Optional device buffers that receive the layer's intermediate results; any
 * NULL member is kept in the workspace instead. */
typedef struct {
  int32_t *topk_ids;        /* [T, k]   */
  float *topk_w;            /* [T, k]   */
  int32_t *logical_counts;  /* [E]      */
  int32_t *phys_counts;     /* [P]      */
  int32_t *phys_offsets;    /* [P + 1]  */
  int32_t *rank_counts;     /* [R]      */
  int32_t *rank_offsets;    /* [R + 1]  */
  int32_t *row_to_token;    /* [N]      */
  int32_t *slot_to_row;     /* [T, k]   */
  moe_load_stats_t *stats;  /* [2]: before, after EPLB */
  int32_t *phys_to_logical; /* [P]      */
  int32_t *phys_rank;       /* [P]      */
  int32_t *replica_count;   /* [E]      */
  int32_t *logical_to_phys; /* [E, 2], or [E, 1 + n_redundant] with eplb_placement 1 */
} moe_layer_aux_t;

/* Static text for a status code. */
const char *moe_status_string(moe_status_t s);

/* Text of the last CUDA error behind a MOE_ERR_CUDA returned to the calling
 * thread ("" when there was none).  The pages have no counterpart; diagnostics. */
const char *moe_last_cuda_error(void);

/* Route ("6.4 ...", section 3.1, step 1 "Route": top-k experts and weights per
 * token).  logits [T, E] fp32.  Experts are chosen by (logit descending, index
 * ascending); -0 and +0 tie.  topk_ids [T, k] int32 in that order; topk_w [T, k]
 * fp32 = softmax over all E renormalised over the k chosen, i.e.
 * exp(l_j - l_max) / sum over the chosen of exp(l_i - l_max).
 * Limits: 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T = 0 queues nothing). */
moe_status_t moe_route(const float *logits, int64_t T, int64_t E, int32_t k,
                       int32_t *topk_ids, float *topk_w, int32_t *err,
                       moe_stream_t stream);

/* moe_route with a per-expert selection bias ("6.4 ...", section 5.1: the
 * bias term that balances expert load without an auxiliary loss).  The experts are
 * picked by logit + selection_bias[e] (fp32 sum; ties to the lower index), and their
 * weights are the softmax of their unbiased logits renormalised over the k picked:
 * w_j = exp(l_j - m) / sum_i exp(l_i - m), m the largest picked logit.
 * selection_bias [E] fp32 (device) or NULL (= moe_route).  A non-finite logit or
 * sum sets MOE_DEV_NONFINITE_LOGIT.  Limits as moe_route. */
moe_status_t moe_route_biased(const float *logits, const float *selection_bias,
                              int64_t T, int64_t E, int32_t k, int32_t *topk_ids,
                              float *topk_w, int32_t *err, moe_stream_t stream);

/* Size of the scratch array built into the library for moe_dispatch_layout_static. */
#define MOE_DISPATCH_STATIC_SCRATCH_BYTES (4u << 20)

/* moe_dispatch_layout for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a deployment convenience of this library).  Some
 * callers receive only their input and output buffers and have no device
 * allocator to take a workspace from -- a plugin whose host runtime owns and
 * pre-budgets all memory, or a latency-critical path where allocating is not
 * allowed.  This entry point computes exactly what moe_dispatch_layout computes
 * (same arguments and results, minus ws/ws_bytes) and allocates nothing: its
 * scratch is a MOE_DISPATCH_STATIC_SCRATCH_BYTES array inside the library, which
 * every GPU that loads the library reserves until the process exits.
 *   - Returns MOE_ERR_WORKSPACE, queuing nothing, when the batch needs more
 *     scratch than that, i.e. moe_dispatch_workspace_size(T, k, P) >
 *     MOE_DISPATCH_STATIC_SCRATCH_BYTES (about 900k slots T*k at P = 256,
 *     500k at P = 2048).
 *   - All calls share the one array and it keeps the previous call's contents;
 *     the kernels overwrite each entry before reading it.  Calls whose work
 *     overlaps on a GPU (different streams or host threads) race on it and give
 *     wrong results: keep them on one stream or synchronise in between.
 *   - The first call on each device (with that device current) looks up the
 *     array's device address, and so does the first call after the device's
 *     context has changed (a cudaDeviceReset gives the device a new context);
 *     make those calls before any stream capture. */
moe_status_t moe_dispatch_layout_static(const int32_t *topk_ids, int64_t T, int32_t k,
                                        int64_t E, int32_t R, const moe_eplb_t *eplb,
                                        int32_t *logical_counts, int32_t *phys_counts,
                                        int32_t *phys_offsets, int32_t *rank_counts,
                                        int32_t *rank_offsets, int32_t *row_to_token,
                                        int32_t *slot_to_row, moe_load_stats_t *stats,
                                        int32_t *err, moe_stream_t stream);

/* EPLB one-step replica map ("6.4 ...", section 5.3: (experts + redundant)/EP
 * physical experts per card; "How Expert Parallelism Works for Mixture-of-Experts
 * Models in vLLM", "MoE Layer Construction": num_physical = E + redundant).
 * logical_counts [E] int32 (tokens per logical expert).  The n_redundant hottest
 * experts (count descending, index ascending) get one replica each.  Rank r holds
 * S = P/R physical slots: slots 0..E/R-1 are logical experts r*E/R + slot, then the
 * replicas, the j-th hottest on rank j mod R in slot E/R + j/R; physical id =
 * r*S + slot.  Outputs: phys_to_logical [P], phys_rank [P], replica_count [E],
 * logical_to_phys [E, 2].  Requires E % R == 0, n_redundant % R == 0,
 * 0 <= n_redundant <= E, E <= 1024. */
moe_status_t moe_eplb_map(const int32_t *logical_counts, int64_t E, int32_t R,
                          int32_t n_redundant, int32_t *phys_to_logical,
                          int32_t *phys_rank, int32_t *replica_count,
                          int32_t *logical_to_phys, moe_stream_t stream);

/* moe_eplb_map with a choice of base placement ("How Expert Parallelism Works for
 * Mixture-of-Experts Models in vLLM", "Configuring Expert Parallelism": the
 * placement strategy is "linear" or "round_robin").  placement 0 = linear, as
 * moe_eplb_map; 1 = round-robin: logical expert e sits on rank e % R in slot e / R
 * (physical id (e % R) * S + e / R).  Replicas are placed as in moe_eplb_map.
 * With n_redundant == 0 the map is the bare placement (P = E, every
 * replica_count 1, logical_to_phys[e][1] = -1) and logical_counts may be NULL.
 * Same outputs and limits as moe_eplb_map; a placement other than 0 or 1 is
 * MOE_ERR_INVALID_ARG. */
moe_status_t moe_placement_map(const int32_t *logical_counts, int64_t E, int32_t R,
                               int32_t n_redundant, int32_t placement,
                               int32_t *phys_to_logical, int32_t *phys_rank,
                               int32_t *replica_count, int32_t *logical_to_phys,
                               moe_stream_t stream);

/* Load-aware EPLB placement ("6.4 Data parallelism and expert parallelism",
 * section 5.2, the placement with redundant slots that the page's simulation
 * compares against the contiguous one).  logical_counts [E] int32.  In the page's
 * order: each of the n_redundant extra slots goes to the expert whose load per
 * replica (count / replicas) is highest, the lowest expert id on a tie; every
 * replica of an expert carries count / replicas; the P = E + n_redundant replicas,
 * heaviest first (equal loads keep expert then replica order), each go to the rank
 * with the smallest load so far among those with one of their S = P / R slots
 * free (the lowest rank on a tie) and take its next slot.  Physical id = rank * S +
 * slot.  Outputs (device): phys_to_logical [P], phys_rank [P], replica_count [E],
 * logical_to_phys [E, 1 + n_redundant] (replica j of expert e in placement order,
 * -1 past replica_count[e]), rank_load [R] fp64 (optional, may be NULL).  Loads
 * are fp64 quotients compared and summed in that order, so the map is exact.  Use it
 * with moe_dispatch_layout through a moe_eplb_t with max_replicas = 1 + n_redundant.
 * Requires E <= 1024, R <= 1024, P <= 2048, P % R == 0.  One CTA; for rebalancing,
 * not for every step. */
moe_status_t moe_eplb_balanced_map(const int32_t *logical_counts, int64_t E, int32_t R,
                                   int32_t n_redundant, int32_t *phys_to_logical,
                                   int32_t *phys_rank, int32_t *replica_count,
                                   int32_t *logical_to_phys, double *rank_load,
                                   moe_stream_t stream);

/* EPLB's sliding window of loads ("6.4 Data parallelism and expert parallelism",
 * section 5.3: the balancer averages per-expert load over window_size recent steps
 * and rebalances every step_interval steps).  window [W, E] int32 is a ring the
 * caller zero-fills once and keeps between calls; this call stores this step's
 * logical_counts [E] (as moe_dispatch_layout writes them) in row step mod W and
 * writes window_sum [E] = the sum over all W rows, i.e. over the last min(step + 1, W)
 * steps (saturating at 2^31 - 1), ready for moe_eplb_balanced_map.  Requires
 * 1 <= W <= 2^20, E <= 1024, step >= 0. */
moe_status_t moe_eplb_window_update(const int32_t *logical_counts, int32_t *window,
                                    int64_t W, int64_t E, int64_t step,
                                    int32_t *window_sum, moe_stream_t stream);

/* Self-test of the failure path shared by the tensor-core kernels (no counterpart
 * on the pages): one thread runs their bounded pipeline wait on an mbarrier that
 * nothing arrives on, with a limit of timeout_ns (1 us .. 100 ms) instead of the
 * kernels' 2 s.  The wait gives up, ORs MOE_DEV_TIMEOUT into *err, writes the time
 * it waited in ms to *waited_ms (may be NULL; -1 had it succeeded) and the kernel
 * returns; the context stays usable.  A test and diagnostic aid, not part of the
 * forward pass. */
moe_status_t moe_selftest_wait_timeout(int32_t *err, int64_t timeout_ns, int32_t *waited_ms,
                                       moe_stream_t stream);

/* Bytes of workspace moe_dispatch_layout needs. */
size_t moe_dispatch_workspace_size(int64_t T, int32_t k, int64_t P);

/* Dispatch layout ("6.4 ...", section 3.1, step 2 "Dispatch" and its figure:
 * each token is copied k times to the cards that own its experts; section 5.1:
 * busiest card / average).  topk_ids [T, k] int32 in [0, E).  Physical expert of
 * slot (t, j): e, or with `eplb` logical_to_phys[e][t mod replica_count[e]] (rows of
 * eplb->max_replicas entries).
 * Physical experts are numbered rank-major (P/R per rank), so rows sorted by
 * physical expert are sorted by (rank, expert); inside an expert, rows are in
 * ascending token order.  Outputs (device, int32):
 *   logical_counts [E], phys_counts [P], phys_offsets [P+1] (exclusive scan),
 *   rank_counts [R], rank_offsets [R+1], row_to_token [N], slot_to_row [T, k];
 *   stats [2] (moe_load_stats_t): [0] logical experts over R ranks in the base
 *   placement (eplb->base_placement; linear without eplb), before replication;
 *   [1] the physical layout (after; equal to [0] when the map only renumbers).
 * ws: moe_dispatch_workspace_size(T, k, P) bytes, 256-byte aligned.
 * Ids out of range set MOE_DEV_ID_RANGE; those slots are left out of the layout.
 * Limits: P <= 2048, P % R == 0, E % R == 0, eplb->base_placement 0 or 1. */
moe_status_t moe_dispatch_layout(const int32_t *topk_ids, int64_t T, int32_t k,
                                 int64_t E, int32_t R, const moe_eplb_t *eplb,
                                 int32_t *logical_counts, int32_t *phys_counts,
                                 int32_t *phys_offsets, int32_t *rank_counts,
                                 int32_t *rank_offsets, int32_t *row_to_token,
                                 int32_t *slot_to_row, moe_load_stats_t *stats,
                                 void *ws, size_t ws_bytes, int32_t *err,
                                 moe_stream_t stream);

/* Dispatch copy ("6.4 ...", section 3.1, step 2: copy each token's hidden state k
 * times; section 3.2: dispatch in FP8).  x [T, d] (MOE_F32 or MOE_BF16) ->
 * x_perm [N, d] with x_perm[slot_to_row[t, j]] = x[t].  perm_dt equal to x_dt is a
 * plain copy; perm_dt = MOE_E4M3 (from bf16) quantises each token per 128-channel
 * group: scale = amax/448 in fp32 (1 when amax = 0), code = e4m3(v / scale) with
 * round-to-nearest-even and saturation; perm_scales [N, d/128] fp32.
 * Requires d % 8 == 0 (d % 128 == 0 for e4m3), 16-byte aligned x and x_perm. */
moe_status_t moe_permute(const void *x, moe_dtype_t x_dt, int64_t T, int64_t d,
                         int32_t k, const int32_t *slot_to_row, void *x_perm,
                         moe_dtype_t perm_dt, float *perm_scales,
                         moe_stream_t stream);

/* Receive side of an FP8 dispatch to bf16 experts ("6.4 ...", section 3.2: tokens
 * are dispatched in FP8, the experts and the combine work in BF16).  codes
 * [rows, d] e4m3 and scales [rows, d/128] fp32, as moe_permute writes them ->
 * out [rows, d] bf16 with out = bf16(code * scale): the product is an IEEE fp32
 * multiply, rounded to bf16 to nearest even.  Requires d % 128 == 0, 16-byte
 * aligned codes and out. */
moe_status_t moe_dequantize_e4m3(const void *codes, const float *scales, int64_t rows,
                                 int64_t d, void *out, moe_stream_t stream);

/* Bytes of workspace moe_expert_ffn needs (the intermediate h and tile tables). */
size_t moe_ffn_workspace_size(int64_t rows, int64_t I, moe_dtype_t expert_dtype);

/* Grouped SwiGLU expert FFN ("6.4 ...", section 2.1: one expert is the three
 * matrices gate, up, down; section 7: the shared expert is a must-pick expert).
 * For physical expert p with logical expert e = phys_to_logical[p] (identity when
 * NULL), rows phys_offsets[p] .. phys_offsets[p+1]-1 of x_perm:
 *   h = silu(x W_gate[e]) * (x W_up[e]);  y = h W_down[e]
 * y_perm [N (+T), d].  With w->has_shared and shared_x != NULL, the shared expert
 * (weight set E) runs on shared_x [T_shared, d] and writes rows N .. N+T_shared-1.
 * Precision: f32 weights -> fp32 FFMA throughout (y fp32).  bf16 -> tensor cores,
 * fp32 accumulate, h stored as bf16, y bf16.  e4m3 -> x_perm e4m3 + x_scales
 * [N, d/128]; tensor cores per 128-deep K block with fp32 promotion by the
 * block scales; h quantised per row per 128 channels (same rule as moe_permute);
 * y bf16.  `rows_hint` is the number of routed rows N (phys_offsets[P] on the
 * device must equal it).  ws: moe_ffn_workspace_size(N + T_shared, I, dtype).
 * Limits (tensor-core paths): d % 128 == 0, I % 128 == 0, P <= 2048.  The tile
 * orientation follows the rows per expert (fewer than 64 rows per physical expert
 * on average: weight rows x token rows; else SM-pair tiles of 256 token rows);
 * MOE_B300_FFN_TILES=swap|wide|pair in the environment forces one (all give the
 * same results within rounding). */
moe_status_t moe_expert_ffn(const void *x_perm, const float *x_scales,
                            const int32_t *phys_offsets, int64_t P,
                            const int32_t *phys_to_logical, int64_t rows_hint,
                            const moe_weights_t *w, const void *shared_x,
                            int64_t T_shared, void *y_perm, void *ws,
                            size_t ws_bytes, int32_t *err, moe_stream_t stream);

/* The expert FFN's first phase on its own ("6.4 ...", section 2.1, the gate and
 * up matrices): h = silu(x W_gate[e]) * (x W_up[e]) for every row of every
 * physical expert (and the shared expert's T_shared rows after row N), as in
 * moe_expert_ffn.  h [N + T_shared, I]: fp32 (f32 weights), bf16, or e4m3 with
 * h_scales [N + T_shared, I/128] (per row per 128 channels, the moe_permute rule). */
moe_status_t moe_expert_gate_up(const void *x_perm, const float *x_scales,
                                const int32_t *phys_offsets, int64_t P,
                                const int32_t *phys_to_logical, int64_t rows_hint,
                                const moe_weights_t *w, const void *shared_x,
                                int64_t T_shared, void *h, float *h_scales,
                                int32_t *err, moe_stream_t stream);

/* The dispatch copy fused into the first phase ("6.4 ...", section 3.1, steps 2
 * and 3: each token's hidden state goes to the experts it picked, and each expert
 * applies its gate and up matrices).  bf16 weights only.  Computes what
 * moe_permute(x, MOE_BF16, T, d, k, slot_to_row, x_perm, MOE_BF16) followed by
 * moe_expert_gate_up(x_perm, ...) computes, bit for bit, without writing x_perm:
 * routed row r (phys_offsets order) reads row row_to_token[r] of x [T, d] bf16
 * (16-byte aligned), row_to_token [rows_hint] int32 being the array
 * moe_dispatch_layout writes.  The other arguments and h [N + T_shared, I] bf16 are
 * those of moe_expert_gate_up.  Always runs the one-SM tiles of 128 token rows, and
 * re-reads each gathered row once per 128 features of h, in 128-byte pieces: on
 * prefill batches that costs more than the separate copy it saves, so the layer
 * forward does not use it.  Returns MOE_ERR_UNSUPPORTED for other weight dtypes; a
 * row_to_token entry outside [0, T) sets MOE_DEV_LAYOUT in *err and leaves that row
 * of h unspecified. */
moe_status_t moe_expert_gate_up_gather(const void *x, int64_t T, const int32_t *row_to_token,
                                       const int32_t *phys_offsets, int64_t P,
                                       const int32_t *phys_to_logical, int64_t rows_hint,
                                       const moe_weights_t *w, const void *shared_x,
                                       int64_t T_shared, void *h, int32_t *err,
                                       moe_stream_t stream);

/* The expert FFN's second phase on its own ("6.4 ...", section 2.1, the down
 * matrix): y = h W_down[e] for the rows moe_expert_gate_up wrote.  y_perm
 * [N + T_shared, d]: fp32 for f32 weights, else bf16. */
moe_status_t moe_expert_down(const void *h, const float *h_scales,
                             const int32_t *phys_offsets, int64_t P,
                             const int32_t *phys_to_logical, int64_t rows_hint,
                             const moe_weights_t *w, int64_t T_shared, void *y_perm,
                             int32_t *err, moe_stream_t stream);

/* The combine fused into the down phase ("6.4 ...", section 3.1, steps 3 and 4:
 * each expert applies its down matrix, then each token's k expert outputs are
 * summed with its route weights).  bf16 weights only.  Writes y_perm as
 * moe_expert_down does (bf16 [rows_hint + T_shared, d]) and out [T, d] bf16
 * identical to moe_combine(y_perm, MOE_BF16, slot_to_row, topk_w, T, k, d,
 * T_shared ? y_perm + rows_hint * d : NULL, out, MOE_BF16): every block of 128 or
 * 256 features of out[t] is summed, in j order with fp32 fused multiply-adds, by
 * whichever tile writes the last of the token's rows for that block.
 * row_to_token [rows_hint] and slot_to_row [T, k] are the arrays moe_dispatch_layout
 * writes; topk_w [T, k] fp32; T_shared is 0 or T (the shared expert's rows, from
 * moe_expert_gate_up, follow the routed ones in h); counts is caller scratch of
 * T * (d / 128) int32, overwritten.  k <= 32; always runs the one-SM tiles of 128
 * token rows; y_perm and out 16-byte aligned.  A block can only be summed after its
 * last row, so most sums fall at the end of the launch: on prefill batches this
 * measured slower than moe_expert_down followed by moe_combine, and the layer
 * forward does not use it.  Returns MOE_ERR_UNSUPPORTED for other weight dtypes.  A
 * row whose token is outside [0, T) sets MOE_DEV_LAYOUT and leaves that token's out
 * unspecified. */
moe_status_t moe_expert_down_combine(const void *h, const int32_t *phys_offsets, int64_t P,
                                     const int32_t *phys_to_logical, int64_t rows_hint,
                                     const moe_weights_t *w, int64_t T_shared,
                                     const int32_t *row_to_token, const int32_t *slot_to_row,
                                     const float *topk_w, int64_t T, int32_t k, void *y_perm,
                                     int32_t *counts, void *out, int32_t *err,
                                     moe_stream_t stream);

/* Combine ("6.4 ...", section 3.1, step 4: weighted-sum by route weights).
 * out[t] = sum_{j<k} topk_w[t, j] * y_perm[slot_to_row[t, j]] (+ shared_y[t]),
 * fp32 accumulation in j order, then rounded to out_dt.  y_perm [N, d] and shared_y
 * [T, d] (nullable) in y_dt (MOE_F32 or MOE_BF16); out [T, d] in out_dt. */
moe_status_t moe_combine(const void *y_perm, moe_dtype_t y_dt,
                         const int32_t *slot_to_row, const float *topk_w,
                         int64_t T, int32_t k, int64_t d, const void *shared_y,
                         void *out, moe_dtype_t out_dt, moe_stream_t stream);

/* One-time weight packing for one expert (not part of the timed forward).
 * Logical w_gate [d, I], w_up [d, I], w_down [I, d] in src_dt (MOE_F32 or
 * MOE_BF16) -> w13_e [2I, d] and w2_e [d, I] in dst_dt (the transposes, tiled
 * for bf16 and e4m3 as moe_weights_t describes).  dst_dt = MOE_E4M3 (from bf16 or f32) quantises per 128x128
 * block of the logical matrices with the moe_permute rule and writes the block
 * scales s13_e [2I/128, d/128] and s2_e [d/128, I/128]. */
moe_status_t moe_pack_weights(const void *w_gate, const void *w_up,
                              const void *w_down, moe_dtype_t src_dt, int64_t d,
                              int64_t I, moe_dtype_t dst_dt, void *w13_e,
                              void *w2_e, float *s13_e, float *s2_e,
                              moe_stream_t stream);

/* Bytes of workspace moe_layer_forward needs. */
size_t moe_layer_workspace_size(const moe_shape_t *shape);

/* The whole layer forward on one stream: route (with w->selection_bias when set)
 * -> dispatch layout (-> EPLB map on this batch's counts, or the round-robin
 * placement, and the physical layout) -> permute (e4m3 + dequantisation with
 * fp8_dispatch) -> expert FFN (+ shared expert) -> combine.  logits [T, E] fp32, x [T, d] in act_dtype,
 * out [T, d] in act_dtype.  `aux` (nullable, host struct) exposes intermediate
 * results.  ws: moe_layer_workspace_size(shape) bytes, 256-byte aligned.  No host
 * synchronisation happens inside. */
moe_status_t moe_layer_forward(const moe_shape_t *shape, const float *logits,
                               const void *x, const moe_weights_t *w, void *out,
                               const moe_layer_aux_t *aux, void *ws,
                               size_t ws_bytes, int32_t *err,
                               moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
