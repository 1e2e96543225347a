// C ABI glue: status strings, the expert-FFN dispatcher and the whole-layer
// forward ("6.4 Data parallelism and expert parallelism", section 3.1: Route ->
// Dispatch -> Expert compute -> Combine, all on one GPU and one stream).
#include "common.cuh"
#include "ffn.cuh"

namespace moe {

size_t dispatch_ws_bytes(int64_t T, int32_t k, int64_t P);
moe_status_t dispatch_layout(const int32_t *, int64_t, int32_t, int64_t, int32_t, const moe_eplb_t *, int32_t *,
                             int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, moe_load_stats_t *,
                             void *, size_t, int32_t *, cudaStream_t);
moe_status_t eplb_balanced_map(const int32_t *, int64_t, int32_t, int32_t, int32_t *, int32_t *, int32_t *,
                               int32_t *, double *, cudaStream_t);
moe_status_t placement_map(const int32_t *, int64_t, int32_t, int32_t, int32_t, int32_t *, int32_t *, int32_t *,
                           int32_t *, cudaStream_t);
moe_status_t route_layout_small(const float *, const float *, int64_t, int64_t, int32_t, int32_t, const moe_eplb_t *,
                                int32_t *, float *, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *,
                                int32_t *, moe_load_stats_t *, int32_t *, cudaStream_t);
moe_status_t eplb_map(const int32_t *, int64_t, int32_t, int32_t, int32_t *, int32_t *, int32_t *, int32_t *,
                      cudaStream_t);
moe_status_t permute(const void *, moe_dtype_t, int64_t, int64_t, int32_t, const int32_t *, void *, moe_dtype_t,
                     float *, cudaStream_t);
moe_status_t dequantize_e4m3(const void *, const float *, int64_t, int64_t, void *, cudaStream_t);
moe_status_t combine(const void *, moe_dtype_t, const int32_t *, const float *, int64_t, int32_t, int64_t,
                     const void *, void *, moe_dtype_t, cudaStream_t);

size_t h_bytes(int64_t rows, int64_t I, moe_dtype_t dt) {
  if (dt == MOE_F32) return (size_t)rows * I * 4;
  if (dt == MOE_BF16) return (size_t)rows * I * 2;
  return align_up((size_t)rows * I, 256) + (size_t)rows * (I / 128) * 4;
}

size_t ffn_ws_bytes(int64_t rows, int64_t I, moe_dtype_t dt) { return align_up(h_bytes(rows, I, dt), 256); }

static moe_status_t check_ffn(const int32_t *offs, int64_t P, int64_t N, const moe_weights_t *w, int64_t T_shared) {
  if (!w || !offs || P < 1 || N < 0 || T_shared < 0) return MOE_ERR_INVALID_ARG;
  if (!w->w13 || !w->w2 || w->d <= 0 || w->I <= 0 || w->E_w < 1) return MOE_ERR_INVALID_ARG;
  if (w->dtype == MOE_E4M3 && (!w->s13 || !w->s2)) return MOE_ERR_INVALID_ARG;
  if (T_shared > 0 && !w->has_shared) return MOE_ERR_INVALID_ARG;
  if (N + T_shared > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (w->dtype == MOE_E4M3 && T_shared > 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static FfnArgs ffn_args(const void *x_perm, const float *x_scales, const int32_t *offs, int64_t P, const int32_t *p2l,
                        int64_t N, const moe_weights_t *w, const void *shared_x, int64_t T_shared, void *h,
                        float *h_scales, void *y, int32_t *err) {
  FfnArgs a;
  a.x_perm = x_perm;
  a.x_scales = x_scales;
  a.offs = offs;
  a.p2l = p2l;
  a.P = P;
  a.N = N;
  a.w = w;
  a.shared_x = shared_x;
  a.T_shared = T_shared;
  a.h = h;
  a.h_scales = h_scales;
  a.y = y;
  a.err = err;
  return a;
}

moe_status_t gate_up(const FfnArgs &a, cudaStream_t st) {
  switch (a.w->dtype) {
    case MOE_F32: return gate_up_f32(a, st);
    case MOE_BF16: return gate_up_bf16(a, st);
    case MOE_E4M3: return gate_up_e4m3(a, st);
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status_t down(const FfnArgs &a, cudaStream_t st) {
  switch (a.w->dtype) {
    case MOE_F32: return down_f32(a, st);
    case MOE_BF16: return down_bf16(a, st);
    case MOE_E4M3: return down_e4m3(a, st);
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status_t expert_ffn(const void *x_perm, const float *x_scales, const int32_t *offs, int64_t P, const int32_t *p2l,
                        int64_t N, const moe_weights_t *w, const void *shared_x, int64_t T_shared, void *y, void *ws,
                        size_t ws_bytes, int32_t *err, cudaStream_t st) {
  moe_status_t r = check_ffn(offs, P, N, w, T_shared);
  if (r != MOE_OK) return r;
  if ((N > 0 && !x_perm) || (T_shared > 0 && !shared_x) || !y) return MOE_ERR_INVALID_ARG;
  if (w->dtype == MOE_E4M3 && N > 0 && !x_scales) return MOE_ERR_INVALID_ARG;
  const int64_t rows = N + T_shared;
  if (!ws || ws_bytes < ffn_ws_bytes(rows, w->I, w->dtype) || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  float *hs = w->dtype == MOE_E4M3
                  ? reinterpret_cast<float *>(static_cast<char *>(ws) + align_up((size_t)rows * w->I, 256))
                  : nullptr;
  const FfnArgs a = ffn_args(x_perm, x_scales, offs, P, p2l, N, w, shared_x, T_shared, ws, hs, y, err);
  if ((r = gate_up(a, st)) != MOE_OK) return r;
  return down(a, st);
}

// ------------------------------------------------------------------ layer forward
struct LayerPlan {
  int64_t T, N, P, d, I, E;
  int32_t k, R;
  size_t act_bytes, perm_bytes, y_bytes;
  bool eplb, shared, balanced, round_robin, mapped, fp8_dispatch;
  // byte offsets into the workspace
  size_t o_ids, o_w, o_lc, o_pc, o_po, o_rc, o_ro, o_r2t, o_s2r, o_stats, o_p2l, o_prank, o_repc, o_l2p, o_disp,
      o_xp, o_xq, o_xs, o_y, o_ffn, total;
};

static bool plan_layer(const moe_shape_t *s, LayerPlan *p) {
  if (!s || s->T < 0 || s->d <= 0 || s->E < 1 || s->I <= 0 || s->k < 1 || s->R < 1) return false;
  if (s->act_dtype == MOE_F32 && s->expert_dtype != MOE_F32) return false;
  if (s->act_dtype == MOE_BF16 && s->expert_dtype == MOE_F32) return false;
  if (s->act_dtype == MOE_E4M3) return false;
  p->T = s->T;
  p->k = s->k;
  p->R = s->R;
  p->E = s->E;
  p->d = s->d;
  p->I = s->I;
  p->N = s->T * s->k;
  p->eplb = s->n_redundant > 0;
  if (s->eplb_placement != 0 && s->eplb_placement != 1) return false;
  p->balanced = p->eplb && s->eplb_placement == 1;
  if (s->expert_placement != 0 && s->expert_placement != 1) return false;
  p->round_robin = s->expert_placement == 1;
  p->mapped = p->eplb || p->round_robin;  // physical ids differ from logical ones
  if (s->fp8_dispatch != 0 && s->fp8_dispatch != 1) return false;
  // bf16 experts fed from an e4m3 dispatch (e4m3 experts always are)
  p->fp8_dispatch = s->fp8_dispatch == 1 && s->expert_dtype == MOE_BF16;
  if (s->fp8_dispatch == 1 && s->expert_dtype == MOE_F32) return false;
  if (p->fp8_dispatch && s->d % 128) return false;
  p->shared = s->shared != 0;
  p->P = s->E + s->n_redundant;
  p->act_bytes = s->act_dtype == MOE_F32 ? 4 : 2;
  p->perm_bytes = s->expert_dtype == MOE_E4M3 ? 1 : p->act_bytes;
  p->y_bytes = s->expert_dtype == MOE_F32 ? 4 : 2;
  const int64_t rows = p->N + (p->shared ? p->T : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o += align_up(bytes, 256);
    return at;
  };
  p->o_ids = take((size_t)p->N * 4);
  p->o_w = take((size_t)p->N * 4);
  p->o_lc = take((size_t)p->E * 4);
  p->o_pc = take((size_t)p->P * 4);
  p->o_po = take((size_t)(p->P + 1) * 4);
  p->o_rc = take((size_t)p->R * 4);
  p->o_ro = take((size_t)(p->R + 1) * 4);
  p->o_r2t = take((size_t)p->N * 4);
  p->o_s2r = take((size_t)p->N * 4);
  p->o_stats = take(2 * sizeof(moe_load_stats_t));
  p->o_p2l = take((size_t)p->P * 4);
  p->o_prank = take((size_t)p->P * 4);
  p->o_repc = take((size_t)p->E * 4);
  p->o_l2p = take((size_t)p->E * 4 * (p->balanced ? 1 + s->n_redundant : 2));
  p->o_disp = take(dispatch_ws_bytes(p->T, p->k, p->P));
  p->o_xp = take((size_t)p->N * p->d * p->perm_bytes);
  p->o_xq = take(p->fp8_dispatch ? (size_t)p->N * p->d : 0);
  p->o_xs = take(s->expert_dtype == MOE_E4M3 || p->fp8_dispatch ? (size_t)p->N * (p->d / 128) * 4 : 0);
  p->o_y = take((size_t)rows * p->d * p->y_bytes);
  p->o_ffn = take(ffn_ws_bytes(rows, p->I, s->expert_dtype));
  p->total = o;
  return true;
}

}  // namespace moe

using namespace moe;

cudaError_t &moe::last_cuda_error() {
  static thread_local cudaError_t e = cudaSuccess;
  return e;
}

MOE_API const char *moe_last_cuda_error(void) {
  const cudaError_t e = last_cuda_error();
  return e == cudaSuccess ? "" : cudaGetErrorString(e);
}

MOE_API const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

MOE_API size_t moe_ffn_workspace_size(int64_t rows, int64_t I, moe_dtype_t dt) {
  if (rows < 0 || I <= 0) return 0;
  return ffn_ws_bytes(rows, I, dt);
}

MOE_API moe_status_t moe_expert_ffn(const void *x_perm, const float *x_scales, const int32_t *phys_offsets, int64_t P,
                                    const int32_t *phys_to_logical, int64_t rows_hint, const moe_weights_t *w,
                                    const void *shared_x, int64_t T_shared, void *y_perm, void *ws, size_t ws_bytes,
                                    int32_t *err, moe_stream_t stream) {
  return expert_ffn(x_perm, x_scales, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x, T_shared, y_perm, ws,
                    ws_bytes, err, as_cuda(stream));
}

MOE_API moe_status_t moe_expert_gate_up(const void *x_perm, const float *x_scales, const int32_t *phys_offsets,
                                        int64_t P, const int32_t *phys_to_logical, int64_t rows_hint,
                                        const moe_weights_t *w, const void *shared_x, int64_t T_shared, void *h,
                                        float *h_scales, int32_t *err, moe_stream_t stream) {
  moe_status_t r = check_ffn(phys_offsets, P, rows_hint, w, T_shared);
  if (r != MOE_OK) return r;
  if ((rows_hint > 0 && !x_perm) || (T_shared > 0 && !shared_x) || !h) return MOE_ERR_INVALID_ARG;
  if (w->dtype == MOE_E4M3 && ((rows_hint > 0 && !x_scales) || !h_scales)) return MOE_ERR_INVALID_ARG;
  return gate_up(ffn_args(x_perm, x_scales, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x, T_shared, h,
                          h_scales, nullptr, err),
                 as_cuda(stream));
}

MOE_API moe_status_t moe_expert_gate_up_gather(const void *x, int64_t T, const int32_t *row_to_token,
                                               const int32_t *phys_offsets, int64_t P,
                                               const int32_t *phys_to_logical, int64_t rows_hint,
                                               const moe_weights_t *w, const void *shared_x, int64_t T_shared,
                                               void *h, int32_t *err, moe_stream_t stream) {
  moe_status_t r = check_ffn(phys_offsets, P, rows_hint, w, T_shared);
  if (r != MOE_OK) return r;
  if (w->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || T > INT32_MAX || (T_shared > 0 && !shared_x) || !h) return MOE_ERR_INVALID_ARG;
  if (rows_hint > 0 && (!x || T < 1 || !row_to_token)) return MOE_ERR_INVALID_ARG;
  FfnArgs a = ffn_args(nullptr, nullptr, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x, T_shared, h,
                       nullptr, nullptr, err);
  if (rows_hint > 0) {
    a.gather_rows = row_to_token;
    a.gather_x = x;
    a.gather_T = T;
  } else {
    a.x_perm = nullptr;  // only the shared expert's rows: the plain kernel
  }
  return gate_up(a, as_cuda(stream));
}

MOE_API moe_status_t moe_expert_down(const void *h, const float *h_scales, const int32_t *phys_offsets, int64_t P,
                                     const int32_t *phys_to_logical, int64_t rows_hint, const moe_weights_t *w,
                                     int64_t T_shared, void *y_perm, int32_t *err, moe_stream_t stream) {
  moe_status_t r = check_ffn(phys_offsets, P, rows_hint, w, T_shared);
  if (r != MOE_OK) return r;
  if (!h || !y_perm || (w->dtype == MOE_E4M3 && !h_scales)) return MOE_ERR_INVALID_ARG;
  return down(ffn_args(nullptr, nullptr, phys_offsets, P, phys_to_logical, rows_hint, w, nullptr, T_shared,
                       const_cast<void *>(h), const_cast<float *>(h_scales), y_perm, err),
              as_cuda(stream));
}

MOE_API moe_status_t moe_expert_down_combine(const void *h, const int32_t *phys_offsets, int64_t P,
                                             const int32_t *phys_to_logical, int64_t rows_hint,
                                             const moe_weights_t *w, int64_t T_shared, const int32_t *row_to_token,
                                             const int32_t *slot_to_row, const float *topk_w, int64_t T, int32_t k,
                                             void *y_perm, int32_t *counts, void *out, int32_t *err,
                                             moe_stream_t stream) {
  moe_status_t r = check_ffn(phys_offsets, P, rows_hint, w, T_shared);
  if (r != MOE_OK) return r;
  if (w->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || k < 1 || k > 32 || rows_hint > T * (int64_t)k || (T_shared != 0 && T_shared != T))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!h || !y_perm || !row_to_token || !slot_to_row || !topk_w || !counts || !out) return MOE_ERR_INVALID_ARG;
  FfnArgs a = ffn_args(nullptr, nullptr, phys_offsets, P, phys_to_logical, rows_hint, w, nullptr, T_shared,
                       const_cast<void *>(h), nullptr, y_perm, err);
  a.c_row_to_token = row_to_token;
  a.c_slot_to_row = slot_to_row;
  a.c_topk_w = topk_w;
  a.c_counts = counts;
  a.c_out = out;
  a.c_T = T;
  a.c_k = k;
  return down(a, as_cuda(stream));
}

MOE_API size_t moe_layer_workspace_size(const moe_shape_t *shape) {
  LayerPlan p;
  if (!plan_layer(shape, &p)) return 0;
  return p.total;
}

MOE_API moe_status_t moe_layer_forward(const moe_shape_t *s, const float *logits, const void *x,
                                       const moe_weights_t *w, void *out, const moe_layer_aux_t *aux, void *ws,
                                       size_t ws_bytes, int32_t *err, moe_stream_t stream) {
  LayerPlan p;
  if (!plan_layer(s, &p) || !w) return MOE_ERR_INVALID_ARG;
  if (w->dtype != s->expert_dtype || w->d != s->d || w->I != s->I) return MOE_ERR_INVALID_ARG;
  if (w->E_w < s->E + (p.shared ? 1 : 0) || (p.shared && !w->has_shared)) return MOE_ERR_INVALID_ARG;
  if (p.T == 0) return MOE_OK;
  if (!logits || !x || !out) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < p.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = as_cuda(stream);
  char *base = static_cast<char *>(ws);
  auto pick = [&](auto *user, size_t off) {
    using Ptr = decltype(user);
    return user ? user : reinterpret_cast<Ptr>(base + off);
  };
  moe_layer_aux_t none{};
  const moe_layer_aux_t &ax = aux ? *aux : none;
  int32_t *ids = pick(ax.topk_ids, p.o_ids);
  float *tw = pick(ax.topk_w, p.o_w);
  int32_t *lc = pick(ax.logical_counts, p.o_lc);
  int32_t *pc = pick(ax.phys_counts, p.o_pc);
  int32_t *po = pick(ax.phys_offsets, p.o_po);
  int32_t *rc = pick(ax.rank_counts, p.o_rc);
  int32_t *ro = pick(ax.rank_offsets, p.o_ro);
  int32_t *r2t = pick(ax.row_to_token, p.o_r2t);
  int32_t *s2r = pick(ax.slot_to_row, p.o_s2r);
  moe_load_stats_t *stats = pick(ax.stats, p.o_stats);
  int32_t *p2l = pick(ax.phys_to_logical, p.o_p2l);
  int32_t *prank = pick(ax.phys_rank, p.o_prank);
  int32_t *repc = pick(ax.replica_count, p.o_repc);
  int32_t *l2p = pick(ax.logical_to_phys, p.o_l2p);
  void *disp = base + p.o_disp;
  void *xp = base + p.o_xp;
  float *xs = reinterpret_cast<float *>(base + p.o_xs);
  char *y = base + p.o_y;
  void *fws = base + p.o_ffn;
  const size_t disp_bytes = dispatch_ws_bytes(p.T, p.k, p.P);

  moe_status_t r;
  moe_eplb_t map{(int32_t)p.P, p2l, repc, l2p, p.balanced ? (int32_t)(1 + p.P - p.E) : 2, p.round_robin ? 1 : 0};
  bool laid_out = false;
  if (!p.eplb) {
    // no replicas: the map (if any) does not depend on the routing, and a batch of
    // at most one count chunk is routed and laid out by one launch
    if (p.round_robin && (r = placement_map(nullptr, p.E, p.R, 0, 1, p2l, prank, repc, l2p, st)) != MOE_OK)
      return r;
    r = route_layout_small(logits, w->selection_bias, p.T, p.E, p.k, p.R, p.mapped ? &map : nullptr, ids, tw, lc,
                           pc, po, rc, ro, r2t, s2r, stats, err, st);
    if (r == MOE_OK)
      laid_out = true;
    else if (r != MOE_ERR_UNSUPPORTED)
      return r;
  }
  if (!laid_out && (r = moe_route_biased(logits, w->selection_bias, p.T, p.E, p.k, ids, tw, err, stream)) != MOE_OK)
    return r;
  if (p.eplb) {
    // counts of this batch's logical routing, then the replica map built on them
    if ((r = dispatch_layout(ids, p.T, p.k, p.E, p.R, nullptr, lc, pc, po, rc, ro, r2t, s2r, stats, disp,
                             disp_bytes, err, st)) != MOE_OK)
      return r;
    r = p.balanced ? eplb_balanced_map(lc, p.E, p.R, (int32_t)(p.P - p.E), p2l, prank, repc, l2p, nullptr, st)
                   : placement_map(lc, p.E, p.R, (int32_t)(p.P - p.E), p.round_robin ? 1 : 0, p2l, prank, repc,
                                   l2p, st);
    if (r != MOE_OK) return r;
  }
  if (!laid_out && (r = dispatch_layout(ids, p.T, p.k, p.E, p.R, p.mapped ? &map : nullptr, lc, pc, po, rc, ro, r2t,
                                        s2r, stats, disp, disp_bytes, err, st)) != MOE_OK)
    return r;
  if (p.fp8_dispatch) {
    // the send buffer holds e4m3 rows and their scales; the receive side rebuilds bf16 rows
    void *xq = base + p.o_xq;
    if ((r = permute(x, s->act_dtype, p.T, p.d, p.k, s2r, xq, MOE_E4M3, xs, st)) != MOE_OK) return r;
    if ((r = dequantize_e4m3(xq, xs, p.N, p.d, xp, st)) != MOE_OK) return r;
  } else {
    const moe_dtype_t perm_dt = s->expert_dtype == MOE_E4M3 ? MOE_E4M3 : s->act_dtype;
    if ((r = permute(x, s->act_dtype, p.T, p.d, p.k, s2r, xp, perm_dt, xs, st)) != MOE_OK) return r;
  }
  const int64_t T_sh = p.shared ? p.T : 0;
  if ((r = expert_ffn(xp, xs, po, p.P, p.mapped ? p2l : nullptr, p.N, w, p.shared ? x : nullptr, T_sh, y, fws,
                      ffn_ws_bytes(p.N + T_sh, p.I, s->expert_dtype), err, st)) != MOE_OK)
    return r;
  const moe_dtype_t y_dt = s->expert_dtype == MOE_F32 ? MOE_F32 : MOE_BF16;
  const void *shared_y = p.shared ? y + (size_t)p.N * p.d * p.y_bytes : nullptr;
  return combine(y, y_dt, s2r, tw, p.T, p.k, p.d, shared_y, out, s->act_dtype, st);
}
