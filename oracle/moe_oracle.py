"""CPU oracle for the routed MoE layer forward (test infrastructure only).

This file is the plain, slow, float64 statement of what the layer computes.
It exists to check the CUDA library: only the tests, the package's smoke check
and the benchmark's CPU-baseline leg may import it.  It shares no code with the
CUDA path; its only inputs are arrays.

Sources (page title, then the section the step follows):

* "6.4 Data parallelism and expert parallelism", section 3.1 "Dataflow inside one
  MoE layer": the four steps Route -> Dispatch -> Expert compute -> Combine.
* same page, section 2.1: one expert is the three matrices gate, up, down.
* same page, section 5.1 and 5.2: per-card load, "busiest card / average".
* same page, section 5.3: EPLB, (experts + redundant) / EP physical experts per card;
  balancedness = average / max.
* same page, section 7: the shared expert is a must-pick expert ("picks 9").
* "Your expert-parallel deployment is slower than the tensor-parallel one. Find out
  why.", "The three causes": compare max rank load against mean rank load.
* "How Expert Parallelism Works for Mixture-of-Experts Models in vLLM", "MoE Layer
  Construction": num_physical_experts = num_experts + num_redundant_experts.
* same page, "Configuring Expert Parallelism": "linear" or "round_robin" placement.

Readings where the pages are silent (each one is listed with its reason in the
design notes): selection is on the fp32 logits, ties go to the lower expert index,
-0 equals +0; weights are the softmax over all E renormalised over the chosen k;
SwiGLU is silu(x W_gate) * (x W_up) then W_down; rows are ordered by physical
expert, then by token; EPLB replicas go to the n_red hottest experts (count desc,
index asc), replica j to rank j mod R, token t uses replica t mod replica_count;
round-robin placement puts expert e on rank e mod R in local slot e div R;
the shared expert has weight 1 and is not renormalised; bf16 workloads round h and
y to bf16 where the kernels store them; fp8 workloads quantise x and h per token per
128-channel group and the weights per 128x128 block with scale = amax/448 (fp32)
and e4m3 round-to-nearest-even with saturation.

Every function here is pinned by a test against something other than itself
(brute force, closed forms, the pages' printed numbers, library special cases);
the dense FFN values beyond those reductions rest on this definition.
"""
from __future__ import annotations

import heapq

import numpy as np

# ============================================================== route
def route(logits: np.ndarray, k: int):
    """Top-k routing ("6.4 ...", section 3.1, step 1 Route).

    For each token, order the experts by (logit descending, expert index ascending)
    and keep the first k.  The weights are the softmax over all E experts,
    renormalised over the chosen k; the full softmax denominator cancels, so
    w_j = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max), in float64.
    Returns (topk_ids int32 [T,k], topk_w float64 [T,k]).
    """
    L = np.asarray(logits, dtype=np.float32)
    if not np.all(np.isfinite(L)):
        raise ValueError("non-finite router logit")
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # A stable sort of -logit keeps equal logits in ascending expert order;
    # numpy compares -0.0 and +0.0 as equal, so they tie as the reading requires.
    order = np.argsort(-L.astype(np.float64), axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    l64 = L.astype(np.float64)
    sel = np.take_along_axis(l64, order[:, :k], axis=1)
    lmax = l64.max(axis=1, keepdims=True)
    e = np.exp(sel - lmax)
    w = e / e.sum(axis=1, keepdims=True)
    return ids, w


def route_softmax_then_renorm(logits: np.ndarray, k: int):
    """The same weights written the long way: softmax over E, take the top-k
    probabilities, divide by their sum.  Used to check route()."""
    l64 = np.asarray(logits, dtype=np.float32).astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ids, _ = route(logits, k)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    return ids, sel / sel.sum(axis=1, keepdims=True)


def route_selection_bias(logits: np.ndarray, bias: np.ndarray, k: int):
    """Top-k routing with a selection bias ("6.4 ...", section 5.1: a bias term
    instead of an auxiliary loss keeps expert counts even).  The experts are chosen
    by the score logit + b_e, summed in float32 as the router's inputs are, ordered
    (score descending, expert index ascending); the weights come from the unbiased
    logits of the chosen experts: w_j = exp(l_j - m) / sum_i exp(l_i - m), m the
    largest chosen logit, in float64.  bias = 0 gives route()."""
    L = np.asarray(logits, dtype=np.float32)
    b = np.asarray(bias, dtype=np.float32)
    score = L + b[None, :]                       # float32 + float32 -> float32
    if not (np.all(np.isfinite(L)) and np.all(np.isfinite(score))):
        raise ValueError("non-finite router logit or score")
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    order = np.argsort(-score.astype(np.float64), axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(L.astype(np.float64), order[:, :k], axis=1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    return ids, e / e.sum(axis=1, keepdims=True)


# ============================================================== load statistics
def rank_stats(rank_counts: np.ndarray, total_copies: int) -> dict:
    """Per-rank load ("Your expert-parallel deployment ...", "The three causes":
    max rank load against mean rank load; "6.4 ...", section 5.3: balancedness =
    average / max).  Counts are token-copies (t, j)."""
    rc = np.asarray(rank_counts, dtype=np.int64)
    R = rc.size
    mean = total_copies / R
    mx = int(rc.max()) if R else 0
    return {
        "max_rank": mx,
        "mean_rank": mean,
        "max_over_mean": (mx / mean) if mean > 0 else 0.0,
        "balancedness": (mean / mx) if mx > 0 else 0.0,
    }


def linear_rank_counts(expert_counts: np.ndarray, R: int) -> np.ndarray:
    """Linear ("contiguous") placement: rank r owns experts r*(P/R) .. (r+1)*(P/R)-1
    ("How Expert Parallelism Works ...", "Configuring Expert Parallelism";
    "6.4 ...", section 5.2, the contiguous placement)."""
    c = np.asarray(expert_counts, dtype=np.int64)
    if c.size % R:
        raise ValueError("experts must divide evenly over ranks")
    return c.reshape(R, c.size // R).sum(axis=1)


def round_robin_rank_counts(expert_counts: np.ndarray, R: int) -> np.ndarray:
    """Round-robin placement: rank r owns experts r, r + R, r + 2R, ... ("How Expert
    Parallelism Works ...", "Configuring Expert Parallelism", "round_robin"; the page
    names the strategy only, so experts are dealt to the ranks in index order)."""
    c = np.asarray(expert_counts, dtype=np.int64)
    if c.size % R:
        raise ValueError("experts must divide evenly over ranks")
    return np.array([c[r::R].sum() for r in range(R)], dtype=np.int64)


def base_rank_counts(expert_counts: np.ndarray, R: int, placement: str = "linear") -> np.ndarray:
    if placement == "linear":
        return linear_rank_counts(expert_counts, R)
    if placement == "round_robin":
        return round_robin_rank_counts(expert_counts, R)
    raise ValueError(f"unknown placement {placement!r}")


def eplb_balanced_map(logical_counts, R: int, n_redundant: int) -> dict:
    """Load-aware placement with redundant slots ("6.4 Data parallelism and expert
    parallelism", section 5.2, the rebalanced placement with one redundant slot per
    card), written out as a physical-expert map in the format of eplb_map.

    The rule, as the section states it: every redundant slot goes to the expert that
    carries the most load per replica, an expert's load is split evenly over its
    replicas, and the replicas are placed heaviest first, each on the least loaded
    card that still has a free slot; each card has S = (E + n_red) / R slots.

    Tie rules (the section leaves them open; these are the readings):
      * equal load per replica: the lower expert id takes the slot;
      * equal replica loads: expert id ascending, then replica index ascending;
      * equal card loads: the lower rank.
    The replica j of expert e is its j-th replica in the placement order, and a card
    fills its slots in the order replicas arrive, so physical id = rank * S + slot.
    Loads are float64 count / replicas, and a card's load is summed in arrival order.
    Returns the map plus rank_load, the per-card load the section tabulates."""
    counts = [int(c) for c in np.asarray(logical_counts).ravel()]
    E = len(counts)
    P = E + n_redundant
    if P % R:
        raise ValueError("physical experts must divide evenly over ranks")
    S = P // R
    # 1. redundant slots: a max-heap on load per replica, lower id first on ties
    replicas = [1] * E
    heap = [(-float(counts[e]), e) for e in range(E)]
    heapq.heapify(heap)
    for _ in range(n_redundant):
        _, e = heapq.heappop(heap)
        replicas[e] += 1
        heapq.heappush(heap, (-(counts[e] / replicas[e]), e))
    # 2. every replica with its load, heaviest first
    pieces = sorted(((counts[e] / replicas[e], e, j) for e in range(E) for j in range(replicas[e])),
                    key=lambda c: (-c[0], c[1], c[2]))
    # 3. cards with a free slot in a min-heap on (load, rank)
    cards = [(0.0, r) for r in range(R)]
    used = [0] * R
    load = [0.0] * R
    phys_to_logical = np.empty(P, dtype=np.int32)
    phys_rank = np.empty(P, dtype=np.int32)
    logical_to_phys = np.full((E, 1 + n_redundant), -1, dtype=np.int32)
    for c, e, j in pieces:
        _, g = heapq.heappop(cards)
        p = g * S + used[g]
        used[g] += 1
        load[g] += c
        if used[g] < S:
            heapq.heappush(cards, (load[g], g))
        phys_to_logical[p] = e
        phys_rank[p] = g
        logical_to_phys[e, j] = p
    return {"P": P, "phys_to_logical": phys_to_logical, "phys_rank": phys_rank,
            "replica_count": np.array(replicas, dtype=np.int32), "logical_to_phys": logical_to_phys,
            "rank_load": np.array(load)}


def eplb_window_sum(history, W: int) -> np.ndarray:
    """EPLB's load window ("6.4 ...", section 5.3: per-expert load over window_size
    recent steps): the per-expert sum of the last W per-step logical count vectors
    (all of them while fewer than W have been seen)."""
    h = [np.asarray(c, dtype=np.int64) for c in history]
    if W < 1 or not h:
        raise ValueError("need W >= 1 and at least one step")
    return np.sum(h[-W:], axis=0)


# ============================================================== EPLB map
def eplb_map(logical_counts: np.ndarray, R: int, n_redundant: int, placement: str = "linear") -> dict:
    """One-step redundant-expert map ("6.4 ...", section 5.3; "How Expert
    Parallelism Works ...", "MoE Layer Construction" and "Configuring Expert
    Parallelism" for the placement strategy).

    P = E + n_red physical experts, S = P / R per rank.  Rank r holds, in its slots
    0 .. E/R-1, its base experts, then replicas: linear placement gives rank r the
    logical experts r*E/R + slot, round-robin the experts r + slot*R.
    The n_red hottest logical experts (count desc, index asc) get one replica each;
    the j-th hottest goes to rank j mod R, slot E/R + j div R.  Physical id = r*S + slot.
    With n_red = 0 this is the bare placement (the counts are not used).
    """
    c = np.asarray(logical_counts, dtype=np.int64)
    E = c.size
    if E % R or n_redundant % R or n_redundant > E:
        raise ValueError("unsupported EPLB geometry")
    if placement not in ("linear", "round_robin"):
        raise ValueError(f"unknown placement {placement!r}")
    P = E + n_redundant
    S, base = P // R, E // R
    hot = np.argsort(-c, kind="stable")[:n_redundant]
    phys_to_logical = np.empty(P, dtype=np.int32)
    phys_rank = np.empty(P, dtype=np.int32)
    logical_to_phys = np.full((E, 2), -1, dtype=np.int32)
    replica_count = np.ones(E, dtype=np.int32)
    for r in range(R):
        for s in range(base):
            e = r * base + s if placement == "linear" else r + s * R
            p = r * S + s
            phys_to_logical[p] = e
            phys_rank[p] = r
            logical_to_phys[e, 0] = p
    for j, e in enumerate(hot):
        r, s = j % R, base + j // R
        p = r * S + s
        phys_to_logical[p] = e
        phys_rank[p] = r
        logical_to_phys[e, 1] = p
        replica_count[e] = 2
    return {"P": P, "phys_to_logical": phys_to_logical, "phys_rank": phys_rank,
            "replica_count": replica_count, "logical_to_phys": logical_to_phys,
            "hot": hot.astype(np.int32)}


# ============================================================== dispatch layout
def dispatch_layout(topk_ids: np.ndarray, E: int, R: int, eplb: dict | None = None,
                    placement: str = "linear") -> dict:
    """Counting, scan and the EP-rank-ordered layout ("6.4 ...", section 3.1 step 2
    Dispatch: each token is copied k times to the cards owning its experts; the
    figure's per-card copy counts).

    Physical id of slot (t, j): the logical id e, or with EPLB
    logical_to_phys[e][t mod replica_count[e]].  Physical ids are numbered
    rank-major, so ordering rows by physical id orders them by (rank, expert);
    inside an expert, rows are in ascending token order.  The "before" statistics
    count the logical experts on the ranks of the base `placement`.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    logical_counts = np.bincount(ids.ravel(), minlength=E).astype(np.int64)
    if eplb is None:
        P = E
        phys = ids
    else:
        P = eplb["P"]
        t = np.arange(T)[:, None]
        rep = t % eplb["replica_count"][ids]
        phys = eplb["logical_to_phys"][ids, rep].astype(np.int64)
    flat = phys.ravel()                       # slot order s = t*k + j
    order = np.argsort(flat, kind="stable")   # rows: physical id asc, then slot asc
    N = flat.size
    row_to_token = (order // k).astype(np.int32)
    slot_to_row = np.empty(N, dtype=np.int32)
    slot_to_row[order] = np.arange(N, dtype=np.int32)
    phys_counts = np.bincount(flat, minlength=P).astype(np.int64)
    phys_offsets = np.concatenate([[0], np.cumsum(phys_counts)]).astype(np.int64)
    rank_counts = linear_rank_counts(phys_counts, R)
    rank_offsets = np.concatenate([[0], np.cumsum(rank_counts)]).astype(np.int64)
    before = rank_stats(base_rank_counts(logical_counts, R, placement), N)
    after = rank_stats(rank_counts, N)
    for st, cnt in ((before, logical_counts), (after, phys_counts)):
        st["max_expert"] = int(cnt.max()) if cnt.size else 0
        st["n_active_experts"] = int((cnt > 0).sum())
    return {
        "P": P, "phys_ids": phys.astype(np.int32),
        "logical_counts": logical_counts, "phys_counts": phys_counts,
        "phys_offsets": phys_offsets, "rank_counts": rank_counts,
        "rank_offsets": rank_offsets, "row_to_token": row_to_token,
        "slot_to_row": slot_to_row.reshape(T, k),
        "stats_before": before, "stats_after": after,
    }


# ============================================================== number formats
def round_bf16(v) -> np.ndarray:
    """Round to bfloat16 (via float32, each step round-to-nearest-even); float64 out."""
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_next_up(r: np.ndarray) -> np.ndarray:
    """The bfloat16 value next above each bfloat16 value r."""
    f = np.ascontiguousarray(np.asarray(r, dtype=np.float32))
    u = f.view(np.uint32).astype(np.int64)
    u = np.where(f > 0, u + 0x10000, np.where(f < 0, u - 0x10000, 0x00010000))
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_bracket(v):
    """The two bfloat16 values around each v: lo <= v <= hi (equal when v is one).
    A computation whose own value of v lies on the other side of the midpoint
    between them rounds to the other one; both are correct roundings of v."""
    v = np.asarray(v, dtype=np.float64)
    r = round_bf16(v)
    lo = np.where(r <= v, r, -_bf16_next_up(-r))
    hi = np.where(r >= v, r, _bf16_next_up(r))
    return lo, hi


def bf16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_value(code: int) -> float:
    """OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (m/8 * 2^-6); 0x7F / 0xFF are NaN; no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    ex, m = (code >> 3) & 0xF, code & 7
    if ex == 15 and m == 7:
        return float("nan")
    if ex == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (ex - 7)


_E4M3_POS = np.array([e4m3_value(c) for c in range(0x7F)])   # codes 0..126, ascending


def e4m3_encode(v) -> np.ndarray:
    """float32 -> e4m3 code, round to nearest (ties to the even code), saturating to
    +-448 (the largest finite magnitude).  Inputs must be finite."""
    a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
    neg = np.signbit(np.asarray(v, dtype=np.float32))
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # first table value >= a
    hi = np.minimum(hi, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(a >= _E4M3_POS[-1], len(_E4M3_POS) - 1, np.where(pick_hi, hi, lo))
    code = np.where(a <= _E4M3_POS[0], 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    tab = np.array([e4m3_value(c) for c in range(256)])
    return tab[np.asarray(codes, dtype=np.uint8)]


def quantize_groups(v, group: int = 128):
    """Per-row, per-`group`-channel e4m3 quantisation (the activation rule):
    scale = amax / 448 in float32 (1 when amax is 0), code = e4m3(v / scale) with the
    division in float32.  Returns (codes uint8 [rows, n], scales float32 [rows, n/group])."""
    f = np.asarray(v, dtype=np.float32)
    rows, n = f.shape
    if n % group:
        raise ValueError("channel count must be a multiple of the group")
    g = f.reshape(rows, n // group, group)
    amax = np.abs(g).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (g / scale[:, :, None]).astype(np.float32)
    return e4m3_encode(q).reshape(rows, n), scale


def quantize_blocks(w, block: int = 128):
    """Per-`block`x`block` e4m3 quantisation of a matrix (the weight rule), with the
    same scale and rounding as quantize_groups.  Returns (codes [r, c], scales
    float32 [r/block, c/block])."""
    f = np.asarray(w, dtype=np.float32)
    r, c = f.shape
    if r % block or c % block:
        raise ValueError("matrix must tile by the block")
    b = f.reshape(r // block, block, c // block, block)
    amax = np.abs(b).max(axis=(1, 3))
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (b / scale[:, None, :, None]).astype(np.float32)
    return e4m3_encode(q).reshape(r, c), scale


def dequantize_blocks(codes, scales, block: int = 128) -> np.ndarray:
    v = e4m3_decode(codes)
    r, c = v.shape
    return (v.reshape(r // block, block, c // block, block)
            * scales.astype(np.float64)[:, None, :, None]).reshape(r, c)


def dequantize_groups_bf16(codes, scales, group: int = 128) -> np.ndarray:
    """The receive side of an FP8 dispatch to bf16 experts ("6.4 ...", section 3.2):
    each code times its group's scale as one IEEE float32 multiply (numpy's float32
    product), then rounded to bf16 to nearest even.  Returns float64 values."""
    v = e4m3_decode(codes).astype(np.float32)                 # exact: e4m3 is a subset of float32
    s = np.repeat(np.asarray(scales, dtype=np.float32), group, axis=1)
    return round_bf16((v * s).astype(np.float32))


def dequantize_groups(codes, scales, group: int = 128) -> np.ndarray:
    v = e4m3_decode(codes)
    rows, n = v.shape
    return (v.reshape(rows, n // group, group) * scales.astype(np.float64)[:, :, None]).reshape(rows, n)


# ============================================================== permute / FFN / combine
def permute(x: np.ndarray, row_to_token: np.ndarray) -> np.ndarray:
    """Dispatch copy ("6.4 ...", section 3.1 step 2): x_perm[r] = x[row_to_token[r]]."""
    return np.asarray(x)[np.asarray(row_to_token, dtype=np.int64)]


def silu(z):
    return z / (1.0 + np.exp(-z))


def stored_h(h, mode: str):
    """The intermediate h as the down projection takes it (the stored tensor between
    gate/up and down): "fp32" unchanged; "bf16" rounded to bf16 (RNE); "fp8"
    quantised to e4m3 per row over each 128-channel group of I and dequantised."""
    if mode == "bf16":
        return round_bf16(h)
    if mode == "fp8":
        q, s = quantize_groups(np.asarray(h).astype(np.float32))
        return dequantize_groups(q, s)
    return h


def stored_y(y, mode: str):
    """An expert's output row as the combine reads it: bf16 (RNE) for the bf16 and
    fp8 workloads ("6.4 ...", section 3.2: BF16 combine), unchanged for fp32."""
    return round_bf16(y) if mode in ("bf16", "fp8") else y


def swiglu_expert_exact(x64, wg64, wu64, wd64, mode: str):
    """One expert's FFN before its output is stored: h = silu(x W_gate) * (x W_up),
    stored as the mode stores it, then y = h W_down in float64."""
    g = x64 @ wg64
    u = x64 @ wu64
    h = stored_h(silu(g) * u, mode)
    return h @ wd64


def swiglu_expert(x64, wg64, wu64, wd64, mode: str):
    """One expert's FFN ("6.4 ...", section 2.1: gate, up, down):
    h = silu(x W_gate) * (x W_up); y = h W_down; float64 matmuls.

    mode "fp32": no intermediate rounding.  "bf16": h and y rounded to bf16 where the
    kernels store them.  "fp8": h quantised per row per 128 channels (e4m3), y
    rounded to bf16.  (x and the weights arrive already dequantised.)"""
    return stored_y(swiglu_expert_exact(x64, wg64, wu64, wd64, mode), mode)


def combine(y_rows: np.ndarray, slot_to_row: np.ndarray, topk_w: np.ndarray, shared=None):
    """Combine ("6.4 ...", section 3.1 step 4): out[t] = sum_j w[t,j] * y[slot_to_row[t,j]]
    (+ shared expert output with weight 1, section 7), in float64."""
    s2r = np.asarray(slot_to_row, dtype=np.int64)
    out = np.einsum("tj,tjd->td", np.asarray(topk_w, dtype=np.float64), y_rows[s2r])
    if shared is not None:
        out = out + shared
    return out


# ============================================================== whole layer
def _as64(a, kind):
    a = np.asarray(a)
    if kind == "bf16" and a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def layer_forward(cfg, logits, x, weight, tokens=None, eplb_enabled=None, selection_bias=None):
    """The layer forward for a workload `cfg` (fields T, d, E, k, I, R, shared,
    n_redundant, dtype, eplb_placement: 1 builds the EPLB map with
    eplb_balanced_map instead of eplb_map, expert_placement: 1 places the
    logical experts round-robin instead of linearly, and fp8_dispatch: 1 sends the
    bf16 workloads' tokens as e4m3 and rebuilds bf16 rows from them).
    selection_bias [E] (optional) routes with route_selection_bias.

    logits: float32 [T, E]; x: [T, d] float32 (fp32) or bf16 bits (uint16);
    weight(which, e) -> logical matrix (which in w_gate, w_up, w_down, ws_gate, ws_up,
    ws_down; float32 or bf16 bits).  Routing and layout always cover all T tokens;
    the expert FFN and combine run for `tokens` (all when None).  Returns a dict with
    the routing, the layout, the quantised x rows (fp8) and out [len(tokens), d]
    (float64, before the final rounding) plus out_rounded (bf16 values for bf16/fp8)."""
    T, E, k, R = cfg.T, cfg.E, cfg.k, cfg.R
    if selection_bias is None:
        ids, w = route(logits, k)
    else:
        ids, w = route_selection_bias(logits, selection_bias, k)
    if eplb_enabled is None:
        eplb_enabled = cfg.n_redundant > 0
    placement = "round_robin" if getattr(cfg, "expert_placement", 0) == 1 else "linear"
    emap = None
    counts = np.bincount(ids.ravel(), minlength=E)
    if eplb_enabled and getattr(cfg, "eplb_placement", 0) == 1:
        emap = eplb_balanced_map(counts, R, cfg.n_redundant)
    elif eplb_enabled:
        emap = eplb_map(counts, R, cfg.n_redundant, placement)
    elif placement == "round_robin":
        emap = eplb_map(counts, R, 0, placement)
    lay = dispatch_layout(ids, E, R, emap, placement)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xin = np.asarray(x)
    kind = "fp32" if cfg.dtype == "fp32" else "bf16"
    mode = cfg.dtype
    xs = _as64(xin[tokens], kind)                          # [n, d]
    res = {"topk_ids": ids, "topk_w": w, "layout": lay, "eplb": emap, "tokens": tokens}
    if mode == "fp8":
        xq, xsc = quantize_groups(xs.astype(np.float32))
        res["x_q"], res["x_scales"] = xq, xsc
        xs = dequantize_groups(xq, xsc)
    x_local = xs          # the shared expert runs where the token lives: never dispatched
    if mode == "bf16" and getattr(cfg, "fp8_dispatch", 0) == 1:
        # the routed rows travel in e4m3 (the x rows' quantisation), rebuilt as bf16 rows
        xq, xsc = quantize_groups(xs.astype(np.float32))
        res["x_q"], res["x_scales"] = xq, xsc
        xs = dequantize_groups_bf16(xq, xsc)

    def wmat(which, e):
        m = weight(which, e)
        if mode == "fp8":
            q, s = quantize_blocks(_as64(m, "bf16").astype(np.float32))
            return dequantize_blocks(q, s)
        return _as64(m, kind)

    phys = lay["phys_ids"][tokens]                         # [n, k] physical ids
    p2l = emap["phys_to_logical"] if emap is not None else np.arange(E)
    logical = p2l[phys]
    y_exact = np.zeros((len(tokens), k, cfg.d))
    for e in np.unique(logical):
        sel = np.nonzero(logical == e)
        y_exact[sel[0], sel[1]] = swiglu_expert_exact(xs[sel[0]], wmat("w_gate", e), wmat("w_up", e),
                                                      wmat("w_down", e), mode)
    y_slots = stored_y(y_exact.reshape(-1, cfg.d), mode).reshape(y_exact.shape)
    wt = w[tokens]
    out = np.einsum("tj,tjd->td", wt, y_slots)
    # the same sum with every stored y at the bf16 value below / above its exact
    # value: a kernel whose own y lies across a rounding midpoint from the exact one
    # stores the other neighbour, which is as correct (the weights are positive)
    lo, hi = (y_exact, y_exact) if mode == "fp32" else bf16_bracket(y_exact)
    out_lo, out_hi = np.einsum("tj,tjd->td", wt, lo), np.einsum("tj,tjd->td", wt, hi)
    if cfg.shared:
        s_exact = swiglu_expert_exact(x_local, wmat("ws_gate", 0), wmat("ws_up", 0), wmat("ws_down", 0), mode)
        out = out + stored_y(s_exact, mode)
        s_lo, s_hi = (s_exact, s_exact) if mode == "fp32" else bf16_bracket(s_exact)
        out_lo, out_hi = out_lo + s_lo, out_hi + s_hi
    res["out"] = out
    res["out_rounded"] = out if mode == "fp32" else round_bf16(out)
    res["out_lo"], res["out_hi"] = out_lo, out_hi
    return res
