"""Python binding of libmoe_b300.so, the B300 (sm_103a) routed MoE layer library.

Argument marshalling only: each function here has the name and the argument
order of the C entry point declared in include/moe.h, takes torch tensors (or
None) for the device pointers, and raises MoeError when the C call returns a
status other than MOE_OK.  Every step of the layer runs in the library's CUDA
kernels; if the library is not built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoeError", "lib", "library_path", "MOE_F32", "MOE_BF16", "MOE_E4M3",
    "MOE_DEV_NONFINITE_LOGIT", "MOE_DEV_ID_RANGE", "MOE_DEV_TIMEOUT", "MOE_DEV_LAYOUT",
    "LoadStats", "Eplb", "Weights", "Shape", "LayerAux",
    "moe_status_string", "moe_route", "moe_route_biased", "moe_eplb_map", "moe_placement_map",
    "moe_eplb_balanced_map", "moe_eplb_window_update", "moe_dispatch_workspace_size",
    "moe_dispatch_layout", "moe_permute", "moe_dequantize_e4m3", "moe_ffn_workspace_size",
    "moe_expert_ffn",
    "moe_combine", "moe_pack_weights", "moe_layer_workspace_size", "moe_layer_forward",
    "moe_expert_gate_up", "moe_expert_gate_up_gather", "moe_expert_down", "moe_expert_down_combine",
    "moe_dispatch_layout_static", "moe_last_cuda_error", "moe_selftest_wait_timeout", "EXPORTED",
    "MOE_DISPATCH_STATIC_SCRATCH_BYTES",
]

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_b300.so")

MOE_F32, MOE_BF16, MOE_E4M3 = 0, 1, 2
MOE_DEV_NONFINITE_LOGIT, MOE_DEV_ID_RANGE, MOE_DEV_TIMEOUT, MOE_DEV_LAYOUT = 1, 2, 4, 8
MOE_DISPATCH_STATIC_SCRATCH_BYTES = 4 << 20
_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
           4: "MOE_ERR_CUDA"}

EXPORTED = ("moe_status_string", "moe_route", "moe_route_biased", "moe_eplb_map", "moe_placement_map",
            "moe_eplb_balanced_map",
            "moe_eplb_window_update", "moe_dispatch_workspace_size",
            "moe_dispatch_layout", "moe_permute", "moe_dequantize_e4m3", "moe_ffn_workspace_size",
    "moe_expert_ffn",
            "moe_combine", "moe_pack_weights", "moe_layer_workspace_size", "moe_layer_forward",
            "moe_expert_gate_up", "moe_expert_gate_up_gather", "moe_expert_down", "moe_expert_down_combine",
            "moe_dispatch_layout_static", "moe_last_cuda_error", "moe_selftest_wait_timeout")


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")


# ------------------------------------------------------------------ structs (moe.h)
c_i32, c_i64, c_vp, c_f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float


class LoadStats(ctypes.Structure):
    _fields_ = [("max_rank", c_i32), ("max_expert", c_i32), ("n_active_experts", c_i32), ("pad_", c_i32),
                ("mean_rank", c_f32), ("max_over_mean", c_f32), ("balancedness", c_f32), ("pad2_", c_f32)]


class Eplb(ctypes.Structure):
    _fields_ = [("P", c_i32), ("phys_to_logical", c_vp), ("replica_count", c_vp), ("logical_to_phys", c_vp),
                ("max_replicas", c_i32), ("base_placement", c_i32)]


class Weights(ctypes.Structure):
    _fields_ = [("dtype", c_i32), ("has_shared", c_i32), ("E_w", c_i64), ("d", c_i64), ("I", c_i64),
                ("w13", c_vp), ("w2", c_vp), ("s13", c_vp), ("s2", c_vp), ("selection_bias", c_vp)]


class Shape(ctypes.Structure):
    _fields_ = [("T", c_i64), ("d", c_i64), ("E", c_i64), ("I", c_i64), ("k", c_i32), ("R", c_i32),
                ("n_redundant", c_i32), ("shared", c_i32), ("act_dtype", c_i32), ("expert_dtype", c_i32),
                ("eplb_placement", c_i32), ("expert_placement", c_i32), ("fp8_dispatch", c_i32)]


class LayerAux(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("topk_ids", "topk_w", "logical_counts", "phys_counts", "phys_offsets",
                                    "rank_counts", "rank_offsets", "row_to_token", "slot_to_row", "stats",
                                    "phys_to_logical", "phys_rank", "replica_count", "logical_to_phys")]


assert ctypes.sizeof(LoadStats) == 32 and ctypes.sizeof(Weights) == 72 and ctypes.sizeof(Shape) == 72
assert ctypes.sizeof(Eplb) == 40

# ------------------------------------------------------------------ loading
_lib = None
_P = ctypes.POINTER


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(f"{library_path} is missing: build it with "
                              "`python -m combine_softmax_top_expert_b300.build`")
        L = ctypes.CDLL(library_path)
        sz, st = ctypes.c_size_t, c_i32
        sig = {
            "moe_status_string": (ctypes.c_char_p, [st]),
            "moe_last_cuda_error": (ctypes.c_char_p, []),
            "moe_route": (st, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp]),
            "moe_route_biased": (st, [c_vp, c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp]),
            "moe_eplb_map": (st, [c_vp, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
            "moe_placement_map": (st, [c_vp, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
            "moe_eplb_balanced_map": (st, [c_vp, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
            "moe_eplb_window_update": (st, [c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp]),
            "moe_selftest_wait_timeout": (st, [c_vp, c_i64, c_vp, c_vp]),
            "moe_dispatch_workspace_size": (sz, [c_i64, c_i32, c_i64]),
            "moe_dispatch_layout": (st, [c_vp, c_i64, c_i32, c_i64, c_i32, _P(Eplb)] + [c_vp] * 8
                                    + [c_vp, sz, c_vp, c_vp]),
            "moe_dispatch_layout_static": (st, [c_vp, c_i64, c_i32, c_i64, c_i32, _P(Eplb)] + [c_vp] * 8
                                           + [c_vp, c_vp]),
            "moe_permute": (st, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp]),
            "moe_dequantize_e4m3": (st, [c_vp, c_vp, c_i64, c_i64, c_vp, c_vp]),
            "moe_ffn_workspace_size": (sz, [c_i64, c_i64, c_i32]),
            "moe_expert_ffn": (st, [c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, _P(Weights), c_vp, c_i64, c_vp,
                                    c_vp, sz, c_vp, c_vp]),
            "moe_expert_gate_up": (st, [c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, _P(Weights), c_vp, c_i64, c_vp,
                                        c_vp, c_vp, c_vp]),
            "moe_expert_gate_up_gather": (st, [c_vp, c_i64, c_vp, c_vp, c_i64, c_vp, c_i64, _P(Weights), c_vp,
                                               c_i64, c_vp, c_vp, c_vp]),
            "moe_expert_down": (st, [c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, _P(Weights), c_i64, c_vp, c_vp, c_vp]),
            "moe_expert_down_combine": (st, [c_vp, c_vp, c_i64, c_vp, c_i64, _P(Weights), c_i64, c_vp, c_vp, c_vp,
                                             c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
            "moe_combine": (st, [c_vp, c_i32, c_vp, c_vp, c_i64, c_i32, c_i64, c_vp, c_vp, c_i32, c_vp]),
            "moe_pack_weights": (st, [c_vp, c_vp, c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp,
                                      c_vp]),
            "moe_layer_workspace_size": (sz, [_P(Shape)]),
            "moe_layer_forward": (st, [_P(Shape), c_vp, c_vp, _P(Weights), c_vp, _P(LayerAux), c_vp, sz,
                                       c_vp, c_vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(t):
    """Device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(name, status):
    if status != 0:
        err = MoeError(name, status)
        if status == 4:
            err.args = (err.args[0] + ": " + moe_last_cuda_error(),)
        raise err


def moe_last_cuda_error() -> str:
    return lib().moe_last_cuda_error().decode()


# ------------------------------------------------------------------ entry points
def moe_status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def moe_route(logits, T, E, k, topk_ids, topk_w, err=None, stream=None):
    _check("moe_route", lib().moe_route(_p(logits), T, E, k, _p(topk_ids), _p(topk_w), _p(err), _s(stream)))


def moe_route_biased(logits, selection_bias, T, E, k, topk_ids, topk_w, err=None, stream=None):
    _check("moe_route_biased", lib().moe_route_biased(_p(logits), _p(selection_bias), T, E, k, _p(topk_ids),
                                                      _p(topk_w), _p(err), _s(stream)))


def moe_placement_map(logical_counts, E, R, n_redundant, placement, phys_to_logical, phys_rank, replica_count,
                      logical_to_phys, stream=None):
    _check("moe_placement_map", lib().moe_placement_map(_p(logical_counts), E, R, n_redundant, placement,
                                                        _p(phys_to_logical), _p(phys_rank), _p(replica_count),
                                                        _p(logical_to_phys), _s(stream)))


def moe_eplb_map(logical_counts, E, R, n_redundant, phys_to_logical, phys_rank, replica_count, logical_to_phys,
                 stream=None):
    _check("moe_eplb_map", lib().moe_eplb_map(_p(logical_counts), E, R, n_redundant, _p(phys_to_logical),
                                              _p(phys_rank), _p(replica_count), _p(logical_to_phys), _s(stream)))


def moe_eplb_balanced_map(logical_counts, E, R, n_redundant, phys_to_logical, phys_rank, replica_count,
                          logical_to_phys, rank_load=None, stream=None):
    _check("moe_eplb_balanced_map",
           lib().moe_eplb_balanced_map(_p(logical_counts), E, R, n_redundant, _p(phys_to_logical), _p(phys_rank),
                                       _p(replica_count), _p(logical_to_phys), _p(rank_load), _s(stream)))


def moe_eplb_window_update(logical_counts, window, W, E, step, window_sum, stream=None):
    _check("moe_eplb_window_update", lib().moe_eplb_window_update(_p(logical_counts), _p(window), W, E, step,
                                                                  _p(window_sum), _s(stream)))


def moe_selftest_wait_timeout(err, timeout_ns, waited_ms=None, stream=None):
    """Run the kernels' bounded pipeline wait on a barrier nothing arrives on; it
    must give up after timeout_ns and OR MOE_DEV_TIMEOUT into err."""
    _check("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(_p(err), timeout_ns, _p(waited_ms),
                                                                        _s(stream)))


def moe_dispatch_workspace_size(T, k, P) -> int:
    return lib().moe_dispatch_workspace_size(T, k, P)


def moe_dispatch_layout(topk_ids, T, k, E, R, eplb, logical_counts, phys_counts, phys_offsets, rank_counts,
                        rank_offsets, row_to_token, slot_to_row, stats, ws, ws_bytes, err=None, stream=None):
    ep = ctypes.byref(eplb) if eplb is not None else None
    _check("moe_dispatch_layout", lib().moe_dispatch_layout(
        _p(topk_ids), T, k, E, R, ep, _p(logical_counts), _p(phys_counts), _p(phys_offsets), _p(rank_counts),
        _p(rank_offsets), _p(row_to_token), _p(slot_to_row), _p(stats), _p(ws), ws_bytes, _p(err), _s(stream)))


def moe_dispatch_layout_static(topk_ids, T, k, E, R, eplb, logical_counts, phys_counts, phys_offsets, rank_counts,
                               rank_offsets, row_to_token, slot_to_row, stats, err=None, stream=None):
    """moe_dispatch_layout without a workspace argument: for callers that cannot
    allocate device memory, the library's built-in scratch array is used (see
    include/moe.h for the size limit and the one-call-at-a-time rule)."""
    ep = ctypes.byref(eplb) if eplb is not None else None
    _check("moe_dispatch_layout_static", lib().moe_dispatch_layout_static(
        _p(topk_ids), T, k, E, R, ep, _p(logical_counts), _p(phys_counts), _p(phys_offsets), _p(rank_counts),
        _p(rank_offsets), _p(row_to_token), _p(slot_to_row), _p(stats), _p(err), _s(stream)))


def moe_permute(x, x_dt, T, d, k, slot_to_row, x_perm, perm_dt, perm_scales=None, stream=None):
    _check("moe_permute", lib().moe_permute(_p(x), x_dt, T, d, k, _p(slot_to_row), _p(x_perm), perm_dt,
                                            _p(perm_scales), _s(stream)))


def moe_dequantize_e4m3(codes, scales, rows, d, out, stream=None):
    _check("moe_dequantize_e4m3", lib().moe_dequantize_e4m3(_p(codes), _p(scales), rows, d, _p(out), _s(stream)))


def moe_ffn_workspace_size(rows, I, dtype) -> int:
    return lib().moe_ffn_workspace_size(rows, I, dtype)


def moe_expert_ffn(x_perm, x_scales, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x, T_shared, y_perm,
                   ws, ws_bytes, err=None, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(
        _p(x_perm), _p(x_scales), _p(phys_offsets), P, _p(phys_to_logical), rows_hint, ctypes.byref(w),
        _p(shared_x), T_shared, _p(y_perm), _p(ws), ws_bytes, _p(err), _s(stream)))


def moe_expert_gate_up(x_perm, x_scales, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x, T_shared, h,
                       h_scales=None, err=None, stream=None):
    _check("moe_expert_gate_up", lib().moe_expert_gate_up(
        _p(x_perm), _p(x_scales), _p(phys_offsets), P, _p(phys_to_logical), rows_hint, ctypes.byref(w),
        _p(shared_x), T_shared, _p(h), _p(h_scales), _p(err), _s(stream)))


def moe_expert_gate_up_gather(x, T, row_to_token, phys_offsets, P, phys_to_logical, rows_hint, w, shared_x,
                              T_shared, h, err=None, stream=None):
    _check("moe_expert_gate_up_gather", lib().moe_expert_gate_up_gather(
        _p(x), T, _p(row_to_token), _p(phys_offsets), P, _p(phys_to_logical), rows_hint, ctypes.byref(w),
        _p(shared_x), T_shared, _p(h), _p(err), _s(stream)))


def moe_expert_down(h, h_scales, phys_offsets, P, phys_to_logical, rows_hint, w, T_shared, y_perm, err=None,
                    stream=None):
    _check("moe_expert_down", lib().moe_expert_down(
        _p(h), _p(h_scales), _p(phys_offsets), P, _p(phys_to_logical), rows_hint, ctypes.byref(w), T_shared,
        _p(y_perm), _p(err), _s(stream)))


def moe_expert_down_combine(h, phys_offsets, P, phys_to_logical, rows_hint, w, T_shared, row_to_token,
                            slot_to_row, topk_w, T, k, y_perm, counts, out, err=None, stream=None):
    _check("moe_expert_down_combine", lib().moe_expert_down_combine(
        _p(h), _p(phys_offsets), P, _p(phys_to_logical), rows_hint, ctypes.byref(w), T_shared, _p(row_to_token),
        _p(slot_to_row), _p(topk_w), T, k, _p(y_perm), _p(counts), _p(out), _p(err), _s(stream)))


def moe_combine(y_perm, y_dt, slot_to_row, topk_w, T, k, d, shared_y, out, out_dt, stream=None):
    _check("moe_combine", lib().moe_combine(_p(y_perm), y_dt, _p(slot_to_row), _p(topk_w), T, k, d,
                                            _p(shared_y), _p(out), out_dt, _s(stream)))


def moe_pack_weights(w_gate, w_up, w_down, src_dt, d, I, dst_dt, w13_e, w2_e, s13_e=None, s2_e=None, stream=None):
    _check("moe_pack_weights", lib().moe_pack_weights(
        _p(w_gate), _p(w_up), _p(w_down), src_dt, d, I, dst_dt, _p(w13_e), _p(w2_e), _p(s13_e), _p(s2_e),
        _s(stream)))


def moe_layer_workspace_size(shape) -> int:
    return lib().moe_layer_workspace_size(ctypes.byref(shape))


def moe_layer_forward(shape, logits, x, w, out, aux, ws, ws_bytes, err=None, stream=None):
    ax = ctypes.byref(aux) if aux is not None else None
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(shape), _p(logits), _p(x), ctypes.byref(w), _p(out), ax, _p(ws), ws_bytes, _p(err),
        _s(stream)))
