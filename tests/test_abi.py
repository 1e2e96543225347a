"""The C-ABI library builds, loads and exports every entry point of include/moe.h;
host-side validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

import combine_softmax_top_expert_b300 as moe
from combine_softmax_top_expert_b300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTED) == names


def test_struct_layouts_match_header():
    assert ctypes.sizeof(moe.LoadStats) == 32
    assert ctypes.sizeof(moe.Weights) == 72
    assert ctypes.sizeof(moe.Shape) == 72
    assert ctypes.sizeof(moe.Eplb) == 40
    assert ctypes.sizeof(moe.LayerAux) == 14 * 8


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert "invalid" in moe.moe_status_string(1)
    assert "workspace" in moe.moe_status_string(3)


def test_host_validation_without_gpu(lib):
    # invalid shapes are rejected on the host before any CUDA call
    L = moe.lib()
    assert L.moe_route(None, -1, 8, 2, None, None, None, None) == 1
    assert L.moe_route(None, 4, 8, 9, None, None, None, None) == 1         # k > E
    assert L.moe_route(None, 4, 2000, 2, None, None, None, None) == 1      # E > 1024
    assert L.moe_route(None, 0, 8, 2, None, None, None, None) == 0         # empty batch: nothing queued
    assert L.moe_eplb_map(None, 256, 32, 33, None, None, None, None, None) == 1  # n_red % R
    assert L.moe_eplb_balanced_map(None, 256, 32, 33, None, None, None, None, None, None) == 1  # P % R
    assert L.moe_eplb_balanced_map(None, 1025, 1, 0, None, None, None, None, None, None) == 1   # E > 1024
    assert L.moe_eplb_balanced_map(None, 1024, 1, 1025, None, None, None, None, None, None) == 1  # P > 2048
    assert L.moe_eplb_window_update(None, None, 0, 8, 0, None, None) == 1      # W < 1
    assert L.moe_eplb_window_update(None, None, 4, 2048, 0, None, None) == 1   # E > 1024
    fake4 = ctypes.c_void_p(256)
    assert L.moe_eplb_balanced_map(fake4, 256, 8, 8, None, fake4, fake4, fake4, None, None) == 1  # null output
    assert L.moe_placement_map(fake4, 256, 32, 32, 2, fake4, fake4, fake4, fake4, None) == 1  # placement 2
    assert L.moe_placement_map(None, 256, 32, 32, 1, fake4, fake4, fake4, fake4, None) == 1   # hot list, no counts
    assert L.moe_placement_map(None, 256, 30, 0, 1, fake4, fake4, fake4, fake4, None) == 1    # E % R
    assert L.moe_dequantize_e4m3(fake4, fake4, 4, 200, fake4, None) == 1        # d % 128
    assert L.moe_dequantize_e4m3(None, None, 0, 128, None, None) == 0           # no rows: nothing queued
    assert L.moe_selftest_wait_timeout(None, 1000000, None, None) == 1          # no error word
    assert L.moe_selftest_wait_timeout(fake4, 10**9, None, None) == 1          # limit above 100 ms
    assert L.moe_permute(None, 1, 0, 128, 2, None, None, 1, None, None) == 0
    assert L.moe_combine(None, 1, None, None, 4, 2, 100, None, None, 1, None) == 1   # d % 8
    ws = L.moe_dispatch_workspace_size(64, 2, 8)
    assert ws > 0 and ws % 256 == 0
    # a too-small workspace is reported as such
    fake = ctypes.c_void_p(256)
    assert L.moe_dispatch_layout(fake, 64, 2, 8, 4, None, fake, fake, fake, fake, fake, fake, fake, None,
                                 fake, 16, None, None) == 3


def test_static_layout_answers_bad_sizes_like_the_workspace_layout(lib):
    # the built-in-scratch layout checks the sizes first, so a bad size gets the same
    # status from both entry points (and no size is computed from an overflowing T * k)
    L = moe.lib()
    fake = ctypes.c_void_p(256)
    outs = [fake] * 7
    for T, k, E, R, want in ((64, 2, 2000, 4, 1),        # E > 1024
                             (64, 2, 8, 3, 1),           # E % R
                             (-1, 2, 8, 4, 1),           # T < 0
                             (64, 0, 8, 4, 1),           # k < 1
                             (2 ** 40, 8, 256, 32, 2),   # T * k beyond the layout's int32 rows
                             (2 ** 62, 8, 256, 32, 2)):  # T * k would overflow int64
        ws_status = L.moe_dispatch_layout(fake, T, k, E, R, None, *outs, None, fake, 1 << 20, None, None)
        st_status = L.moe_dispatch_layout_static(fake, T, k, E, R, None, *outs, None, None, None)
        assert ws_status == st_status == want, (T, k, E, R, ws_status, st_status)
    assert L.moe_dispatch_workspace_size(2 ** 62, 8, 256) == 0


def test_layer_workspace_sizes(lib):
    import moe_inputs as mi
    for cfg in mi.CONFIGS:
        s = moe.Shape()
        s.T, s.d, s.E, s.I, s.k, s.R = cfg.T, cfg.d, cfg.E, cfg.I, cfg.k, cfg.R
        s.n_redundant, s.shared = cfg.n_redundant, int(cfg.shared)
        s.act_dtype = moe.MOE_F32 if cfg.dtype == "fp32" else moe.MOE_BF16
        s.expert_dtype = {"fp32": moe.MOE_F32, "bf16": moe.MOE_BF16, "fp8": moe.MOE_E4M3}[cfg.dtype]
        n = moe.moe_layer_workspace_size(s)
        rows = cfg.N + (cfg.T if cfg.shared else 0)
        # at least x_perm + y_perm + h
        elem = {"fp32": 4, "bf16": 2, "fp8": 1}[cfg.dtype]
        assert n >= cfg.N * cfg.d * elem + rows * cfg.d * (4 if cfg.dtype == "fp32" else 2) + rows * cfg.I * elem
    s = moe.Shape()
    s.T, s.d, s.E, s.I, s.k, s.R, s.act_dtype, s.expert_dtype = 4, 128, 8, 64, 2, 4, moe.MOE_F32, moe.MOE_BF16
    assert moe.moe_layer_workspace_size(s) == 0    # fp32 activations need fp32 experts


def test_empty_batch_and_unsupported_shapes_without_gpu(lib):
    """Calls the library answers on the host, before any CUDA call."""
    L = moe.lib()
    fake = ctypes.c_void_p(256)
    w = moe.Weights()
    w.dtype, w.has_shared, w.E_w, w.d, w.I = moe.MOE_BF16, 0, 8, 256, 256
    w.w13, w.w2 = 256, 256
    s = moe.Shape()
    s.T, s.d, s.E, s.I, s.k, s.R, s.act_dtype, s.expert_dtype = 0, 256, 8, 256, 2, 4, moe.MOE_BF16, moe.MOE_BF16
    # an empty batch is a no-op
    assert L.moe_layer_forward(ctypes.byref(s), None, None, ctypes.byref(w), None, None, None, 0, None, None) == 0
    # an unknown EPLB placement or base placement is rejected
    s.T, s.n_redundant, s.eplb_placement = 16, 4, 7
    assert moe.moe_layer_workspace_size(s) == 0
    s.eplb_placement, s.expert_placement = 0, 2
    assert moe.moe_layer_workspace_size(s) == 0
    s.expert_placement = 1
    assert moe.moe_layer_workspace_size(s) > 0
    # FP8 dispatch: bf16 experts take it (workspace grows by the e4m3 rows and scales),
    # fp32 layers and d % 128 != 0 do not
    plain = moe.moe_layer_workspace_size(s)
    s.fp8_dispatch = 1
    assert moe.moe_layer_workspace_size(s) >= plain + 16 * 2 * 256 + 16 * 2 * 2 * 4
    s.d = 200
    assert moe.moe_layer_workspace_size(s) == 0
    s.d, s.fp8_dispatch = 256, 2
    assert moe.moe_layer_workspace_size(s) == 0
    # e4m3 experts need d % 256 == 0 (the pair tiles' 256 output features)
    w8 = moe.Weights()
    w8.dtype, w8.has_shared, w8.E_w, w8.d, w8.I = moe.MOE_E4M3, 0, 8, 384, 256
    w8.w13 = w8.w2 = w8.s13 = w8.s2 = 256
    ws = moe.moe_ffn_workspace_size(64, 256, moe.MOE_E4M3)
    assert L.moe_expert_ffn(fake, fake, fake, 8, None, 64, ctypes.byref(w8), None, 0, fake, fake, ws, None,
                            None) == 2
    # the gathered gate/up: bf16 weights only, a row map and a 16-byte aligned x
    assert L.moe_expert_gate_up_gather(fake, 64, fake, fake, 8, None, 64, ctypes.byref(w8), None, 0, fake, None,
                                       None) == 2
    assert L.moe_expert_gate_up_gather(fake, 64, None, fake, 8, None, 64, ctypes.byref(w), None, 0, fake, None,
                                       None) == 1
    assert L.moe_expert_gate_up_gather(ctypes.c_void_p(264), 64, fake, fake, 8, None, 64, ctypes.byref(w), None,
                                       0, fake, None, None) == 1
    assert L.moe_expert_gate_up_gather(None, 0, None, fake, 8, None, 0, ctypes.byref(w), None, 0, fake, None,
                                       None) == 0      # no rows: nothing queued
    # the down phase with the combine fused: bf16 weights only, T_shared 0 or T, k <= 32
    dc = lambda ww, T_sh, T, k, N=64: L.moe_expert_down_combine(fake, fake, 8, None, N, ctypes.byref(ww), T_sh, fake,
                                                                fake, fake, T, k, fake, fake, fake, None, None)
    assert dc(w8, 0, 32, 2) == 2
    assert dc(w, 5, 32, 2) == 1          # a shared expert over part of the batch
    assert dc(w, 0, 32, 33) == 1         # k above 32
    assert dc(w, 0, 16, 2) == 1          # more rows than T * k
    assert dc(w, 0, 0, 2, N=0) == 0      # empty batch: nothing queued
    # the shared expert needs its weight set
    assert L.moe_expert_ffn(fake, None, fake, 8, None, 64, ctypes.byref(w), fake, 16, fake, fake, 1 << 30, None,
                            None) == 1
