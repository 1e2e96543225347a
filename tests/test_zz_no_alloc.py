"""moe_dispatch_layout_static: the dispatch layout for callers that cannot
allocate device memory (they hold only their input and output buffers, so they
cannot hand moe_dispatch_layout a workspace).  It must produce exactly what
moe_dispatch_layout produces, call after call, although every call reuses the
same scratch array built into the library.

This file is collected last on purpose: if it fails, every other test has
already run."""
import numpy as np
import pytest
import torch

import combine_softmax_top_expert_b300 as moe
import moe_inputs as mi
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
I32 = dict(dtype=torch.int32, device="cuda")


def run_layout(static, ids_np, E, R, eplb_np=None):
    T, k = ids_np.shape
    P = E if eplb_np is None else eplb_np["P"]
    N = T * k
    ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    outs = [torch.full((n,), -5, **I32) for n in (E, P, P + 1, R, R + 1, N, N)]
    stats = torch.full((16,), -5, **I32)
    err = torch.zeros(1, **I32)
    ep, keep = None, []
    if eplb_np is not None:
        keep = [torch.from_numpy(eplb_np[n]).cuda() for n in ("phys_to_logical", "replica_count", "logical_to_phys")]
        ep = moe.Eplb(P, *(t.data_ptr() for t in keep))
    if static:
        moe.moe_dispatch_layout_static(ids, T, k, E, R, ep, *outs, stats, err)
    else:
        wsb = moe.moe_dispatch_workspace_size(T, k, P)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        moe.moe_dispatch_layout(ids, T, k, E, R, ep, *outs, stats, ws, wsb, err)
    torch.cuda.synchronize()
    del keep
    res = [t.cpu().numpy() for t in outs] + [stats.cpu().numpy(), err.cpu().numpy()]
    return res


def case(workload, T=None, eplb=False):
    cfg = mi.config(workload) if T is None else mi.config(workload).scaled(T=T)
    ids, _ = O.route(mi.make_logits(cfg), cfg.k)
    emap = O.eplb_map(np.bincount(ids.ravel(), minlength=cfg.E), cfg.R, cfg.n_redundant) if eplb else None
    return ids, cfg.E, cfg.R, emap


def test_static_scratch_layout_matches_workspace_layout_call_after_call():
    # a large skewed batch with EPLB, then a small decode batch, then the large one
    # again: each call overwrites what the previous one left in the shared scratch
    cases = [case("prefill_bf16_skew_eplb", eplb=True), case("decode_bf16"), case("prefill_fp8_skew", T=4096),
             case("prefill_bf16_skew_eplb", eplb=True)]
    for ids, E, R, emap in cases:
        ref = run_layout(False, ids, E, R, emap)
        got = run_layout(True, ids, E, R, emap)
        assert int(got[-1][0]) == 0
        for a, b in zip(ref, got):
            assert np.array_equal(a, b)


def test_static_scratch_rejects_a_batch_beyond_its_size():
    need = moe.moe_dispatch_workspace_size(200000, 8, 256)
    assert need > moe.MOE_DISPATCH_STATIC_SCRATCH_BYTES
    L = moe.lib()
    status = L.moe_dispatch_layout_static(None, 200000, 8, 256, 32, None, *([None] * 8), None, None)
    assert status == 3    # MOE_ERR_WORKSPACE, nothing queued
