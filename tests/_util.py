"""Shared helpers for the tests: moving seeded inputs to the device and
building packed weight sets from the counter-based generator."""
import functools

import numpy as np
import torch

import moe_inputs as mi

BF16_TOL = (1e-2, 2e-2)     # |gpu - oracle| <= atol + rtol*|oracle| (bf16 outputs)
F32_TOL = (1e-5, 1e-5)      # fp32 outputs and route weights
FP8_RMS = 5e-2              # rms(gpu - oracle) <= 5e-2 * rms(oracle)
# Both sides quantise x and h at the same points (the same codes but where a value of h
# lies at an e4m3 rounding boundary), so over a whole output the error sits far below
# FP8_RMS (1.6e-4 to 1.75e-3 measured).  A block scale 5-10 % off on one of 48 K
# blocks moves the output by 2.4-3.5 % (rms, on the oracle: test_fp8_tolerance.py):
# within FP8_RMS, not within this.
FP8_CONSISTENCY = 1e-2


def dev_f32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_bf16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(device).view(torch.bfloat16)


def host_bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_x(cfg, x):
    return dev_f32(x) if cfg.dtype == "fp32" else dev_bf16(x)


def close(got, ref, tol):
    atol, rtol = tol
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = np.abs(got - ref) > atol + rtol * np.abs(ref)
    return int(bad.sum()), float(np.abs(got - ref).max()) if got.size else 0.0


def fill_weights(cfg, packed, experts=None):
    """Generate the logical weights on the device and pack them expert by expert."""
    experts = range(cfg.E) if experts is None else experts
    for e in experts:
        packed.pack(e, *(mi.make_weight_device(cfg, w, e, "cuda") for w in ("w_gate", "w_up", "w_down")))
    if cfg.shared:
        packed.pack(cfg.E, *(mi.make_weight_device(cfg, w, 0, "cuda") for w in ("ws_gate", "ws_up", "ws_down")))
    torch.cuda.synchronize()


def host_weights(cfg):
    """weight(which, e) for the oracle, from the host generator (cached)."""
    @functools.lru_cache(maxsize=None)
    def weight(which, e):
        return mi.make_weight_host(cfg, which, int(e))
    return weight
