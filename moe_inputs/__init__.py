"""Seeded synthetic inputs for the routed MoE layer.

This module is the only code that both the CPU oracle and the CUDA path see.
It draws numbers and holds none of the layer's arithmetic: no routing, no
counting, no expert math, no quantisation.

Generator (counter-based, so any element can be drawn on its own, on the host
with numpy or on the device with torch, and both give the same value):

  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014; the finaliser constants are Vigna's).  The value
    for element ``i`` of stream ``s`` is the SplitMix64 output after the state
    ``s`` has been advanced ``i + 1`` times by the golden gamma.
  * Box-Muller in float64: ``u1 = (hi32 + 1) / 2^32`` in (0, 1],
    ``u2 = lo32 / 2^32`` in [0, 1), ``n = sqrt(-2 ln u1) * cos(2 pi u2)``.
  * Rounding to the stored dtype: float64 -> float32 (round to nearest even),
    then float32 -> bfloat16 (round to nearest even) for bf16 tensors.

Workloads (the five layer shapes the pages' deployments use; the fields are the
pages' notation: T tokens, d hidden, E routed experts, k experts per token,
I expert intermediate size, R logical expert-parallel ranks):

  ========================  =====  ====  ===  =  ====  ==  ======  ====  =====
  name                      T      d     E    k  I     R   shared  red.  dtype
  ========================  =====  ====  ===  =  ====  ==  ======  ====  =====
  tiny_fp32                 64     128   8    2  64    4   no      0     fp32
  decode_bf16               128    6144  256  8  2048  64  no      0     bf16
  prefill_bf16_skew         8192   7168  256  8  2048  32  yes     0     bf16
  prefill_bf16_skew_eplb    8192   7168  256  8  2048  32  yes     32    bf16
  prefill_fp8_skew          16384  6144  256  8  2048  64  no      0     fp8
  ========================  =====  ====  ===  =  ====  ==  ======  ====  =====

Router logits are N(0,1) in fp32, plus, for the skewed workloads, a per-expert
bias ``b_e = 1.5 * ln(1 / r_e^1.2)`` where ``r_e`` is a seeded random
permutation of 1..E (Fisher-Yates), so a few experts are hot (Zipf-like).
Weights are N(0, 1/fan_in) (fan_in = d for gate/up, I for down), x is N(0,1).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "LayerConfig", "CONFIGS", "config", "stream_id", "normal_host",
    "bf16_bits_from_f32", "f32_from_bf16_bits", "zipf_rank_perm", "expert_bias",
    "make_logits", "make_x", "make_weight_host", "make_weight_device",
    "normal_device", "TAG",
]

# ---------------------------------------------------------------- streams
GOLDEN = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)

TAG = {
    "logits": 1, "x": 2, "w_gate": 3, "w_up": 4, "w_down": 5,
    "ws_gate": 6, "ws_up": 7, "ws_down": 8, "rank_perm": 9,
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * MIX1
    z = (z ^ (z >> np.uint64(27))) * MIX2
    return z ^ (z >> np.uint64(31))


def stream_id(seed: int, tag: int) -> int:
    """64-bit stream key for (seed, tag): one SplitMix64 output of seed*2^16+tag."""
    with np.errstate(over="ignore"):
        z = np.array([(int(seed) << 16) + int(tag)], dtype=np.uint64) + GOLDEN
        return int(_mix(z)[0])


def _bits_host(stream: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(stream) + idx * GOLDEN
        return _mix(z)


def _box_muller(z: np.ndarray) -> np.ndarray:
    hi = (z >> np.uint64(32)).astype(np.float64)
    lo = (z & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1 = (hi + 1.0) * (1.0 / 4294967296.0)
    u2 = lo * (1.0 / 4294967296.0)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * math.pi) * u2)


_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def normal_host(stream: int, start: int, count: int) -> np.ndarray:
    """float64 N(0,1) draws for elements start..start+count-1 of a stream."""
    chunk = 1 << 22
    if count <= chunk:
        return _box_muller(_bits_host(stream, start, count))
    out = np.empty(count, dtype=np.float64)

    def work(lo):
        n = min(chunk, count - lo)
        out[lo:lo + n] = _box_muller(_bits_host(stream, start + lo, n))

    list(_pool().map(work, range(0, count, chunk)))
    return out


# ---------------------------------------------------------------- rounding
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- configs
@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    R: int
    shared: bool = False
    n_redundant: int = 0
    eplb_placement: int = 0      # 0: replicas for the hottest experts; 1: load-aware placement
    expert_placement: int = 0    # 0: linear (rank e // (E/R)); 1: round-robin (rank e % R)
    fp8_dispatch: int = 0        # 1: bf16 workloads dispatch tokens as e4m3 (+ scales)
    dtype: str = "bf16"          # "fp32", "bf16" or "fp8" (e4m3 experts, bf16 in/out)
    zipf_bias: bool = False
    seed: int = 0

    @property
    def P(self) -> int:
        return self.E + self.n_redundant

    @property
    def N(self) -> int:
        return self.T * self.k

    def scaled(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


CONFIGS = [
    LayerConfig("tiny_fp32", T=64, d=128, E=8, k=2, I=64, R=4, dtype="fp32"),
    LayerConfig("decode_bf16", T=128, d=6144, E=256, k=8, I=2048, R=64),
    LayerConfig("prefill_bf16_skew", T=8192, d=7168, E=256, k=8, I=2048, R=32,
                shared=True, zipf_bias=True),
    LayerConfig("prefill_bf16_skew_eplb", T=8192, d=7168, E=256, k=8, I=2048, R=32,
                shared=True, zipf_bias=True, n_redundant=32),
    LayerConfig("prefill_fp8_skew", T=16384, d=6144, E=256, k=8, I=2048, R=64,
                dtype="fp8", zipf_bias=True),
]


NAMES = tuple(c.name for c in CONFIGS)


def config(name_or_index) -> LayerConfig:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    for c in CONFIGS:
        if c.name == name_or_index:
            return c
    raise KeyError(name_or_index)


# ---------------------------------------------------------------- tensors
def zipf_rank_perm(seed: int, E: int) -> np.ndarray:
    """r_e: a permutation of 1..E by Fisher-Yates driven by the rank_perm stream."""
    z = _bits_host(stream_id(seed, TAG["rank_perm"]), 0, E)
    r = np.arange(1, E + 1, dtype=np.int64)
    for i in range(E - 1, 0, -1):
        j = int(z[i] % np.uint64(i + 1))
        r[i], r[j] = r[j], r[i]
    return r


def expert_bias(cfg: LayerConfig) -> np.ndarray:
    """b_e = 1.5 * ln(1 / r_e^1.2), float64; zeros when the workload has no skew."""
    if not cfg.zipf_bias:
        return np.zeros(cfg.E, dtype=np.float64)
    r = zipf_rank_perm(cfg.seed, cfg.E).astype(np.float64)
    return 1.5 * np.log(1.0 / r ** 1.2)


def make_logits(cfg: LayerConfig) -> np.ndarray:
    """Router logits [T, E] float32 = round_f32(N(0,1) + b_e)."""
    n = normal_host(stream_id(cfg.seed, TAG["logits"]), 0, cfg.T * cfg.E).reshape(cfg.T, cfg.E)
    return (n + expert_bias(cfg)[None, :]).astype(np.float32)


def _round(v64: np.ndarray, dtype: str) -> np.ndarray:
    f32 = v64.astype(np.float32)
    if dtype == "fp32":
        return f32
    return bf16_bits_from_f32(f32)


def make_x(cfg: LayerConfig, rows=None) -> np.ndarray:
    """Hidden states x [T, d]: float32 for fp32 workloads, else bf16 bits (uint16)."""
    st = stream_id(cfg.seed, TAG["x"])
    dt = "fp32" if cfg.dtype == "fp32" else "bf16"
    if rows is None:
        return _round(normal_host(st, 0, cfg.T * cfg.d), dt).reshape(cfg.T, cfg.d)
    out = [_round(normal_host(st, int(t) * cfg.d, cfg.d), dt) for t in rows]
    return np.stack(out) if out else np.zeros((0, cfg.d), dtype=np.float32 if dt == "fp32" else np.uint16)


def _weight_geom(cfg: LayerConfig, which: str):
    shared = which.startswith("ws_")
    base = which[3:] if shared else which[2:]
    rows, cols = (cfg.d, cfg.I) if base in ("gate", "up") else (cfg.I, cfg.d)
    fan_in = rows
    return rows, cols, 1.0 / math.sqrt(fan_in)


def make_weight_host(cfg: LayerConfig, which: str, e: int) -> np.ndarray:
    """Logical weight matrix of expert e: which in w_gate/w_up (d x I), w_down (I x d),
    or the shared expert's ws_gate/ws_up/ws_down (e must be 0).  float32 for fp32
    workloads, else bf16 bits (fp8 workloads draw bf16 weights and quantise them)."""
    rows, cols, std = _weight_geom(cfg, which)
    n = normal_host(stream_id(cfg.seed, TAG[which]), e * rows * cols, rows * cols)
    dt = "fp32" if cfg.dtype == "fp32" else "bf16"
    return _round(n * std, dt).reshape(rows, cols)


# ---------------------------------------------------------------- device side
def _i64(v: int) -> int:
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def _lsr(t, s):
    import torch
    return torch.bitwise_and(torch.bitwise_right_shift(t, s), (1 << (64 - s)) - 1)


def normal_device(stream: int, start: int, count: int, device):
    """The same draws as normal_host, computed with torch int64/float64 ops."""
    import torch
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = idx * _i64(int(GOLDEN)) + _i64(stream)
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _i64(int(MIX1))
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _i64(int(MIX2))
    z = torch.bitwise_xor(z, _lsr(z, 31))
    hi = _lsr(z, 32).to(torch.float64)
    lo = torch.bitwise_and(z, 0xFFFFFFFF).to(torch.float64)
    del z, idx
    u1 = (hi + 1.0) * (1.0 / 4294967296.0)
    u2 = lo * (1.0 / 4294967296.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def make_weight_device(cfg: LayerConfig, which: str, e: int, device, out=None):
    """Device copy of make_weight_host(cfg, which, e): torch float32 or bfloat16 [rows, cols]."""
    import torch
    rows, cols, std = _weight_geom(cfg, which)
    n = normal_device(stream_id(cfg.seed, TAG[which]), e * rows * cols, rows * cols, device)
    f32 = (n * std).to(torch.float32)
    del n
    v = f32 if cfg.dtype == "fp32" else f32.to(torch.bfloat16)
    v = v.view(rows, cols)
    if out is not None:
        out.copy_(v)
        return out
    return v
