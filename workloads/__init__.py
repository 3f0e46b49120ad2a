"""Seeded synthetic workloads for the routed MoE FFN layer.

Holds the five layer configurations and a ctypes front end to ``gen.c``, the
counter-based generator.  Nothing here computes any part of the layer: it only
draws x, the router weights and bias, and the fp32 expert weights that are then
quantised by whichever side (oracle or CUDA) consumes them.

Shapes follow the Laguna-S-2.1 MoE layer as the decode commit of
thewafflehaus/butter PR #69 ("feat(laguna): Laguna-S-2.1 decode on the CUDA
engine") describes it: sigmoid router scores with a correction bias choose ten
of 256 routed experts per token, and one shared expert always runs; here
d_model 4096 and expert FFN 1024.
Value recipe (the layer statement that accompanies the pages):
  x ~ N(0, 1) rounded to bf16; W_r ~ N(0, 1/d) fp32; bias ~ N(0, 0.5) fp32;
  expert weights ~ N(0, 1/K) fp32, K the contraction length (d for gate/up,
  F for down).  N(0, v) names the variance v.
The skewed prefill case replaces the bias by 2 ln p(rank) with p the Zipf(1.2)
law over a seeded permutation of the experts.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libmoegen.so")
_lock = threading.Lock()
_lib = None

# tensor ids of the counter-based streams
TID_X = 1
TID_WR = 2
TID_BIAS = 3
TID_BIAS_PERM = 4
TID_WGU = 0x10000      # + expert id
TID_WD = 0x20000       # + expert id
TID_WGU_SHARED = 0x30000
TID_WD_SHARED = 0x30001


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    Fs: int
    group: int
    seed: int
    bias: str  # "normal" or "zipf"
    zipf_s: float = 1.2
    zipf_scale: float = 2.0

    @property
    def slots(self) -> int:
        return self.T * self.k

    @property
    def rows(self) -> int:
        """Rows of the expert intermediates: T*k routed slots then T shared rows."""
        return self.T * self.k + self.T

    def packed_expert_bytes(self) -> int:
        gu = 2 * self.F * self.d // 2 + 2 * self.F * (self.d // self.group) * 2
        dn = self.d * self.F // 2 + self.d * (self.F // self.group) * 2
        return gu + dn

    def packed_shared_bytes(self) -> int:
        gu = 2 * self.Fs * self.d // 2 + 2 * self.Fs * (self.d // self.group) * 2
        dn = self.d * self.Fs // 2 + self.d * (self.Fs // self.group) * 2
        return gu + dn

    def flops(self) -> float:
        """Expert GEMM flops of one layer pass: 2 * (2F*d + d*F) per (slot) + shared."""
        return 2.0 * 3.0 * self.d * (self.F * self.slots + self.Fs * self.T)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=4, d=256, E=16, k=2, F=128, Fs=128, group=32, seed=0,
                        bias="normal"),
    "decode1": LayerConfig("decode1", T=1, d=4096, E=256, k=10, F=1024, Fs=1024, group=128,
                           seed=1, bias="normal"),
    "decode32": LayerConfig("decode32", T=32, d=4096, E=256, k=10, F=1024, Fs=1024, group=128,
                            seed=2, bias="normal"),
    "prefill2048": LayerConfig("prefill2048", T=2048, d=4096, E=256, k=10, F=1024, Fs=1024,
                               group=128, seed=3, bias="normal"),
    "skew8192": LayerConfig("skew8192", T=8192, d=4096, E=256, k=10, F=1024, Fs=1024,
                            group=128, seed=4, bias="zipf"),
}


def build(force: bool = False) -> str:
    """Compile gen.c into libmoegen.so next to it (gcc, no host-specific flags)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                                   "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, p = ctypes.c_uint64, ctypes.c_void_p
        lib.gen_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, p]
        lib.gen_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_double, p]
        lib.gen_permutation.argtypes = [u64, u64, ctypes.c_int32, p]
        lib.gen_zipf_bias.argtypes = [u64, u64, ctypes.c_int32, ctypes.c_double,
                                      ctypes.c_double, p, p]
        for f in (lib.gen_normal_f32, lib.gen_normal_bf16, lib.gen_permutation,
                  lib.gen_zipf_bias):
            f.restype = None
        _lib = lib
    return _lib


_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _fill(fn, seed: int, tid: int, n: int, std: float, dtype, out=None, chunk: int = 1 << 20):
    lib = _get()
    if out is None:
        out = np.empty(n, dtype=dtype)
    flat = out.reshape(-1)
    assert flat.size == n and flat.flags["C_CONTIGUOUS"]
    base = flat.ctypes.data
    esz = flat.itemsize
    f = getattr(lib, fn)
    jobs = []
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        jobs.append(_pool().submit(f, seed, tid, s, m, std, base + s * esz))
    for j in jobs:
        j.result()
    return out


def normal_f32(seed: int, tid: int, shape, std: float, out=None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is not None:
        _fill("gen_normal_f32", seed, tid, n, std, np.float32, out=out)
        return out
    return _fill("gen_normal_f32", seed, tid, n, std, np.float32).reshape(shape)


def normal_bf16_bits(seed: int, tid: int, shape, std: float) -> np.ndarray:
    n = int(np.prod(shape))
    return _fill("gen_normal_bf16", seed, tid, n, std, np.uint16).reshape(shape)


def gen_x(cfg: LayerConfig, batch: int = 0) -> np.ndarray:
    """Activations x [T][d] as bf16 bit patterns (uint16).  batch > 0 draws a fresh batch."""
    return normal_bf16_bits(cfg.seed, TID_X + (batch << 32), (cfg.T, cfg.d), 1.0)


def gen_router(cfg: LayerConfig):
    """Router weight W_r [E][d] fp32 and correction bias b [E] fp32."""
    wr = normal_f32(cfg.seed, TID_WR, (cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d))
    if cfg.bias == "zipf":
        lib = _get()
        b = np.empty(cfg.E, np.float32)
        scratch = np.empty(cfg.E, np.int32)
        lib.gen_zipf_bias(cfg.seed, TID_BIAS_PERM, cfg.E, cfg.zipf_s, cfg.zipf_scale,
                          scratch.ctypes.data, b.ctypes.data)
    else:
        b = normal_f32(cfg.seed, TID_BIAS, (cfg.E,), math.sqrt(0.5))
    return wr, b


def gen_gateup(cfg: LayerConfig, e: int, out=None) -> np.ndarray:
    """fp32 gate+up weight of routed expert e (rows 0..F-1 gate, F..2F-1 up), [2F][d].
    e = -1 selects the shared expert, [2Fs][d]."""
    if e < 0:
        return normal_f32(cfg.seed, TID_WGU_SHARED, (2 * cfg.Fs, cfg.d), 1.0 / math.sqrt(cfg.d),
                          out=out)
    return normal_f32(cfg.seed, TID_WGU + e, (2 * cfg.F, cfg.d), 1.0 / math.sqrt(cfg.d), out=out)


def gen_down(cfg: LayerConfig, e: int, out=None) -> np.ndarray:
    """fp32 down weight of routed expert e, [d][F]; e = -1 selects the shared expert [d][Fs]."""
    if e < 0:
        return normal_f32(cfg.seed, TID_WD_SHARED, (cfg.d, cfg.Fs), 1.0 / math.sqrt(cfg.Fs),
                          out=out)
    return normal_f32(cfg.seed, TID_WD + e, (cfg.d, cfg.F), 1.0 / math.sqrt(cfg.F), out=out)


def permutation(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _get().gen_permutation(seed, tid, n, out.ctypes.data)
    return out
