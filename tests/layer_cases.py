"""Shared cases for the GPU parity tests: one generated layer per configuration,
uploaded and packed on the device by the library, plus the oracle's own
quantisation of the same fp32 weights and its reference results.

Nothing the oracle sees comes from the CUDA path: both sides draw their inputs
from the seeded generator, and each side quantises the fp32 weights itself.
"""
from __future__ import annotations

import functools
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import workloads
from workloads.device import upload

THREADS = max(1, min(32, os.cpu_count() or 1))

# tokens checked one by one against the oracle at the large sizes
SAMPLE_TOKENS = {"prefill2048": 24, "skew8192": 24}


class Case:
    def __init__(self, cfg):
        if isinstance(cfg, str):
            cfg = workloads.CONFIGS[cfg]
        self.cfg = cfg
        name = cfg.name
        E, F, Fs, d, g = cfg.E, cfg.F, cfg.Fs, cfg.d, cfg.group
        q_gu = np.empty((E, 2 * F, d // 2), np.uint8)
        s_gu = np.empty((E, 2 * F, d // g), np.uint16)
        q_dn = np.empty((E, d, F // 2), np.uint8)
        s_dn = np.empty((E, d, F // g), np.uint16)
        shared = {}
        pool = ThreadPoolExecutor(THREADS)
        jobs = []

        def pack(e, wgu, wdn):
            if e >= 0:
                oracle.pack_w4_into(wgu, g, q_gu[e], s_gu[e])
                oracle.pack_w4_into(wdn, g, q_dn[e], s_dn[e])
            else:
                shared["gu"] = oracle.pack_w4(wgu, g)
                shared["dn"] = oracle.pack_w4(wdn, g)

        slots = threading.BoundedSemaphore(2 * THREADS)  # bounds host fp32 held at once

        def pack_release(e, wgu, wdn):
            try:
                pack(e, wgu, wdn)
            finally:
                slots.release()

        def on_expert(e, wgu, wdn):
            slots.acquire()
            jobs.append(pool.submit(pack_release, e, wgu, wdn))

        self.dev = upload(cfg, on_expert=on_expert)
        for j in jobs:
            j.result()
        pool.shutdown()
        self.W = oracle.PackedLayer(q_gu, s_gu, q_dn, s_dn, *shared["gu"], *shared["dn"], g)
        # the oracle's inputs come straight from the generator
        self.x = workloads.gen_x(cfg)
        self.W_r, self.bias = workloads.gen_router(cfg)
        idx, w, margin, _ = oracle.router(self.x, self.W_r, self.bias, cfg.k, threads=THREADS)
        self.topk_idx, self.topk_w, self.margin = idx, w, margin
        self.desc = oracle.descriptors(idx, E)
        n_sample = SAMPLE_TOKENS.get(name)
        if n_sample is None or n_sample >= cfg.T:
            self.tokens = np.arange(cfg.T)
        else:
            rng = np.random.default_rng(1234 + cfg.seed)
            pick = rng.choice(np.arange(1, cfg.T - 1), n_sample - 2, replace=False)
            self.tokens = np.sort(np.concatenate([[0, cfg.T - 1], pick]))
        self.out, self.h_routed, self.h_shared = oracle.layer_tokens(
            self.x, self.W, idx, w, self.tokens, threads=THREADS, want_h=True)


@functools.lru_cache(maxsize=2)
def case(cfg) -> Case:
    """A cached Case for a configuration name or a LayerConfig."""
    return Case(cfg)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def within_layer_bound(got_bits, ref_bits):
    """The layer gate: relative L2 error <= 1e-3 and max-abs error <= 1e-2 * max|ref|."""
    g = bf16_to_f64(got_bits)
    r = bf16_to_f64(ref_bits)
    rel_l2 = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    max_abs = np.abs(g - r).max() if g.size else 0.0
    bound = 1e-2 * (np.abs(r).max() if r.size else 0.0)
    return rel_l2 <= 1e-3 and max_abs <= bound, rel_l2, max_abs, bound


def to_i16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
