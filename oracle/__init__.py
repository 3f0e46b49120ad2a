"""ORACLE -- test infrastructure, not part of the product.

Python front end (ctypes + numpy) to ``moe_oracle.c``, the plain C definition
of the routed MoE FFN layer.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package; the CUDA
library and its binding never do.

Every function here is a thin marshalling layer: the arithmetic is in the C
file, single-threaded per call.  Helpers that take a ``threads`` argument run
the same C routine over disjoint token (or expert) ranges in parallel threads;
per-token arithmetic is unchanged, so results are bit-identical to one thread.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "libmoeoracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    with _lock:
        stale = (not os.path.exists(_LIB) or
                 os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                                   "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data


def _get():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "orc_pack_w4": [p, i64, i64, i32, p, p],
        "orc_dequant_w4": [p, p, i64, i64, i32, p],
        "orc_dequant_q4_blocks": [p, i64, i64, p],
        "orc_import_q4_blocks": [p, i64, i64, i32, p, p],
        "orc_router": [p, p, p, i64, i32, i32, i32, i64, i64, p, p, p, p],
        "orc_descriptors": [p, i64, i32, i32, p, p, p, p, p],
        "orc_expert_token": [p, i32, i32, i32, p, p, p, p, p, p],
        "orc_layer_tokens": [p, i32, i32, i32, i32, i32, i32, p, p, p, p, p, p, p, p, p, p, p,
                             p, i64, p, p, p],
        "orc_f32_to_f16_array": [p, i64, p],
        "orc_f16_to_f32_array": [p, i64, p],
        "orc_f32_to_bf16_array": [p, i64, p],
        "orc_f64_to_bf16_array": [p, i64, p],
        "orc_bf16_to_f32_array": [p, i64, p],
        "orc_pack_w8": [p, i64, i64, p, p],
        "orc_quant_rows_fp8": [p, i64, i64, p, p],
        "orc_expert_token_w8a8": [p, i32, i32, p, p, p, p, p, p],
        "orc_layer_w8a8_tokens": [p, i32, i32, i32, i32, p, p, p, p, p, p, p, p, p, p, p, i64,
                                  p, p, p],
        "orc_f32_to_e4m3_array": [p, i64, p],
        "orc_e4m3_to_f32_array": [p, i64, p],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = None
    _lib = lib
    return lib


def _threads(n):
    return max(1, min(n or (os.cpu_count() or 1), 64))


# ---------------------------------------------------------------- formats

def f32_to_f16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _get().orc_f32_to_f16_array(_p(x), x.size, _p(out))
    return out


def f16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _get().orc_f16_to_f32_array(_p(h), h.size, _p(out))
    return out


def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _get().orc_f32_to_bf16_array(_p(x), x.size, _p(out))
    return out


def f64_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _get().orc_f64_to_bf16_array(_p(x), x.size, _p(out))
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _get().orc_bf16_to_f32_array(_p(h), h.size, _p(out))
    return out


# ---------------------------------------------------------------- int4

def pack_w4(w, group: int):
    """w fp32 [rows][K] -> (q uint8 [rows][K/2], s fp16 bits uint16 [rows][K/group])."""
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // group), np.uint16)
    _get().orc_pack_w4(_p(w), rows, K, group, _p(q), _p(s))
    return q, s


def pack_w4_into(w, group: int, q_out: np.ndarray, s_out: np.ndarray):
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    assert q_out.flags["C_CONTIGUOUS"] and s_out.flags["C_CONTIGUOUS"]
    assert q_out.shape == (rows, K // 2) and s_out.shape == (rows, K // group)
    _get().orc_pack_w4(_p(w), rows, K, group, _p(q_out), _p(s_out))


def dequant_w4(q, s, group: int) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint16)
    rows, half = q.shape
    out = np.empty((rows, 2 * half), np.float32)
    _get().orc_dequant_w4(_p(q), _p(s), rows, 2 * half, group, _p(out))
    return out


# ---------------------------------------------------------------- router

def dequant_q4_blocks(blocks, K: int) -> np.ndarray:
    """GGUF-style Q4 blocks uint8 [rows][K/32*18] -> fp32 [rows][K]."""
    blocks = np.ascontiguousarray(blocks, np.uint8)
    rows = blocks.shape[0]
    assert K % 32 == 0 and blocks.shape[1] == K // 32 * 18
    w = np.empty((rows, K), np.float32)
    _get().orc_dequant_q4_blocks(_p(blocks), rows, K, _p(w))
    return w


def import_q4_blocks(blocks, K: int, group: int):
    """GGUF-style Q4 blocks -> the canonical packed int4 (q [rows][K/2], s fp16 bits)."""
    blocks = np.ascontiguousarray(blocks, np.uint8)
    rows = blocks.shape[0]
    assert K % 32 == 0 and blocks.shape[1] == K // 32 * 18 and K % group == 0
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // group), np.uint16)
    _get().orc_import_q4_blocks(_p(blocks), rows, K, group, _p(q), _p(s))
    return q, s


def router(x, W_r, bias, k: int, t0: int = 0, t1: int | None = None, threads: int = 1,
           want_scores: bool = False):
    """Returns (topk_idx int32 [T][k], topk_w fp32 [T][k], margin fp64 [T], scores or None).
    Rows outside [t0, t1) are left as zeros."""
    x = np.ascontiguousarray(x, np.uint16)
    W_r = np.ascontiguousarray(W_r, np.float32)
    bias = np.ascontiguousarray(bias, np.float32)
    T, d = x.shape
    E = W_r.shape[0]
    t1 = T if t1 is None else t1
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    margin = np.zeros(T, np.float64)
    scores = np.zeros((T, E), np.float64) if want_scores else None
    lib = _get()
    n = _threads(threads)
    bounds = np.linspace(t0, t1, n + 1).astype(np.int64) if t1 > t0 else [t0, t1]

    def run(a, b):
        if b > a:
            lib.orc_router(_p(x), _p(W_r), _p(bias), T, d, E, k, int(a), int(b), _p(idx), _p(w),
                           _p(margin), _p(scores))

    if n == 1 or t1 - t0 < 2:
        run(t0, t1)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(lambda ab: run(*ab), zip(bounds[:-1], bounds[1:])))
    return idx, w, margin, scores


def descriptors(topk_idx, E: int) -> dict:
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pos = np.empty(T * k, np.int32)
    sched = np.empty(E, np.int32)
    _get().orc_descriptors(_p(topk_idx), T, E, k, _p(counts), _p(offsets), _p(perm), _p(pos),
                           _p(sched))
    return dict(counts=counts, offsets=offsets, perm=perm, pos=pos, sched=sched)


# ---------------------------------------------------------------- experts

def expert_token(x_row, q_gu, s_gu, q_dn, s_dn, group: int):
    """One expert on one token: returns (h bf16 bits [F], y fp32 [d])."""
    x_row = np.ascontiguousarray(x_row, np.uint16)
    d = x_row.shape[0]
    F = q_gu.shape[0] // 2
    h = np.empty(F, np.uint16)
    y = np.empty(d, np.float32)
    _get().orc_expert_token(_p(x_row), d, F, group, _p(np.ascontiguousarray(q_gu)),
                            _p(np.ascontiguousarray(s_gu)), _p(np.ascontiguousarray(q_dn)),
                            _p(np.ascontiguousarray(s_dn)), _p(h), _p(y))
    return h, y


class PackedLayer:
    """Oracle-packed weights of one layer, stacked over experts."""

    def __init__(self, q_gu, s_gu, q_dn, s_dn, qs_gu, ss_gu, qs_dn, ss_dn, group: int):
        self.q_gu, self.s_gu, self.q_dn, self.s_dn = q_gu, s_gu, q_dn, s_dn
        self.qs_gu, self.ss_gu, self.qs_dn, self.ss_dn = qs_gu, ss_gu, qs_dn, ss_dn
        self.group = group
        self.E = q_gu.shape[0]
        self.F = q_gu.shape[1] // 2
        self.d = q_gu.shape[2] * 2
        self.Fs = qs_gu.shape[0] // 2

    @staticmethod
    def from_float(Wgu, Wd, Wgu_s, Wd_s, group: int, threads: int = 1) -> "PackedLayer":
        """Wgu [E][2F][d], Wd [E][d][F], shared [2Fs][d] and [d][Fs], all fp32."""
        E, twoF, d = Wgu.shape
        F = twoF // 2
        q_gu = np.empty((E, 2 * F, d // 2), np.uint8)
        s_gu = np.empty((E, 2 * F, d // group), np.uint16)
        q_dn = np.empty((E, d, F // 2), np.uint8)
        s_dn = np.empty((E, d, F // group), np.uint16)

        def one(e):
            pack_w4_into(Wgu[e], group, q_gu[e], s_gu[e])
            pack_w4_into(Wd[e], group, q_dn[e], s_dn[e])

        _map(one, range(E), threads)
        qs_gu, ss_gu = pack_w4(Wgu_s, group)
        qs_dn, ss_dn = pack_w4(Wd_s, group)
        return PackedLayer(q_gu, s_gu, q_dn, s_dn, qs_gu, ss_gu, qs_dn, ss_dn, group)

    @staticmethod
    def from_generator(make_gu, make_dn, E, F, Fs, d, group: int, threads: int = 1):
        """Build from per-expert fp32 producers (expert -1 = shared) without holding
        every fp32 matrix at once."""
        q_gu = np.empty((E, 2 * F, d // 2), np.uint8)
        s_gu = np.empty((E, 2 * F, d // group), np.uint16)
        q_dn = np.empty((E, d, F // 2), np.uint8)
        s_dn = np.empty((E, d, F // group), np.uint16)

        def one(e):
            pack_w4_into(make_gu(e), group, q_gu[e], s_gu[e])
            pack_w4_into(make_dn(e), group, q_dn[e], s_dn[e])

        _map(one, range(E), threads)
        qs_gu, ss_gu = pack_w4(make_gu(-1), group)
        qs_dn, ss_dn = pack_w4(make_dn(-1), group)
        return PackedLayer(q_gu, s_gu, q_dn, s_dn, qs_gu, ss_gu, qs_dn, ss_dn, group)


def _map(fn, items, threads):
    items = list(items)
    n = _threads(threads)
    if n == 1:
        for it in items:
            fn(it)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(fn, items))


def layer_tokens(x, W: PackedLayer, topk_idx, topk_w, tokens, threads: int = 1,
                 want_h: bool = False, residual=None):
    """Layer output for the listed tokens.  Returns (out bf16 bits [n][d],
    h_routed [n][k][F] or None, h_shared [n][Fs] or None).  ``residual``
    (bf16 bits [T][d], optional) is added after the routed + shared sum."""
    x = np.ascontiguousarray(x, np.uint16)
    if residual is not None:
        residual = np.ascontiguousarray(residual, np.uint16)
        assert residual.shape == x.shape
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    topk_w = np.ascontiguousarray(topk_w, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int64)
    n = tokens.shape[0]
    T, d = x.shape
    k = topk_idx.shape[1]
    out = np.empty((n, d), np.uint16)
    h_r = np.empty((n, k, W.F), np.uint16) if want_h else None
    h_s = np.empty((n, W.Fs), np.uint16) if want_h else None
    lib = _get()

    def run(a, b):
        if b <= a:
            return
        lib.orc_layer_tokens(
            _p(x), d, W.E, k, W.F, W.Fs, W.group, _p(topk_idx), _p(topk_w),
            _p(W.q_gu), _p(W.s_gu), _p(W.q_dn), _p(W.s_dn),
            _p(W.qs_gu), _p(W.ss_gu), _p(W.qs_dn), _p(W.ss_dn), _p(residual),
            tokens.ctypes.data + a * 8, b - a,
            out.ctypes.data + a * d * 2,
            None if h_r is None else h_r.ctypes.data + a * k * W.F * 2,
            None if h_s is None else h_s.ctypes.data + a * W.Fs * 2)

    nt = _threads(threads)
    if nt == 1 or n < 2:
        run(0, n)
    else:
        b = np.linspace(0, n, min(nt, n) + 1).astype(np.int64)
        with ThreadPoolExecutor(len(b) - 1) as ex:
            list(ex.map(lambda ab: run(int(ab[0]), int(ab[1])), zip(b[:-1], b[1:])))
    return out, h_r, h_s


def layer(x, W_r, bias, W: PackedLayer, k: int, threads: int = 1, want_h: bool = False,
          residual=None):
    """The whole layer on every token: router, descriptors, experts, combine
    (plus the residual row when given)."""
    idx, w, margin, _ = router(x, W_r, bias, k, threads=threads)
    desc = descriptors(idx, W.E)
    T = x.shape[0]
    out, h_r, h_s = layer_tokens(x, W, idx, w, np.arange(T), threads=threads, want_h=want_h,
                                 residual=residual)
    return dict(topk_idx=idx, topk_w=w, margin=margin, out=out, h_routed=h_r, h_shared=h_s,
                **desc)


# ---------------------------------------------------------------- W8A8 (fp8 E4M3)

def f32_to_e4m3(x) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _get().orc_f32_to_e4m3_array(_p(x), x.size, _p(out))
    return out


def e4m3_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, np.uint8)
    out = np.empty(b.shape, np.float32)
    _get().orc_e4m3_to_f32_array(_p(b), b.size, _p(out))
    return out


def pack_w8(w):
    """w fp32 [rows][K] -> (q E4M3 codes uint8 [rows][K], s fp32 [rows])."""
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty(rows, np.float32)
    _get().orc_pack_w8(_p(w), rows, K, _p(q), _p(s))
    return q, s


def quant_rows_fp8(x):
    """x fp32 [n][K] (activation values) -> (codes uint8 [n][K], a fp32 [n])."""
    x = np.ascontiguousarray(x, np.float32)
    n, K = x.shape
    q = np.empty((n, K), np.uint8)
    a = np.empty(n, np.float32)
    _get().orc_quant_rows_fp8(_p(x), n, K, _p(q), _p(a))
    return q, a


def expert_token_w8a8(x_row, q_gu, s_gu, q_dn, s_dn):
    """One W8A8 expert on one token: returns (h bf16 bits [F], y fp32 [d])."""
    x_row = np.ascontiguousarray(x_row, np.uint16)
    d = x_row.shape[0]
    F = q_gu.shape[0] // 2
    h = np.empty(F, np.uint16)
    y = np.empty(d, np.float32)
    _get().orc_expert_token_w8a8(_p(x_row), d, F, _p(np.ascontiguousarray(q_gu)),
                                 _p(np.ascontiguousarray(s_gu, np.float32)),
                                 _p(np.ascontiguousarray(q_dn)),
                                 _p(np.ascontiguousarray(s_dn, np.float32)), _p(h), _p(y))
    return h, y


class PackedLayerW8:
    """Oracle-packed W8A8 weights of one layer: codes [E][2F][d], [E][d][F] and the
    shared expert's [2Fs][d], [d][Fs], with one fp32 scale per row."""

    def __init__(self, q_gu, s_gu, q_dn, s_dn, qs_gu, ss_gu, qs_dn, ss_dn):
        self.q_gu, self.s_gu, self.q_dn, self.s_dn = q_gu, s_gu, q_dn, s_dn
        self.qs_gu, self.ss_gu, self.qs_dn, self.ss_dn = qs_gu, ss_gu, qs_dn, ss_dn
        self.E, twoF, self.d = q_gu.shape
        self.F = twoF // 2
        self.Fs = qs_gu.shape[0] // 2

    @staticmethod
    def from_generator(make_gu, make_dn, E, F, Fs, d, threads: int = 1) -> "PackedLayerW8":
        """Build from per-expert fp32 producers (expert -1 = shared)."""
        q_gu = np.empty((E, 2 * F, d), np.uint8)
        s_gu = np.empty((E, 2 * F), np.float32)
        q_dn = np.empty((E, d, F), np.uint8)
        s_dn = np.empty((E, d), np.float32)

        def one(e):
            q_gu[e], s_gu[e] = pack_w8(make_gu(e))
            q_dn[e], s_dn[e] = pack_w8(make_dn(e))

        _map(one, range(E), threads)
        qs_gu, ss_gu = pack_w8(make_gu(-1))
        qs_dn, ss_dn = pack_w8(make_dn(-1))
        return PackedLayerW8(q_gu, s_gu, q_dn, s_dn, qs_gu, ss_gu, qs_dn, ss_dn)

    @staticmethod
    def from_float(Wgu, Wd, Wgu_s, Wd_s, threads: int = 1) -> "PackedLayerW8":
        E, twoF, d = Wgu.shape
        return PackedLayerW8.from_generator(lambda e: Wgu[e] if e >= 0 else Wgu_s,
                                            lambda e: Wd[e] if e >= 0 else Wd_s,
                                            E, twoF // 2, Wgu_s.shape[0] // 2, d, threads)


def layer_w8a8_tokens(x, W: PackedLayerW8, topk_idx, topk_w, tokens, threads: int = 1,
                      want_h: bool = False):
    """W8A8 layer output for the listed tokens: (out bf16 bits [n][d], h_routed, h_shared)."""
    x = np.ascontiguousarray(x, np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    topk_w = np.ascontiguousarray(topk_w, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int64)
    n = tokens.shape[0]
    T, d = x.shape
    k = topk_idx.shape[1]
    out = np.empty((n, d), np.uint16)
    h_r = np.empty((n, k, W.F), np.uint16) if want_h else None
    h_s = np.empty((n, W.Fs), np.uint16) if want_h else None
    lib = _get()

    def run(a, b):
        if b <= a:
            return
        lib.orc_layer_w8a8_tokens(
            _p(x), d, k, W.F, W.Fs, _p(topk_idx), _p(topk_w),
            _p(W.q_gu), _p(W.s_gu), _p(W.q_dn), _p(W.s_dn),
            _p(W.qs_gu), _p(W.ss_gu), _p(W.qs_dn), _p(W.ss_dn),
            tokens.ctypes.data + a * 8, b - a, out.ctypes.data + a * d * 2,
            None if h_r is None else h_r.ctypes.data + a * k * W.F * 2,
            None if h_s is None else h_s.ctypes.data + a * W.Fs * 2)

    nt = _threads(threads)
    if nt == 1 or n < 2:
        run(0, n)
    else:
        b = np.linspace(0, n, min(nt, n) + 1).astype(np.int64)
        with ThreadPoolExecutor(len(b) - 1) as ex:
            list(ex.map(lambda ab: run(int(ab[0]), int(ab[1])), zip(b[:-1], b[1:])))
    return out, h_r, h_s


def layer_w8a8(x, W_r, bias, W: PackedLayerW8, k: int, threads: int = 1, want_h: bool = False):
    """The whole W8A8 layer on every token (the router and descriptors are the W4A16
    layer's)."""
    idx, w, margin, _ = router(x, W_r, bias, k, threads=threads)
    out, h_r, h_s = layer_w8a8_tokens(x, W, idx, w, np.arange(x.shape[0]), threads=threads,
                                      want_h=want_h)
    return dict(topk_idx=idx, topk_w=w, margin=margin, out=out, h_routed=h_r, h_shared=h_s)
