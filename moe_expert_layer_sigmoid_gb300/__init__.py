"""Python binding of libmoe.so, the GB300 routed MoE FFN layer.

Argument marshalling only: every function here checks tensor shapes, dtypes
and devices, passes raw pointers and the current CUDA stream to the C ABI
declared in include/moe.h, and raises MoeError on a non-OK status.  All
arithmetic runs in the library's CUDA kernels; there is no other path.  If
libmoe.so has not been built, importing works but every call raises.

PyTorch supplies device memory and streams.  bf16 / fp16 tensors are passed
as their bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_CHECK = 5

MOE_FLAG_FORCE_GEMV = 0x1
MOE_FLAG_FORCE_GROUPED = 0x2
MOE_FLAG_NO_SCHED = 0x4
MOE_FLAG_DECODE_MMA = 0x8

# every extern "C" symbol include/moe.h declares
EXPORTS = (
    "moe_status_string", "moe_pack_w4", "moe_workspace_bytes", "moe_router_topk",
    "moe_build_descriptors", "moe_gateup_swiglu_w4a16", "moe_down_w4a16", "moe_combine_shared",
    "moe_layer_workspace_bytes", "moe_layer_forward", "moe_layer_forward_host",
    "moe_check_device_status", "moe_router_topk_noalloc", "moe_pack_w4_bytes",
    "moe_combine_shared_residual", "moe_layer_forward_residual", "moe_import_q4_blocks",
    "moe_down_combine_w4a16", "moe_pack_w8", "moe_quant_rows_fp8",
    "moe_layer_workspace_bytes_w8a8", "moe_layer_forward_w8a8", "moe_gateup_swiglu_w8a8",
    "moe_down_w8a8", "moe_debug_set_waits",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class Dims(ctypes.Structure):
    """moe_dims_t."""
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("F_s", ctypes.c_int32),
                ("group", ctypes.c_int32), ("flags", ctypes.c_uint32)]

    def replace(self, **kw) -> "Dims":
        vals = {f: getattr(self, f) for f, _ in self._fields_}
        vals.update(kw)
        return Dims(**vals)


class W4(ctypes.Structure):
    """moe_w4_t: packed int4 bytes and fp16 scales (device pointers)."""
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class W8(ctypes.Structure):
    """moe_w8_t: E4M3 codes and fp32 row scales (device pointers)."""
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(Dims)
    sigs = {
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_pack_w4": ([p, i64, i64, i32, p, p, p], i32),
        "moe_workspace_bytes": ([D], sz),
        "moe_layer_workspace_bytes": ([D], sz),
        "moe_router_topk": ([p, p, p, D, p, p, p, p, sz, p], i32),
        "moe_build_descriptors": ([p, D, p, p, p, p, p, p, sz, p], i32),
        "moe_gateup_swiglu_w4a16": ([p, D, p, p, p, W4, W4, p, p, sz, p], i32),
        "moe_down_w4a16": ([p, D, p, p, W4, W4, p, p, sz, p], i32),
        "moe_down_combine_w4a16": ([p, D, p, p, p, p, W4, W4, p, p, p, sz, p], i32),
        "moe_pack_w8": ([p, i64, i64, p, p, p], i32),
        "moe_quant_rows_fp8": ([p, i64, i64, p, p, p], i32),
        "moe_layer_workspace_bytes_w8a8": ([D], sz),
        "moe_layer_forward_w8a8": ([p, p, p, D, W8, W8, W8, W8, p, p, sz, p], i32),
        "moe_gateup_swiglu_w8a8": ([p, D, p, W8, W8, p, p, sz, p], i32),
        "moe_down_w8a8": ([p, D, W8, W8, p, p, sz, p], i32),
        "moe_debug_set_waits": ([p, sz, ctypes.c_uint64, i32, p], i32),
        "moe_pack_w4_bytes": ([i64, i64, i32, ctypes.POINTER(sz)], sz),
        "moe_import_q4_blocks": ([p, i64, i64, i32, p, p, p, p], i32),
        "moe_combine_shared": ([p, p, p, D, p, p], i32),
        "moe_combine_shared_residual": ([p, p, p, D, p, p, p], i32),
        "moe_layer_forward_residual": ([p, p, p, D, W4, W4, W4, W4, p, p, p, sz, p], i32),
        "moe_layer_forward": ([p, p, p, D, W4, W4, W4, W4, p, p, sz, p], i32),
        "moe_layer_forward_host": ([p, p, p, D, W4, W4, W4, W4, p, p, sz, p], i32),
        "moe_check_device_status": ([p, sz, p], i32),
        "moe_router_topk_noalloc": ([p, p, p, D, p, p, p, p], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


# 16-bit float patterns may travel as int16 or as the matching torch dtype
_ALIASES = {torch.int16: (torch.int16, torch.bfloat16, torch.float16)}


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in _ALIASES.get(dtype, (dtype,)):
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def w4(q: torch.Tensor, s: torch.Tensor) -> W4:
    return W4(_dev(q, torch.uint8, "q"), _dev(s, torch.int16, "s"))


def w8(q: torch.Tensor, s: torch.Tensor) -> W8:
    return W8(_dev(q, torch.uint8, "q"), _dev(s, torch.float32, "s"))


# ------------------------------------------------------------------ entry points

def moe_pack_w4(w: torch.Tensor, group: int, q: torch.Tensor | None = None,
                s: torch.Tensor | None = None, stream=None):
    """fp32 [rows][K] -> (q uint8 [rows][K/2], s fp16 bits as int16 [rows][K/group])."""
    rows, K = w.shape
    if q is None:
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((rows, K // group), dtype=torch.int16, device=w.device)
    _check(lib().moe_pack_w4(_dev(w, torch.float32, "w"), rows, K, group,
                             _dev(q, torch.uint8, "q"), _dev(s, torch.int16, "s"),
                             _stream(stream)), "moe_pack_w4")
    return q, s


def moe_pack_w8(w: torch.Tensor, q: torch.Tensor | None = None, s: torch.Tensor | None = None,
                stream=None):
    """fp32 [rows][K] -> (E4M3 codes uint8 [rows][K], fp32 row scales [rows])."""
    rows, K = w.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().moe_pack_w8(_dev(w, torch.float32, "w"), rows, K, _dev(q, torch.uint8, "q"),
                             _dev(s, torch.float32, "s"), _stream(stream)), "moe_pack_w8")
    return q, s


def moe_quant_rows_fp8(x: torch.Tensor, q: torch.Tensor | None = None,
                       a: torch.Tensor | None = None, stream=None):
    """bf16 rows (int16 bits) [rows][K] -> (E4M3 codes uint8 [rows][K], fp32 scales [rows])."""
    rows, K = x.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    if a is None:
        a = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(lib().moe_quant_rows_fp8(_dev(x, torch.int16, "x"), rows, K, _dev(q, torch.uint8, "q"),
                                    _dev(a, torch.float32, "a"), _stream(stream)),
           "moe_quant_rows_fp8")
    return q, a


def moe_layer_workspace_bytes_w8a8(dims: Dims) -> int:
    return lib().moe_layer_workspace_bytes_w8a8(ctypes.byref(dims))


def moe_layer_forward_w8a8(x, W_r, bias, dims: Dims, Wgu: W8, Wd: W8, Wgu_s: W8, Wd_s: W8, out,
                           ws, stream=None):
    _check(lib().moe_layer_forward_w8a8(
        _dev(x, torch.int16, "x"), _dev(W_r, torch.float32, "W_r"), _dev(bias, torch.float32, "bias"),
        ctypes.byref(dims), Wgu, Wd, Wgu_s, Wd_s, _dev(out, torch.int16, "out"), _ptr(ws),
        ws.numel(), _stream(stream)), "moe_layer_forward_w8a8")


def moe_gateup_swiglu_w8a8(x, dims: Dims, perm, Wgu: W8, Wgu_s: W8, H, ws, stream=None):
    _check(lib().moe_gateup_swiglu_w8a8(
        _dev(x, torch.int16, "x"), ctypes.byref(dims), _dev(perm, torch.int32, "perm"), Wgu, Wgu_s,
        _dev(H, torch.int16, "H"), _ptr(ws), ws.numel(), _stream(stream)), "moe_gateup_swiglu_w8a8")


def moe_down_w8a8(H, dims: Dims, Wd: W8, Wd_s: W8, Y, ws, stream=None):
    _check(lib().moe_down_w8a8(
        _dev(H, torch.int16, "H"), ctypes.byref(dims), Wd, Wd_s, _dev(Y, torch.float32, "Y"),
        _ptr(ws), ws.numel(), _stream(stream)), "moe_down_w8a8")


def moe_debug_set_waits(ws, wait_ns: int, withhold_stage: int, stream=None):
    """Test hook: the bounded waits' limit and a withheld pipeline stage (see moe.h)."""
    _check(lib().moe_debug_set_waits(_ptr(ws), ws.numel(), wait_ns, withhold_stage,
                                     _stream(stream)), "moe_debug_set_waits")


def moe_import_q4_blocks(blocks: torch.Tensor, K: int, group: int, w_scratch=None,
                         q: torch.Tensor | None = None, s: torch.Tensor | None = None,
                         stream=None):
    """GGUF-style Q4 blocks uint8 [rows][K/32*18] -> (q uint8 [rows][K/2], s fp16 bits as
    int16 [rows][K/group], w_scratch fp32 [rows][K] holding the decoded weights)."""
    rows = blocks.shape[0]
    if blocks.dim() != 2 or blocks.shape[1] != (K // 32) * 18:
        raise ValueError("blocks must be [rows][K/32*18] bytes")
    dev = blocks.device
    if w_scratch is None:
        w_scratch = torch.empty((rows, K), dtype=torch.float32, device=dev)
    if q is None:
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    if s is None:
        s = torch.empty((rows, K // group), dtype=torch.int16, device=dev)
    _check(lib().moe_import_q4_blocks(
        _dev(blocks, torch.uint8, "blocks"), rows, K, group,
        _dev(w_scratch, torch.float32, "w_scratch"), _dev(q, torch.uint8, "q"),
        _dev(s, torch.int16, "s"), _stream(stream)), "moe_import_q4_blocks")
    return q, s, w_scratch


def moe_workspace_bytes(dims: Dims) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(dims))


def moe_layer_workspace_bytes(dims: Dims) -> int:
    return lib().moe_layer_workspace_bytes(ctypes.byref(dims))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace buffer (256-byte aligned by the allocator)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def moe_router_topk(x, W_r, bias, dims: Dims, topk_idx, topk_w, margin, ws, stream=None):
    _check(lib().moe_router_topk(
        _dev(x, torch.int16, "x"), _dev(W_r, torch.float32, "W_r"),
        _dev(bias, torch.float32, "bias"), ctypes.byref(dims),
        _dev(topk_idx, torch.int32, "topk_idx"), _dev(topk_w, torch.float32, "topk_w"),
        None if margin is None else _dev(margin, torch.float32, "margin"),
        _ptr(ws), ws.numel(), _stream(stream)), "moe_router_topk")


def moe_router_topk_noalloc(x, W_r, bias, dims: Dims, topk_idx, topk_w, margin, stream=None):
    """The router without a workspace: its scratch is a fixed device array inside the
    library (see include/moe.h for the size limit and the sharing rules)."""
    _check(lib().moe_router_topk_noalloc(
        _dev(x, torch.int16, "x"), _dev(W_r, torch.float32, "W_r"),
        _dev(bias, torch.float32, "bias"), ctypes.byref(dims),
        _dev(topk_idx, torch.int32, "topk_idx"), _dev(topk_w, torch.float32, "topk_w"),
        None if margin is None else _dev(margin, torch.float32, "margin"), _stream(stream)),
        "moe_router_topk_noalloc")


def moe_build_descriptors(topk_idx, dims: Dims, counts, offsets, perm, pos, sched, ws,
                          stream=None):
    _check(lib().moe_build_descriptors(
        _dev(topk_idx, torch.int32, "topk_idx"), ctypes.byref(dims),
        _dev(counts, torch.int32, "counts"), _dev(offsets, torch.int32, "offsets"),
        _dev(perm, torch.int32, "perm"), _dev(pos, torch.int32, "pos"),
        _dev(sched, torch.int32, "sched"), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_build_descriptors")


def moe_gateup_swiglu_w4a16(x, dims: Dims, offsets, perm, sched, Wgu: W4, Wgu_s: W4, H, ws,
                            stream=None):
    _check(lib().moe_gateup_swiglu_w4a16(
        _dev(x, torch.int16, "x"), ctypes.byref(dims), _dev(offsets, torch.int32, "offsets"),
        _dev(perm, torch.int32, "perm"), _dev(sched, torch.int32, "sched"), Wgu, Wgu_s,
        _dev(H, torch.int16, "H"), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_gateup_swiglu_w4a16")


def moe_down_w4a16(H, dims: Dims, offsets, sched, Wd: W4, Wd_s: W4, Y, ws, stream=None):
    _check(lib().moe_down_w4a16(
        _dev(H, torch.int16, "H"), ctypes.byref(dims), _dev(offsets, torch.int32, "offsets"),
        _dev(sched, torch.int32, "sched"), Wd, Wd_s, _dev(Y, torch.float32, "Y"), _ptr(ws),
        ws.numel(), _stream(stream)), "moe_down_w4a16")


def moe_down_combine_w4a16(H, dims: Dims, offsets, sched, topk_w, pos, Wd: W4, Wd_s: W4,
                           residual, out, ws, stream=None):
    """Down projection with the weighted combine (and an optional residual) fused in;
    ws is a layer-sized workspace (it holds Y)."""
    _check(lib().moe_down_combine_w4a16(
        _dev(H, torch.int16, "H"), ctypes.byref(dims), _dev(offsets, torch.int32, "offsets"),
        _dev(sched, torch.int32, "sched"), _dev(topk_w, torch.float32, "topk_w"),
        _dev(pos, torch.int32, "pos"), Wd, Wd_s,
        None if residual is None else _dev(residual, torch.int16, "residual"),
        _dev(out, torch.int16, "out"), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_down_combine_w4a16")


def moe_combine_shared(Y, topk_w, pos, dims: Dims, out, stream=None):
    _check(lib().moe_combine_shared(
        _dev(Y, torch.float32, "Y"), _dev(topk_w, torch.float32, "topk_w"),
        _dev(pos, torch.int32, "pos"), ctypes.byref(dims), _dev(out, torch.int16, "out"),
        _stream(stream)), "moe_combine_shared")


def moe_combine_shared_residual(Y, topk_w, pos, dims: Dims, residual, out, stream=None):
    """out = bf16(residual + (routed + shared)); out may be residual itself."""
    _check(lib().moe_combine_shared_residual(
        _dev(Y, torch.float32, "Y"), _dev(topk_w, torch.float32, "topk_w"),
        _dev(pos, torch.int32, "pos"), ctypes.byref(dims), _dev(residual, torch.int16, "residual"),
        _dev(out, torch.int16, "out"), _stream(stream)), "moe_combine_shared_residual")


def moe_layer_forward_residual(x, W_r, bias, dims: Dims, Wgu: W4, Wd: W4, Wgu_s: W4, Wd_s: W4,
                               residual, out, ws, stream=None):
    """The layer with the residual add in its last kernel; out may be residual itself."""
    _check(lib().moe_layer_forward_residual(
        _dev(x, torch.int16, "x"), _dev(W_r, torch.float32, "W_r"),
        _dev(bias, torch.float32, "bias"), ctypes.byref(dims), Wgu, Wd, Wgu_s, Wd_s,
        _dev(residual, torch.int16, "residual"), _dev(out, torch.int16, "out"), _ptr(ws),
        ws.numel(), _stream(stream)), "moe_layer_forward_residual")


def moe_pack_w4_bytes(rows: int, K: int, group: int) -> tuple[int, int]:
    """(packed bytes, scale bytes) of moe_pack_w4's output; (0, 0) for arguments it
    rejects."""
    sb = ctypes.c_size_t(0)
    qb = lib().moe_pack_w4_bytes(rows, K, group, ctypes.byref(sb))
    return int(qb), int(sb.value)


def moe_layer_forward(x, W_r, bias, dims: Dims, Wgu: W4, Wd: W4, Wgu_s: W4, Wd_s: W4, out, ws,
                      stream=None):
    _check(lib().moe_layer_forward(
        _dev(x, torch.int16, "x"), _dev(W_r, torch.float32, "W_r"),
        _dev(bias, torch.float32, "bias"), ctypes.byref(dims), Wgu, Wd, Wgu_s, Wd_s,
        _dev(out, torch.int16, "out"), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_layer_forward")


def moe_layer_forward_host(x_host, W_r, bias, dims: Dims, Wgu: W4, Wd: W4, Wgu_s: W4, Wd_s: W4,
                           out_host, ws, stream=None):
    """x_host / out_host: pinned CPU int16 tensors [T][d].  Asynchronous."""
    for t, n in ((x_host, "x_host"), (out_host, "out_host")):
        if t.is_cuda or t.dtype != torch.int16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU int16 tensor")
    _check(lib().moe_layer_forward_host(
        x_host.data_ptr(), _dev(W_r, torch.float32, "W_r"), _dev(bias, torch.float32, "bias"),
        ctypes.byref(dims), Wgu, Wd, Wgu_s, Wd_s, out_host.data_ptr(), _ptr(ws), ws.numel(),
        _stream(stream)), "moe_layer_forward_host")


def moe_check_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns the status (MOE_ERR_DEVICE_CHECK if a device check
    tripped since the last call) without raising."""
    return lib().moe_check_device_status(_ptr(ws), ws.numel(), _stream(stream))
