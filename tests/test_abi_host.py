"""Host-side checks of the C ABI (no GPU): the library builds and loads, every
symbol include/moe.h declares is exported, and argument validation returns its
documented status codes before anything would be launched."""
import ctypes
import os
import re

import pytest

import moe_expert_layer_sigmoid_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import moe_expert_layer_sigmoid_gb300.build as b
    b.build()
    return moe.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTS)


def test_status_strings(L):
    for code in range(6):
        assert moe.status_string(code).startswith("MOE_")
    assert "unknown" in moe.status_string(99)


def _dims(**kw):
    base = dict(T=4, d=256, E=16, k=2, F=128, F_s=128, group=32, flags=0)
    base.update(kw)
    return moe.Dims(**base)


def test_workspace_bytes(L):
    d = _dims()
    a = moe.moe_workspace_bytes(d)
    b = moe.moe_layer_workspace_bytes(d)
    assert 256 <= a < b
    assert moe.moe_workspace_bytes(_dims(T=4096)) > a
    assert moe.moe_workspace_bytes(_dims(group=48)) == 0
    assert moe.moe_workspace_bytes(_dims(k=17, E=16)) == 0
    # weight-row counts E * 2F and E * d must stay below 2^31
    assert moe.moe_workspace_bytes(_dims(E=1024, k=4, F=(1 << 20) - 128)) > 0
    assert moe.moe_workspace_bytes(_dims(E=1024, k=4, F=1 << 20)) == 0
    assert moe.moe_workspace_bytes(_dims(E=1024, k=4, d=(1 << 21) - 256)) > 0
    assert moe.moe_workspace_bytes(_dims(E=1024, k=4, d=1 << 21)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(group=48), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=300), moe.MOE_ERR_UNSUPPORTED),
    (dict(F=96), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(k=20, E=16), moe.MOE_ERR_INVALID_ARG),
    (dict(k=33, E=64), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=2048, k=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(flags=3), moe.MOE_ERR_INVALID_ARG),
    (dict(E=1024, k=4, F=1 << 20), moe.MOE_ERR_UNSUPPORTED),   # E * 2F = 2^31 weight rows
    (dict(E=1024, k=4, d=1 << 21), moe.MOE_ERR_UNSUPPORTED),   # E * d = 2^31 weight rows
])
def test_dims_validation(L, kw, code):
    d = _dims(**kw)
    ws = ctypes.create_string_buffer(1 << 20)
    got = L.moe_router_topk(None, None, None, ctypes.byref(d), None, None, None,
                            ctypes.addressof(ws), 1 << 20, None)
    assert got == code


def test_workspace_too_small(L):
    d = _dims()
    need = moe.moe_workspace_bytes(d)
    got = L.moe_build_descriptors(None, ctypes.byref(d), None, None, None, None, None, None,
                                  need, None)
    assert got == moe.MOE_ERR_WORKSPACE
    got = L.moe_build_descriptors(None, ctypes.byref(d), None, None, None, None, None, 256, 16,
                                  None)
    assert got == moe.MOE_ERR_WORKSPACE


def test_null_pointers_rejected(L):
    d = _dims()
    need = moe.moe_layer_workspace_bytes(d)
    fake_ws = 1 << 20  # never dereferenced: validation fails first
    assert L.moe_layer_forward(None, None, None, ctypes.byref(d), moe.W4(), moe.W4(), moe.W4(),
                               moe.W4(), None, fake_ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine_shared(None, None, None, ctypes.byref(d), None,
                                None) == moe.MOE_ERR_INVALID_ARG


def test_pack_validation(L):
    assert L.moe_pack_w4(None, 4, 96, 48, None, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_pack_w4(None, 4, 100, 32, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_w4(None, 0, 128, 32, None, None, None) == moe.MOE_OK
    assert L.moe_pack_w4(None, 4, 128, 32, None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_zero_tokens_validates_then_returns_ok(L):
    d = _dims(T=0)
    need = moe.moe_layer_workspace_bytes(d)
    ws = 1 << 20
    assert L.moe_layer_forward(None, None, None, ctypes.byref(d), moe.W4(), moe.W4(), moe.W4(),
                               moe.W4(), None, ws, need, None) == moe.MOE_OK
    bad = _dims(T=0, group=48)
    assert L.moe_layer_forward(None, None, None, ctypes.byref(bad), moe.W4(), moe.W4(), moe.W4(),
                               moe.W4(), None, ws, need, None) == moe.MOE_ERR_UNSUPPORTED


def test_pack_w4_bytes(L):
    assert moe.moe_pack_w4_bytes(6, 256, 32) == (6 * 128, 6 * 8 * 2)
    assert moe.moe_pack_w4_bytes(0, 128, 128) == (0, 0)
    assert moe.moe_pack_w4_bytes(4, 100, 32) == (0, 0)   # K % group != 0
    assert moe.moe_pack_w4_bytes(4, 96, 48) == (0, 0)    # unsupported group
    assert moe.moe_pack_w4_bytes(-1, 128, 32) == (0, 0)
    big = moe.moe_pack_w4_bytes(256 * 2048, 4096, 128)  # every routed gate+up row of a layer
    assert big == (256 * 2048 * 2048, 256 * 2048 * 32 * 2)


def test_residual_calls_validate_before_launch(L):
    d = _dims()
    need = moe.moe_layer_workspace_bytes(d)
    ws = 1 << 20  # never dereferenced: validation fails first
    assert L.moe_layer_forward_residual(None, None, None, ctypes.byref(d), moe.W4(), moe.W4(),
                                        moe.W4(), moe.W4(), None, None, ws, need,
                                        None) == moe.MOE_ERR_INVALID_ARG
    # misaligned residual or out
    assert L.moe_layer_forward_residual(None, None, None, ctypes.byref(d), moe.W4(), moe.W4(),
                                        moe.W4(), moe.W4(), 4096 + 8, 8192, ws, need,
                                        None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine_shared_residual(4096, 4096, 4096, ctypes.byref(d), 4096 + 2, 8192,
                                         None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine_shared_residual(None, None, None, ctypes.byref(_dims(group=48)), None,
                                         None, None) == moe.MOE_ERR_UNSUPPORTED
    d0 = _dims(T=0)
    assert L.moe_layer_forward_residual(None, None, None, ctypes.byref(d0), moe.W4(), moe.W4(),
                                        moe.W4(), moe.W4(), None, None, ws,
                                        moe.moe_layer_workspace_bytes(d0), None) == moe.MOE_OK
    assert L.moe_combine_shared_residual(None, None, None, ctypes.byref(d0), None, None,
                                         None) == moe.MOE_OK


def test_misaligned_activation_pointers_rejected(L):
    """x, W_r, H, Y and out are accessed with 16-byte vector loads and stores: a pointer
    off a 16-byte boundary is an argument error before anything is enqueued."""
    d = _dims()
    step = moe.moe_workspace_bytes(d)
    layer = moe.moe_layer_workspace_bytes(d)
    ws = 1 << 20              # never dereferenced
    ok, bad = 1 << 21, (1 << 21) + 8
    INV = moe.MOE_ERR_INVALID_ARG
    assert L.moe_router_topk(bad, ok, ok, ctypes.byref(d), ok, ok, None, ws, step, None) == INV
    assert L.moe_router_topk(ok, bad, ok, ctypes.byref(d), ok, ok, None, ws, step, None) == INV
    assert L.moe_router_topk_noalloc(bad, ok, ok, ctypes.byref(d), ok, ok, None, None) == INV
    w4 = moe.W4(ok, ok)
    assert L.moe_gateup_swiglu_w4a16(bad, ctypes.byref(d), ok, ok, ok, w4, w4, ok, ws, step,
                                     None) == INV
    assert L.moe_gateup_swiglu_w4a16(ok, ctypes.byref(d), ok, ok, ok, w4, w4, bad, ws, step,
                                     None) == INV
    assert L.moe_down_w4a16(bad, ctypes.byref(d), ok, ok, w4, w4, ok, ws, step, None) == INV
    assert L.moe_down_w4a16(ok, ctypes.byref(d), ok, ok, w4, w4, bad, ws, step, None) == INV
    assert L.moe_combine_shared(bad, ok, ok, ctypes.byref(d), ok, None) == INV
    assert L.moe_combine_shared(ok, ok, ok, ctypes.byref(d), bad, None) == INV
    assert L.moe_layer_forward(bad, ok, ok, ctypes.byref(d), w4, w4, w4, w4, ok, ws, layer,
                               None) == INV
    assert L.moe_layer_forward(ok, ok, ok, ctypes.byref(d), w4, w4, w4, w4, bad, ws, layer,
                               None) == INV


def test_import_q4_blocks_validation(L):
    ok = 1 << 21
    INV, UNS = moe.MOE_ERR_INVALID_ARG, moe.MOE_ERR_UNSUPPORTED
    assert L.moe_import_q4_blocks(None, 0, 64, 32, None, None, None, None) == moe.MOE_OK
    assert L.moe_import_q4_blocks(ok, 2, 48, 16, ok, ok, ok, None) == INV      # K % 32
    assert L.moe_import_q4_blocks(ok, 2, 96, 64, ok, ok, ok, None) == INV      # K % group
    assert L.moe_import_q4_blocks(ok, 2, 96, 48, ok, ok, ok, None) == UNS      # group
    assert L.moe_import_q4_blocks(ok, -1, 64, 32, ok, ok, ok, None) == INV
    assert L.moe_import_q4_blocks(None, 2, 64, 32, ok, ok, ok, None) == INV
    assert L.moe_import_q4_blocks(ok, 2, 64, 32, ok + 4, ok, ok, None) == INV  # w_scratch align
    assert L.moe_import_q4_blocks(ok, 2, 64, 32, ok, ok + 2, ok, None) == INV  # q align


def test_down_combine_validation(L):
    d = _dims()
    step, layer = moe.moe_workspace_bytes(d), moe.moe_layer_workspace_bytes(d)
    ws, ok, bad = 1 << 20, 1 << 21, (1 << 21) + 8
    w4 = moe.W4(ok, ok)
    INV = moe.MOE_ERR_INVALID_ARG

    def call(H=ok, topk_w=ok, pos=ok, residual=None, out=ok, nbytes=layer, dims=d):
        return L.moe_down_combine_w4a16(H, ctypes.byref(dims), ok, ok, topk_w, pos, w4, w4,
                                        residual, out, ws, nbytes, None)

    assert call(nbytes=step) == moe.MOE_ERR_WORKSPACE  # Y lives in the layer workspace
    assert call(H=bad) == INV
    assert call(out=bad) == INV
    assert call(residual=bad) == INV
    assert call(topk_w=None) == INV
    assert call(pos=None) == INV
    assert call(dims=_dims(group=48)) == moe.MOE_ERR_UNSUPPORTED
    d0 = _dims(T=0)
    assert call(H=None, topk_w=None, pos=None, out=None, dims=d0,
                nbytes=moe.moe_layer_workspace_bytes(d0)) == moe.MOE_OK


def test_w8a8_entries_validate_before_launch(L):
    ok, INV = 1 << 21, moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_w8(None, 0, 64, None, None, None) == moe.MOE_OK
    assert L.moe_pack_w8(ok, 4, 60, ok, ok, None) == INV          # K % 8
    assert L.moe_pack_w8(ok + 8, 4, 64, ok, ok, None) == INV      # w alignment
    assert L.moe_pack_w8(ok, 4, 64, ok + 4, ok, None) == INV      # q alignment
    assert L.moe_quant_rows_fp8(ok, 4, 64, ok, ok + 2, None) == INV
    d = _dims()
    need = moe.moe_layer_workspace_bytes_w8a8(d)
    assert need > moe.moe_layer_workspace_bytes(d)
    assert moe.moe_layer_workspace_bytes_w8a8(_dims(group=48)) == 0
    w8 = moe.W8(ok, ok)
    ws = 1 << 22
    assert L.moe_layer_forward_w8a8(ok, ok, ok, ctypes.byref(d), w8, w8, w8, w8, ok, ws, need - 1,
                                    None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_layer_forward_w8a8(ok, ok, ok, ctypes.byref(d), moe.W8(ok, ok + 2), w8, w8, w8,
                                    ok, ws, need, None) == INV
    assert L.moe_layer_forward_w8a8(ok + 8, ok, ok, ctypes.byref(d), w8, w8, w8, w8, ok, ws, need,
                                    None) == INV


def test_debug_set_waits_validation(L):
    assert L.moe_debug_set_waits(None, 1 << 20, 0, 0, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_debug_set_waits(256 + 8, 1 << 20, 0, 0, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_debug_set_waits(1 << 20, 16, 0, 0, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_debug_set_waits(1 << 20, 1 << 20, 0, -1, None) == moe.MOE_ERR_INVALID_ARG
