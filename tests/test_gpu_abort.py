"""GPU: the bounded-wait abort path of the grouped kernels, made to run on purpose.

moe_debug_set_waits sets a 1 ms limit on every mbarrier wait and has CTA 0 of
the gate+up launch skip the copies of its first pipeline stage, so that stage's
consumers wait until the limit.  No memory access changes: the copies of the
skipped stage are simply not issued.  The call must then report
MOE_ERR_DEVICE_CHECK (the wait-timeout flag), and after the hook is switched off
the same workspace must give a normal call whose output is bit-identical to a
call on a fresh workspace and, on the W4A16 path, within the bound of the
oracle: the aborted kernel freed its TMEM and left no copy or MMA in flight.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import workloads
from layer_cases import case, within_layer_bound
from workloads.device import upload

pytestmark = pytest.mark.gpu

GROUPED = moe.MOE_FLAG_FORCE_GROUPED
LIMIT_NS = 1_000_000  # 1 ms: every other wait of these small launches takes microseconds


def _run(fwd, dev, dims, weights, ws):
    out = torch.empty((dev.cfg.T, dev.cfg.d), dtype=torch.int16, device="cuda")
    fwd(dev.x, dev.W_r, dev.bias, dims, *weights, out, ws)
    status = moe.moe_check_device_status(ws)
    return status, out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["w4", "w8"])
def test_withheld_stage_times_out_and_the_workspace_recovers(fmt):
    cfg = workloads.CONFIGS["tiny"]
    if fmt == "w4":
        C = case(cfg)
        dev, fwd, weights = C.dev, moe.moe_layer_forward, C.dev.w4s()
        ws_bytes = moe.moe_layer_workspace_bytes
    else:
        C = None
        dev = upload(cfg, fmt="w8")
        fwd, weights = moe.moe_layer_forward_w8a8, dev.w8s()
        ws_bytes = moe.moe_layer_workspace_bytes_w8a8
    dims = dev.dims(GROUPED)
    ws = moe.workspace(ws_bytes(dims))
    moe.moe_debug_set_waits(ws, LIMIT_NS, 1)
    status, _ = _run(fwd, dev, dims, weights, ws)
    assert status == moe.MOE_ERR_DEVICE_CHECK
    moe.moe_debug_set_waits(ws, 0, 0)
    status, got = _run(fwd, dev, dims, weights, ws)
    assert status == moe.MOE_OK
    status, fresh = _run(fwd, dev, dims, weights, moe.workspace(ws_bytes(dims)))
    assert status == moe.MOE_OK
    assert np.array_equal(got, fresh)
    if C is not None:
        ok, rel, mx, bound = within_layer_bound(got[C.tokens], C.out)
        assert ok, (rel, mx, bound)


def test_short_limit_alone_changes_nothing():
    """A 1 ms limit with no withheld stage: every wait ends in time, same bits."""
    C = case(workloads.CONFIGS["tiny"])
    dims = C.dev.dims(GROUPED)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    moe.moe_debug_set_waits(ws, LIMIT_NS, 0)
    status, got = _run(moe.moe_layer_forward, C.dev, dims, C.dev.w4s(), ws)
    assert status == moe.MOE_OK
    status, fresh = _run(moe.moe_layer_forward, C.dev, dims, C.dev.w4s(),
                         moe.workspace(moe.moe_layer_workspace_bytes(dims)))
    assert status == moe.MOE_OK and np.array_equal(got, fresh)
