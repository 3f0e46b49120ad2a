"""GPU: the single-token layer on the warp-level tensor cores (MOE_FLAG_DECODE_MMA),
through the C ABI.

  - the one-launch step (router, descriptors, gate+up SwiGLU, down, combine in a
    cooperative kernel) against the oracle, at the decode shapes and at odd
    shapes (k = E, F != F_s, groups 32 / 64 / 128), one token per call;
  - the step-by-step calls with the flag (the separate router and descriptor
    calls, then the tensor-core gate+up and down kernels and the combine)
    reproduce the one-launch step bit for bit;
  - repeated calls on one workspace (the grid barrier's counter advances) and a
    CUDA-graph capture replay to the same bits;
  - the residual form against the oracle, and in place.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import oracle
import workloads
from layer_cases import case, to_i16, within_layer_bound

pytestmark = pytest.mark.gpu

MMA = moe.MOE_FLAG_DECODE_MMA
TINY = workloads.CONFIGS["tiny"]

# (d, E, k, F, Fs, group); F and F_s multiples of 256 take the path.  Each shape
# has NTOK tokens, run as NTOK separate T = 1 calls, and the layer bound holds over
# them together: rel-L2 over one token's d outputs is a noisy statistic (at the
# first shape below one token reaches 1.10e-3 on both expert paths).
NTOK = 4
SHAPES = [
    (2048, 16, 16, 512, 256, 128),   # k == E
    (1024, 64, 8, 512, 256, 64),     # F != F_s, group 64
    (512, 32, 4, 256, 512, 32),      # F_s > F, group 32
    (4096, 256, 10, 1024, 1024, 32),  # the decode shapes at group 32
]


def _cfg(i, spec):
    d, E, k, F, Fs, g = spec
    return dataclasses.replace(TINY, name=f"mma{i}", T=NTOK, d=d, E=E, k=k, F=F, Fs=Fs,
                               group=g, seed=300 + i)


@pytest.fixture(scope="module", params=["decode1"] + [f"s{i}" for i in range(len(SHAPES))])
def C(request):
    p = request.param
    return case(p) if not p.startswith("s") else case(_cfg(int(p[1:]), SHAPES[int(p[1:])]))


def _forward(C, flags=MMA, ws=None, x=None):
    """Every token of the case through its own T = 1 layer call."""
    dev = C.dev
    dims = dev.dims(flags, T=1)
    if ws is None:
        ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    x = dev.x if x is None else x
    out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
    for t in range(C.cfg.T):
        moe.moe_layer_forward(x[t:t + 1], dev.W_r, dev.bias, dims, *dev.w4s(), out[t:t + 1], ws)
        assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


def test_mma_step_matches_oracle(C):
    got = _forward(C)
    keep = C.margin[C.tokens] >= 1e-5
    ok, rel, mx, bound = within_layer_bound(got[C.tokens[keep]], C.out[keep])
    core = _forward(C, 0)
    _, rel_c, mx_c, _ = within_layer_bound(core[C.tokens[keep]], C.out[keep])
    print(f"[{C.cfg.name}] mma rel_l2 {rel:.3e} max_abs {mx:.3e}; cuda-core rel_l2 {rel_c:.3e} "
          f"max_abs {mx_c:.3e} (bound {bound:.3e})")
    assert ok
    # and the CUDA-core path computes the same layer
    ok, rel, mx, bound = within_layer_bound(got, _forward(C, 0))
    assert ok, (rel, mx, bound)


def test_mma_stepwise_calls_reproduce_the_step(C):
    dev, cfg = C.dev, C.cfg
    k, E, d = cfg.k, cfg.E, cfg.d
    dims = dev.dims(MMA, T=1)
    ws = moe.workspace(moe.moe_workspace_bytes(dims))
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.empty((1, k), **i32)
    w = torch.empty((1, k), dtype=torch.float32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    perm, pos, sched = torch.empty(k, **i32), torch.empty(k, **i32), torch.empty(E, **i32)
    H = torch.empty((k + 1, max(cfg.F, cfg.Fs)), dtype=torch.int16, device="cuda")
    Y = torch.empty((k + 1, d), dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.T, d), dtype=torch.int16, device="cuda")
    Wgu, Wd, Wgu_s, Wd_s = dev.w4s()
    for t in range(cfg.T):
        x = dev.x[t:t + 1]
        moe.moe_router_topk(x, dev.W_r, dev.bias, dims, idx, w, None, ws)
        moe.moe_build_descriptors(idx, dims, counts, offsets, perm, pos, sched, ws)
        moe.moe_gateup_swiglu_w4a16(x, dims, offsets, perm, sched, Wgu, Wgu_s, H, ws)
        moe.moe_down_w4a16(H, dims, offsets, sched, Wd, Wd_s, Y, ws)
        moe.moe_combine_shared(Y, w, pos, dims, out[t:t + 1])
        assert moe.moe_check_device_status(ws) == moe.MOE_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint16), _forward(C))


def test_mma_repeated_calls_and_graph_replay(C):
    dev = C.dev
    dims = dev.dims(MMA, T=1)
    ref = _forward(C)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    for _ in range(3):  # the grid barrier's counter keeps advancing on one workspace
        assert np.array_equal(_forward(C, ws=ws), ref)
    x = dev.x.clone()
    out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):  # every token's call in one graph
        for t in range(C.cfg.T):
            moe.moe_layer_forward(x[t:t + 1], dev.W_r, dev.bias, dims, *dev.w4s(), out[t:t + 1], ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), ref)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK


def _forward_residual(C, res, out, ws):
    dev = C.dev
    dims = dev.dims(MMA, T=1)
    for t in range(C.cfg.T):
        moe.moe_layer_forward_residual(dev.x[t:t + 1], dev.W_r, dev.bias, dims, *dev.w4s(),
                                       res[t:t + 1], out[t:t + 1], ws)
        assert moe.moe_check_device_status(ws) == moe.MOE_OK


def test_mma_residual_matches_oracle_and_in_place(C):
    dev = C.dev
    dims = dev.dims(MMA, T=1)
    scale = float(np.std((C.out.astype(np.uint32) << 16).view(np.float32)))
    rng = np.random.default_rng(60 + C.cfg.seed)
    r = torch.from_numpy(rng.standard_normal((C.cfg.T, C.cfg.d)).astype(np.float32) * max(scale, 1e-3))
    r_bits = r.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    res = to_i16(r_bits).cuda()
    out = torch.empty_like(res)
    _forward_residual(C, res, out, ws)
    got = out.cpu().numpy().view(np.uint16)
    ref, _, _ = oracle.layer_tokens(C.x, C.W, C.topk_idx, C.topk_w, C.tokens, residual=r_bits)
    keep = C.margin[C.tokens] >= 1e-5
    ok, rel, mx, bound = within_layer_bound(got[C.tokens[keep]], ref[keep])
    assert ok, (rel, mx, bound)
    _forward_residual(C, res, res, ws)
    assert np.array_equal(res.cpu().numpy().view(np.uint16), got)
