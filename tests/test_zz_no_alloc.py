"""moe_router_topk_noalloc: the router for callers that cannot allocate device
memory when they call it (a framework that owns every allocation through its
own pool, or a server that reserved all of HBM up front), so cannot pass a
workspace.  Its scratch is a fixed array inside libmoe.so.

Checked through the C ABI against the workspace form, moe_router_topk, on two
calls in a row with different activations: the second call must not see
anything the first left in the shared array.  Collected last, so a stop at
the first failure has already run every other test; it also passes alone in a
fresh process (it builds its own inputs).
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import workloads

pytestmark = pytest.mark.gpu

BASE = workloads.CONFIGS["tiny"]
SHAPES = [
    # decode form of the router (split-K partials): T <= 64
    dataclasses.replace(BASE, name="na_decode", T=8, d=4096, E=256, k=10, F=1024, Fs=1024,
                        group=128, seed=71),
    # prefill form (one partial per logit): T > 64, ragged tiles
    dataclasses.replace(BASE, name="na_prefill", T=300, d=1024, E=64, k=6, F=256, Fs=256,
                        group=64, seed=72),
]


def _route(cfg, x, wr, b, noalloc):
    dims = moe.Dims(T=cfg.T, d=cfg.d, E=cfg.E, k=cfg.k, F=cfg.F, F_s=cfg.Fs, group=cfg.group,
                    flags=0)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    m = torch.empty(cfg.T, dtype=torch.float32, device="cuda")
    if noalloc:
        moe.moe_router_topk_noalloc(x, wr, b, dims, idx, w, m)
    else:
        ws = moe.workspace(moe.moe_workspace_bytes(dims))
        moe.moe_router_topk(x, wr, b, dims, idx, w, m, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), m.cpu().numpy()


@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
def test_noalloc_router_matches_workspace_router_on_two_calls(cfg):
    wr_h, b_h = workloads.gen_router(cfg)
    wr, b = torch.from_numpy(wr_h).cuda(), torch.from_numpy(b_h).cuda()
    for call in range(2):
        x = torch.from_numpy(workloads.gen_x(cfg, batch=call).view(np.int16)).cuda()
        i_ref, w_ref, m_ref = _route(cfg, x, wr, b, noalloc=False)
        i_got, w_got, m_got = _route(cfg, x, wr, b, noalloc=True)
        # the two forms may sum the logit partials in a different order (the
        # workspace form splits K above 64 tokens), so a token whose top-k margin
        # is below 1e-5 may select differently: the matching rule leaves it out
        keep = (m_ref >= 1e-5) & (m_got >= 1e-5)
        assert keep.sum() >= cfg.T - 2, f"call {call}: too many near-ties"
        assert np.array_equal(i_got[keep], i_ref[keep]), f"call {call}: expert ids differ"
        assert np.max(np.abs(w_got[keep] - w_ref[keep])) <= 2e-6, f"call {call}: weights differ"
        assert np.max(np.abs(m_got[keep] - m_ref[keep])) <= 1e-5, f"call {call}: margins differ"


def test_noalloc_router_rejects_sizes_beyond_its_scratch():
    cfg = dataclasses.replace(SHAPES[1], T=5000, d=1024, E=256, k=8)  # 5000 * 256 > 1 Mi floats
    dims = moe.Dims(T=cfg.T, d=cfg.d, E=cfg.E, k=cfg.k, F=cfg.F, F_s=cfg.Fs, group=cfg.group,
                    flags=0)
    x = torch.zeros((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    wr = torch.zeros((cfg.E, cfg.d), dtype=torch.float32, device="cuda")
    b = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as exc:
        moe.moe_router_topk_noalloc(x, wr, b, dims, idx, w, None)
    assert exc.value.status == moe.MOE_ERR_UNSUPPORTED
