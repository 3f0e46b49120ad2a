"""GPU: the W8A8 variant (fp8 E4M3 weights and activations, reading R16) through the
C ABI against the oracle.

  - moe_pack_w8: codes and row scales bit-exact against the oracle's packing of the
    same fp32 weights, for every expert the checked tokens use and the shared one;
  - moe_quant_rows_fp8: activation codes and row scales bit-exact (the scale and
    every code are decided in fp32 on both sides);
  - moe_layer_forward_w8a8: within the layer bound of the oracle's W8A8 layer on the
    checked tokens (every token up to T = 64, a seeded sample at the prefill sizes),
    at the workloads' shapes and at an odd one (k = E, F != F_s, ragged T), and
    bit-identical when repeated.
"""
import dataclasses
import functools
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import oracle
import workloads
from layer_cases import THREADS, within_layer_bound
from workloads.device import upload

pytestmark = pytest.mark.gpu

ODD = dataclasses.replace(workloads.CONFIGS["tiny"], name="w8_odd", T=37, d=512, E=8, k=8,
                          F=256, Fs=128, group=32, seed=41)
CONFIGS = ["tiny", "decode1", "decode32", "prefill2048", "skew8192", ODD]
SAMPLE = {"prefill2048": 16, "skew8192": 16}


class W8Case:
    def __init__(self, cfg):
        if isinstance(cfg, str):
            cfg = workloads.CONFIGS[cfg]
        self.cfg = cfg
        self.x = workloads.gen_x(cfg)
        W_r, b = workloads.gen_router(cfg)
        idx, w, margin, _ = oracle.router(self.x, W_r, b, cfg.k, threads=THREADS)
        n = SAMPLE.get(cfg.name)
        if n is None or n >= cfg.T:
            self.tokens = np.arange(cfg.T)
        else:
            rng = np.random.default_rng(99 + cfg.seed)
            pick = rng.choice(np.arange(1, cfg.T - 1), n - 2, replace=False)
            self.tokens = np.sort(np.concatenate([[0, cfg.T - 1], pick]))
        self.margin = margin
        self.experts = sorted(set(idx[self.tokens].ravel().tolist()))
        local = {e: i for i, e in enumerate(self.experts)}
        packed = {}
        pool = ThreadPoolExecutor(THREADS)
        slots = threading.BoundedSemaphore(2 * THREADS)  # bounds host fp32 held at once
        jobs = []

        def pack(e, wgu, wdn):
            try:
                packed[e] = (oracle.pack_w8(wgu), oracle.pack_w8(wdn))
            finally:
                slots.release()

        def on_expert(e, wgu, wdn):
            if e < 0 or e in local:
                slots.acquire()
                jobs.append(pool.submit(pack, e, wgu, wdn))

        self.dev = upload(cfg, on_expert=on_expert, fmt="w8")
        for j in jobs:
            j.result()
        pool.shutdown()
        self.packed = packed
        ex = self.experts
        self.W = oracle.PackedLayerW8(
            np.stack([packed[e][0][0] for e in ex]), np.stack([packed[e][0][1] for e in ex]),
            np.stack([packed[e][1][0] for e in ex]), np.stack([packed[e][1][1] for e in ex]),
            *packed[-1][0], *packed[-1][1])
        local_idx = np.vectorize(lambda e: local.get(int(e), 0))(idx).astype(np.int32)
        self.out, _, _ = oracle.layer_w8a8_tokens(self.x, self.W, local_idx, w, self.tokens,
                                                  threads=THREADS)


@functools.lru_cache(maxsize=1)
def w8_case(cfg) -> W8Case:
    return W8Case(cfg)


@pytest.fixture(scope="module", params=CONFIGS, ids=lambda c: c if isinstance(c, str) else c.name)
def C(request):
    return w8_case(request.param)


def _forward(C):
    dims = C.dev.dims()
    ws = moe.workspace(moe.moe_layer_workspace_bytes_w8a8(dims))
    out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
    moe.moe_layer_forward_w8a8(C.dev.x, C.dev.W_r, C.dev.bias, dims, *C.dev.w8s(), out, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


def test_pack_w8_bit_exact(C):
    dev = C.dev
    for e in C.experts[:8] + [-1]:
        (qg, sg), (qd, sd) = C.packed[e]
        gq, gs = (dev.gu_q[e], dev.gu_s[e]) if e >= 0 else (dev.sgu_q, dev.sgu_s)
        dq, ds = (dev.dn_q[e], dev.dn_s[e]) if e >= 0 else (dev.sdn_q, dev.sdn_s)
        assert np.array_equal(gq.cpu().numpy(), qg), e
        assert np.array_equal(gs.cpu().numpy().view(np.uint32), sg.view(np.uint32)), e
        assert np.array_equal(dq.cpu().numpy(), qd), e
        assert np.array_equal(ds.cpu().numpy().view(np.uint32), sd.view(np.uint32)), e


def test_quant_rows_bit_exact(C):
    rows = C.tokens[:64]
    x = C.dev.x[torch.from_numpy(rows).cuda()].contiguous()
    q, a = moe.moe_quant_rows_fp8(x)
    xf = oracle.bf16_to_f32(C.x[rows])
    qo, ao = oracle.quant_rows_fp8(xf)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ao.view(np.uint32))


def test_layer_w8a8_matches_oracle(C):
    got = _forward(C)
    keep = C.margin[C.tokens] >= 1e-5
    ok, rel, mx, bound = within_layer_bound(got[C.tokens[keep]], C.out[keep])
    print(f"[{C.cfg.name}] w8a8 tokens {keep.sum()}: rel_l2 {rel:.3e} max_abs {mx:.3e} "
          f"(bound {bound:.3e})")
    assert ok
    assert np.array_equal(_forward(C), got)  # deterministic


def test_w8a8_stepwise_calls_reproduce_the_layer(C):
    """router, descriptors, moe_gateup_swiglu_w8a8, moe_down_w8a8, moe_combine_shared
    on one W8A8 workspace give moe_layer_forward_w8a8's bits."""
    dev, cfg = C.dev, C.cfg
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    dims = dev.dims()
    ws = moe.workspace(moe.moe_layer_workspace_bytes_w8a8(dims))
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.empty((T, k), **i32)
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    perm, pos, sched = torch.empty(T * k, **i32), torch.empty(T * k, **i32), torch.empty(E, **i32)
    H = torch.empty((T * k + T, max(cfg.F, cfg.Fs)), dtype=torch.int16, device="cuda")
    Y = torch.empty((T * k + T, d), dtype=torch.float32, device="cuda")
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    Wgu, Wd, Wgu_s, Wd_s = dev.w8s()
    moe.moe_router_topk(dev.x, dev.W_r, dev.bias, dims, idx, w, None, ws)
    moe.moe_build_descriptors(idx, dims, counts, offsets, perm, pos, sched, ws)
    moe.moe_gateup_swiglu_w8a8(dev.x, dims, perm, Wgu, Wgu_s, H, ws)
    moe.moe_down_w8a8(H, dims, Wd, Wd_s, Y, ws)
    moe.moe_combine_shared(Y, w, pos, dims, out)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint16), _forward(C))


def test_w8a8_rejects_unsupported_and_small_workspace():
    cfg = workloads.CONFIGS["tiny"]
    dims = moe.Dims(T=4, d=256, E=16, k=2, F=128, F_s=128, group=32, flags=0)
    need = moe.moe_layer_workspace_bytes_w8a8(dims)
    assert need > moe.moe_layer_workspace_bytes(dims)
    ws = moe.workspace(need - 256)
    x = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    W_r = torch.zeros((16, 256), device="cuda")
    b = torch.zeros(16, device="cuda")
    q = torch.zeros(16 * 256 * 256, dtype=torch.uint8, device="cuda")
    s = torch.zeros(16 * 256, dtype=torch.float32, device="cuda")
    W = moe.w8(q, s)
    out = torch.empty((4, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(moe.MoeError) as exc:
        moe.moe_layer_forward_w8a8(x, W_r, b, dims, W, W, W, W, out, ws)
    assert exc.value.status == moe.MOE_ERR_WORKSPACE
    del cfg
