"""GPU edge cases through the C ABI: ragged and odd shapes against the oracle,
T = 0, k = E, the device check flag, and both expert paths on shapes that
span several tiles with a ragged tail."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import workloads
from layer_cases import Case, within_layer_bound

pytestmark = pytest.mark.gpu

TINY = workloads.CONFIGS["tiny"]

EDGE_CONFIGS = [
    # (T, d, E, k, F, Fs, group)
    (1, 256, 16, 2, 128, 128, 32),
    (3, 512, 24, 3, 256, 128, 64),       # E not a multiple of 8, F != Fs
    (17, 256, 16, 16, 128, 256, 32),     # k == E: every expert selected, margin = inf
    (65, 512, 40, 5, 128, 128, 128),     # just above the GEMV limit
    (130, 256, 16, 1, 256, 128, 32),     # k = 1, ragged token tiles
    (300, 768, 64, 6, 384, 256, 128),    # several 128-token tiles + ragged tail
    # decode-sized batches at group 128: F != F_s, k == E, several tokens
    # per expert, K from 512 to 4096
    (2, 512, 24, 3, 256, 128, 128),
    (5, 1024, 40, 4, 384, 256, 128),
    (8, 768, 32, 8, 128, 384, 128),
    (1, 2048, 16, 16, 256, 128, 128),    # k == E at T = 1
    (7, 4096, 32, 10, 1024, 1024, 128),  # decode shapes, several tokens per expert
    (9, 256, 1024, 32, 128, 128, 32),    # the largest E and k the library accepts
    # grouped-kernel tile and layout boundaries: 64 tokens per expert on the
    # small-tile layout (64-column accumulators), and 385 tokens per expert on
    # the 192-token layout (tiles of 192, 192 and 1)
    (64, 256, 8, 8, 128, 128, 32),
    (385, 256, 2, 2, 128, 128, 64),
]


def _cfg(i, spec):
    T, d, E, k, F, Fs, g = spec
    return dataclasses.replace(TINY, name=f"edge{i}", T=T, d=d, E=E, k=k, F=F, Fs=Fs, group=g,
                               seed=100 + i)


@pytest.fixture(scope="module", params=list(range(len(EDGE_CONFIGS))))
def E_(request):
    return Case(_cfg(request.param, EDGE_CONFIGS[request.param]))


def _forward(C, flags):
    dims = C.dev.dims(flags)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
    moe.moe_layer_forward(C.dev.x, C.dev.W_r, C.dev.bias, dims, *C.dev.w4s(), out, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("flags", [0, moe.MOE_FLAG_FORCE_GEMV, moe.MOE_FLAG_FORCE_GROUPED])
def test_edge_layer_matches_oracle(E_, flags):
    out = _forward(E_, flags)
    assert E_.margin.min() >= 1e-5 or E_.cfg.k == E_.cfg.E
    ok, rel, mx, bound = within_layer_bound(out[E_.tokens], E_.out)
    assert ok, (E_.cfg, rel, mx, bound)


def test_zero_tokens_is_a_noop():
    dims = moe.Dims(T=0, d=256, E=16, k=2, F=128, F_s=128, group=32, flags=0)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    z = torch.empty(0, dtype=torch.int16, device="cuda")
    f = torch.empty(16, 256, dtype=torch.float32, device="cuda")
    b = torch.empty(16, dtype=torch.float32, device="cuda")
    q = torch.empty(16, dtype=torch.uint8, device="cuda")
    s = torch.empty(16, dtype=torch.int16, device="cuda")
    w = moe.w4(q, s)
    moe.moe_layer_forward(z, f, b, dims, w, w, w, w, z, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK


def test_bad_expert_id_sets_device_flag():
    T, k, E = 8, 2, 16
    dims = moe.Dims(T=T, d=256, E=E, k=k, F=128, F_s=128, group=32, flags=0)
    ws = moe.workspace(moe.moe_workspace_bytes(dims))
    idx = torch.tensor([[0, 1]] * (T - 1) + [[3, 99]], dtype=torch.int32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    perm, pos, sched = torch.zeros(T * k, **i32), torch.zeros(T * k, **i32), torch.empty(E, **i32)
    moe.moe_build_descriptors(idx, dims, counts, offsets, perm, pos, sched, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert moe.moe_check_device_status(ws) == moe.MOE_OK  # the flag was cleared
    assert counts.cpu().numpy().sum() == T * k - 1


def test_pack_odd_shapes_match_oracle():
    import oracle
    rng = np.random.default_rng(5)
    for rows, K, g in ((1, 32, 32), (7, 64, 64), (33, 384, 128), (5, 128, 32)):
        w = (rng.standard_normal((rows, K)) * rng.uniform(1e-6, 10)).astype(np.float32)
        w[0, :g] = 0.0
        q, s = moe.moe_pack_w4(torch.from_numpy(w).cuda(), g)
        qo, so = oracle.pack_w4(w, g)
        assert np.array_equal(q.cpu().numpy(), qo)
        assert np.array_equal(s.cpu().numpy().view(np.uint16), so)


def test_pack_hand_worked_fixture_on_gpu():
    from conftest import read_golden
    gold = read_golden("pack_w4_example.txt")
    K, g = int(gold["K"][0][0]), int(gold["group"][0][0])
    w = np.array([float(v) for row in gold["w"] for v in row], np.float32).reshape(1, K)
    q, s = moe.moe_pack_w4(torch.from_numpy(w).cuda(), g)
    assert q.cpu().numpy().tobytes().hex().upper() == "".join(gold["bytes"][0])
    assert [f"{v:04X}" for v in s.cpu().numpy().view(np.uint16)[0]] == gold["scales"][0]
