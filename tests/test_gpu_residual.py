"""GPU: the residual add folded into the layer's last kernel (the residual +
routed + shared add of thewafflehaus/FFAI PR #72, Nemotron commit
"ffai_add3", with routed and shared summed first), through the C ABI.

  - moe_layer_forward_residual against the oracle's residual form, on the
    default path and both forced expert paths (the decode down kernel's fused
    combine and the standalone combine kernel);
  - a residual of -0 (the additive identity) reproduces moe_layer_forward bit
    for bit, and the in-place form (out is the residual buffer) reproduces the
    out-of-place one;
  - moe_combine_shared_residual bit for bit against a plain fp32 evaluation on
    inputs whose products are exact, with residuals chosen so that the other
    grouping would round differently.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import oracle
from layer_cases import case, to_i16, within_layer_bound

pytestmark = pytest.mark.gpu

PATHS = [0, moe.MOE_FLAG_FORCE_GEMV, moe.MOE_FLAG_FORCE_GROUPED]


def _bf16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _residual(C, seed):
    """Seeded bf16 residual rows on the scale of the layer output."""
    scale = float(np.std((C.out.astype(np.uint32) << 16).view(np.float32)))
    rng = np.random.default_rng(seed)
    return _bf16_bits(rng.standard_normal((C.cfg.T, C.cfg.d)) * max(scale, 1e-3))


def _forward_residual(C, flags, r_bits, in_place=False):
    dev = C.dev
    dims = dev.dims(flags)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    res = to_i16(r_bits).cuda()
    out = res if in_place else torch.empty_like(res)
    moe.moe_layer_forward_residual(dev.x, dev.W_r, dev.bias, dims, *dev.w4s(), res, out, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


def _forward_plain(C, flags):
    dev = C.dev
    dims = dev.dims(flags)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
    moe.moe_layer_forward(dev.x, dev.W_r, dev.bias, dims, *dev.w4s(), out, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module", params=["tiny", "decode1", "decode32"])
def C(request):
    return case(request.param)


@pytest.mark.parametrize("flags", PATHS)
def test_layer_residual_matches_oracle(C, flags):
    if flags == moe.MOE_FLAG_FORCE_GEMV and C.cfg.T > 64:
        pytest.skip("the GEMV path takes at most 64 tokens")
    r = _residual(C, 50 + C.cfg.seed)
    got = _forward_residual(C, flags, r)
    ref, _, _ = oracle.layer_tokens(C.x, C.W, C.topk_idx, C.topk_w, C.tokens, residual=r)
    keep = C.margin[C.tokens] >= 1e-5  # near-ties may select differently (margin rule)
    ok, rel, mx, bound = within_layer_bound(got[C.tokens[keep]], ref[keep])
    print(f"[{C.cfg.name} flags {flags}] rel_l2 {rel:.3e}, max_abs {mx:.3e} (bound {bound:.3e})")
    assert ok


@pytest.mark.parametrize("flags", PATHS)
def test_negative_zero_residual_and_in_place_are_exact(C, flags):
    if flags == moe.MOE_FLAG_FORCE_GEMV and C.cfg.T > 64:
        pytest.skip("the GEMV path takes at most 64 tokens")
    plain = _forward_plain(C, flags)
    neg0 = np.full((C.cfg.T, C.cfg.d), 0x8000, np.uint16)
    assert np.array_equal(_forward_residual(C, flags, neg0), plain)
    r = _residual(C, 70 + C.cfg.seed)
    assert np.array_equal(_forward_residual(C, flags, r, in_place=True),
                          _forward_residual(C, flags, r))


def test_combine_residual_bit_exact_on_exact_products():
    """Weights 1/4 (a power of two) make every product exact, so the kernel's fused
    multiply-adds equal plain fp32 adds in the stated order; the rows are full fp32
    values, so the sums round and the grouping shows."""
    T, d, k, E = 6, 512, 4, 16
    rng = np.random.default_rng(90)
    Yf = rng.standard_normal((T * k + T, d)).astype(np.float32)
    topk_w = np.full((T, k), 0.25, np.float32)
    pos = rng.permutation(T * k).astype(np.int32)
    routed = np.zeros((T, d), np.float32)
    for j in range(k):
        routed = routed + topk_w[:, j:j + 1] * Yf[pos.reshape(T, k)[:, j]]
    shared = Yf[T * k:]
    # residuals that make (r + routed) + shared round differently, where one exists
    cand = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    cand = cand[np.isfinite(cand) & (np.abs(cand) >= 2.0 ** -6) & (np.abs(cand) < 2.0 ** 8)]
    r = rng.standard_normal((T, d)).astype(np.float32)
    r = (_bf16_bits(r).astype(np.uint32) << 16).view(np.float32)
    sep = np.zeros((T, d), bool)
    for t in range(T):
        for c in range(d):
            hit = np.nonzero(_bf16_bits(cand + (routed[t, c] + shared[t, c])) !=
                             _bf16_bits((cand + routed[t, c]) + shared[t, c]))[0]
            if hit.size:
                r[t, c], sep[t, c] = cand[hit[0]], True
    assert sep.sum() >= 1
    expect = _bf16_bits(r + (routed + shared))
    dims = moe.Dims(T=T, d=d, E=E, k=k, F=128, F_s=128, group=32, flags=0)
    Yd = torch.from_numpy(Yf.copy()).cuda()
    wd = torch.from_numpy(topk_w).cuda()
    pd = torch.from_numpy(pos).cuda()
    rd = to_i16(_bf16_bits(r)).cuda()
    out = torch.empty_like(rd)
    moe.moe_combine_shared_residual(Yd, wd, pd, dims, rd, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, expect)
    plain = torch.empty_like(rd)
    moe.moe_combine_shared(Yd, wd, pd, dims, plain)
    torch.cuda.synchronize()
    assert np.array_equal(plain.cpu().numpy().view(np.uint16), _bf16_bits(routed + shared))
