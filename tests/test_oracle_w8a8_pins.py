"""Pins of the oracle's W8A8 variant (reading R16), each against something other
than the oracle itself:

  - E4M3 decode of all 256 codes and encode of a sweep of fp32 values (midpoints
    between neighbours, one ulp either side of them, subnormals, signed zeros)
    against PyTorch's independent float8_e4m3fn conversion; saturation by hand;
  - hand-worked weight rows (tests/golden/w8_rows_example.txt);
  - the per-row activation quantisation against the format's error bound;
  - one expert against an fp64 evaluation of the definition from independently
    decoded codes, within the fp32 accumulation bound;
  - an identity-like W8A8 layer against its closed form, whose only lossy step
    (the H row's quantisation) is taken with PyTorch's conversion.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _torch_decode(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn) \
        .float().numpy()


def test_e4m3_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got, ref = oracle.e4m3_to_f32(codes), _torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_an_independent_conversion():
    finite = _torch_decode(np.arange(256, dtype=np.uint8))
    vals = np.unique(finite[~np.isnan(finite)].astype(np.float64))
    mids = (vals[:-1] + vals[1:]) / 2                       # ties: to even
    up = np.nextafter(mids.astype(np.float32), np.float32(np.inf))
    dn = np.nextafter(mids.astype(np.float32), np.float32(-np.inf))
    rng = np.random.default_rng(3)
    rand = (rng.standard_normal(100000) * np.exp(rng.uniform(-12, 6, 100000))).astype(np.float32)
    x = np.concatenate([vals, mids, up, dn, rand, [0.0, -0.0]]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(oracle.f32_to_e4m3(x), _torch_e4m3(x))


def test_e4m3_saturates_to_the_largest_finite():
    x = np.array([448, 449, 464, 465, 1e6, np.inf, -470, -np.inf], np.float32)
    assert list(oracle.f32_to_e4m3(x)) == [0x7E] * 6 + [0xFE] * 2


def test_pack_w8_hand_worked_rows():
    g = read_golden("w8_rows_example.txt")
    for r in range(3):
        w = np.array([[float(v) for v in g[f"row{r}"][0]]], np.float32)
        q, s = oracle.pack_w8(w)
        assert [f"{b:02X}" for b in q[0]] == g[f"codes{r}"][0], r
        if f"scale{r}" in g:
            assert s[0] == np.float32(float(g[f"scale{r}"][0][0]))
        else:
            assert s[0] == np.float32(1.0) / np.float32(448.0)


def test_quant_rows_error_bound_and_the_row_maximum():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 3, (64, 1)))).astype(np.float32)
    x[3] = 0.0
    q, a = oracle.quant_rows_fp8(x)
    assert a[3] == 0 and not q[3].any()
    back = _torch_decode(q).astype(np.float64) * a[:, None]
    # E4M3 with 3 fraction bits: rounding error <= 2^-4 relative for normal codes,
    # <= half the subnormal spacing 2^-10 (times the scale) below 2^-6
    bound = np.maximum(np.abs(x) * 2.0 ** -4, a[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(back - x) <= bound)
    imax = np.argmax(np.abs(x), axis=1)
    rows = np.arange(64)[np.any(x != 0, axis=1)]
    assert np.all(np.abs(_torch_decode(q[rows, imax[rows]])) == 448.0)


def test_expert_token_within_the_fp32_bound_of_an_fp64_evaluation():
    """Evaluate the definition in fp64 from codes decoded by PyTorch; the oracle may
    differ by the fp32 accumulation (d and F terms) and the bf16 rounding of h."""
    rng = np.random.default_rng(9)
    d, F = 256, 64
    x = torch.from_numpy(rng.standard_normal(d).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q_gu, s_gu = oracle.pack_w8((rng.standard_normal((2 * F, d)) / 16).astype(np.float32))
    q_dn, s_dn = oracle.pack_w8((rng.standard_normal((d, F)) / 8).astype(np.float32))
    h, y = oracle.expert_token_w8a8(xb, q_gu, s_gu, q_dn, s_dn)
    xq, a = oracle.quant_rows_fp8(x.float().numpy()[None])
    wg = _torch_decode(q_gu).astype(np.float64)
    xv = _torch_decode(xq[0]).astype(np.float64)
    acc = wg @ xv
    gu = acc * float(a[0]) * s_gu.astype(np.float64)
    tol = 2.0 ** -22 * (np.abs(wg) @ np.abs(xv)) * float(a[0]) * s_gu + 1e-30
    g, u = gu[:F], gu[F:]
    hf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    h64 = g / (1 + np.exp(-g)) * u
    assert np.all(np.abs(hf - h64) <= np.abs(h64) * 2.0 ** -8 + 4 * (tol[:F] + tol[F:]) * 4)
    hq, ah = oracle.quant_rows_fp8(hf.astype(np.float32)[None])
    wd = _torch_decode(q_dn).astype(np.float64)
    hv = _torch_decode(hq[0]).astype(np.float64)
    y64 = (wd @ hv) * float(ah[0]) * s_dn.astype(np.float64)
    ytol = 2.0 ** -22 * (np.abs(wd) @ np.abs(hv)) * float(ah[0]) * s_dn * 4 + 1e-30
    assert np.all(np.abs(y - y64) <= ytol)


def _silu_u(x, sign):
    g = 0.875 * x
    return g / (1.0 + math.exp(-g)) * 0.4375 * x * sign


def test_identity_like_w8a8_layer_closed_form():
    """gate rows 0.875 P_e, up rows +-0.4375 P_e, down rows 0.875 P_e^T: per-row scales
    0.875 / 448 = 2^-9 and 0.4375 / 448 = 2^-10 make every weight code 448, exact.  x
    rows take values k/4 (k = 0..7) with one 1.75 each, so a = 1.75 / 448 = 2^-8 and
    every x code is exact too; g = 0.875 x_i and u = +-0.4375 x_i exactly.  The H row is
    then quantised (the one lossy step): y_i = (448 * hq_i * a_h) * 2^-9 in fp32."""
    d, E, k, F = 64, 4, 2, 16
    rng = np.random.default_rng(12)
    coords = [rng.permutation(d)[:F] for _ in range(E)]
    sign = [1.0, -1.0, 1.0, -1.0]
    Wgu = np.zeros((E, 2 * F, d), np.float32)
    Wd = np.zeros((E, d, F), np.float32)
    for e in range(E):
        Wgu[e, np.arange(F), coords[e]] = 0.875
        Wgu[e, F + np.arange(F), coords[e]] = 0.4375 * sign[e]
        Wd[e, coords[e], np.arange(F)] = 0.875
    W = oracle.PackedLayerW8.from_float(Wgu, Wd, np.zeros((2 * F, d), np.float32),
                                        np.zeros((d, F), np.float32))
    assert np.all(W.s_gu[:, :F] == 2.0 ** -9) and np.all(W.s_gu[:, F:] == 2.0 ** -10)
    T = 3
    x = rng.integers(0, 8, (T, d)) / 4.0 * rng.choice([-1.0, 1.0], (T, d))
    x[:, 0] = 1.75
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    b = np.zeros(E, np.float32)
    b[[1, 2]] = 10.0
    res = oracle.layer_w8a8(xb, np.zeros((E, d), np.float32), b, W, k, want_h=True)
    assert np.all(np.sort(res["topk_idx"], 1) == [1, 2])
    for t in range(T):
        acc = np.zeros(d, np.float32)
        for j in range(k):
            e = int(res["topk_idx"][t, j])
            # + 0.0: a zero h is +0, as every fp32 sum that starts at +0 gives
            hrow = np.array([_silu_u(float(x[t, i]), sign[e]) for i in coords[e]]) + 0.0
            hb = torch.from_numpy(hrow).to(torch.bfloat16).float().numpy()
            assert np.array_equal(res["h_routed"][t, j].view(np.int16),
                                  torch.from_numpy(hb).to(torch.bfloat16).view(torch.int16).numpy())
            a_h = np.float32(np.abs(hb).max()) / np.float32(448)
            hq = _torch_decode(_torch_e4m3(hb / a_h if a_h else hb * 0))
            y = np.zeros(d, np.float32)
            y[coords[e]] = (np.float32(448) * hq * a_h) * np.float32(2.0 ** -9)
            acc = acc + np.float32(0.5) * y
        want = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(res["out"][t], want), t
