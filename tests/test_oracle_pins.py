"""Pins for the CPU oracle: each test ties an oracle function to something other
than itself -- a library routine on a case that reduces to it, a closed form,
an invariant of the definition, a brute force on tiny inputs, or a
hand-worked fixture under tests/golden/.  No GPU.

The routed MoE layer these functions define: thewafflehaus/butter PR #69,
commits "feat(laguna): Laguna-S-2.1 decode on the CUDA engine" (sigmoid top-10
router with score-correction bias, shared expert, Q4 experts, fused gate+up)
and "feat(laguna): batched prefill with tensor-core projections, fused MoE,
CTA scheduling" (grouped-GEMM MoE with on-device descriptors).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden

# ------------------------------------------------------------------ formats


def _special_f32():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e-8, 5.96e-8,
            2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -15 * 1.5, 1e30, -1e30,
            float("inf"), float("-inf"), 3.4e38]
    # halfway points between neighbouring fp16 values (ties)
    for e in (-20, -10, -3, 0, 4, 14):
        base = 2.0 ** e
        q = base * 2.0 ** -10
        for m in (0, 1, 2, 3, 1021, 1022):
            vals.append(base + (m + 0.5) * q)
    return np.array(vals, np.float32)


def test_f32_to_f16_matches_ieee_library(oracle_lib):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        _special_f32(),
        (rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000)).astype(np.float32),
    ])
    got = oracle_lib.f32_to_f16(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    nan = oracle_lib.f32_to_f16(np.array([np.nan], np.float32))
    assert np.isnan(nan.view(np.float16)[0])


def test_f16_to_f32_all_patterns(oracle_lib):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_lib.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_bf16_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _special_f32(),
        (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32),
        # exact bf16 ties: low 16 bits 0x8000
        (rng.integers(0x00800000, 0x7F000000, 2000).astype(np.uint32) & 0xFFFF0000 |
         0x8000).view(np.float32),
    ])
    got = oracle_lib.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_to_f32_is_top_half_of_f32(oracle_lib):
    h = np.arange(65536, dtype=np.uint32)
    got = oracle_lib.bf16_to_f32(h.astype(np.uint16))
    ref = (h << 16).astype(np.uint32).view(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _bf16_nearest_exact(v: float) -> int:
    """Brute force: the bf16 pattern nearest to v, by exact rational distance."""
    f = Fraction(v)
    sign = 0x8000 if v < 0 else 0
    a = abs(f)
    best = None
    # candidates: the bf16 values just below and above, from the fp32 neighbours
    b = int(np.float32(abs(v)).view(np.uint32)) >> 16
    for c in range(max(0, b - 2), min(0x7F80, b + 3)):
        val = Fraction(float((np.uint32(c) << np.uint32(16)).view(np.float32)))
        dist = abs(val - a)
        key = (dist, c & 1)  # ties go to the even pattern
        if best is None or key < best[0]:
            best = (key, c)
    return sign | best[1]


def test_f64_to_bf16_single_rounding(oracle_lib):
    rng = np.random.default_rng(2)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-5, 5, 3000))
    # just above a bf16 midpoint by far less than fp32 resolution: a double
    # rounding through fp32 would tie to even (down); one rounding goes up
    for m in (1.0 + 2 ** -8, 3.0 + 2 ** -7, 0.75 + 2 ** -9 * 3):
        vals.append(m + 2.0 ** -40)
        vals.append(-(m + 2.0 ** -40))
    x = np.array(vals, np.float64)
    got = oracle_lib.f64_to_bf16(x)
    ref = np.array([_bf16_nearest_exact(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    # the planted midpoint cases really distinguish one rounding from two
    assert oracle_lib.f64_to_bf16(np.array([1.0 + 2 ** -8 + 2.0 ** -40]))[0] == 0x3F81


# ------------------------------------------------------------------ int4 pack


def test_pack_hand_worked_fixture(oracle_lib):
    g = read_golden("pack_w4_example.txt")
    K = int(g["K"][0][0])
    group = int(g["group"][0][0])
    w = np.array([float(v) for row in g["w"] for v in row], np.float32).reshape(1, K)
    q, s = oracle_lib.pack_w4(w, group)
    assert q.tobytes().hex().upper() == "".join(g["bytes"][0])
    assert [f"{v:04X}" for v in s[0]] == g["scales"][0]


@pytest.mark.parametrize("m", [0, 3, 7, 12])
def test_pack_closed_form_power_of_two(oracle_lib, m):
    # w = +-7 * 2^-m at the absmax gives s = 2^-m exactly and q = +-7
    group = 32
    rng = np.random.default_rng(m)
    w = (rng.uniform(-1, 1, (4, 64)) * 7 * 2.0 ** -m * 0.9).astype(np.float32)
    w[:, 5] = 7 * 2.0 ** -m
    w[:, 40] = -7 * 2.0 ** -m
    q, s = oracle_lib.pack_w4(w, group)
    expect_s = (15 - m) << 10  # fp16 pattern of 2^-m
    assert np.all(s == expect_s)
    wh = oracle_lib.dequant_w4(q, s, group)
    assert np.all(wh[:, 5] == 7 * 2.0 ** -m) and np.all(wh[:, 40] == -7 * 2.0 ** -m)


def test_pack_roundtrip_error_bound(oracle_lib):
    rng = np.random.default_rng(3)
    group = 32
    w = (rng.standard_normal((64, 256)) / 16).astype(np.float32)
    w[3, :32] = 0.0  # an all-zero group
    q, s = oracle_lib.pack_w4(w, group)
    wh = oracle_lib.dequant_w4(q, s, group)
    sf = np.repeat(s.view(np.float16).astype(np.float64), group, axis=1)
    err = np.abs(w.astype(np.float64) - wh)
    assert np.all(err <= sf / 2 * (1 + 1e-6) + 1e-30)
    # the absmax element of each group lands on |q| = 7
    qv = wh / np.where(sf == 0, 1, sf)
    wg = np.abs(w).reshape(64, -1, group)
    amax_pos = wg.argmax(axis=2)
    qg = np.abs(qv.reshape(64, -1, group))
    picked = np.take_along_axis(qg, amax_pos[..., None], axis=2)[..., 0]
    nonzero = s.view(np.float16) != 0
    assert np.all(picked[nonzero] == 7)
    assert s[3, 0] == 0 and np.all(q[3, :16] == 0)
    # q is integral and within [-8, 7]
    assert np.all(qv == np.round(qv)) and qv.min() >= -8 and qv.max() <= 7


def test_unpack_every_byte_pattern(oracle_lib):
    # one row holding all 256 byte values with scale 1.0 (fp16 0x3C00)
    q = np.arange(256, dtype=np.uint8).reshape(1, 256)
    s = np.full((1, 512 // 32), 0x3C00, np.uint16)
    wh = oracle_lib.dequant_w4(q, s, 32)[0]

    def sext(n):
        return n - 16 if n >= 8 else n

    expect = []
    for b in range(256):
        expect += [sext(b & 15), sext(b >> 4)]
    assert np.array_equal(wh, np.array(expect, np.float32))


# ------------------------------------------------------------------ router


def _router_inputs(T=24, d=64, E=16, seed=0, bias_scale=0.7):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    x = x.view(torch.int16).numpy().view(np.uint16)
    Wr = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    b = (rng.standard_normal(E) * bias_scale).astype(np.float32)
    return x, Wr, b


def _x_f64(x_bits):
    return (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_router_brute_force_sort(oracle_lib):
    x, Wr, b = _router_inputs()
    k = 4
    idx, w, margin, scores = oracle_lib.router(x, Wr, b, k, want_scores=True)
    logits = _x_f64(x) @ Wr.astype(np.float64).T
    s_ref = 1.0 / (1.0 + np.exp(-logits))
    assert np.allclose(scores, s_ref, rtol=0, atol=1e-14)
    for t in range(x.shape[0]):
        keys = s_ref[t] + b.astype(np.float64)
        order = sorted(range(len(keys)), key=lambda e: (-keys[e], e))
        assert list(idx[t]) == order[:k]
        assert abs(margin[t] - (keys[order[k - 1]] - keys[order[k]])) < 1e-12
        sel = s_ref[t, order[:k]]
        assert np.allclose(w[t], (sel / sel.sum()).astype(np.float32), rtol=1e-6, atol=0)


def test_router_weights_sum_to_one(oracle_lib):
    x, Wr, b = _router_inputs(T=64, E=32, seed=5)
    _, w, _, _ = oracle_lib.router(x, Wr, b, 8)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    assert np.all(w > 0)


def test_router_closed_form_one_hot_input(oracle_lib):
    # x = one-hot 1.0 at coordinate i, so logit_e = W_r[e][i] exactly
    E, d, k = 8, 16, 3
    x = np.zeros((d, d), np.uint16)
    for i in range(d):
        x[i, i] = 0x3F80  # bf16 1.0
    rng = np.random.default_rng(7)
    Wr = rng.uniform(-3, 3, (E, d)).astype(np.float32)
    b = np.zeros(E, np.float32)
    _, _, _, scores = oracle_lib.router(x, Wr, b, k, want_scores=True)
    for i in range(d):
        for e in range(E):
            assert scores[i, e] == 1.0 / (1.0 + math.exp(-float(Wr[e, i])))


def test_router_one_hot_bias_forces_selection(oracle_lib):
    x, Wr, b = _router_inputs(T=16, E=16, seed=9, bias_scale=0.0)
    chosen = [3, 11, 7, 0]
    b2 = np.zeros(16, np.float32)
    b2[chosen] = 10.0
    idx, _, margin, scores = oracle_lib.router(x, Wr, b2, 4, want_scores=True)
    for t in range(16):
        assert sorted(idx[t]) == sorted(chosen)
        # within the forced set the order follows s (bias equal)
        assert list(idx[t]) == sorted(chosen, key=lambda e: (-scores[t, e], e))
        assert margin[t] > 8.0


def test_router_bias_is_for_selection_only(oracle_lib):
    x, Wr, _ = _router_inputs(T=16, E=16, seed=11)
    chosen = [1, 2, 3]
    b1 = np.zeros(16, np.float32)
    b1[chosen] = 10.0
    b2 = b1.copy()
    b2[chosen] = [20.0, 35.0, 12.5]  # same selected set, different bias values
    b2[[5, 6]] = [-3.0, 2.0]
    i1, w1, _, _ = oracle_lib.router(x, Wr, b1, 3)
    i2, w2, _, _ = oracle_lib.router(x, Wr, b2, 3)
    for t in range(16):
        m1 = dict(zip(i1[t], w1[t]))
        m2 = dict(zip(i2[t], w2[t]))
        assert m1 == m2


def test_router_zero_weights_give_uniform_combine(oracle_lib):
    x, _, b = _router_inputs(T=8, E=16, seed=13)
    Wr = np.zeros((16, x.shape[1]), np.float32)
    for k in (1, 2, 4, 10):
        _, w, _, _ = oracle_lib.router(x, Wr, b, k)
        assert np.all(w == np.float32(1.0 / k))


def test_router_ties_go_to_lower_id(oracle_lib):
    x, _, _ = _router_inputs(T=4, E=8, seed=17)
    Wr = np.zeros((8, x.shape[1]), np.float32)  # all scores 0.5
    b = np.array([0, 1, 1, 0, 1, 0, 0, 1], np.float32)
    idx, _, margin, _ = oracle_lib.router(x, Wr, b, 3)
    assert np.all(idx == np.array([1, 2, 4]))
    assert np.all(margin == 0.0)


# ------------------------------------------------------------------ descriptors


def test_descriptors_hand_worked_fixture(oracle_lib):
    g = read_golden("descriptors_example.txt")
    T, k, E = (int(g[n][0][0]) for n in ("T", "k", "E"))
    idx = np.array(g["topk_idx"][0], np.int32).reshape(T, k)
    desc = oracle_lib.descriptors(idx, E)
    for name in ("counts", "offsets", "perm", "pos", "sched"):
        assert list(desc[name]) == [int(v) for v in g[name][0]], name


@pytest.mark.parametrize("seed", range(5))
def test_descriptors_invariants_brute_force(oracle_lib, seed):
    rng = np.random.default_rng(seed)
    T, E, k = int(rng.integers(1, 40)), int(rng.integers(2, 20)), 0
    k = int(rng.integers(1, min(E, 6) + 1))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    desc = oracle_lib.descriptors(idx, E)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(desc["counts"], counts)
    assert desc["offsets"][0] == 0 and np.array_equal(np.diff(desc["offsets"]), counts)
    perm = desc["perm"]
    assert sorted(perm) == list(range(T * k))
    keys = [(idx.ravel()[s], s // k) for s in perm]
    assert keys == sorted(keys)
    assert np.array_equal(desc["pos"][perm], np.arange(T * k))
    brute_sched = sorted(range(E), key=lambda e: (-counts[e], e))
    assert list(desc["sched"]) == brute_sched


# ------------------------------------------------------------------ experts / layer


def _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group):
    return oracle_lib.PackedLayer.from_float(Wgu, Wd, Wgu_s, Wd_s, group)


def test_identity_like_experts_closed_form(oracle_lib):
    """W_r = 0 (all scores 0.5, weights 1/k), bias one-hot on the chosen experts,
    gate = 0.875 P_e, up = 0.4375 P_e, down = 0.875 P_e^T with P_e selecting F
    coordinates; shared expert zero.  Every weight is exact in int4 (s = 2^-m),
    so out_i = bf16( sum_{j: i in P_ej} (1/k) * 0.875 * bf16(silu(0.875 x_i) * 0.4375 x_i) )."""
    d, E, k, F, group = 64, 4, 2, 8, 8
    coords = [list(range(e * 16, e * 16 + F)) for e in range(E)]  # disjoint coordinates
    coords[3] = coords[0][:4] + list(range(56, 60))                # overlap with expert 0
    Wgu = np.zeros((E, 2 * F, d), np.float32)
    Wd = np.zeros((E, d, F), np.float32)
    for e in range(E):
        for f, i in enumerate(coords[e]):
            Wgu[e, f, i] = 0.875
            Wgu[e, F + f, i] = 0.4375
            Wd[e, i, f] = 0.875
    Wgu_s = np.zeros((2 * F, d), np.float32)
    Wd_s = np.zeros((d, F), np.float32)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    rng = np.random.default_rng(21)
    T = 5
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xf = x.float().numpy().astype(np.float64)
    Wr = np.zeros((E, d), np.float32)
    b = np.zeros(E, np.float32)
    b[[0, 3]] = 10.0
    res = oracle_lib.layer(xb, Wr, b, W, k)
    assert np.all(np.sort(res["topk_idx"], 1) == [0, 3])
    assert np.all(res["topk_w"] == np.float32(0.5))
    for t in range(T):
        expect = np.zeros(d)
        for e in (0, 3):
            for i in coords[e]:
                z = 0.875 * xf[t, i]
                hv = z / (1 + math.exp(-z)) * 0.4375 * xf[t, i]
                hb = float(torch.tensor(hv, dtype=torch.float64).to(torch.bfloat16).float())
                expect[i] += 0.5 * (0.875 * hb)
        expect_bf = torch.from_numpy(expect.astype(np.float32)).to(torch.bfloat16)
        expect_bits = expect_bf.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(res["out"][t], expect_bits), t


def test_closed_form_layer_of_the_gpu_tests_on_the_oracle(oracle_lib):
    """The GPU suite's larger identity-like layer (alternating up-row signs, overlapping
    coordinate sets, group 32) gives the closed form bit for bit on the oracle too."""
    from closed_form import (CF, CF_CHOSEN, bf16_bits, closed_form_expect, closed_form_inputs,
                             closed_form_weights)
    coords, sign, Wgu, Wd, Wgu_s, Wd_s = closed_form_weights(31)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, CF["group"])
    x = closed_form_inputs(5, 32)
    b = np.zeros(CF["E"], np.float32)
    b[list(CF_CHOSEN)] = 10.0
    res = oracle_lib.layer(bf16_bits(x), np.zeros((CF["E"], CF["d"]), np.float32), b, W, CF["k"])
    assert np.all(np.sort(res["topk_idx"], 1) == list(CF_CHOSEN))
    assert np.array_equal(res["out"], closed_form_expect(x, coords, sign))


def _random_layer(oracle_lib, T=6, d=64, E=8, k=3, F=32, Fs=32, group=16, seed=0):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    Wr = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    b = (rng.standard_normal(E) * 0.7).astype(np.float32)
    Wgu = (rng.standard_normal((E, 2 * F, d)) / math.sqrt(d)).astype(np.float32)
    Wd = (rng.standard_normal((E, d, F)) / math.sqrt(F)).astype(np.float32)
    Wgu_s = (rng.standard_normal((2 * Fs, d)) / math.sqrt(d)).astype(np.float32)
    Wd_s = (rng.standard_normal((d, Fs)) / math.sqrt(Fs)).astype(np.float32)
    return xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s


def test_layer_within_fp32_bound_of_exact_result(oracle_lib):
    """Exact (fp64) evaluation of the same definition from an independent unpack of
    the bytes; the oracle may differ only by fp32 accumulation and the bf16
    rounding points."""
    d, E, k, F, Fs, group = 64, 8, 3, 32, 32, 16
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, d=d, E=E, k=k, F=F, Fs=Fs,
                                                     group=group)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    res = oracle_lib.layer(xb, Wr, b, W, k, want_h=True)

    def unpack(q, s):
        lo = (q & 15).astype(np.int64)
        hi = (q >> 4).astype(np.int64)
        n = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
        n = np.where(n >= 8, n - 16, n).astype(np.float64)
        sc = np.repeat(s.view(np.float16).astype(np.float64), group, axis=1)
        return n * sc

    xf = _x_f64(xb)
    for t in range(xb.shape[0]):
        acc = np.zeros(d)
        hs = []
        for j in range(k):
            e = res["topk_idx"][t, j]
            gu = unpack(W.q_gu[e], W.s_gu[e])
            dn = unpack(W.q_dn[e], W.s_dn[e])
            g = gu[:F] @ xf[t]
            u = gu[F:] @ xf[t]
            h = g / (1 + np.exp(-g)) * u
            hs.append(h)
            h_or = _x_f64(res["h_routed"][t, j])
            assert np.all(np.abs(h_or - h) <= 2 ** -8 * np.abs(h) + 1e-5)
            acc += float(res["topk_w"][t, j]) * (dn @ h_or)
        gu = unpack(W.qs_gu, W.ss_gu)
        dn = unpack(W.qs_dn, W.ss_dn)
        g, u = gu[:Fs] @ xf[t], gu[Fs:] @ xf[t]
        h = g / (1 + np.exp(-g)) * u
        h_or = _x_f64(res["h_shared"][t])
        assert np.all(np.abs(h_or - h) <= 2 ** -8 * np.abs(h) + 1e-5)
        acc += dn @ h_or
        out = _x_f64(res["out"][t])
        assert np.all(np.abs(out - acc) <= 2 ** -8 * np.abs(acc) + 1e-5)


def test_layer_dense_masked_equals_sparse(oracle_lib):
    """Every expert on every token, masked by the selection, equals the routed path."""
    d, E, k, F, Fs, group = 64, 8, 3, 32, 32, 16
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=4, d=d, E=E, k=k, F=F,
                                                     Fs=Fs, group=group)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    res = oracle_lib.layer(xb, Wr, b, W, k)
    T = xb.shape[0]
    Y = np.zeros((T, E, d), np.float32)
    for t in range(T):
        for e in range(E):
            _, Y[t, e] = oracle_lib.expert_token(xb[t], W.q_gu[e], W.s_gu[e], W.q_dn[e],
                                                 W.s_dn[e], group)
    for t in range(T):
        _, ys = oracle_lib.expert_token(xb[t], W.qs_gu, W.ss_gu, W.qs_dn, W.ss_dn, group)
        acc = np.float32(0) * np.zeros(d, np.float32)
        for j in range(k):
            mask = np.zeros(E, np.float32)
            mask[res["topk_idx"][t, j]] = 1.0
            contrib = (mask[:, None] * Y[t]).sum(0, dtype=np.float32)  # exactly one term
            acc = acc + res["topk_w"][t, j] * contrib
        acc = acc + ys
        expect = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(res["out"][t], expect.view(np.uint16))


def test_layer_relabel_invariance(oracle_lib):
    d, E, k, F, Fs, group = 64, 8, 3, 32, 32, 16
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=6, d=d, E=E, k=k, F=F,
                                                     Fs=Fs, group=group)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    res = oracle_lib.layer(xb, Wr, b, W, k)
    p = np.random.default_rng(1).permutation(E)
    W2 = _pack_expert_stack(oracle_lib, Wgu[p], Wd[p], Wgu_s, Wd_s, group)
    res2 = oracle_lib.layer(xb, Wr[p], b[p], W2, k)
    assert np.array_equal(res["out"], res2["out"])
    assert np.array_equal(p[res2["topk_idx"]], res["topk_idx"])


def test_layer_down_scale_power_of_two(oracle_lib):
    """Doubling every down-projection scale doubles the output exactly."""
    d, E, k, F, Fs, group = 64, 8, 3, 32, 32, 16
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=8, d=d, E=E, k=k, F=F,
                                                     Fs=Fs, group=group)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    res = oracle_lib.layer(xb, Wr, b, W, k)

    def dbl(s):  # fp16 pattern of 2*s (normal, finite values)
        out = s.copy()
        nz = (s & 0x7C00) != 0
        out[nz] = s[nz] + (1 << 10)
        return out

    assert np.all((W.s_dn & 0x7C00) != 0) and np.all((W.ss_dn & 0x7C00) != 0)
    W2 = oracle_lib.PackedLayer(W.q_gu, W.s_gu, W.q_dn, dbl(W.s_dn), W.qs_gu, W.ss_gu, W.qs_dn,
                                dbl(W.ss_dn), group)
    res2 = oracle_lib.layer(xb, Wr, b, W2, k)
    o1 = _x_f64(res["out"])
    o2 = _x_f64(res2["out"])
    assert np.array_equal(o2, 2 * o1)


# ------------------------------------------------------------------ residual add (add3)


def _bf16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_residual_negative_zero_is_identity(oracle_lib):
    """-0 is the additive identity of IEEE addition (x + -0 == x bit for bit,
    -0 included), so a residual of -0 leaves every output bit unchanged."""
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=10)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, 16)
    plain = oracle_lib.layer(xb, Wr, b, W, 3)["out"]
    neg0 = np.full(xb.shape, 0x8000, np.uint16)
    assert np.array_equal(oracle_lib.layer(xb, Wr, b, W, 3, residual=neg0)["out"], plain)


def test_residual_with_zero_experts_is_the_residual(oracle_lib):
    """All expert weights zero: the routed + shared sum is +0, and r + 0 = r is
    already a bf16 value, so the output is the residual itself."""
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=11)
    W = _pack_expert_stack(oracle_lib, 0 * Wgu, 0 * Wd, 0 * Wgu_s, 0 * Wd_s, 16)
    r = _bf16_bits(np.random.default_rng(12).standard_normal(xb.shape) * 3)
    assert np.array_equal(oracle_lib.layer(xb, Wr, b, W, 3, residual=r)["out"], r)


def test_residual_added_after_routed_plus_shared(oracle_lib):
    """out = bf16(r + (routed + shared)) with the bracket summed first, against the
    dense-masked route.  Residuals are chosen per element, where one exists, so that
    the other grouping, (r + routed) + shared, would round to a different bf16
    value: a kernel or oracle that adds in the wrong order fails there."""
    d, E, k, F, Fs, group = 64, 8, 3, 32, 32, 16
    xb, Wr, b, Wgu, Wd, Wgu_s, Wd_s = _random_layer(oracle_lib, seed=13, d=d, E=E, k=k, F=F,
                                                     Fs=Fs, group=group)
    W = _pack_expert_stack(oracle_lib, Wgu, Wd, Wgu_s, Wd_s, group)
    sel = oracle_lib.layer(xb, Wr, b, W, k)
    T = xb.shape[0]
    routed = np.zeros((T, d), np.float32)
    shared = np.zeros((T, d), np.float32)
    for t in range(T):
        for j in range(k):
            e = sel["topk_idx"][t, j]
            _, y = oracle_lib.expert_token(xb[t], W.q_gu[e], W.s_gu[e], W.q_dn[e], W.s_dn[e],
                                           group)
            routed[t] = routed[t] + sel["topk_w"][t, j] * y
        _, shared[t] = oracle_lib.expert_token(xb[t], W.qs_gu, W.ss_gu, W.qs_dn, W.ss_dn, group)
    # candidate residuals: every bf16 value with 2^-6 <= |r| < 2^8
    cand = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    cand = cand[np.isfinite(cand) & (np.abs(cand) >= 2.0 ** -6) & (np.abs(cand) < 2.0 ** 8)]
    r = np.full((T, d), 1.0, np.float32)
    separating = np.zeros((T, d), bool)
    for t in range(T):
        for c in range(d):
            first = _bf16_bits(cand + (routed[t, c] + shared[t, c]))
            other = _bf16_bits((cand + routed[t, c]) + shared[t, c])
            hit = np.nonzero(first != other)[0]
            if hit.size:
                r[t, c] = cand[hit[0]]
                separating[t, c] = True
    assert separating.sum() >= 1
    rb = _bf16_bits(r)
    out = oracle_lib.layer(xb, Wr, b, W, k, residual=rb)["out"]
    assert np.array_equal(out, _bf16_bits(r + (routed + shared)))
    assert not np.array_equal(out[separating], _bf16_bits((r + routed) + shared)[separating])


# ------------------------------------------------------------------ GGUF-style Q4 import


def test_q4_blocks_hand_worked_fixture(oracle_lib):
    g = read_golden("q4_block_example.txt")
    # case A: group 32, the block kept exactly (s = d, q = n - 8)
    K, group = int(g["K"][0][0]), int(g["group"][0][0])
    block = np.array([int(v, 16) for v in g["block"][0]], np.uint8).reshape(1, 18)
    w_ref = np.array([float(v) for row in g["w"] for v in row], np.float32).reshape(1, K)
    assert np.array_equal(oracle_lib.dequant_q4_blocks(block, K), w_ref)
    # the fixture's q and bytes agree with each other (element 2j in the low nibble)
    qv = [int(v) for v in g["q"][0]]
    assert [f"{(qv[2 * j] & 15) | ((qv[2 * j + 1] & 15) << 4):02X}" for j in range(K // 2)] \
        == g["bytes"][0]
    q, s = oracle_lib.import_q4_blocks(block, K, group)
    assert q.tobytes().hex().upper() == "".join(g["bytes"][0])
    assert [f"{v:04X}" for v in s[0]] == g["scales"][0]
    assert np.array_equal(oracle_lib.dequant_w4(q, s, group), w_ref)
    # case B: group 64 over two blocks, re-quantised at absmax / 7
    K, group = int(g["K64"][0][0]), int(g["group64"][0][0])
    block = np.array([int(v, 16) for v in g["block64"][0]], np.uint8).reshape(1, 36)
    qv = [int(v) for row in g["q64"] for v in row]
    assert [f"{(qv[2 * j] & 15) | ((qv[2 * j + 1] & 15) << 4):02X}" for j in range(K // 2)] \
        == g["bytes64"][0]
    q, s = oracle_lib.import_q4_blocks(block, K, group)
    assert q.tobytes().hex().upper() == "".join(g["bytes64"][0])
    assert [f"{v:04X}" for v in s[0]] == g["scales64"][0]


def _q4_blocks(rng, rows, K, codes=None):
    nb = K // 32
    if codes is None:
        codes = rng.integers(0, 16, size=(rows, nb, 32))
    mag = np.exp2(rng.integers(-10, 5, size=(rows, nb))) * (1 + rng.integers(0, 1024, (rows, nb)) / 1024)
    d = (mag * rng.choice([-1.0, 1.0], size=(rows, nb))).astype(np.float16)
    blocks = np.zeros((rows, nb, 18), np.uint8)
    dbits = d.view(np.uint16)
    blocks[:, :, 0] = dbits & 0xFF
    blocks[:, :, 1] = dbits >> 8
    blocks[:, :, 2:] = (codes[:, :, :16] | (codes[:, :, 16:] << 4)).astype(np.uint8)
    return blocks.reshape(rows, nb * 18), d, codes


@pytest.mark.parametrize("group", [8, 16, 32])
def test_q4_import_is_exact_at_groups_within_a_block(oracle_lib, group):
    """At a group of at most 32 the import is lossless for every code, n = 0 (q = -8)
    included, and for scales of either sign: q * s reproduces every block weight bit
    for bit, the scales are d's bits and the nibbles are n ^ 8."""
    rng = np.random.default_rng(31 + group)
    rows, K = 6, 256
    codes = rng.integers(0, 16, size=(rows, K // 32, 32))
    codes[:, :, 0] = 0  # every block holds the weight -8 * d
    blocks, d, codes = _q4_blocks(rng, rows, K, codes)
    w = oracle_lib.dequant_q4_blocks(blocks, K)
    q, s = oracle_lib.import_q4_blocks(blocks, K, group)
    assert np.array_equal(oracle_lib.dequant_w4(q, s, group), w)
    assert np.array_equal(s, np.repeat(d.view(np.uint16), 32 // group, axis=1))
    flat = codes.reshape(rows, K)  # element e of a block: code index e
    assert np.array_equal(q & 15, (flat[:, 0::2] ^ 8).astype(np.uint8))
    assert np.array_equal(q >> 4, (flat[:, 1::2] ^ 8).astype(np.uint8))


def test_q4_import_requantises_groups_spanning_blocks(oracle_lib):
    """At group 64 / 128 a group spans blocks with their own scales: the rows are
    decoded exactly and packed as moe_pack_w4 packs fp32 weights."""
    rng = np.random.default_rng(77)
    rows, K = 4, 512
    blocks, _, _ = _q4_blocks(rng, rows, K)
    w = oracle_lib.dequant_q4_blocks(blocks, K)
    for group in (64, 128):
        q, s = oracle_lib.import_q4_blocks(blocks, K, group)
        qp, sp = oracle_lib.pack_w4(w, group)
        assert np.array_equal(q, qp) and np.array_equal(s, sp)
