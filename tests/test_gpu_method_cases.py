"""GPU: cases whose result the method fixes exactly, through the C ABI.

  - Exact ties in the router: W_r = 0 makes every score sigmoid(0) = 0.5, and
    the bias takes a few repeated values, so many experts tie at the k-th
    place.  The expert lists must equal the oracle's element by element, order
    included (equal scores go to the lower id), on every router form: T = 1,
    T <= 8, T <= 64 and the prefill form; and the whole layer must route the
    same way on every expert path (its output matches the oracle's layer on the
    tie-resolved experts).
  - Identity-like experts, a closed form: expert e's gate rows are 0.875 P_e,
    its up rows +-0.4375 P_e and its down rows 0.875 P_e^T, where P_e picks F of
    the d coordinates; the shared expert is zero; W_r = 0 and a bias of 10 on
    two experts routes every token to them with weight 1/2.  Every weight is
    exact in int4 (one 0.875 per group gives s = 2^-3, q = 7), so
        out_i = bf16( sum_{e : i in P_e} 0.5 * 0.875 * bf16(silu(0.875 x_i) * (+-0.4375 x_i)) ).
    The activations are drawn so that every sum the kernels form is exact in
    fp32 (x on a 2^-7 grid below 4, every nonzero h in one binade) and every
    h lies far from a bf16 rounding boundary; then each expert path must give
    the closed form bit for bit.
  - The grouped kernel without its CTA scheduling (MOE_FLAG_NO_SCHED) on the
    skewed-routing workload: bit-identical to the scheduled order (the order
    of the tiles changes, not the arithmetic of a row) and within the layer
    bound of the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_expert_layer_sigmoid_gb300 as moe
import oracle
import workloads
from closed_form import CF, CF_CHOSEN, bf16_bits, closed_form_expect, closed_form_inputs, \
    closed_form_weights
from layer_cases import case, within_layer_bound

pytestmark = pytest.mark.gpu

TINY = workloads.CONFIGS["tiny"]
GEMV, GROUPED = moe.MOE_FLAG_FORCE_GEMV, moe.MOE_FLAG_FORCE_GROUPED
MMA, NO_SCHED = moe.MOE_FLAG_DECODE_MMA, moe.MOE_FLAG_NO_SCHED


def _i16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _tie_bias(E: int, k: int, seed: int) -> np.ndarray:
    """Three repeated values, the top one shared by more than k experts (so the k-th
    place is a tie) at random ids."""
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 2, E) * 0.25
    n_top = min(E, k + 1 + int(rng.integers(0, k + 1)))
    b[rng.permutation(E)[:n_top]] = 0.5
    return b.astype(np.float32)


# ------------------------------------------------------------------ router ties

TIE_ROUTER = [  # (T, d, E, k): the T = 1, T <= 8, T <= 64 and prefill forms (fp32 SGEMM at
    # E = 64, the tensor-core form at E = 256)
    (1, 4096, 256, 10), (5, 1024, 64, 6), (8, 512, 16, 4), (40, 4096, 256, 10),
    (300, 1024, 64, 8), (300, 1024, 256, 8),
]


@pytest.mark.parametrize("T,d,E,k", TIE_ROUTER)
def test_router_exact_ties_match_oracle_order(T, d, E, k):
    rng = np.random.default_rng(1000 + T)
    x = bf16_bits(rng.standard_normal((T, d)))
    W_r = np.zeros((E, d), np.float32)
    b = _tie_bias(E, k, T)
    idx_o, w_o, m_o, _ = oracle.router(x, W_r, b, k)
    top = np.sort(b)[::-1]
    assert top[k - 1] == top[k], "the k-th place must be a tie"
    dims = moe.Dims(T=T, d=d, E=E, k=k, F=256, F_s=256, group=128, flags=0)
    ws = moe.workspace(moe.moe_workspace_bytes(dims))
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m = torch.empty(T, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(_i16(x), torch.from_numpy(W_r).cuda(), torch.from_numpy(b).cuda(), dims,
                        idx, w, m, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    assert np.array_equal(idx.cpu().numpy(), idx_o)  # ids and their order
    assert np.array_equal(w.cpu().numpy(), w_o)      # 0.5 / (k * 0.5), one rounding
    assert np.all(m.cpu().numpy() == 0.0) and np.all(m_o == 0.0)


TIE_LAYER = dataclasses.replace(TINY, name="ties", T=40, d=512, E=64, k=6, F=256, Fs=256,
                                group=32, seed=77)


@pytest.fixture(scope="module")
def tie_case():
    return case(TIE_LAYER)


def _layer(C, x, W_r, b, flags, T):
    dims = C.dev.dims(flags, T=T)
    ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
    out = torch.empty((T, C.cfg.d), dtype=torch.int16, device="cuda")
    moe.moe_layer_forward(x, W_r, b, dims, *C.dev.w4s(), out, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_OK
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("form", ["t1", "t1_mma", "t3", "t40", "t40_gemv"])
def test_layer_routes_exact_ties_like_the_oracle(tie_case, form):
    """The router inside each layer form: the fused decode router (T = 1 on the decode
    chain, T = 3 and T = 40 forced onto it), the single-launch step's own router, and
    the standalone router before the grouped path (T = 40)."""
    C = tie_case
    cfg = C.cfg
    W_r = np.zeros((cfg.E, cfg.d), np.float32)
    b = _tie_bias(cfg.E, cfg.k, 5)
    idx_o, w_o, _, _ = oracle.router(C.x, W_r, b, cfg.k)
    ref, _, _ = oracle.layer_tokens(C.x, C.W, idx_o, w_o, np.arange(cfg.T))
    W_r_d, b_d = torch.from_numpy(W_r).cuda(), torch.from_numpy(b).cuda()
    x = C.dev.x
    if form in ("t1", "t1_mma"):
        flags = MMA if form == "t1_mma" else 0
        got = np.concatenate([_layer(C, x[t:t + 1], W_r_d, b_d, flags, 1) for t in range(4)])
        want = ref[:4]
    elif form == "t3":
        got, want = _layer(C, x[:3], W_r_d, b_d, GEMV, 3), ref[:3]
    else:
        got = _layer(C, x, W_r_d, b_d, GEMV if form == "t40_gemv" else 0, cfg.T)
        want = ref
    ok, rel, mx, bound = within_layer_bound(got, want)
    assert ok, (form, rel, mx, bound)


# ------------------------------------------------------------------ closed form

@pytest.fixture(scope="module")
def closed_form():
    d, E, k, F, Fs, g = (CF[n] for n in ("d", "E", "k", "F", "Fs", "group"))
    coords, sign, Wgu, Wd, Wgu_s, Wd_s = closed_form_weights(31)
    pk = lambda w: moe.moe_pack_w4(torch.from_numpy(w.reshape(-1, w.shape[-1])).cuda(), g)
    gq, gs = pk(Wgu)
    dq, ds = pk(Wd)
    sgq, sgs = pk(Wgu_s)
    sdq, sds = pk(Wd_s)
    W = (moe.w4(gq.view(E, 2 * F, d // 2), gs.view(E, 2 * F, d // g)),
         moe.w4(dq.view(E, d, F // 2), ds.view(E, d, F // g)),
         moe.w4(sgq, sgs), moe.w4(sdq, sds))
    T = 5
    x = closed_form_inputs(T, 32)
    xb = bf16_bits(x)
    assert np.array_equal(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float().numpy(),
                          x), "x must be exact in bf16"
    b = np.zeros(E, np.float32)
    b[list(CF_CHOSEN)] = 10.0
    keep = (W, gq, gs, dq, ds, sgq, sgs, sdq, sds)
    return dict(T=T, xb=xb, W=W, W_r=torch.zeros((E, d), device="cuda"),
                b=torch.from_numpy(b).cuda(), expect=closed_form_expect(x, coords, sign),
                keep=keep)


@pytest.mark.parametrize("path", ["default", "gemv", "grouped", "t1", "t1_mma"])
def test_identity_like_experts_closed_form_bit_exact(closed_form, path):
    cf = closed_form
    T = cf["T"]
    d, E, k, F, Fs, g = (CF[n] for n in ("d", "E", "k", "F", "Fs", "group"))

    def run(x_bits, flags):
        n = x_bits.shape[0]
        dims = moe.Dims(T=n, d=d, E=E, k=k, F=F, F_s=Fs, group=g, flags=flags)
        ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
        out = torch.empty((n, d), dtype=torch.int16, device="cuda")
        moe.moe_layer_forward(_i16(x_bits), cf["W_r"], cf["b"], dims, *cf["W"], out, ws)
        assert moe.moe_check_device_status(ws) == moe.MOE_OK
        return out.cpu().numpy().view(np.uint16)

    if path in ("t1", "t1_mma"):
        flags = MMA if path == "t1_mma" else 0
        got = np.concatenate([run(cf["xb"][t:t + 1], flags) for t in range(T)])
    else:
        got = run(cf["xb"], {"default": 0, "gemv": GEMV, "grouped": GROUPED}[path])
    bad = np.argwhere(got != cf["expect"])
    assert bad.size == 0, f"{path}: {len(bad)} outputs differ, first {bad[:4].tolist()}"
    assert np.count_nonzero(cf["expect"]) > T * 100  # the case is not mostly zeros


# ------------------------------------------------------------------ scheduling A/B

def test_no_sched_is_bit_identical_and_within_the_layer_bound():
    C = case("skew8192")
    dims = C.dev.dims(0)
    outs = []
    for flags in (0, NO_SCHED):
        dims = C.dev.dims(flags)
        ws = moe.workspace(moe.moe_layer_workspace_bytes(dims))
        out = torch.empty((C.cfg.T, C.cfg.d), dtype=torch.int16, device="cuda")
        moe.moe_layer_forward(C.dev.x, C.dev.W_r, C.dev.bias, dims, *C.dev.w4s(), out, ws)
        assert moe.moe_check_device_status(ws) == moe.MOE_OK
        outs.append(out.cpu().numpy().view(np.uint16))
    assert np.array_equal(outs[0], outs[1])
    keep = C.margin[C.tokens] >= 1e-5
    ok, rel, mx, bound = within_layer_bound(outs[1][C.tokens[keep]], C.out[keep])
    assert ok, (rel, mx, bound)
