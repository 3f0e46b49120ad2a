// Device pieces of the sigmoid top-k router shared by the two router forms
// (router.cu: logits then a top-k kernel; decode.cu: one fused launch).
//
// The Laguna MoE router (thewafflehaus/butter PR #69, commit "feat(laguna):
// Laguna-S-2.1 decode on the CUDA engine"): sigmoid scores s = sigmoid(x . W_r[e]),
// k experts per token chosen by s + bias, the bias shifting the choice only;
// the combine weights are the chosen s normalised to sum 1.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace moe {

// Split-K logit partial of expert e over K range [k0, k0 + kchunk) for every
// token, one warp; partial[(kc * T + t) * E + e].  kchunk is 256 or 512.
constexpr int kRouterTokTile = 16;

__device__ __forceinline__ void router_gemv_warp(const uint16_t* __restrict__ x,
                                                 const float* __restrict__ W_r, int T, int d,
                                                 int E, int e, int kc, int kchunk,
                                                 float* __restrict__ partial, int lane) {
    const int k0 = kc * kchunk;
    const int nvec = kchunk / 128;  // float4 loads per lane
    float4 wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i < nvec)
            wv[i] = __ldg(reinterpret_cast<const float4*>(W_r + (int64_t)e * d + k0) + lane + 32 * i);
        else
            wv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int t0 = 0; t0 < T; t0 += kRouterTokTile) {
        float acc[kRouterTokTile];
#pragma unroll
        for (int tt = 0; tt < kRouterTokTile; ++tt) acc[tt] = 0.f;
#pragma unroll
        for (int tt = 0; tt < kRouterTokTile; ++tt) {
            const int t = t0 + tt;
            if (t < T) {
                const uint2* xr = reinterpret_cast<const uint2*>(x + (int64_t)t * d + k0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < nvec) {
                        const uint2 xv = __ldg(xr + lane + 32 * i);
                        float a = acc[tt];
                        a = fmaf(bf16_lo(xv.x), wv[i].x, a);
                        a = fmaf(bf16_hi(xv.x), wv[i].y, a);
                        a = fmaf(bf16_lo(xv.y), wv[i].z, a);
                        a = fmaf(bf16_hi(xv.y), wv[i].w, a);
                        acc[tt] = a;
                    }
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < kRouterTokTile; ++tt) {
            const int t = t0 + tt;
            if (t < T) {  // warp-uniform
                float v = acc[tt];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) partial[((int64_t)kc * T + t) * E + e] = v;
            }
        }
    }
}

// Logit of (t, e): its ksplit partials summed in kc order.  The loads are
// independent (unrolled), the adds in order.
__device__ __forceinline__ float router_logit(const float* partial, int ksplit, int T, int E, int t,
                                              int e) {
    const float* p = partial + (int64_t)t * E + e;
    const int64_t step = (int64_t)T * E;
    float l = 0.f;
#pragma unroll 8
    for (int kc = 0; kc < ksplit; ++kc) l += __ldcg(p + kc * step);
    return l;
}

struct RouterCand {
    float key;
    float s;
    int e;
};

__device__ __forceinline__ bool router_better(float ka, int ea, float kb, int eb) {
    return ka > kb || (ka == kb && ea < eb);
}

__device__ __forceinline__ RouterCand router_warp_argmax(RouterCand c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RouterCand o_c;
        o_c.key = __shfl_xor_sync(0xffffffffu, c.key, o);
        o_c.s = __shfl_xor_sync(0xffffffffu, c.s, o);
        o_c.e = __shfl_xor_sync(0xffffffffu, c.e, o);
        if (router_better(o_c.key, o_c.e, c.key, c.e)) c = o_c;
    }
    return c;
}

// Bitonic sort of one (key, e, v) per lane across a warp.  DESC: best first
// by (key, then lower e); otherwise by ascending e alone.
template <bool DESC>
__device__ __forceinline__ void warp_bitonic(float& key, int& e, float& v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float pk = __shfl_xor_sync(0xffffffffu, key, stride);
            const int pe = __shfl_xor_sync(0xffffffffu, e, stride);
            const float pv = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool partner_first = DESC ? router_better(pk, pe, key, e) : pe < e;
            const bool lower = (lane & stride) == 0;
            const bool dir = (lane & size) == 0;  // this run is sorted first-to-last
            if (lower == dir ? partner_first : !partner_first) {
                key = pk;
                e = pe;
                v = pv;
            }
        }
    }
}

// Top-k of token t, one warp; lane l holds experts l, l + 32, ...  The logit
// of expert e is the sum of its ksplit partials in kc order.  Selection is k
// rounds of a warp arg-max of s + bias (ties to the lower id).  Lane j < k
// ends with the j-th choice in (*sel_e, *sel_w); the margin (k-th key minus
// the best unselected key, +inf when k == E) goes to margin[t] if non-null.
// `partial` may have been written by other CTAs of the same grid, so it is
// read through L2.
template <int NV>
__device__ __forceinline__ void router_topk_warp(const float* partial, int ksplit,
                                                 const float* __restrict__ bias, int T, int E,
                                                 int k, int t, int lane,
                                                 int32_t* __restrict__ topk_idx,
                                                 float* __restrict__ topk_w,
                                                 float* __restrict__ margin, int* sel_e) {
    float key[NV], sv[NV], lg[NV];
    // the lane's NV logits, each summed over its partials in kc order (as
    // router_logit); one round of NV independent loads per partial, so the
    // loads of all NV experts are in flight together
#pragma unroll
    for (int i = 0; i < NV; ++i) lg[i] = 0.f;
    {
        const float* p = partial + (int64_t)t * E + lane;
        const int64_t step = (int64_t)T * E;
#pragma unroll 2
        for (int kc = 0; kc < ksplit; ++kc) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (lane + 32 * i < E) lg[i] += __ldcg(p + kc * step + 32 * i);
        }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float l = lg[i];
            const float s = 1.0f / (1.0f + expf(-l));
            sv[i] = s;
            key[i] = s + __ldg(bias + e);
        } else {
            sv[i] = 0.f;
            key[i] = -FLT_MAX;
        }
    }
    int my_e = -1;
    float my_s = 0.f, kth_key = 0.f;
    for (int j = 0; j < k; ++j) {
        RouterCand c{-INFINITY, 0.f, 0x7fffffff};
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (e < E && key[i] != -INFINITY && router_better(key[i], e, c.key, c.e))
                c = RouterCand{key[i], sv[i], e};
        }
        c = router_warp_argmax(c);
        if (lane == j) {
            my_e = c.e;
            my_s = c.s;
        }
        kth_key = c.key;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (lane + 32 * i == c.e) key[i] = -INFINITY;
    }
    if (margin) {
        float m = INFINITY;
        if (k < E) {
            RouterCand c{-INFINITY, 0.f, 0x7fffffff};
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = lane + 32 * i;
                if (e < E && key[i] != -INFINITY && router_better(key[i], e, c.key, c.e))
                    c = RouterCand{key[i], sv[i], e};
            }
            c = router_warp_argmax(c);
            m = kth_key - c.key;
        }
        if (lane == 0) margin[t] = m;
    }
    // normaliser: sum of the selected scores in selection order
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, my_s, j);
    if (lane < k) {
        topk_idx[(int64_t)t * k + lane] = my_e;
        topk_w[(int64_t)t * k + lane] = __fdiv_rn(my_s, sum);
    }
    *sel_e = my_e;
}

}  // namespace moe
