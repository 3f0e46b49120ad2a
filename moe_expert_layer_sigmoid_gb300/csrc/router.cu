// Sigmoid top-k router with a score-correction bias.
//
// The Laguna MoE router (thewafflehaus/butter PR #69, commit "feat(laguna):
// Laguna-S-2.1 decode on the CUDA engine"): sigmoid scores s = sigmoid(x . W_r[e]),
// ten experts per token chosen by s + bias, the bias shifting the choice only;
// the combine weights are the chosen s normalised to sum 1.
//
// Two kernels: router logits (fp32 accumulate) into a partial-sum buffer, then
// a warp-per-token kernel that sums the partials in a fixed order, applies the
// sigmoid and the bias, and extracts the top k by k rounds of a warp shuffle
// arg-max (ties to the lower expert id).
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// Small T (decode): split-K GEMV.  Grid (E / 8, ksplit); warp w of block b owns
// expert 8b + w over K range [kc * kchunk, (kc + 1) * kchunk) and every token.
// W_r is read once, with 16-byte coalesced loads spread over E/8 * ksplit CTAs.
constexpr int kRouterTokTile = 16;

__global__ void __launch_bounds__(256) router_logits_gemv(const uint16_t* __restrict__ x,
                                                         const float* __restrict__ W_r, int T,
                                                         int d, int E, int kchunk,
                                                         float* __restrict__ partial) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    const int kc = blockIdx.y;
    if (e >= E) return;
    const int k0 = kc * kchunk;
    const int nvec = kchunk / 128;  // float4 loads per lane (kchunk in {256, 512})
    // this lane's W_r slice: float4 at k0 + 4 * (lane + 32 * i)
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
                        uint2 xv = __ldg(xr + lane + 32 * i);
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
            float v = acc[tt];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            const int t = t0 + tt;
            if (lane == 0 && t < T) partial[((int64_t)kc * T + t) * E + e] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// Large T (prefill): 64 x 64 register-tiled SGEMM, logits[t][e] = x[t] . W_r[e].
constexpr int kBM = 64, kBN = 64, kBK = 16;

__global__ void __launch_bounds__(256) router_logits_sgemm(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ W_r, int T,
                                                          int d, int E, float* __restrict__ out) {
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Bs[kBK][kBN + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.y * kBM, e0 = blockIdx.x * kBN;
    const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4 x 4 outputs each
    float acc[4][4] = {};
    // loader mapping: 64 rows x 16 k = 1024 elements = 256 threads x 4
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    for (int kb = 0; kb < d; kb += kBK) {
        {
            const int t = t0 + lr;
            float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
            if (t < T) {
                uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (int64_t)t * d + kb + lk));
                v0 = bf16_lo(xv.x); v1 = bf16_hi(xv.x); v2 = bf16_lo(xv.y); v3 = bf16_hi(xv.y);
            }
            As[lk + 0][lr] = v0; As[lk + 1][lr] = v1; As[lk + 2][lr] = v2; As[lk + 3][lr] = v3;
            const int e = e0 + lr;
            float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E) wv = __ldg(reinterpret_cast<const float4*>(W_r + (int64_t)e * d + kb + lk));
            Bs[lk + 0][lr] = wv.x; Bs[lk + 1][lr] = wv.y; Bs[lk + 2][lr] = wv.z; Bs[lk + 3][lr] = wv.w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) out[(int64_t)t * E + e] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------------------------
// Top-k: one warp per token; lane l holds experts l, l + 32, ...
struct Cand {
    float key;
    float s;
    int e;
};

__device__ __forceinline__ bool better(float ka, int ea, float kb, int eb) {
    return ka > kb || (ka == kb && ea < eb);
}

__device__ __forceinline__ Cand warp_argmax(Cand c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Cand o_c;
        o_c.key = __shfl_xor_sync(0xffffffffu, c.key, o);
        o_c.s = __shfl_xor_sync(0xffffffffu, c.s, o);
        o_c.e = __shfl_xor_sync(0xffffffffu, c.e, o);
        if (better(o_c.key, o_c.e, c.key, c.e)) c = o_c;
    }
    return c;
}

template <int NV>
__global__ void __launch_bounds__(256) router_topk(const float* __restrict__ partial, int ksplit,
                                                  const float* __restrict__ bias, int T, int E,
                                                  int k, int32_t* __restrict__ topk_idx,
                                                  float* __restrict__ topk_w,
                                                  float* __restrict__ margin) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float key[NV], sv[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            float l = 0.f;
            for (int kc = 0; kc < ksplit; ++kc) l += partial[((int64_t)kc * T + t) * E + e];
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
        Cand c{-INFINITY, 0.f, 0x7fffffff};
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (e < E && key[i] != -INFINITY && better(key[i], e, c.key, c.e)) c = Cand{key[i], sv[i], e};
        }
        c = warp_argmax(c);
        if (lane == j) { my_e = c.e; my_s = c.s; }
        kth_key = c.key;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (lane + 32 * i == c.e) key[i] = -INFINITY;
    }
    if (margin) {
        float m = INFINITY;
        if (k < E) {
            Cand c{-INFINITY, 0.f, 0x7fffffff};
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = lane + 32 * i;
                if (e < E && key[i] != -INFINITY && better(key[i], e, c.key, c.e)) c = Cand{key[i], sv[i], e};
            }
            c = warp_argmax(c);
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
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, const float* W_r, const float* bias,
                          const moe_dims_t& dm, int32_t* topk_idx, float* topk_w, float* margin,
                          float* logits, int ksplit, cudaStream_t st) {
    const int T = dm.T, d = dm.d, E = dm.E, k = dm.k;
    int ks = 1;
    if (T <= kRouterSmallT) {
        ks = ksplit;  // d / ks is 256 or 512
        dim3 grid((E + 7) / 8, ks);
        router_logits_gemv<<<grid, 256, 0, st>>>(x, W_r, T, d, E, d / ks, logits);
    } else {
        dim3 grid((E + kBN - 1) / kBN, (T + kBM - 1) / kBM);
        router_logits_sgemm<<<grid, 256, 0, st>>>(x, W_r, T, d, E, logits);
    }
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int warps = 8;
    const unsigned blocks = (unsigned)((T + warps - 1) / warps);
    if (E <= 256)
        router_topk<8><<<blocks, 32 * warps, 0, st>>>(logits, ks, bias, T, E, k, topk_idx, topk_w, margin);
    else if (E <= 512)
        router_topk<16><<<blocks, 32 * warps, 0, st>>>(logits, ks, bias, T, E, k, topk_idx, topk_w, margin);
    else
        router_topk<32><<<blocks, 32 * warps, 0, st>>>(logits, ks, bias, T, E, k, topk_idx, topk_w, margin);
    return cudaGetLastError();
}

}  // namespace moe
