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
#include "router_dev.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// Small T (decode): split-K GEMV.  Grid (E / 8, ksplit); warp w of block b owns
// expert 8b + w over one K range and every token.  W_r is read once, with
// 16-byte coalesced loads spread over E/8 * ksplit CTAs.
__global__ void __launch_bounds__(256) router_logits_gemv(const uint16_t* __restrict__ x,
                                                         const float* __restrict__ W_r, int T,
                                                         int d, int E, int kchunk,
                                                         float* __restrict__ partial) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    router_gemv_warp(x, W_r, T, d, E, e, blockIdx.y, kchunk, partial, lane);
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
// Top-k: one warp per token.
template <int NV>
__global__ void __launch_bounds__(256) router_topk(const float* __restrict__ partial, int ksplit,
                                                  const float* __restrict__ bias, int T, int E,
                                                  int k, int32_t* __restrict__ topk_idx,
                                                  float* __restrict__ topk_w,
                                                  float* __restrict__ margin) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int sel;
    router_topk_warp<NV>(partial, ksplit, bias, T, E, k, t, lane, topk_idx, topk_w, margin, &sel);
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
