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
// Large T (prefill): register-blocked SGEMM, logits partial [kz][t][e] =
// sum over the kz-th K slice of x[t][k] * W_r[e][k], fp32 products and sums.
// CTA tile 128 tokens x 128 experts, 256 threads with 8 x 8 outputs each
// (rows ty*4 + {0..3, 64..67}, columns tx*4 + {0..3, 64..67}), K step 8,
// double-buffered shared memory filled from registers loaded one step ahead.
// The K dimension is split over gridDim.z slices so that the grid covers the
// GPU; the top-k sums the slices in order.
constexpr int kSgBM = 128, kSgBN = 128, kSgBK = 16;

__global__ void __launch_bounds__(256) router_logits_sgemm(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ W_r, int T,
                                                          int d, int E, int kchunk,
                                                          float* __restrict__ partial) {
    __shared__ __align__(16) float As[2][kSgBK][kSgBM];
    __shared__ __align__(16) float Bs[2][kSgBK][kSgBN];
    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * kSgBN, t0 = blockIdx.y * kSgBM;
    const int kz = blockIdx.z, kbeg = kz * kchunk;
    const int tx = tid & 15, ty = tid >> 4;
    // loader: row lr (token / expert) of the tile, 8 consecutive k at lk
    const int lr = tid >> 1, lk = (tid & 1) * 8;
    const int lt = t0 + lr, le = e0 + lr;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    auto load = [&](int k, uint4& xa, float4* wb) {
        xa = lt < T ? __ldg(reinterpret_cast<const uint4*>(x + (int64_t)lt * d + k + lk)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            wb[i] = le < E ? __ldg(reinterpret_cast<const float4*>(W_r + (int64_t)le * d + k + lk) + i)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto store = [&](int buf, uint4 xa, const float4* wb) {
        const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            As[buf][lk + 2 * i][lr] = bf16_lo(xw[i]);
            As[buf][lk + 2 * i + 1][lr] = bf16_hi(xw[i]);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            Bs[buf][lk + 4 * i + 0][lr] = wb[i].x;
            Bs[buf][lk + 4 * i + 1][lr] = wb[i].y;
            Bs[buf][lk + 4 * i + 2][lr] = wb[i].z;
            Bs[buf][lk + 4 * i + 3][lr] = wb[i].w;
        }
    };
    uint4 xa;
    float4 wb[2];
    load(kbeg, xa, wb);
    store(0, xa, wb);
    __syncthreads();
    const int nsteps = kchunk / kSgBK;
    for (int s = 0; s < nsteps; ++s) {
        const int buf = s & 1;
        if (s + 1 < nsteps) load(kbeg + (s + 1) * kSgBK, xa, wb);
#pragma unroll
        for (int kk = 0; kk < kSgBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4 + 64]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; j += 2) ffma2(acc[i][j], acc[i][j + 1], av[i], bv[j], bv[j + 1]);
        }
        if (s + 1 < nsteps) store(buf ^ 1, xa, wb);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (t >= T) continue;
        float* row = partial + ((int64_t)kz * T + t) * E;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
            const int e = e0 + tx * 4 + jh * 64;
            if (e + 3 < E) {
                *reinterpret_cast<float4*>(row + e) =
                    make_float4(acc[i][4 * jh], acc[i][4 * jh + 1], acc[i][4 * jh + 2], acc[i][4 * jh + 3]);
            } else {
                for (int j = 0; j < 4; ++j)
                    if (e + j < E) row[e + j] = acc[i][4 * jh + j];
            }
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

int router_ksplit_large(const moe_dims_t& d) {
    if (router_tc_supported(d)) return router_tc_ksplit(d);
    const int64_t tiles = (int64_t)((d.T + kSgBM - 1) / kSgBM) * ((d.E + kSgBN - 1) / kSgBN);
    int ks = 1;
    while (ks * 2 <= d.d / 256 && tiles * ks * 2 <= 320) ks *= 2;
    return ks;
}

cudaError_t launch_router(const uint16_t* x, const float* W_r, const float* bias,
                          const moe_dims_t& dm, int32_t* topk_idx, float* topk_w, float* margin,
                          float* logits, int ksplit, int ksplit_large, uint16_t* planes,
                          WsHeader* hdr, cudaStream_t st) {
    const int T = dm.T, d = dm.d, E = dm.E, k = dm.k;
    int ks = 1;
    if (T <= kRouterSmallT) {
        ks = ksplit;  // d / ks is 256 or 512
        dim3 grid((E + 7) / 8, ks);
        router_logits_gemv<<<grid, 256, 0, st>>>(x, W_r, T, d, E, d / ks, logits);
    } else if (planes && router_tc_supported(dm)) {
        ks = ksplit_large;
        cudaError_t e = launch_router_logits_tc(x, W_r, dm, planes, logits, ks, hdr, st);
        if (e != cudaSuccess) return e;
    } else {
        ks = ksplit_large;  // a power of two dividing d / 256
        dim3 grid((E + kSgBN - 1) / kSgBN, (T + kSgBM - 1) / kSgBM, ks);
        router_logits_sgemm<<<grid, 256, 0, st>>>(x, W_r, T, d, E, d / ks, logits);
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
