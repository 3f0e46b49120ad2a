// Decode-side expert projections: int4 GEMV on CUDA cores.
//
// The Laguna decode path runs the MoE gate+up projection fused (SwiGLU) and the
// shared expert through the same gathered kernel (thewafflehaus/butter PR #69,
// commit "feat(laguna): Laguna-S-2.1 decode on the CUDA engine").  Here one CTA
// owns a band of output rows of one expert (or of the shared expert) and
// every token routed to it; weights stream from HBM once per token tile with
// coalesced 16-byte loads (32 nibbles per load, one group scale per load),
// activations are gathered through the descriptor permutation into shared
// memory.
//
// Arithmetic: a 32-element chunk is contracted against exact integer q values
// (q = nibble, made an fp32 integer by the 2^23 exponent trick) and the
// chunk's fp32 partial sum is multiplied by its group scale; since q * s is the
// dequantised weight exactly, this computes sum_i x_i * (q_i * s) with only
// fp32 summation rounding.
#include "common.cuh"

namespace moe {
namespace {

// Offset-binary nibble u = q + 8 in the low mantissa bits of 2^23: value 2^23 + u.
constexpr float kMagicOffset = 8388616.0f;  // 2^23 + 8

__device__ __forceinline__ float dot8_q4(uint32_t w, uint4 xv) {
    const uint32_t u = w ^ 0x88888888u;  // two's complement nibble -> offset binary
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = __uint_as_float(0x4B000000u | ((u >> (4 * j)) & 0xFu)) - kMagicOffset;
    float a = q[0] * bf16_lo(xv.x);
    a = fmaf(q[1], bf16_hi(xv.x), a);
    a = fmaf(q[2], bf16_lo(xv.y), a);
    a = fmaf(q[3], bf16_hi(xv.y), a);
    a = fmaf(q[4], bf16_lo(xv.z), a);
    a = fmaf(q[5], bf16_hi(xv.z), a);
    a = fmaf(q[6], bf16_lo(xv.w), a);
    a = fmaf(q[7], bf16_hi(xv.w), a);
    return a;
}

// 32 nibbles (one 16-byte load) against 32 bf16 activations (four 16-byte words).
__device__ __forceinline__ float dot32_q4(uint4 w, const uint4* xs) {
    float a = dot8_q4(w.x, xs[0]);
    a += dot8_q4(w.y, xs[1]);
    a += dot8_q4(w.z, xs[2]);
    a += dot8_q4(w.w, xs[3]);
    return a;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Group descriptor of blockIdx.y: a routed expert in schedule order, or the
// shared expert after the last routed group.
struct GroupRef {
    int64_t row0;  // first row of H / Y
    int count;     // rows (tokens) in the group
    int Fg;        // FFN width of the group
    int expert;    // -1 for the shared expert
};

__device__ __forceinline__ GroupRef group_of(int y, int n_route_groups, int T, int k, int F,
                                             int Fs, const int32_t* offsets, const int32_t* sched) {
    GroupRef g;
    if (y < n_route_groups) {
        const int e = sched[y];
        g.expert = e;
        g.row0 = offsets[e];
        g.count = offsets[e + 1] - offsets[e];
        g.Fg = F;
    } else {
        g.expert = -1;
        g.row0 = (int64_t)T * k;
        g.count = T;
        g.Fg = Fs;
    }
    return g;
}

constexpr int kGuRowPairsPerWarp = 2;
constexpr int kGuRowsPerCta = 8 * kGuRowPairsPerWarp;  // gate rows (and as many up rows) per CTA

template <int TOK>
__global__ void __launch_bounds__(256)
gateup_gemv_kernel(const uint16_t* __restrict__ x, int T, int d, int k, int F, int Fs, int group,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
                   const int32_t* __restrict__ sched, const uint8_t* __restrict__ q_r,
                   const __half* __restrict__ s_r, const uint8_t* __restrict__ q_sh,
                   const __half* __restrict__ s_sh, uint16_t* __restrict__ H, int ldh,
                   int n_route_groups) {
    extern __shared__ uint4 xs[];  // [TOK][d / 8]
    const GroupRef g = group_of(blockIdx.y, n_route_groups, T, k, F, Fs, offsets, sched);
    if (g.count == 0) return;
    const int f0 = blockIdx.x * kGuRowsPerCta;
    if (f0 >= g.Fg) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d8 = d / 8, nchunk = d / 32, ngr = d / group;
    const uint8_t* qg = g.expert >= 0 ? q_r + (int64_t)g.expert * 2 * F * (d / 2) : q_sh;
    const __half* sg = g.expert >= 0 ? s_r + (int64_t)g.expert * 2 * F * ngr : s_sh;

    for (int i0 = 0; i0 < g.count; i0 += TOK) {
        const int ntok = min(TOK, g.count - i0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < ntok * d8; idx += blockDim.x) {
            const int tt = idx / d8, c8 = idx - tt * d8;
            const int64_t row = g.row0 + i0 + tt;
            const int tok = g.expert >= 0 ? perm[row] / k : (int)(row - g.row0);
            xs[tt * d8 + c8] = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)tok * d) + c8);
        }
        __syncthreads();
#pragma unroll
        for (int p = 0; p < kGuRowPairsPerWarp; ++p) {
            const int f = f0 + warp * kGuRowPairsPerWarp + p;
            const uint4* gq = reinterpret_cast<const uint4*>(qg + (int64_t)f * (d / 2));
            const uint4* uq = reinterpret_cast<const uint4*>(qg + (int64_t)(g.Fg + f) * (d / 2));
            const __half* gsc = sg + (int64_t)f * ngr;
            const __half* usc = sg + (int64_t)(g.Fg + f) * ngr;
            float accg[TOK], accu[TOK];
#pragma unroll
            for (int tt = 0; tt < TOK; ++tt) accg[tt] = accu[tt] = 0.f;
            for (int c = lane; c < nchunk; c += 32) {
                const uint4 wg = __ldg(gq + c), wu = __ldg(uq + c);
                const float scg = __half2float(gsc[(32 * c) / group]);
                const float scu = __half2float(usc[(32 * c) / group]);
#pragma unroll
                for (int tt = 0; tt < TOK; ++tt) {
                    if (tt < ntok) {
                        const uint4* xv = xs + tt * d8 + 4 * c;
                        accg[tt] = fmaf(scg, dot32_q4(wg, xv), accg[tt]);
                        accu[tt] = fmaf(scu, dot32_q4(wu, xv), accu[tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < TOK; ++tt) {
                const float gv = warp_sum(accg[tt]);
                const float uv = warp_sum(accu[tt]);
                if (lane == 0 && tt < ntok) {
                    const float h = gv / (1.0f + expf(-gv)) * uv;
                    H[(g.row0 + i0 + tt) * ldh + f] = float_to_bf16_bits(h);
                }
            }
        }
    }
}

constexpr int kDnRowsPerWarp = 4;
constexpr int kDnRowsPerCta = 8 * kDnRowsPerWarp;

template <int TOK>
__global__ void __launch_bounds__(256)
down_gemv_kernel(const uint16_t* __restrict__ H, int ldh, int T, int d, int k, int F, int Fs,
                 int group, const int32_t* __restrict__ offsets, const int32_t* __restrict__ sched,
                 const uint8_t* __restrict__ q_r, const __half* __restrict__ s_r,
                 const uint8_t* __restrict__ q_sh, const __half* __restrict__ s_sh,
                 float* __restrict__ Y, int n_route_groups) {
    extern __shared__ uint4 hs[];  // [TOK][Fg / 8]
    const GroupRef g = group_of(blockIdx.y, n_route_groups, T, k, F, Fs, offsets, sched);
    if (g.count == 0) return;
    const int c0 = blockIdx.x * kDnRowsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = g.Fg, k8 = K / 8, nchunk = K / 32, ngr = K / group;
    const uint8_t* qd = g.expert >= 0 ? q_r + (int64_t)g.expert * d * (F / 2) : q_sh;
    const __half* sd = g.expert >= 0 ? s_r + (int64_t)g.expert * d * (F / group) : s_sh;

    for (int i0 = 0; i0 < g.count; i0 += TOK) {
        const int ntok = min(TOK, g.count - i0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < ntok * k8; idx += blockDim.x) {
            const int tt = idx / k8, c8 = idx - tt * k8;
            hs[tt * k8 + c8] =
                __ldg(reinterpret_cast<const uint4*>(H + (g.row0 + i0 + tt) * ldh) + c8);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kDnRowsPerWarp; ++r) {
            const int c = c0 + warp * kDnRowsPerWarp + r;
            const uint4* wq = reinterpret_cast<const uint4*>(qd + (int64_t)c * (K / 2));
            const __half* wsc = sd + (int64_t)c * ngr;
            float acc[TOK];
#pragma unroll
            for (int tt = 0; tt < TOK; ++tt) acc[tt] = 0.f;
            for (int ch = lane; ch < nchunk; ch += 32) {
                const uint4 w = __ldg(wq + ch);
                const float sc = __half2float(wsc[(32 * ch) / group]);
#pragma unroll
                for (int tt = 0; tt < TOK; ++tt)
                    if (tt < ntok) acc[tt] = fmaf(sc, dot32_q4(w, hs + tt * k8 + 4 * ch), acc[tt]);
            }
#pragma unroll
            for (int tt = 0; tt < TOK; ++tt) {
                const float v = warp_sum(acc[tt]);
                if (lane == 0 && tt < ntok) Y[(g.row0 + i0 + tt) * d + c] = v;
            }
        }
    }
}

constexpr int kGemvTok = 4;

}  // namespace

cudaError_t launch_gateup_gemv(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                               const int32_t* perm, const int32_t* sched, moe_w4_t Wgu,
                               moe_w4_t Wgu_s, uint16_t* H, WsHeader* hdr, cudaStream_t st) {
    (void)hdr;
    const int n_route = (int)std::min<int64_t>(d.E, (int64_t)d.T * d.k);
    const int Fmax = std::max(d.F, d.F_s);
    dim3 grid((Fmax + kGuRowsPerCta - 1) / kGuRowsPerCta, n_route + 1);
    const size_t smem = (size_t)kGemvTok * d.d * 2;
    cudaError_t err = ensure_dynamic_smem((const void*)gateup_gemv_kernel<kGemvTok>, smem);
    if (err != cudaSuccess) return err;
    gateup_gemv_kernel<kGemvTok><<<grid, 256, smem, st>>>(
        x, d.T, d.d, d.k, d.F, d.F_s, d.group, offsets, perm, sched, Wgu.q,
        reinterpret_cast<const __half*>(Wgu.s), Wgu_s.q, reinterpret_cast<const __half*>(Wgu_s.s),
        H, Fmax, n_route);
    return cudaGetLastError();
}

cudaError_t launch_down_gemv(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                             WsHeader* hdr, cudaStream_t st) {
    (void)hdr;
    const int n_route = (int)std::min<int64_t>(d.E, (int64_t)d.T * d.k);
    const int Fmax = std::max(d.F, d.F_s);
    dim3 grid(d.d / kDnRowsPerCta, n_route + 1);
    const size_t smem = (size_t)kGemvTok * Fmax * 2;
    cudaError_t err = ensure_dynamic_smem((const void*)down_gemv_kernel<kGemvTok>, smem);
    if (err != cudaSuccess) return err;
    down_gemv_kernel<kGemvTok><<<grid, 256, smem, st>>>(
        H, Fmax, d.T, d.d, d.k, d.F, d.F_s, d.group, offsets, sched, Wd.q,
        reinterpret_cast<const __half*>(Wd.s), Wd_s.q, reinterpret_cast<const __half*>(Wd_s.s), Y,
        n_route);
    return cudaGetLastError();
}

}  // namespace moe
