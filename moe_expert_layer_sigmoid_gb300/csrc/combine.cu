// Weighted combine of the routed expert rows plus the shared expert row, and
// optionally a residual row.
//
// Deterministic: each output element sums its k routed rows in selection
// order j = 0..k-1 and then adds the shared row, in fp32, with a fixed order
// that does not depend on scheduling (the deterministic scatter-add and the
// residual + routed + shared add of thewafflehaus/FFAI PR #72, Nemotron
// commits "ffai_add3" and W4A16 Marlin MoE, keep a fixed summation order for
// the same reason).  The residual, when given, is added last, to the finished
// routed + shared sum, before the one bf16 rounding (the "ffai_add3" order).
// `out` may be the residual buffer itself: each thread reads its residual
// elements before it writes the same elements of out.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ Y, const float* __restrict__ topk_w,
               const int32_t* __restrict__ pos, int T, int d, int k, const uint16_t* residual,
               uint16_t* out) {
    const int t = blockIdx.y;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const float w = __ldg(topk_w + (int64_t)t * k + j);
        const int64_t r = __ldg(pos + (int64_t)t * k + j);
        const float4 y = __ldg(reinterpret_cast<const float4*>(Y + r * d + c));
        acc.x = fmaf(w, y.x, acc.x);
        acc.y = fmaf(w, y.y, acc.y);
        acc.z = fmaf(w, y.z, acc.z);
        acc.w = fmaf(w, y.w, acc.w);
    }
    const float4 ys = __ldg(reinterpret_cast<const float4*>(Y + ((int64_t)T * k + t) * d + c));
    acc.x += ys.x;
    acc.y += ys.y;
    acc.z += ys.z;
    acc.w += ys.w;
    if (residual) {
        const uint2 r = *reinterpret_cast<const uint2*>(residual + (int64_t)t * d + c);
        acc.x = bf16_lo(r.x) + acc.x;
        acc.y = bf16_hi(r.x) + acc.y;
        acc.z = bf16_lo(r.y) + acc.z;
        acc.w = bf16_hi(r.y) + acc.w;
    }
    uint2 o;
    o.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
    o.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
    *reinterpret_cast<uint2*>(out + (int64_t)t * d + c) = o;
}

}  // namespace

cudaError_t launch_combine(const float* Y, const float* topk_w, const int32_t* pos,
                           const moe_dims_t& d, const uint16_t* residual, uint16_t* out,
                           cudaStream_t st) {
    const int threads = 256;
    dim3 grid((d.d / 4 + threads - 1) / threads, d.T);
    combine_kernel<<<grid, threads, 0, st>>>(Y, topk_w, pos, d.T, d.d, d.k, residual, out);
    return cudaGetLastError();
}

}  // namespace moe
