// Router logits for many tokens on the tcgen05 tensor cores.
//
// The router scores every token against every expert, l = x . W_r[e], with x
// bf16 and W_r fp32 (the layer statement: fp32 router, fp32 accumulation).
// The fp32 weights are split exactly into three bf16 parts, w = hi + mid + lo
// (hi = bf16(w), mid = bf16(w - hi), lo = w - hi - mid; each difference is
// exact in fp32 and the last one fits in bf16), so
//     l = x . hi + x . mid + x . lo
// with every product exact (8 x 8 significant bits) and the sums in fp32 in the
// TMEM accumulator.  That is the fp32 router's definition up to the order of
// the fp32 additions, at the bf16 tensor rate: 3 x 2 x T x E x d flop instead
// of an fp32 SGEMM on the CUDA cores (the pages' prefill computes its router
// projection as a GEMM too).
//
// One CTA per (128 experts, 128 tokens, K slice): the three planes form one K
// loop of 3 d / 64 stages, split over the CTAs of a tile into contiguous
// slices; each CTA writes its fp32 partial logits [slice][T][E], which the
// top-k kernel sums in slice order (deterministic).  Warp 0 issues the TMA
// copies (weight rows and token rows, 128 x 128 B each, 128-byte swizzle),
// warp 1 allocates TMEM and issues four K = 16 MMAs per stage, warps 2-5 read
// the accumulator and store the partials.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tma.cuh"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kRtWarps = 6;
constexpr int kRtThreads = kRtWarps * 32;
constexpr int kRtStages = 6;
constexpr int kRtK = 64;                   // bf16 K elements per stage (128-byte rows)
constexpr int kRtTileBytes = 128 * 128;    // 128 rows x 128 B
constexpr int kRtOffA = 0;
constexpr int kRtOffB = kRtOffA + kRtStages * kRtTileBytes;
constexpr int kRtOffBar = kRtOffB + kRtStages * kRtTileBytes;
// FULL[stages], EMPTY[stages], ACC, TD
constexpr int kRtBarFull = 0, kRtBarEmpty = kRtStages, kRtBarAcc = 2 * kRtStages,
              kRtBarTd = kRtBarAcc + 1, kRtNumBars = kRtBarTd + 1;
constexpr int kRtOffMisc = kRtOffBar + kRtNumBars * 8;
constexpr int kRtSmem = kRtOffMisc + 16 + 1024;
static_assert(kRtSmem <= 227 * 1024, "shared memory budget");

struct RtParams {
    CUtensorMap tm_w;  // weight planes [3E][d] bf16, box {64, 128}
    CUtensorMap tm_x;  // tokens [T][d] bf16, box {64, 128}
    float* logits;     // partials [ks][T][E]
    WsHeader* hdr;
    int T, d, E, ks;
};

__global__ void __launch_bounds__(kRtThreads, 1)
router_tc_kernel(const __grid_constant__ RtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRtOffBar);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kRtOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kRtOffMisc + 4);

    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128, slice = blockIdx.z;
    const int per_plane = p.d / kRtK, total = 3 * per_plane;
    const int q0 = (int)((int64_t)slice * total / p.ks), q1 = (int)((int64_t)(slice + 1) * total / p.ks);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init(bar(kRtBarFull + s), 1);
            mbar_init(bar(kRtBarEmpty + s), 1);
        }
        mbar_init(bar(kRtBarAcc), 1);
        mbar_init(bar(kRtBarTd), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tm_w);
        prefetch_tmap(&p.tm_x);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            for (int q = q0; q < q1; ++q, ++it) {
                const int s = it % kRtStages;
                if (!mbar_wait(bar(kRtBarEmpty + s), ((it / kRtStages) & 1) ^ 1, abort_flag, p.hdr))
                    break;
                const int plane = q / per_plane, kk = (q - plane * per_plane) * kRtK;
                mbar_expect_tx(bar(kRtBarFull + s), 2u * kRtTileBytes);
                tma_load_2d(sbase + kRtOffA + s * kRtTileBytes, &p.tm_w, kk, plane * p.E + m0,
                            bar(kRtBarFull + s));
                tma_load_2d(sbase + kRtOffB + s * kRtTileBytes, &p.tm_x, kk, n0, bar(kRtBarFull + s));
            }
            // no copies in flight at exit (bounded, whatever the abort flag)
            for (uint32_t j = (it >= kRtStages ? it - kRtStages : 0); j < it; ++j)
                mbar_drain(bar(kRtBarFull + j % kRtStages), (j / kRtStages) & 1, p.hdr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, 128);
            uint32_t it = 0;
            bool ok = true;
            for (int q = q0; q < q1; ++q, ++it) {
                const int s = it % kRtStages;
                if (!mbar_wait(bar(kRtBarFull + s), (it / kRtStages) & 1, abort_flag, p.hdr)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = smem_desc_sw128(sbase + kRtOffA + s * kRtTileBytes);
                const uint64_t bd = smem_desc_sw128(sbase + kRtOffB + s * kRtTileBytes);
#pragma unroll
                for (int k = 0; k < kRtK / 16; ++k)  // 32 bytes = 2 address units per K step
                    mma_ss_bf16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                                   (q > q0 || k > 0) ? 1u : 0u);
                mma_commit(bar(kRtBarEmpty + s));
            }
            if (ok) mma_commit(bar(kRtBarAcc));
            mma_commit(bar(kRtBarTd));
            mbar_drain(bar(kRtBarTd), 0, p.hdr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp & 3;
        const int m = qd * 32 + lane;  // expert row = TMEM lane
        if (q1 > q0 && mbar_wait(bar(kRtBarAcc), 0, abort_flag, p.hdr)) {
            tc_fence_after();
            float* out = p.logits + (int64_t)slice * p.T * p.E;
            const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
            for (int c0 = 0; c0 < 128 && n0 + c0 < p.T; c0 += 32) {
                uint32_t v[32];
                tmem_ld_x32(tmem + lane_base + (uint32_t)c0, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = n0 + c0 + j;
                    if (n < p.T && m0 + m < p.E) out[(int64_t)n * p.E + m0 + m] = __uint_as_float(v[j]);
                }
            }
        } else if (q1 <= q0) {
            // an empty slice still owns its partials: zeros
            float* out = p.logits + (int64_t)slice * p.T * p.E;
            for (int n = n0; n < min(n0 + 128, p.T); ++n) out[(int64_t)n * p.E + m0 + m] = 0.f;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128)
                     : "memory");
    }
}

// W_r fp32 [E][d] -> three bf16 planes [3][E][d] with w = hi + mid + lo exactly.
__global__ void __launch_bounds__(256) split_router_kernel(const float4* __restrict__ w,
                                                           int64_t n4, uint2* __restrict__ planes) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = __ldg(w + i);
        const float a[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4], mi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(a[j]);
            const float r1 = a[j] - __bfloat162float(hb);  // exact
            const __nv_bfloat16 mb = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mb);    // exact, fits in bf16
            const __nv_bfloat16 lb = __float2bfloat16_rn(r2);
            h[j] = *reinterpret_cast<const uint16_t*>(&hb);
            mi[j] = *reinterpret_cast<const uint16_t*>(&mb);
            lo[j] = *reinterpret_cast<const uint16_t*>(&lb);
        }
        planes[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        planes[n4 + i] = make_uint2(mi[0] | (mi[1] << 16), mi[2] | (mi[3] << 16));
        planes[2 * n4 + i] = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
}

bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kRtK, 128};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 2, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool router_tc_supported(const moe_dims_t& d) {
    return d.T > kRouterSmallT && d.E % 128 == 0 && d.d % kRtK == 0;
}

// K slices per (128 x 128) tile.  The tensor core's accumulation keeps fewer
// bits than an fp32 FMA chain, and its error grows with the number of MMAs one
// accumulator takes; the slices' partials are summed in fp32 by the top-k
// kernel.  So at least 4 slices (48 stages of K = 64 each at d = 4096: the
// combine weights then stay within 2e-6 of the fp64 router at T = 2048), up to
// 8 while the grid stays at or under 320 CTAs.
int router_tc_ksplit(const moe_dims_t& d) {
    const int64_t tiles = (int64_t)(d.E / 128) * ((d.T + 127) / 128);
    int ks = 4;
    while (ks < 8 && tiles * ks * 2 <= 320) ks *= 2;
    return ks;
}

cudaError_t launch_router_logits_tc(const uint16_t* x, const float* W_r, const moe_dims_t& d,
                                    uint16_t* planes, float* logits, int ks, WsHeader* hdr,
                                    cudaStream_t st) {
    const int64_t n4 = (int64_t)d.E * d.d / 4;
    split_router_kernel<<<(unsigned)std::min<int64_t>((n4 + 255) / 256, 1184), 256, 0, st>>>(
        reinterpret_cast<const float4*>(W_r), n4, reinterpret_cast<uint2*>(planes));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    RtParams prm;
    memset(&prm, 0, sizeof(prm));
    if (!make_bf16_map(&prm.tm_w, planes, d.d, 3ull * d.E) ||
        !make_bf16_map(&prm.tm_x, x, d.d, (uint64_t)d.T))
        return cudaErrorInvalidValue;
    prm.logits = logits;
    prm.hdr = hdr;
    prm.T = d.T; prm.d = d.d; prm.E = d.E; prm.ks = ks;
    if ((err = ensure_dynamic_smem((const void*)router_tc_kernel, kRtSmem)) != cudaSuccess) return err;
    dim3 grid(d.E / 128, (d.T + 127) / 128, ks);
    router_tc_kernel<<<grid, kRtThreads, kRtSmem, st>>>(prm);
    return cudaGetLastError();
}

}  // namespace moe
