// Decode-side expert projections: int4 GEMV on CUDA cores.
//
// The Laguna decode path runs the MoE gate+up projection fused (SwiGLU) and the
// shared expert through the same gathered kernel (thewafflehaus/butter PR #69,
// commit "feat(laguna): Laguna-S-2.1 decode on the CUDA engine").  Here both
// projections are persistent kernels with one CTA per SM:
//
//   gate+up  work item = one gate row and its up row of one group (a routed
//            expert in schedule order, or the shared expert) against every
//            token of the group; each CTA takes an equal contiguous share of
//            the items, the shared expert's before the routed experts'.  The
//            shared expert depends on x alone, so it runs before the kernel
//            waits for the router (programmatic dependent launch).
//   down     each CTA owns a contiguous range of output channels for every
//            group; work item = four channels of one group.  With the combine
//            fused in, the CTA then sums its channels' routed rows and shared
//            row in the fixed order of moe_combine_shared.
//
// Loads.  Each lane reads 16 bytes (32 nibbles, one quantisation-group scale)
// per load, the 32 lanes of a warp a contiguous 512 bytes, straight into
// registers; every warp loads its next item while it computes the current one
// (two register buffers), so each SM keeps about 64 KB of reads in flight.
// Streaming from HBM this way measured ~6.2 TB/s on GB300, against ~4 TB/s
// for the same bytes moved by cp.async.bulk in 8-16 KB pieces.  For T = 1 the
// token's x (and its 32-element chunk sums) sit in shared memory,
// lane-interleaved so a warp's 16-byte reads are conflict-free.
//
// Launch order (programmatic dependent launch): the gate+up kernel requests
// its shared-expert stages and loads x before it waits for the router, and
// lets the down kernel launch once the routing is complete; the down kernel
// requests its first two items' weights before it waits for H.
//
// Arithmetic.  Decode streams about two int4 weights per HBM byte, so the
// kernel has only a few lane-operations per weight.  One lop3 turns bits 0-3
// and 16-19 of a word into the bf16 pair {136 + q, 136 + q'} exactly (mantissa
// field of 128.0 = 0x4300, nibble xor 8 = q + 8), so a 32-bit word of eight
// nibbles costs three shifts and four lop3; the products use the mixed
// fma.rn.f32.bf16 (bf16 x bf16 + fp32), exact products with fp32 accumulation.
//   T = 1:  the offset is taken out per 32-element chunk, sum x * q =
//           sum x * (136 + q) - 136 * sum x, with the chunk sums of x kept in
//           registers beside x itself.
//   T > 1:  each pair is first made exact q by one fma.rn.bf16x2 (t - 136),
//           then reused for every token of the pass.
// Each chunk's fp32 partial is multiplied by its fp16 scale and accumulated,
// so the result is sum x * (q * s) with fp32 summation rounding only.
#include "common.cuh"

namespace moe {
namespace {

// Warps per gate+up CTA: 16 for one token (112 registers, 57K of the 64K
// register file), 12 for several (160 registers: the multi-token passes keep
// more values live).  At T = 1 the 16-warp CTA cannot sit beside the decode
// router's last CTA, so the one on that SM starts when the router ends; the
// extra loads in flight on every other SM outweigh that (measured 17.2 against
// 18.4 us for the launch, 35.8 against 37.0 us for the step).  Down: 16 warps.
__host__ __device__ constexpr int gu_warps(bool one) { return one ? 16 : 12; }
constexpr int kDnWarps = 16;
constexpr int kDnThreads = kDnWarps * 32;
constexpr int kGuTokPass = 4;  // tokens per pass of the gate+up kernel (T > 1)
constexpr int kDnTokPass = 2;  // tokens per pass of the down kernel (T > 1)
constexpr int kDnQuad = 4;     // output channels per down work item

// 16-byte load of streamed weights: read once, so no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// bits 0-3 and 16-19 of v -> bf16 pair {136 + q_lo, 136 + q_hi}
__device__ __forceinline__ uint32_t nib_pair(uint32_t v) {
    uint32_t t;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(t) : "r"(v), "r"(0x000F000Fu), "r"(0x43084308u));
    return t;
}

// exact q pair: t * 1 - 136 in bf16x2 (both values are small integers)
__device__ __forceinline__ uint32_t q_pair(uint32_t v) {
    uint32_t q;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(nib_pair(v)), "r"(0x3F803F80u), "r"(0xC308C308u));
    return q;
}

// acc += lo(p) * half_S(xa) + hi(p) * half_S(xb), S = 0 low halves, 1 high.
template <int S>
__device__ __forceinline__ float fma_pair(float acc, uint32_t p, uint32_t xa, uint32_t xb) {
    if (S == 0)
        asm("{\n .reg .b16 pl, ph, al, ah, bl, bh;\n mov.b32 {pl, ph}, %1;\n mov.b32 {al, ah}, %2;\n"
            " mov.b32 {bl, bh}, %3;\n fma.rn.f32.bf16 %0, pl, al, %0;\n fma.rn.f32.bf16 %0, ph, bl, %0;\n}"
            : "+f"(acc)
            : "r"(p), "r"(xa), "r"(xb));
    else
        asm("{\n .reg .b16 pl, ph, al, ah, bl, bh;\n mov.b32 {pl, ph}, %1;\n mov.b32 {al, ah}, %2;\n"
            " mov.b32 {bl, bh}, %3;\n fma.rn.f32.bf16 %0, pl, ah, %0;\n fma.rn.f32.bf16 %0, ph, bh, %0;\n}"
            : "+f"(acc)
            : "r"(p), "r"(xa), "r"(xb));
    return acc;
}

// Eight nibbles of w (element 2j in the low nibble of byte j) against the
// eight bf16 activations xv.  Element pairs are (j, j + 4): word w >> 4j gives
// element j in bits 0-3 and element j + 4 in bits 16-19.  Four accumulators
// (one per j) keep four independent FMA chains.
// Offset form: acc[j] += x * (136 + q).
__device__ __forceinline__ void dot8_off(uint32_t w, uint4 xv, float* acc) {
    acc[0] = fma_pair<0>(acc[0], nib_pair(w), xv.x, xv.z);
    acc[1] = fma_pair<1>(acc[1], nib_pair(w >> 4), xv.x, xv.z);
    acc[2] = fma_pair<0>(acc[2], nib_pair(w >> 8), xv.y, xv.w);
    acc[3] = fma_pair<1>(acc[3], nib_pair(w >> 12), xv.y, xv.w);
}

// Exact form on pre-made q pairs qp[0..3] of one word.
__device__ __forceinline__ void dot8_q(const uint32_t* qp, uint4 xv, float* acc) {
    acc[0] = fma_pair<0>(acc[0], qp[0], xv.x, xv.z);
    acc[1] = fma_pair<1>(acc[1], qp[1], xv.x, xv.z);
    acc[2] = fma_pair<0>(acc[2], qp[2], xv.y, xv.w);
    acc[3] = fma_pair<1>(acc[3], qp[3], xv.y, xv.w);
}

__device__ __forceinline__ void q_pairs32(uint4 w, uint32_t* qp) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        qp[4 * i + 0] = q_pair(ws[i]);
        qp[4 * i + 1] = q_pair(ws[i] >> 4);
        qp[4 * i + 2] = q_pair(ws[i] >> 8);
        qp[4 * i + 3] = q_pair(ws[i] >> 12);
    }
}

__device__ __forceinline__ float sum4(const float* a) { return (a[0] + a[1]) + (a[2] + a[3]); }

// sum over a 32-element chunk of x * (136 + q)
__device__ __forceinline__ float dot32_off(uint4 w, const uint4* xv) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    dot8_off(w.x, xv[0], acc);
    dot8_off(w.y, xv[1], acc);
    dot8_off(w.z, xv[2], acc);
    dot8_off(w.w, xv[3], acc);
    return sum4(acc);
}

// sum over a 32-element chunk of x * q
__device__ __forceinline__ float dot32_q(const uint32_t* qp, const uint4* xv) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    dot8_q(qp, xv[0], acc);
    dot8_q(qp + 4, xv[1], acc);
    dot8_q(qp + 8, xv[2], acc);
    dot8_q(qp + 12, xv[3], acc);
    return sum4(acc);
}

__device__ __forceinline__ float sum32_bf16(const uint4* xv) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t p[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) s += bf16_lo(p[j]) + bf16_hi(p[j]);
    }
    return s;
}

// Sums of four per-lane values over the warp, transposed: lane L ends with the
// total of value ((L >> 4) & 1) * 2 + ((L >> 3) & 1), in 7 shuffles.
__device__ __forceinline__ float reduce4(float v0, float v1, float v2, float v3, int lane) {
    const bool h16 = lane & 16, h8 = lane & 8;
    const float a = (h16 ? v0 : v2) + 0.f, b = (h16 ? v1 : v3) + 0.f;
    const float w0 = (h16 ? v2 : v0) + __shfl_xor_sync(0xffffffffu, a, 16);
    const float w1 = (h16 ? v3 : v1) + __shfl_xor_sync(0xffffffffu, b, 16);
    float z = (h8 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, h8 ? w0 : w1, 8);
    z += __shfl_xor_sync(0xffffffffu, z, 4);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    return z;
}

__device__ __forceinline__ void load_chunk(const uint16_t* row, int c, uint4* xv) {
    const uint4* p = reinterpret_cast<const uint4*>(row) + 4 * c;
#pragma unroll
    for (int v = 0; v < 4; ++v) xv[v] = __ldg(p + v);
}

__device__ __forceinline__ float swiglu(float g, float u) { return swiglu_f32(g, u); }

// ---------------------------------------------------------------------------
constexpr size_t kMaxStagedH = 64 * 1024;  // H rows staged by the down kernel, at most

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const __half* p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float half_lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// Rows [row0, row0 + count) of H / Y belong to a group: a routed expert's rows
// (offsets) or the shared expert's (after the T*k routed rows).
__device__ __forceinline__ void group_rows(const int32_t* offsets, int T, int k, int expert,
                                           int* row0, int* count) {
    if (expert >= 0) {
        *row0 = offsets[expert];
        *count = offsets[expert + 1] - *row0;
    } else {
        *row0 = T * k;
        *count = T;
    }
}

// Routed groups with rows, counted by one warp (no block barrier), or read
// from the header.
__device__ __forceinline__ int warp_active_groups(const int32_t* n_active, const int32_t* offsets,
                                                  const int32_t* sched, int n_route_max, int lane) {
    if (n_active) return *n_active;
    int n = 0;
    for (int y0 = 0; y0 < n_route_max; y0 += 32) {
        const int y = y0 + lane;
        bool act = false;
        if (y < n_route_max) {
            const int e = sched[y];
            act = offsets[e + 1] > offsets[e];
        }
        n += __popc(__ballot_sync(0xffffffffu, act));
    }
    return n;
}

// x of a single token in shared memory, lane-interleaved: 16-byte sub-vector
// v of chunk lane + 32 i at slot (4 i + v) * 32 + lane; chunk sums after it.
template <int CPL>
__device__ __forceinline__ void stage_x(const uint16_t* x, int d, uint4* xs, float* xsum) {
    const int nc = d >> 5;
    for (int i = threadIdx.x; i < 32 * CPL; i += blockDim.x) {
        const int ln = i & 31, ci = i >> 5, c = ln + 32 * ci;
        uint4 xv[4];
        if (c < nc) {
            load_chunk(x, c, xv);
            xsum[i] = sum32_bf16(xv);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) xv[v] = make_uint4(0, 0, 0, 0);
            xsum[i] = 0.f;
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) xs[(4 * ci + v) * 32 + ln] = xv[v];
    }
}

// Sum over the warp of g (lanes 0-15 after the first step) and u (16-31);
// lane 0 ends with the gate total, lane 16 with the up total.
__device__ __forceinline__ float reduce2(float g, float u, int lane) {
    const bool hi = lane & 16;
    float z = (hi ? u : g) + __shfl_xor_sync(0xffffffffu, hi ? g : u, 16);
    z += __shfl_xor_sync(0xffffffffu, z, 8);
    z += __shfl_xor_sync(0xffffffffu, z, 4);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    return z;
}

// ---------------------------------------------------------------------------
// Gate+up.
struct GuArgs {
    const uint16_t* x;
    int T, d, k, F, Fs, gsh;  // chunk c (32 elements) uses scale index c >> gsh
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* sched;
    const uint8_t* q_r;
    const __half* s_r;
    const uint8_t* q_sh;
    const __half* s_sh;
    uint16_t* H;
    int ldh;
    int n_route_max;
    const int32_t* n_active;
    WsHeader* hdr;
};

// One item in registers: the lane's words of a gate row and its up row (row
// pair f of `expert`, -1 for the shared expert) and their scales.
template <int CPL>
struct GuBuf {
    uint4 g[CPL], u[CPL];
    uint32_t sc[CPL];  // gate scale bits | up scale bits << 16
    int expert, f;
};

template <int CPL>
__device__ __forceinline__ void gu_load(const GuArgs& a, int expert, int f, int lane,
                                        GuBuf<CPL>& B) {
    const int nc = a.d >> 5, ngr = nc >> a.gsh;
    const int Fg = expert >= 0 ? a.F : a.Fs;
    const int64_t rowb = a.d / 2;
    const uint8_t* qb = expert >= 0 ? a.q_r + (int64_t)expert * 2 * a.F * rowb : a.q_sh;
    const __half* sb = expert >= 0 ? a.s_r + (int64_t)expert * 2 * a.F * ngr : a.s_sh;
    const uint4* gq = reinterpret_cast<const uint4*>(qb + (int64_t)f * rowb);
    const uint4* uq = reinterpret_cast<const uint4*>(qb + (int64_t)(Fg + f) * rowb);
    const __half* gs = sb + (int64_t)f * ngr;
    const __half* us = sb + (int64_t)(Fg + f) * ngr;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) {
            B.g[i] = ld_stream(gq + c);
            B.u[i] = ld_stream(uq + c);
            B.sc[i] = ldg_u16(gs + (c >> a.gsh)) | (ldg_u16(us + (c >> a.gsh)) << 16);
        }
    }
    B.expert = expert;
    B.f = f;
}

// Compute one loaded item and write SwiGLU(gate, up) to H.  ONE: T == 1, x
// and its chunk sums in shared memory at xs / xsum.
template <int CPL, bool ONE>
__device__ __forceinline__ void gu_compute(const GuArgs& a, const GuBuf<CPL>& B, uint32_t xs,
                                           const float* xsum, int lane) {
    const int nc = a.d >> 5;
    int row0, count;
    group_rows(a.offsets, a.T, a.k, B.expert, &row0, &count);
    if constexpr (ONE) {
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < nc) {
                uint4 xv[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) xv[v] = lds128(xs + 16u * (uint32_t)((4 * i + v) * 32 + lane));
                const float xsm = xsum[32 * i + lane];
                g = fmaf(half_lo(B.sc[i]), fmaf(-136.f, xsm, dot32_off(B.g[i], xv)), g);
                u = fmaf(half_hi(B.sc[i]), fmaf(-136.f, xsm, dot32_off(B.u[i], xv)), u);
            }
        }
        const float z = reduce2(g, u, lane);
        const float zu = __shfl_down_sync(0xffffffffu, z, 16);
        if (lane == 0 && count > 0)
            a.H[(int64_t)row0 * a.ldh + B.f] = float_to_bf16_bits(swiglu(z, zu));
    } else {
        for (int i0 = 0; i0 < count; i0 += kGuTokPass) {
            const int ntok = min(kGuTokPass, count - i0);
            const uint16_t* xrow[kGuTokPass];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                const int r = row0 + i0 + min(tt, ntok - 1);
                const int tok = B.expert >= 0 ? a.perm[r] / a.k : r - row0;
                xrow[tt] = a.x + (int64_t)tok * a.d;
            }
            float g[kGuTokPass], u[kGuTokPass];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) g[tt] = u[tt] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = lane + 32 * i;
                if (c >= nc) continue;
                uint32_t qg[16], qu[16];
                q_pairs32(B.g[i], qg);
                q_pairs32(B.u[i], qu);
#pragma unroll
                for (int tt = 0; tt < kGuTokPass; ++tt) {
                    if (tt < ntok) {
                        uint4 xv[4];
                        load_chunk(xrow[tt], c, xv);
                        g[tt] = fmaf(half_lo(B.sc[i]), dot32_q(qg, xv), g[tt]);
                        u[tt] = fmaf(half_hi(B.sc[i]), dot32_q(qu, xv), u[tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                if (tt < ntok) {
                    const float z = reduce2(g[tt], u[tt], lane);
                    const float zu = __shfl_down_sync(0xffffffffu, z, 16);
                    if (lane == 0)
                        a.H[(int64_t)(row0 + i0 + tt) * a.ldh + B.f] = float_to_bf16_bits(swiglu(z, zu));
                }
            }
        }
    }
}

// Items of one warp, two register buffers: item u + 1 is loaded before item u
// is computed.  item(u, e, f) gives the items in load order.
template <int CPL, bool ONE, typename ItemFn>
__device__ __forceinline__ void gu_pipeline(const GuArgs& a, int n, ItemFn item, uint32_t xs,
                                            const float* xsum, int lane) {
    GuBuf<CPL> A, B;
    int e, f;
    if (n > 0) {
        item(0, &e, &f);
        gu_load<CPL>(a, e, f, lane, A);
    }
    for (int u = 0; u < n; u += 2) {
        if (u + 1 < n) {
            item(u + 1, &e, &f);
            gu_load<CPL>(a, e, f, lane, B);
        }
        gu_compute<CPL, ONE>(a, A, xs, xsum, lane);
        if (u + 2 < n) {
            item(u + 2, &e, &f);
            gu_load<CPL>(a, e, f, lane, A);
        }
        if (u + 1 < n) gu_compute<CPL, ONE>(a, B, xs, xsum, lane);
    }
}

// Persistent: CTA b takes an equal contiguous share of the shared expert's row
// pairs, then (after the router) of the routed row pairs (group y, row f) =
// y * F + f; warp w takes the items w, w + 12, ... of each share.
template <int CPL, bool ONE>
__global__ void __maxnreg__(ONE ? 112 : 160) gateup_gemv_kernel(const GuArgs a) {
    extern __shared__ __align__(16) uint4 gu_xs[];  // ONE: x, lane-interleaved
    __shared__ float s_xsum[32 * CPL];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    if (ONE) {  // x is an input of the layer
        stage_x<CPL>(a.x, a.d, gu_xs, s_xsum);
        __syncthreads();
    }
    const uint32_t xs = ONE ? (uint32_t)__cvta_generic_to_shared(gu_xs) : 0u;
    {   // the shared expert reads only x: it runs before the wait for the router
        const int lo = (int)((int64_t)b * a.Fs / G), hi = (int)((int64_t)(b + 1) * a.Fs / G);
        const int first = lo + warp;
        constexpr int kGuWarps = gu_warps(ONE);
        const int n = first < hi ? (hi - first + kGuWarps - 1) / kGuWarps : 0;
        gu_pipeline<CPL, ONE>(
            a, n,
            [&](int u, int* e, int* f) {
                *e = -1;
                *f = first + u * kGuWarps;
            },
            xs, s_xsum, lane);
    }
    pdl_wait();
    pdl_trigger();  // dependents launch once the routing is complete and may read it early
    const int n_act = warp_active_groups(a.n_active, a.offsets, a.sched, a.n_route_max, lane);
    const int64_t R = (int64_t)n_act * a.F;
    const int64_t lo = (int64_t)b * R / G, hi = (int64_t)(b + 1) * R / G;
    const int64_t first = lo + warp;
    constexpr int kGuWarps = gu_warps(ONE);
    const int n = first < hi ? (int)((hi - first + kGuWarps - 1) / kGuWarps) : 0;
    // cursor (group, row) in load order
    int cy = n ? (int)(first / a.F) : 0;
    int cf = n ? (int)(first - (int64_t)cy * a.F) : 0;
    gu_pipeline<CPL, ONE>(
        a, n,
        [&](int, int* e, int* f) {
            *e = a.sched[cy];
            *f = cf;
            cf += kGuWarps;
            while (cf >= a.F) {
                cf -= a.F;
                ++cy;
            }
        },
        xs, s_xsum, lane);
}

// ---------------------------------------------------------------------------
// Down projection.
struct DnArgs {
    const uint16_t* H;
    int ldh;
    int T, d, k, F, Fs, gsh;
    const int32_t* offsets;
    const int32_t* sched;
    const uint8_t* q_r;
    const __half* s_r;
    const uint8_t* q_sh;
    const __half* s_sh;
    float* Y;
    int n_route_max;
    const int32_t* n_active;
    const float* topk_w;  // fused combine when out is non-null
    const int32_t* pos;
    const uint16_t* residual;  // added after routed + shared when non-null; may alias out
    uint16_t* out;
    WsHeader* hdr;
};

// One item in registers: the lane's words of output channels c0 .. c0 + 3 of
// `expert` (-1: shared) and their scales.
template <int CPL>
struct DnBuf {
    uint4 w[kDnQuad][CPL];
    uint32_t sc[kDnQuad / 2][CPL];  // channel 2j scale bits | channel 2j + 1 << 16
    int expert, c0;
};

template <int CPL>
__device__ __forceinline__ void dn_load(const DnArgs& a, int expert, int c0, int lane,
                                        DnBuf<CPL>& B) {
    const int K = expert >= 0 ? a.F : a.Fs;
    const int nc = K >> 5, ngr = nc >> a.gsh;
    const int64_t rowb = K / 2;
    const uint8_t* qb = (expert >= 0 ? a.q_r + (int64_t)expert * a.d * rowb : a.q_sh) + (int64_t)c0 * rowb;
    const __half* sb = (expert >= 0 ? a.s_r + (int64_t)expert * a.d * ngr : a.s_sh) + (int64_t)c0 * ngr;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) {
#pragma unroll
            for (int ch = 0; ch < kDnQuad; ++ch)
                B.w[ch][i] = ld_stream(reinterpret_cast<const uint4*>(qb + ch * rowb) + c);
#pragma unroll
            for (int j = 0; j < kDnQuad / 2; ++j)
                B.sc[j][i] = ldg_u16(sb + (2 * j) * ngr + (c >> a.gsh)) |
                             (ldg_u16(sb + (2 * j + 1) * ngr + (c >> a.gsh)) << 16);
        }
    }
    B.expert = expert;
    B.c0 = c0;
}

// Compute one loaded item and write Y.  hs (ONE only): shared-memory address
// of the staged H rows (0: read H from global memory); hsum: their 32-element
// chunk sums, [row][ldh / 32] fp32.
template <int CPL, bool ONE>
__device__ __forceinline__ void dn_compute(const DnArgs& a, const DnBuf<CPL>& B, uint32_t hs,
                                           uint32_t hsum, int lane) {
    const int K = B.expert >= 0 ? a.F : a.Fs;
    const int nc = K >> 5;
    int row0, count;
    group_rows(a.offsets, a.T, a.k, B.expert, &row0, &count);
    constexpr int TP = ONE ? 1 : kDnTokPass;
    for (int i0 = 0; i0 < count; i0 += TP) {
        const int ntok = min(TP, count - i0);
        float acc[TP][kDnQuad];
#pragma unroll
        for (int tt = 0; tt < TP; ++tt)
#pragma unroll
            for (int ch = 0; ch < kDnQuad; ++ch) acc[tt][ch] = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c >= nc) continue;
            float sc[kDnQuad];
#pragma unroll
            for (int j = 0; j < kDnQuad / 2; ++j) {
                sc[2 * j] = half_lo(B.sc[j][i]);
                sc[2 * j + 1] = half_hi(B.sc[j][i]);
            }
            if constexpr (ONE) {
                uint4 hv[4];
                float hsm;
                if (hs) {
                    const uint32_t h = hs + (uint32_t)(row0 * a.ldh + 32 * c) * 2u;
#pragma unroll
                    for (int v = 0; v < 4; ++v) hv[v] = lds128(h + 16u * v);
                    hsm = lds_f32(hsum + 4u * (uint32_t)(row0 * (a.ldh >> 5) + c));
                } else {
                    load_chunk(a.H + (int64_t)row0 * a.ldh, c, hv);
                    hsm = sum32_bf16(hv);
                }
#pragma unroll
                for (int ch = 0; ch < kDnQuad; ++ch)
                    acc[0][ch] = fmaf(sc[ch], fmaf(-136.f, hsm, dot32_off(B.w[ch][i], hv)), acc[0][ch]);
            } else {
                uint4 hv[TP][4];
#pragma unroll
                for (int tt = 0; tt < TP; ++tt)
                    load_chunk(a.H + (int64_t)(row0 + i0 + min(tt, ntok - 1)) * a.ldh, c, hv[tt]);
#pragma unroll
                for (int ch = 0; ch < kDnQuad; ++ch) {
                    uint32_t qp[16];
                    q_pairs32(B.w[ch][i], qp);
#pragma unroll
                    for (int tt = 0; tt < TP; ++tt) acc[tt][ch] = fmaf(sc[ch], dot32_q(qp, hv[tt]), acc[tt][ch]);
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < TP; ++tt) {
            if (tt < ntok) {
                // lanes 0 / 8 / 16 / 24 hold channels c0 .. c0 + 3
                const float z = reduce4(acc[tt][0], acc[tt][1], acc[tt][2], acc[tt][3], lane);
                if ((lane & 7) == 0) a.Y[(int64_t)(row0 + i0 + tt) * a.d + B.c0 + (lane >> 3)] = z;
            }
        }
    }
}

// Output-channel share of CTA b: quads [q_lo, q_hi) of d / 4.
__device__ __forceinline__ void dn_share(int d, int* q_lo, int* q_hi) {
    const int nq = d / kDnQuad, G = gridDim.x, b = blockIdx.x;
    *q_lo = (int)((int64_t)b * nq / G);
    *q_hi = (int)((int64_t)(b + 1) * nq / G);
}

// Fused combine over this CTA's channels: routed rows in selection order, then
// the shared row (the order of moe_combine_shared).  Y was written by this
// CTA, so it is read with plain loads after the barrier.
__device__ __forceinline__ void dn_combine(const DnArgs& a, int q_lo, int nqc) {
    __syncthreads();
    const int T = a.T, k = a.k, d = a.d;
    for (int idx = threadIdx.x; idx < T * nqc; idx += blockDim.x) {
        const int t = idx / nqc;
        const int c = kDnQuad * (q_lo + (idx - t * nqc));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float w = __ldg(a.topk_w + (int64_t)t * k + j);
            const int64_t r = __ldg(a.pos + (int64_t)t * k + j);
            const float4 y = *reinterpret_cast<const float4*>(a.Y + r * d + c);
            acc.x = fmaf(w, y.x, acc.x);
            acc.y = fmaf(w, y.y, acc.y);
            acc.z = fmaf(w, y.z, acc.z);
            acc.w = fmaf(w, y.w, acc.w);
        }
        const float4 ys = *reinterpret_cast<const float4*>(a.Y + ((int64_t)T * k + t) * d + c);
        acc.x += ys.x;
        acc.y += ys.y;
        acc.z += ys.z;
        acc.w += ys.w;
        if (a.residual) {
            const uint2 r = *reinterpret_cast<const uint2*>(a.residual + (int64_t)t * d + c);
            acc.x = bf16_lo(r.x) + acc.x;
            acc.y = bf16_hi(r.x) + acc.y;
            acc.z = bf16_lo(r.y) + acc.z;
            acc.w = bf16_hi(r.y) + acc.w;
        }
        uint2 o;
        o.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
        o.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
        *reinterpret_cast<uint2*>(a.out + (int64_t)t * d + c) = o;
    }
}

// Persistent: CTA b owns output-channel quads [q_lo, q_hi) of every group;
// its items are (group y, quad) group-major, group 0 being the shared expert
// and group y > 0 the routed expert sched[y - 1]; warp w takes items w,
// w + 16, ...  The routing is complete at launch (the gate+up kernel lets this
// kernel launch only after its own wait for the router), so the first two
// items' weights are requested before the wait for H.  For T == 1 the token's H rows (k
// routed + 1 shared) and their chunk sums are staged in shared memory.
template <int CPL, bool ONE>
__global__ void __launch_bounds__(kDnThreads, 1) down_gemv_kernel(const DnArgs a, int h_rows) {
    extern __shared__ __align__(16) uint4 dn_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int q_lo, q_hi;
    dn_share(a.d, &q_lo, &q_hi);
    const int nqc = q_hi - q_lo;
    pdl_trigger();
    const int n_act = warp_active_groups(a.n_active, a.offsets, a.sched, a.n_route_max, lane);
    const int items = (1 + n_act) * nqc;
    const int n = warp < items ? (items - warp + kDnWarps - 1) / kDnWarps : 0;
    int cy = n ? warp / nqc : 0, cq = n ? warp - (warp / nqc) * nqc : 0;  // cursor, load order
    auto next = [&](int* e, int* c0) {
        *e = cy == 0 ? -1 : a.sched[cy - 1];
        *c0 = kDnQuad * (q_lo + cq);
        cq += kDnWarps;
        while (cq >= nqc) {
            cq -= nqc;
            ++cy;
        }
    };
    DnBuf<CPL> A, B;
    int e, c0;
    if (n > 0) {  // the first two items' weights do not depend on H
        next(&e, &c0);
        dn_load<CPL>(a, e, c0, lane, A);
    }
    if (n > 1) {
        next(&e, &c0);
        dn_load<CPL>(a, e, c0, lane, B);
    }
    pdl_wait();  // H is written by the gate+up kernel
    uint32_t hs = 0, hsum = 0;
    if (h_rows) {
        const uint32_t h_bytes = (uint32_t)h_rows * a.ldh * 2u;
        const uint4* src = reinterpret_cast<const uint4*>(a.H);
        for (uint32_t i = threadIdx.x; i < h_bytes / 16; i += kDnThreads) dn_smem[i] = __ldg(src + i);
        __syncthreads();
        const int ncr = a.ldh >> 5;  // chunks per row
        float* sums = reinterpret_cast<float*>(dn_smem + h_bytes / 16);
        for (int i = threadIdx.x; i < h_rows * ncr; i += kDnThreads) sums[i] = sum32_bf16(dn_smem + 4 * i);
        __syncthreads();
        hs = (uint32_t)__cvta_generic_to_shared(dn_smem);
        hsum = (uint32_t)__cvta_generic_to_shared(sums);
    }
    for (int u = 0; u < n; u += 2) {
        dn_compute<CPL, ONE>(a, A, hs, hsum, lane);
        if (u + 2 < n) {
            next(&e, &c0);
            dn_load<CPL>(a, e, c0, lane, A);
        }
        if (u + 1 < n) {
            dn_compute<CPL, ONE>(a, B, hs, hsum, lane);
            if (u + 3 < n) {
                next(&e, &c0);
                dn_load<CPL>(a, e, c0, lane, B);
            }
        }
    }
    if (a.out) dn_combine(a, q_lo, nqc);
}

// ---------------------------------------------------------------------------
int log2_group_chunks(int group) { return group == 32 ? 0 : group == 64 ? 1 : 2; }

// 16-byte loads per lane and row: one pass covers K <= 1024 * CPL.
int chunks_per_lane(int K) {
    const int c = (K / 32 + 31) / 32;
    return c <= 1 ? 1 : c <= 2 ? 2 : 4;
}

// Shared memory of the staged H rows and their chunk sums (down kernel, T == 1).
size_t staged_h_bytes(int rows, int ldh) {
    return (size_t)rows * ldh * 2 + (size_t)rows * (ldh / 32) * 4;
}

template <typename Kern, typename... Args>
cudaError_t launch_persistent(Kern kern, int threads, size_t smem, bool pdl, cudaStream_t st,
                              Args... args) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (smem) {
        cudaError_t err = ensure_dynamic_smem((const void*)kern, smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int CPL>
cudaError_t launch_gu(const GuArgs& a, bool one, bool pdl, cudaStream_t st) {
    const size_t smem = one ? (size_t)CPL * 4 * 32 * 16 : 0;
    return one ? launch_persistent(gateup_gemv_kernel<CPL, true>, gu_warps(true) * 32, smem, pdl, st, a)
               : launch_persistent(gateup_gemv_kernel<CPL, false>, gu_warps(false) * 32, smem, pdl, st, a);
}

template <int CPL>
cudaError_t launch_dn(const DnArgs& a, bool one, int h_rows, bool pdl, cudaStream_t st) {
    const size_t smem = staged_h_bytes(h_rows, a.ldh);
    return one ? launch_persistent(down_gemv_kernel<CPL, true>, kDnThreads, smem, pdl, st, a, h_rows)
               : launch_persistent(down_gemv_kernel<CPL, false>, kDnThreads, smem, pdl, st, a, h_rows);
}

}  // namespace

cudaError_t launch_gateup_gemv(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                               const int32_t* perm, const int32_t* sched, moe_w4_t Wgu,
                               moe_w4_t Wgu_s, uint16_t* H, const int32_t* n_active,
                               WsHeader* hdr, bool pdl, cudaStream_t st) {
    GuArgs a;
    a.x = x;
    a.T = d.T;
    a.d = d.d;
    a.k = d.k;
    a.F = d.F;
    a.Fs = d.F_s;
    a.gsh = log2_group_chunks(d.group);
    a.offsets = offsets;
    a.perm = perm;
    a.sched = sched;
    a.q_r = Wgu.q;
    a.s_r = reinterpret_cast<const __half*>(Wgu.s);
    a.q_sh = Wgu_s.q;
    a.s_sh = reinterpret_cast<const __half*>(Wgu_s.s);
    a.H = H;
    a.ldh = std::max(d.F, d.F_s);
    a.n_route_max = (int)std::min<int64_t>(d.E, (int64_t)d.T * d.k);
    a.n_active = n_active;
    a.hdr = hdr;
    if (!gemv_supported(d)) return cudaErrorInvalidValue;
    const int cpl = chunks_per_lane(d.d);
    const bool one = d.T == 1;
    switch (cpl) {
        case 1: return launch_gu<1>(a, one, pdl, st);
        case 2: return launch_gu<2>(a, one, pdl, st);
        default: return launch_gu<4>(a, one, pdl, st);
    }
}

cudaError_t launch_down_gemv(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                             const int32_t* n_active, const float* topk_w, const int32_t* pos,
                             const uint16_t* residual, uint16_t* out, WsHeader* hdr, bool pdl,
                             cudaStream_t st) {
    DnArgs a;
    a.H = H;
    a.ldh = std::max(d.F, d.F_s);
    a.T = d.T;
    a.d = d.d;
    a.k = d.k;
    a.F = d.F;
    a.Fs = d.F_s;
    a.gsh = log2_group_chunks(d.group);
    a.offsets = offsets;
    a.sched = sched;
    a.q_r = Wd.q;
    a.s_r = reinterpret_cast<const __half*>(Wd.s);
    a.q_sh = Wd_s.q;
    a.s_sh = reinterpret_cast<const __half*>(Wd_s.s);
    a.Y = Y;
    a.n_route_max = (int)std::min<int64_t>(d.E, (int64_t)d.T * d.k);
    a.n_active = n_active;
    a.topk_w = topk_w;
    a.pos = pos;
    a.residual = residual;
    a.out = out;
    a.hdr = hdr;
    if (!gemv_supported(d)) return cudaErrorInvalidValue;
    const int cpl = chunks_per_lane(std::max(d.F, d.F_s));
    const bool one = d.T == 1;
    // a single token's H rows (k routed + 1 shared) are staged in shared memory
    const int h_rows = (one && staged_h_bytes(d.k + 1, a.ldh) <= kMaxStagedH) ? d.k + 1 : 0;
    return cpl == 1 ? launch_dn<1>(a, one, h_rows, pdl, st) : launch_dn<2>(a, one, h_rows, pdl, st);
}

bool gemv_supported(const moe_dims_t& d) {
    return d.d <= kGemvMaxD && std::max(d.F, d.F_s) <= kGemvMaxF;
}

}  // namespace moe
