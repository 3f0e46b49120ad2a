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
// Staging.  Each warp runs its own ring of shared-memory stages filled by the
// TMA unit (cp.async.bulk, completion on one mbarrier per stage): while it
// computes one item, the rows of its next items are already in flight, so
// each SM keeps about 190 KB of weight reads outstanding.  A lane then reads
// 16 bytes (32 nibbles, one quantisation-group scale) per shared-memory load.
// Shapes whose scale rows are not 16-byte multiples use the same arithmetic
// with 16-byte global loads instead (the load path).
//
// Launch order (programmatic dependent launch): the gate+up kernel requests
// its shared-expert stages and loads x before it waits for the router, and
// lets the down kernel launch once the routing is complete; the down kernel
// requests its first weight stages before it waits for H.
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
#include "async.cuh"

namespace moe {
namespace {

// Gate+up: 8 warps at up to 128 registers (32K of the 64K-register file) and
// a 135 KB ring, so a CTA fits beside the decode router's last CTA and every
// CTA is resident (and stages its shared-expert rows) when the routing lands.
// Down: 16 warps.
constexpr int kGuWarps = 8;
constexpr int kGuRP = 2;  // row pairs per ring unit of the gate+up kernel
constexpr int kGuThreads = kGuWarps * 32;
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
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

__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Number of routed groups with rows: from the header, or counted (sched is
// ordered by count, so the active experts are a prefix).  Block-uniform.
__device__ __forceinline__ int active_groups(const int32_t* n_active, const int32_t* offsets,
                                             const int32_t* sched, int n_route_max) {
    if (n_active) return *n_active;
    int n = 0;
    for (int y0 = 0; y0 < n_route_max; y0 += blockDim.x) {
        const int y = y0 + threadIdx.x;
        bool act = false;
        if (y < n_route_max) {
            const int e = sched[y];
            act = offsets[e + 1] > offsets[e];
        }
        n += __syncthreads_count(act);
    }
    return n;
}

// ---------------------------------------------------------------------------
constexpr int kMaxRing = 6;                     // stages per warp, at most
constexpr int kGuRingBudget = 152 * 1024;       // dynamic shared memory of the gate+up ring
constexpr int kDnRingBudget = 200 * 1024;       // dynamic shared memory of the down ring
constexpr size_t kMaxStagedH = 64 * 1024;       // H rows staged by the down kernel, at most

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
__device__ __forceinline__ float lds_f16(uint32_t addr) {
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
    return __half2float(__ushort_as_half(h));
}

// A row (16-byte words) and its scale row, in global memory (load path) or in
// a ring stage (shared-memory addresses).
struct RowRef {
    const uint4* q;
    const __half* s;
    uint32_t sq, ss;
};

template <bool SMEM>
__device__ __forceinline__ uint4 row_word(const RowRef& r, int c) {
    if constexpr (SMEM)
        return lds128(r.sq + 16u * (uint32_t)c);
    else
        return ld_stream(r.q + c);
}
template <bool SMEM>
__device__ __forceinline__ float row_scale(const RowRef& r, int i) {
    if constexpr (SMEM)
        return lds_f16(r.ss + 2u * (uint32_t)i);
    else
        return __half2float(r.s[i]);
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

// Where the gate and up rows of one item are, with their scale rows.
struct GuRows {
    RowRef g, u;
};

__device__ __forceinline__ GuRows gu_rows_global(const GuArgs& a, int expert, int f) {
    const int ngr = (a.d >> 5) >> a.gsh;
    const int Fg = expert >= 0 ? a.F : a.Fs;
    const int64_t rowb = a.d / 2;
    const uint8_t* qb = expert >= 0 ? a.q_r + (int64_t)expert * 2 * a.F * rowb : a.q_sh;
    const __half* sb = expert >= 0 ? a.s_r + (int64_t)expert * 2 * a.F * ngr : a.s_sh;
    GuRows r;
    r.g.q = reinterpret_cast<const uint4*>(qb + (int64_t)f * rowb);
    r.u.q = reinterpret_cast<const uint4*>(qb + (int64_t)(Fg + f) * rowb);
    r.g.s = sb + (int64_t)f * ngr;
    r.u.s = sb + (int64_t)(Fg + f) * ngr;
    r.g.sq = r.g.ss = r.u.sq = r.u.ss = 0;
    return r;
}

// One gate+up item: row pair f of `expert` (-1: the shared expert) against the
// group's rows [row0, row0 + count), writing SwiGLU(gate, up) to H.
// ONE: T == 1 and the lane's x chunks (and their sums) are in xr / xs.
template <int CPL, bool ONE, bool SMEM>
__device__ __forceinline__ void gu_compute(const GuArgs& a, int expert, int f, const GuRows& w,
                                           int row0, int count, const uint4 (&xr)[CPL][4],
                                           const float (&xs)[CPL], int lane) {
    const int nc = a.d >> 5;
    if constexpr (ONE) {
        float ag = 0.f, au = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < nc) {
                const uint4 wg = row_word<SMEM>(w.g, c), wu = row_word<SMEM>(w.u, c);
                const float sg = row_scale<SMEM>(w.g, c >> a.gsh);
                const float su = row_scale<SMEM>(w.u, c >> a.gsh);
                const float pg = fmaf(-136.f, xs[i], dot32_off(wg, xr[i]));
                const float pu = fmaf(-136.f, xs[i], dot32_off(wu, xr[i]));
                ag = fmaf(sg, pg, ag);
                au = fmaf(su, pu, au);
            }
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0 && count > 0)
            a.H[(int64_t)row0 * a.ldh + f] = float_to_bf16_bits(swiglu(ag, au));
    } else {
        for (int i0 = 0; i0 < count; i0 += kGuTokPass) {
            const int ntok = min(kGuTokPass, count - i0);
            const uint16_t* xrow[kGuTokPass];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                const int r = row0 + i0 + min(tt, ntok - 1);
                const int tok = expert >= 0 ? a.perm[r] / a.k : r - row0;
                xrow[tt] = a.x + (int64_t)tok * a.d;
            }
            float ag[kGuTokPass], au[kGuTokPass];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) ag[tt] = au[tt] = 0.f;
            for (int cb = 0; cb < nc; cb += 32 * CPL) {
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int c = cb + lane + 32 * i;
                    if (c >= nc) continue;
                    uint32_t qg[16], qu[16];
                    q_pairs32(row_word<SMEM>(w.g, c), qg);
                    q_pairs32(row_word<SMEM>(w.u, c), qu);
                    const float sg = row_scale<SMEM>(w.g, c >> a.gsh);
                    const float su = row_scale<SMEM>(w.u, c >> a.gsh);
#pragma unroll
                    for (int tt = 0; tt < kGuTokPass; ++tt) {
                        if (tt < ntok) {
                            uint4 xv[4];
                            load_chunk(xrow[tt], c, xv);
                            ag[tt] = fmaf(sg, dot32_q(qg, xv), ag[tt]);
                            au[tt] = fmaf(su, dot32_q(qu, xv), au[tt]);
                        }
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                if (tt < ntok) {
                    const float g = warp_sum(ag[tt]);
                    const float u = warp_sum(au[tt]);
                    if (lane == 0)
                        a.H[(int64_t)(row0 + i0 + tt) * a.ldh + f] = float_to_bf16_bits(swiglu(g, u));
                }
            }
        }
    }
}

// x chunks of the lane (chunk c = lane + 32 i) and their sums, for T == 1.
template <int CPL>
__device__ __forceinline__ void load_x_regs(const uint16_t* x, int d, int lane, uint4 (&xr)[CPL][4],
                                            float (&xs)[CPL]) {
    const int nc = d >> 5;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) {
            load_chunk(x, c, xr[i]);
            xs[i] = sum32_bf16(xr[i]);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) xr[i][v] = make_uint4(0, 0, 0, 0);
            xs[i] = 0.f;
        }
    }
}

// Item of the routed phase: (expert, row pair).
__device__ __forceinline__ void gu_routed_item(const GuArgs& a, int64_t it, int* expert, int* f) {
    const int y = (int)(it / a.F);
    *f = (int)(it - (int64_t)y * a.F);
    *expert = a.sched[y];
}

// Load path.
template <int CPL, bool ONE>
__global__ void __maxnreg__(128) gateup_gemv_kernel(const GuArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    uint4 xr[CPL][4];
    float xs[CPL];
    if (ONE) load_x_regs<CPL>(a.x, a.d, lane, xr, xs);
    // the shared expert reads only x: it runs before the wait for the router
    {
        const int lo = (int)((int64_t)b * a.Fs / G), hi = (int)((int64_t)(b + 1) * a.Fs / G);
        for (int f = lo + warp; f < hi; f += kGuWarps) {
            int row0, count;
            group_rows(a.offsets, a.T, a.k, -1, &row0, &count);
            gu_compute<CPL, ONE, false>(a, -1, f, gu_rows_global(a, -1, f), row0, count, xr, xs, lane);
        }
    }
    pdl_wait();
    pdl_trigger();  // after the wait: dependents may read the routing early
    const int n_act = active_groups(a.n_active, a.offsets, a.sched, a.n_route_max);
    const int64_t R = (int64_t)n_act * a.F;
    const int64_t lo = (int64_t)b * R / G, hi = (int64_t)(b + 1) * R / G;
    for (int64_t it = lo + warp; it < hi; it += kGuWarps) {
        int e, f, row0, count;
        gu_routed_item(a, it, &e, &f);
        group_rows(a.offsets, a.T, a.k, e, &row0, &count);
        gu_compute<CPL, ONE, false>(a, e, f, gu_rows_global(a, e, f), row0, count, xr, xs, lane);
    }
}

// One ring unit of the gate+up kernel: row pairs f0 .. f0 + kGuRP - 1 of
// `expert` (-1: shared) from a stage laid out as [gate q rows | up q rows |
// gate scale rows | up scale rows], against the group's rows [row0, row0 +
// count), writing SwiGLU(gate, up) to H.
template <int CPL, bool ONE>
__device__ __forceinline__ void gu_unit(const GuArgs& a, int expert, int f0, uint32_t st,
                                        int row0, int count, const uint4 (&xr)[CPL][4],
                                        const float (&xs)[CPL], int lane) {
    static_assert(kGuRP == 2, "the reduction below pairs two row pairs");
    const int nc = a.d >> 5;
    const uint32_t rowb = (uint32_t)(a.d / 2), scb = (uint32_t)(((a.d >> 5) >> a.gsh) * 2);
    RowRef rg[kGuRP], ru[kGuRP];
#pragma unroll
    for (int r = 0; r < kGuRP; ++r) {
        rg[r].q = ru[r].q = nullptr;
        rg[r].s = ru[r].s = nullptr;
        rg[r].sq = st + r * rowb;
        ru[r].sq = st + (kGuRP + r) * rowb;
        rg[r].ss = st + 2 * kGuRP * rowb + r * scb;
        ru[r].ss = st + 2 * kGuRP * rowb + (kGuRP + r) * scb;
    }
    if constexpr (ONE) {
        float g[kGuRP], u[kGuRP];
#pragma unroll
        for (int r = 0; r < kGuRP; ++r) g[r] = u[r] = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < nc) {
#pragma unroll
                for (int r = 0; r < kGuRP; ++r) {
                    const uint4 wg = row_word<true>(rg[r], c), wu = row_word<true>(ru[r], c);
                    const float sg = row_scale<true>(rg[r], c >> a.gsh);
                    const float su = row_scale<true>(ru[r], c >> a.gsh);
                    g[r] = fmaf(sg, fmaf(-136.f, xs[i], dot32_off(wg, xr[i])), g[r]);
                    u[r] = fmaf(su, fmaf(-136.f, xs[i], dot32_off(wu, xr[i])), u[r]);
                }
            }
        }
        // lanes 0 / 8 / 16 / 24 hold gate 0 / up 0 / gate 1 / up 1
        const float z = reduce4(g[0], u[0], g[1], u[1], lane);
        const float zu = __shfl_down_sync(0xffffffffu, z, 8);
        if ((lane & 15) == 0 && count > 0)
            a.H[(int64_t)row0 * a.ldh + f0 + (lane >> 4)] = float_to_bf16_bits(swiglu(z, zu));
    } else {
        for (int i0 = 0; i0 < count; i0 += kGuTokPass) {
            const int ntok = min(kGuTokPass, count - i0);
            const uint16_t* xrow[kGuTokPass];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                const int r = row0 + i0 + min(tt, ntok - 1);
                const int tok = expert >= 0 ? a.perm[r] / a.k : r - row0;
                xrow[tt] = a.x + (int64_t)tok * a.d;
            }
            float g[kGuTokPass][kGuRP], u[kGuTokPass][kGuRP];
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt)
#pragma unroll
                for (int r = 0; r < kGuRP; ++r) g[tt][r] = u[tt][r] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = lane + 32 * i;
                if (c >= nc) continue;
#pragma unroll
                for (int r = 0; r < kGuRP; ++r) {
                    uint32_t qg[16], qu[16];
                    q_pairs32(row_word<true>(rg[r], c), qg);
                    q_pairs32(row_word<true>(ru[r], c), qu);
                    const float sg = row_scale<true>(rg[r], c >> a.gsh);
                    const float su = row_scale<true>(ru[r], c >> a.gsh);
#pragma unroll
                    for (int tt = 0; tt < kGuTokPass; ++tt) {
                        if (tt < ntok) {
                            uint4 xv[4];
                            load_chunk(xrow[tt], c, xv);
                            g[tt][r] = fmaf(sg, dot32_q(qg, xv), g[tt][r]);
                            u[tt][r] = fmaf(su, dot32_q(qu, xv), u[tt][r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kGuTokPass; ++tt) {
                if (tt < ntok) {
                    const float z = reduce4(g[tt][0], u[tt][0], g[tt][1], u[tt][1], lane);
                    const float zu = __shfl_down_sync(0xffffffffu, z, 8);
                    if ((lane & 15) == 0)
                        a.H[(int64_t)(row0 + i0 + tt) * a.ldh + f0 + (lane >> 4)] =
                            float_to_bf16_bits(swiglu(z, zu));
                }
            }
        }
    }
}

// Ring path.  A unit is kGuRP consecutive row pairs of one group; its stage
// holds [gate q rows | up q rows | gate scale rows | up scale rows].
template <int CPL, bool ONE>
__global__ void __maxnreg__(128) gateup_ring_kernel(const GuArgs a, int S) {
    extern __shared__ __align__(128) uint8_t ring_smem[];
    __shared__ __align__(8) uint64_t s_bar[kGuWarps * kMaxRing];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int64_t rowb = a.d / 2;
    const int scb = ((a.d >> 5) >> a.gsh) * 2;
    const uint32_t stage_bytes = (uint32_t)(kGuRP * (2 * rowb + 2 * scb));
    uint8_t* wbuf = ring_smem + (size_t)warp * S * stage_bytes;
    const uint32_t bar0 = smem_u32(&s_bar[warp * kMaxRing]);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kGuWarps * kMaxRing; ++i) mbar_init(smem_u32(&s_bar[i]), 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Units of this warp, in order: its shared-expert units, then its routed
    // units.  The shared expert depends on x alone, so its first stages are
    // requested before the wait for the router; nothing routed is touched
    // before that wait.  Routed units are walked with cursors (group, unit),
    // one for the stages being requested and one for the stages being used.
    const int Fu = a.F / kGuRP, Fsu = a.Fs / kGuRP;  // units per group
    const int s_first = (int)((int64_t)b * Fsu / G) + warp, s_hi = (int)((int64_t)(b + 1) * Fsu / G);
    const int n_sh = s_first < s_hi ? (s_hi - s_first + kGuWarps - 1) / kGuWarps : 0;
    int n_units = n_sh;
    struct Cursor {
        int y, j;
    };
    Cursor pc{0, 0}, cc{0, 0};  // producer (lane 0) and consumer cursors
    // expert and first row pair of unit u; routed units advance the cursor
    auto item = [&](int u, Cursor& c, int* e, int* f0) {
        if (u < n_sh) {
            *e = -1;
            *f0 = kGuRP * (s_first + u * kGuWarps);
        } else {
            *e = a.sched[c.y];
            *f0 = kGuRP * c.j;
            c.j += kGuWarps;
            while (c.j >= Fu) {
                c.j -= Fu;
                ++c.y;
            }
        }
    };
    auto issue = [&](int u) {  // lane 0
        int e, f0;
        item(u, pc, &e, &f0);
        const GuRows g = gu_rows_global(a, e, f0);
        const uint32_t slot = u % S;
        const uint32_t dst = smem_u32(wbuf + slot * stage_bytes);
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t qb = (uint32_t)(kGuRP * rowb), sb = (uint32_t)(kGuRP * scb);
        mbar_expect_tx(bar, stage_bytes);
        bulk_load(dst, g.g.q, qb, bar);
        bulk_load(dst + qb, g.u.q, qb, bar);
        bulk_load(dst + 2 * qb, g.g.s, sb, bar);
        bulk_load(dst + 2 * qb + sb, g.u.s, sb, bar);
    };
    if (lane == 0)
        for (int u = 0; u < n_sh && u < S; ++u) issue(u);

    uint4 xr[CPL][4];
    float xs[CPL];
    if (ONE) load_x_regs<CPL>(a.x, a.d, lane, xr, xs);

    pdl_wait();
    // dependents launch only once the routing is complete, so they may read it
    // before their own wait
    pdl_trigger();
    const int n_act = active_groups(a.n_active, a.offsets, a.sched, a.n_route_max);
    {
        const int64_t R = (int64_t)n_act * Fu;
        const int64_t lo = (int64_t)b * R / G, hi = (int64_t)(b + 1) * R / G;
        const int64_t r_first = lo + warp;
        if (r_first < hi) {
            n_units += (int)((hi - r_first + kGuWarps - 1) / kGuWarps);
            pc.y = cc.y = (int)(r_first / Fu);
            pc.j = cc.j = (int)(r_first - (int64_t)pc.y * Fu);
        }
    }
    if (lane == 0)
        for (int u = n_sh; u < n_units && u < S; ++u) issue(u);
    for (int u = 0; u < n_units; ++u) {
        const uint32_t slot = u % S;
        if (!mbar_wait(bar0 + 8 * slot, (u / S) & 1, &s_abort, a.hdr)) return;
        int e, f0, row0, count;
        item(u, cc, &e, &f0);
        group_rows(a.offsets, a.T, a.k, e, &row0, &count);
        gu_unit<CPL, ONE>(a, e, f0, smem_u32(wbuf + slot * stage_bytes), row0, count, xr, xs, lane);
        __syncwarp();
        if (lane == 0 && u + S < n_units) {
            fence_proxy_async_smem();  // the stage was read with plain loads
            issue(u + S);
        }
    }
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
    uint16_t* out;
    WsHeader* hdr;
};

// The kDnQuad consecutive down rows c0 .. c0 + 3 of one group and their scale
// rows: row ch at q + ch * rowb bytes, its scales at s + ch * ngr (global), or
// at sq + ch * rowb and ss + 2 * ch * ngr (a ring stage).
struct DnRows {
    const uint8_t* q;
    const __half* s;
    uint32_t sq, ss;
};

__device__ __forceinline__ DnRows dn_rows_global(const DnArgs& a, int expert, int c0) {
    const int K = expert >= 0 ? a.F : a.Fs;
    const int ngr = (K >> 5) >> a.gsh;
    const int64_t rowb = K / 2;
    DnRows r;
    r.q = (expert >= 0 ? a.q_r + (int64_t)expert * a.d * rowb : a.q_sh) + (int64_t)c0 * rowb;
    r.s = (expert >= 0 ? a.s_r + (int64_t)expert * a.d * ngr : a.s_sh) + (int64_t)c0 * ngr;
    r.sq = r.ss = 0;
    return r;
}

__device__ __forceinline__ RowRef dn_channel(const DnRows& w, int ch, int64_t rowb, int ngr) {
    RowRef r;
    r.q = reinterpret_cast<const uint4*>(w.q + ch * rowb);
    r.s = w.s + ch * ngr;
    r.sq = w.sq + (uint32_t)(ch * rowb);
    r.ss = w.ss + (uint32_t)(2 * ch * ngr);
    return r;
}

// One down item: channels c0 .. c0 + 3 of `expert` (-1: shared) for the
// group's rows [row0, row0 + count), writing Y.
// hs (ONE only): shared-memory address of the staged H rows (0: read H from
// global memory); hsum: their 32-element chunk sums, [row][K / 32] fp32.
template <int CPL, bool ONE, bool SMEM>
__device__ __forceinline__ void dn_compute(const DnArgs& a, int expert, int c0, const DnRows& w,
                                           int row0, int count, int lane, uint32_t hs = 0,
                                           uint32_t hsum = 0) {
    const int K = expert >= 0 ? a.F : a.Fs;
    const int nc = K >> 5, ngr = nc >> a.gsh;
    const int64_t rowb = K / 2;
    constexpr int TP = ONE ? 1 : kDnTokPass;
    for (int i0 = 0; i0 < count; i0 += TP) {
        const int ntok = min(TP, count - i0);
        float acc[TP][kDnQuad];
#pragma unroll
        for (int tt = 0; tt < TP; ++tt)
#pragma unroll
            for (int ch = 0; ch < kDnQuad; ++ch) acc[tt][ch] = 0.f;
        for (int cb = 0; cb < nc; cb += 32 * CPL) {
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = cb + lane + 32 * i;
                if (c >= nc) continue;
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
                    for (int ch = 0; ch < kDnQuad; ++ch) {
                        const RowRef r = dn_channel(w, ch, rowb, ngr);
                        const uint4 wq = row_word<SMEM>(r, c);
                        const float sc = row_scale<SMEM>(r, c >> a.gsh);
                        const float p = fmaf(-136.f, hsm, dot32_off(wq, hv));
                        acc[0][ch] = fmaf(sc, p, acc[0][ch]);
                    }
                } else {
                    uint4 hv[TP][4];
#pragma unroll
                    for (int tt = 0; tt < TP; ++tt)
                        load_chunk(a.H + (int64_t)(row0 + i0 + min(tt, ntok - 1)) * a.ldh, c, hv[tt]);
#pragma unroll
                    for (int ch = 0; ch < kDnQuad; ++ch) {
                        uint32_t qp[16];
                        const RowRef r = dn_channel(w, ch, rowb, ngr);
                        q_pairs32(row_word<SMEM>(r, c), qp);
                        const float sc = row_scale<SMEM>(r, c >> a.gsh);
#pragma unroll
                        for (int tt = 0; tt < TP; ++tt)
                            acc[tt][ch] = fmaf(sc, dot32_q(qp, hv[tt]), acc[tt][ch]);
                    }
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < TP; ++tt) {
            if (tt < ntok) {
                // lanes 0 / 8 / 16 / 24 hold channels c0 .. c0 + 3
                const float z = reduce4(acc[tt][0], acc[tt][1], acc[tt][2], acc[tt][3], lane);
                if ((lane & 7) == 0) a.Y[(int64_t)(row0 + i0 + tt) * a.d + c0 + (lane >> 3)] = z;
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

// Item it of the CTA's list, group-major: group 0 is the shared expert,
// group y > 0 the routed expert sched[y - 1].
__device__ __forceinline__ void dn_item(const DnArgs& a, int it, int nqc, int q_lo, int* expert,
                                        int* c0) {
    const int y = it / nqc;
    *c0 = kDnQuad * (q_lo + (it - y * nqc));
    *expert = y == 0 ? -1 : a.sched[y - 1];
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
        uint2 o;
        o.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
        o.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
        *reinterpret_cast<uint2*>(a.out + (int64_t)t * d + c) = o;
    }
}

// Load path.
template <int CPL, bool ONE>
__global__ void __launch_bounds__(kDnThreads, 1) down_gemv_kernel(const DnArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int q_lo, q_hi;
    dn_share(a.d, &q_lo, &q_hi);
    const int nqc = q_hi - q_lo;
    pdl_trigger();
    pdl_wait();
    const int n_act = active_groups(a.n_active, a.offsets, a.sched, a.n_route_max);
    const int items = (1 + n_act) * nqc;
    for (int it = warp; it < items; it += kDnWarps) {
        int e, c0, row0, count;
        dn_item(a, it, nqc, q_lo, &e, &c0);
        group_rows(a.offsets, a.T, a.k, e, &row0, &count);
        dn_compute<CPL, ONE, false>(a, e, c0, dn_rows_global(a, e, c0), row0, count, lane);
    }
    if (a.out) dn_combine(a, q_lo, nqc);
}

// Ring path.  Stage of one item: [4 down rows | their scale rows], the rows
// of the widest group (max(F, F_s)).  Shared memory: [H rows (h_rows of ldh,
// T == 1 only) | per-warp rings].
template <int CPL, bool ONE>
__global__ void __launch_bounds__(kDnThreads, 1) down_ring_kernel(const DnArgs a, int S,
                                                                    int h_rows) {
    extern __shared__ __align__(128) uint8_t ring_smem[];
    __shared__ __align__(8) uint64_t s_bar[kDnWarps * kMaxRing];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Kmax = max(a.F, a.Fs);
    const uint32_t q_bytes = (uint32_t)(kDnQuad * (Kmax / 2));
    const uint32_t stage_bytes = q_bytes + (uint32_t)(kDnQuad * (((Kmax >> 5) >> a.gsh) * 2));
    const uint32_t h_bytes = (uint32_t)h_rows * a.ldh * 2u;
    const uint32_t hsum_bytes = (uint32_t)h_rows * (a.ldh >> 5) * 4u;
    uint8_t* wbuf = ring_smem + h_bytes + hsum_bytes + (size_t)warp * S * stage_bytes;
    const uint32_t bar0 = smem_u32(&s_bar[warp * kMaxRing]);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kDnWarps * kMaxRing; ++i) mbar_init(smem_u32(&s_bar[i]), 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    int q_lo, q_hi;
    dn_share(a.d, &q_lo, &q_hi);
    const int nqc = q_hi - q_lo;
    pdl_trigger();
    // The routing is complete here: the gate+up kernel lets this kernel launch
    // only after its own wait for the router.  So the weight stages are
    // requested now, and only H (written by the gate+up kernel) waits.
    const int n_act = active_groups(a.n_active, a.offsets, a.sched, a.n_route_max);
    const int items = (1 + n_act) * nqc;
    const int n = warp < items ? (items - warp + kDnWarps - 1) / kDnWarps : 0;
    // items walked with cursors (group, quad): producer (lane 0) and consumer
    struct Cursor {
        int y, qd;
    };
    Cursor pc{0, 0}, cc{0, 0};
    if (n) pc.y = cc.y = warp / nqc, pc.qd = cc.qd = warp - (warp / nqc) * nqc;
    auto item = [&](Cursor& c, int* e, int* c0) {
        *e = c.y == 0 ? -1 : a.sched[c.y - 1];
        *c0 = kDnQuad * (q_lo + c.qd);
        c.qd += kDnWarps;
        while (c.qd >= nqc) {
            c.qd -= nqc;
            ++c.y;
        }
    };
    auto issue = [&](int u) {  // lane 0
        int e, c0;
        item(pc, &e, &c0);
        const DnRows g = dn_rows_global(a, e, c0);
        const int K = e >= 0 ? a.F : a.Fs;
        const uint32_t qb = (uint32_t)(kDnQuad * (K / 2));
        const uint32_t sb = (uint32_t)(kDnQuad * (((K >> 5) >> a.gsh) * 2));
        const uint32_t slot = u % S;
        const uint32_t dst = smem_u32(wbuf + slot * stage_bytes);
        const uint32_t bar = bar0 + 8 * slot;
        mbar_expect_tx(bar, qb + sb);
        bulk_load(dst, g.q, qb, bar);
        bulk_load(dst + q_bytes, g.s, sb, bar);
    };
    if (lane == 0)
        for (int u = 0; u < n && u < S; ++u) issue(u);
    pdl_wait();
    uint32_t hs = 0, hsum = 0;
    if (h_rows) {  // H rows of a single token and their chunk sums, staged once
        const uint4* src = reinterpret_cast<const uint4*>(a.H);
        uint4* dst = reinterpret_cast<uint4*>(ring_smem);
        for (uint32_t i = threadIdx.x; i < h_bytes / 16; i += kDnThreads) dst[i] = __ldg(src + i);
        __syncthreads();
        const int ncr = a.ldh >> 5;  // chunks per row
        float* sums = reinterpret_cast<float*>(ring_smem + h_bytes);
        for (int i = threadIdx.x; i < h_rows * ncr; i += kDnThreads) sums[i] = sum32_bf16(dst + 4 * i);
        __syncthreads();
        hs = smem_u32(ring_smem);
        hsum = smem_u32(sums);
    }
    for (int u = 0; u < n; ++u) {
        const uint32_t slot = u % S;
        if (!mbar_wait(bar0 + 8 * slot, (u / S) & 1, &s_abort, a.hdr)) break;
        int e, c0, row0, count;
        item(cc, &e, &c0);
        group_rows(a.offsets, a.T, a.k, e, &row0, &count);
        DnRows w;
        w.q = nullptr;
        w.s = nullptr;
        w.sq = smem_u32(wbuf + slot * stage_bytes);
        w.ss = w.sq + q_bytes;
        dn_compute<CPL, ONE, true>(a, e, c0, w, row0, count, lane, hs, hsum);
        __syncwarp();
        if (lane == 0 && u + S < n) {
            fence_proxy_async_smem();  // the stage was read with plain loads
            issue(u + S);
        }
    }
    if (a.out) dn_combine(a, q_lo, nqc);
}

// ---------------------------------------------------------------------------
int log2_group_chunks(int group) { return group == 32 ? 0 : group == 64 ? 1 : 2; }

// 16-byte loads per lane and row in one pass over K; longer rows take several
// passes (register budget of 128 per thread at 512 threads).
int chunks_per_lane(int K, int cap) {
    const int nc = K / 32;
    const int c = (nc + 31) / 32;
    return std::min(cap, c <= 1 ? 1 : c <= 2 ? 2 : 4);
}

// Shared memory of the staged H rows and their chunk sums (down kernel, T == 1).
size_t staged_h_bytes(int rows, int ldh) {
    return (size_t)rows * ldh * 2 + (size_t)rows * (ldh / 32) * 4;
}

// Stages per warp that fit `budget` less `other` bytes over `warps` rings (0:
// the ring path does not apply).
int ring_stages(size_t stage_bytes, size_t budget, int warps, size_t other = 0) {
    if (other >= budget) return 0;
    const size_t per_warp = (budget - other) / warps;
    return (int)std::min<size_t>(kMaxRing, per_warp / stage_bytes);
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
cudaError_t launch_gu(const GuArgs& a, bool one, int S, size_t stage, bool pdl, cudaStream_t st) {
    if (S >= 2) {
        const size_t smem = (size_t)kGuWarps * S * stage;
        return one ? launch_persistent(gateup_ring_kernel<CPL, true>, kGuThreads, smem, pdl, st, a, S)
                   : launch_persistent(gateup_ring_kernel<CPL, false>, kGuThreads, smem, pdl, st, a, S);
    }
    return one ? launch_persistent(gateup_gemv_kernel<CPL, true>, kGuThreads, 0, pdl, st, a)
               : launch_persistent(gateup_gemv_kernel<CPL, false>, kGuThreads, 0, pdl, st, a);
}

template <int CPL>
cudaError_t launch_dn(const DnArgs& a, bool one, int S, size_t stage, int h_rows, bool pdl,
                      cudaStream_t st) {
    if (S >= 2) {
        const size_t smem = staged_h_bytes(h_rows, a.ldh) + (size_t)kDnWarps * S * stage;
        return one ? launch_persistent(down_ring_kernel<CPL, true>, kDnThreads, smem, pdl, st, a, S,
                                       h_rows)
                   : launch_persistent(down_ring_kernel<CPL, false>, kDnThreads, smem, pdl, st, a, S,
                                       h_rows);
    }
    return one ? launch_persistent(down_gemv_kernel<CPL, true>, kDnThreads, 0, pdl, st, a)
               : launch_persistent(down_gemv_kernel<CPL, false>, kDnThreads, 0, pdl, st, a);
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

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
    const int cpl = chunks_per_lane(d.d, 4);
    const bool single_pass = d.d / 32 <= 32 * cpl;
    // the register-resident x form needs the whole row in one pass
    const bool one = d.T == 1 && single_pass;
    // ring: one stage holds a whole row pair, scale rows are 16-byte multiples
    const int scb = d.d / d.group * 2;
    const size_t stage = (size_t)kGuRP * (d.d + 2 * scb);
    const bool ring_ok = single_pass && scb % 16 == 0 && aligned16(Wgu.s) && aligned16(Wgu_s.s);
    const int S = ring_ok ? ring_stages(stage, kGuRingBudget, kGuWarps) : 0;
    switch (cpl) {
        case 1: return launch_gu<1>(a, one, S, stage, pdl, st);
        case 2: return launch_gu<2>(a, one, S, stage, pdl, st);
        default: return launch_gu<4>(a, one, S, stage, pdl, st);
    }
}

cudaError_t launch_down_gemv(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                             const int32_t* n_active, const float* topk_w, const int32_t* pos,
                             uint16_t* out, WsHeader* hdr, bool pdl, cudaStream_t st) {
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
    a.out = out;
    a.hdr = hdr;
    const int Kmax = std::max(d.F, d.F_s);
    const int cpl = chunks_per_lane(Kmax, 2);
    const bool single_pass = Kmax / 32 <= 32 * cpl;
    const bool one = d.T == 1;
    // ring: one stage holds four whole rows; four scale rows are 16-byte multiples
    const int sb_F = kDnQuad * (d.F / d.group) * 2, sb_Fs = kDnQuad * (d.F_s / d.group) * 2;
    const size_t stage = (size_t)kDnQuad * (Kmax / 2) + kDnQuad * (Kmax / d.group) * 2;
    const bool ring_ok = single_pass && sb_F % 16 == 0 && sb_Fs % 16 == 0 && aligned16(Wd.s) &&
                         aligned16(Wd_s.s);
    // a single token's H rows (k routed + 1 shared) are staged in shared memory
    const int h_rows = (one && staged_h_bytes(d.k + 1, a.ldh) <= kMaxStagedH) ? d.k + 1 : 0;
    const int S = ring_ok ? ring_stages(stage, kDnRingBudget, kDnWarps, staged_h_bytes(h_rows, a.ldh)) : 0;
    return cpl == 1 ? launch_dn<1>(a, one, S, stage, h_rows, pdl, st)
                    : launch_dn<2>(a, one, S, stage, h_rows, pdl, st);
}

}  // namespace moe
