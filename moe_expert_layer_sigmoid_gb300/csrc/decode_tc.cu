// Single-token decode on the warp-level tensor cores: the expert projections,
// and the whole step (router, descriptors, gate+up, down, combine) in one
// launch.
//
// The Laguna decode step runs the gathered Q4 expert GEMVs: gate+up fused with
// SwiGLU, the shared expert through the same kernel, then the down projection
// (thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1 decode on
// the CUDA engine"), and sums the expert outputs back per token in a fixed
// order (thewafflehaus/FFAI PR #72, Nemotron W4A16 MoE commit, the
// deterministic scatter-add).  At T = 1 the step streams ~71 MB of int4
// weights, two weights per byte, so at HBM rate an SM must retire ~43 weights
// per clock.  A CUDA-core dot product spends ~3 lane-instructions per weight
// (unpack, convert, FMA) and caps the stream below the HBM rate; here the
// multiply-add goes to mma.sync m16n8k16 (bf16 in, fp32 accumulate), 256
// weight-activation products per instruction, and the CUDA cores only unpack.
//
// Exact int4 operands without a per-weight conversion.  One lop3 turns a
// 32-bit word of eight two's-complement nibbles into two bf16 values:
// (w ^ 0x88888888) & 0x000F000F leaves u = q + 8 (0..15) of nibbles 0 and 4
// in bits 0-3 and 16-19, and a bf16 whose exponent field is zero is the
// subnormal u * 2^-133, exactly; mask 0x00F000F0 gives nibbles 1 and 5 as
// u * 2^-129, and the same two masks on w >> 8 give nibbles 2, 6 and 3, 7.
// The tensor core takes these subnormal operands exactly (measured on GB300:
// products and sums agree with an fp64 reference to fp32 rounding).  The
// activation operand carries the matching power-of-two scale: x * 2^sigma
// against the nibbles in bits 0-3, x * 2^(sigma - 4) against those in bits
// 4-7, so every product is u * x * 2^(sigma - 133).  sigma is chosen per row
// from the row's largest |x| so that x * 2^sigma stays finite and the products
// stay normal fp32 numbers.  The offset u = q + 8 is taken out by starting the
// accumulator at -8 * sum(x) * 2^(sigma - 133), so each quantisation group's
// accumulator holds sum x * q * 2^(sigma - 133); it is multiplied by the
// group's fp16 scale and added into an fp32 total, and the total is rescaled
// by 2^(133 - sigma).  The result is sum x * (q * s) up to fp32 rounding.
//
// Fragment layout (m16n8k16, A row-major 16 x 16, B 16 x 8): lane (g, t) =
// (lane / 4, lane % 4) holds A rows g and g + 8.  A unit is 16 weight rows x
// one span pair (256 K elements, 128 bytes per row); lane t takes 16 bytes of
// each row per 128-element span (for groups of 64 or 32: two 8-byte or four
// 4-byte pieces, one per quantisation group, so that every MMA stays inside
// one group); one 8-nibble word feeds two MMAs.  The logical k order inside an
// MMA is a permutation of the physical K order; the activation operand is
// staged once per CTA in shared memory in that permuted order, already
// scaled.  Only column 0 of the MMA's eight token columns carries the token.
//
// Data movement.  Each warp owns a ring of unit slots in shared memory, so
// the bytes in flight are bounded by shared memory, not by registers: gate+up
// weights arrive by TMA (a tensor map viewing [E][2F][d/2] as {d/2 bytes,
// 8 rows, gate/up, F/8 row blocks, E}, one box per unit, 128-byte swizzle),
// down weights and every unit's fp16 scales by cp.async; a slot is refilled as
// soon as it has been read.  Streamed weights carry an evict-first L2 policy.
// The code is kept compact on purpose: a step executes most of its code once,
// and code that does not stay in the SM's instruction cache is fetched again
// at several cycles per instruction, so the unit loops are not unrolled and
// every phase body exists once (non-inlined), shared by the three kernels.
//
// gate+up:  a unit's rows g are gate rows f0 + pi(g) and rows g + 8 the up
//           rows F + f0 + pi(g), pi(g) = (g >> 1) | ((g & 1) << 2) (with the
//           swizzle this makes each quarter-warp's 16-byte reads cover all
//           banks once), so lane (g, 0) ends with the gate and up sums of one
//           row pair.  A CTA owns a contiguous range of row blocks (8 row
//           pairs); warp w takes span pair w % P of every (16 / P)-th block,
//           partial sums go to shared memory and are summed over the pairs in
//           order, then SwiGLU and one bf16 rounding.
// down:     a CTA owns a contiguous range of output channels for every group
//           (shared expert, then the routed experts in schedule order); units
//           are (group, 16-channel block, span pair).  Each group's channel
//           values are summed over the pairs in order, and the fused combine
//           adds them in the fixed order of moe_combine_shared: routed slots
//           j = 0..k-1, then the shared expert, then (optionally) the residual.
#include <cstring>

#include "router_dev.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kTcWarps = 16;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTile = 2048;        // weight bytes of a unit: 16 rows x 128 bytes
constexpr int kTcMaxRoute = 64;    // routed groups of one token (k <= 32)

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ uint32_t ob_pair(uint32_t w, uint32_t mask) {
    // (w ^ 0x88888888) & mask: two's-complement nibbles to offset-binary u = q + 8
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(r) : "r"(w), "r"(0x88888888u), "r"(mask));
    return r;
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Routing data written by an earlier kernel of the step: read through L2.
__device__ __forceinline__ int ld_cg_i32(const int32_t* p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ float h2f_lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float h2f_hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// cp.async of N bytes (4, 8 or 16) global -> shared, L1-allocating (scales:
// the warps of a CTA read different pieces of the same scale lines).
template <int N>
__device__ __forceinline__ void cp_async_ca(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(N) : "memory");
}

// cp.async of N bytes (4, 8 or 16) global -> shared with an L2 policy.
template <int N>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src, uint64_t pol) {
    if constexpr (N == 16)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                     "l"(pol)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], %2, %3;" ::"r"(dst), "l"(src),
                     "n"(N), "l"(pol)
                     : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One unit in registers: lane t's words of two weight rows for a span pair
// (span 0: words 0-3, span 1: words 4-7) and the rows' fp16 scales of the
// pair's 2 * (128 / G) groups.
template <int G>
struct TcUnit {
    uint32_t w0[8], w1[8];
    uint32_t s0[128 / G], s1[128 / G];
};

// The pair's MMAs.  frag: shared address of the activation fragments of the
// row ([span][word i][lane t] uint4); cin: accumulator starts of the pair's
// groups.  p0 / p1 += scale * (group sum) for rows g / g + 8 (column 0 on the
// t = 0 lanes).
template <int G>
__device__ __forceinline__ void tc_mma(const TcUnit<G>& U, uint32_t frag, int pair, int t,
                                       const float* cin, float& p0, float& p1) {
    constexpr int NG = 128 / G, MPG = 8 / NG;
#pragma unroll
    for (int sp = 0; sp < 2; ++sp) {
        uint32_t b[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = lds_v4(frag + (uint32_t)(((2 * pair + sp) * 4 + i) * 4 + t) * 16u);
            b[4 * i] = v.x;
            b[4 * i + 1] = v.y;
            b[4 * i + 2] = v.z;
            b[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int q = sp * NG + j;  // group within the pair
            const float ci = cin[q];
            float acc[4] = {ci, ci, ci, ci};
#pragma unroll
            for (int m = 0; m < MPG; ++m) {
                const int mi = j * MPG + m, i = 4 * sp + (mi >> 1);
                const uint32_t wa = (mi & 1) ? U.w0[i] >> 8 : U.w0[i];
                const uint32_t wb = (mi & 1) ? U.w1[i] >> 8 : U.w1[i];
                mma16816(acc, ob_pair(wa, 0x000F000Fu), ob_pair(wb, 0x000F000Fu),
                         ob_pair(wa, 0x00F000F0u), ob_pair(wb, 0x00F000F0u), b[2 * mi], b[2 * mi + 1]);
            }
            const float sa = (q & 1) ? h2f_hi(U.s0[q >> 1]) : h2f_lo(U.s0[q >> 1]);
            const float sb = (q & 1) ? h2f_hi(U.s1[q >> 1]) : h2f_lo(U.s1[q >> 1]);
            p0 = fmaf(sa, acc[0], p0);
            p1 = fmaf(sb, acc[2], p1);
        }
    }
}

// Scale exponent of a row whose largest |value| has fp32 bits `mbits`:
// |v| * 2^sigma < 2^126, and sigma <= 100 keeps products of small values
// normal.
__device__ __forceinline__ int row_sigma(int mbits) {
    const int e = ((mbits >> 23) & 0xFF) - 126;  // max |v| < 2^e
    return min(100, 126 - e);
}

// ---------------------------------------------------------------- layout
// One shared-memory layout for the three kernels (offsets from a 1024-aligned
// base; parts a kernel does not use have size zero).
struct DecSmem {
    size_t wring, sring, bars;                     // rings: weight tiles, scales, barriers
    size_t xfrag, xcin, xtmp;                      // x: fragments, accumulator starts, scratch
    size_t gpart, coord, soff, sched, srow;        // gate+up: partials and tables
    size_t hfrag, hcin, htmp, dpart, yc, qe, hrow, yrow;  // down: staged H, partials, tables
    size_t cand, route;                            // routing scratch and results
    size_t misc;                                   // Misc, then the warps' ring parities
    size_t total;
    int R, S, Smax, P, PF, max_rb, max_groups, nrb_max;
};
struct DecDims {
    int d, F, Fs, group, max_rb, max_groups, max_ch, rows;
    bool gu, dn, route;
};
__host__ __device__ inline DecSmem dec_smem(const DecDims& q) {
    DecSmem L;
    const int NG = 128 / q.group;
    L.R = q.group == 128 ? 4 : 3;  // slots per warp
    const int Fm = q.F > q.Fs ? q.F : q.Fs;
    L.S = q.d / 128;
    L.Smax = Fm / 128;
    L.P = q.d / 256;
    L.PF = Fm / 256;
    L.max_rb = q.max_rb;
    L.max_groups = q.max_groups;
    L.nrb_max = (q.max_ch + 15) / 16;
    size_t o = 0;
    auto take = [&](size_t& at, size_t bytes, size_t align) {
        o = (o + align - 1) / align * align;
        at = o;
        o += bytes;
    };
    take(L.wring, (size_t)kTcWarps * L.R * kTile, 1024);
    take(L.sring, (size_t)kTcWarps * L.R * 32 * 8 * NG, 16);
    take(L.bars, (size_t)kTcWarps * L.R * 8, 8);
    take(L.xfrag, q.gu ? (size_t)L.S * 256 : 0, 16);
    take(L.xcin, q.gu ? (size_t)(q.d / q.group) * 4 : 0, 16);
    take(L.xtmp, q.gu ? (size_t)(q.d / 8) * 4 : 0, 16);
    take(L.gpart, q.gu ? (size_t)q.max_rb * L.P * 64 : 0, 16);
    take(L.coord, q.gu ? (size_t)q.max_rb * 8 : 0, 8);
    take(L.soff, q.gu ? (size_t)q.max_rb * 8 : 0, 8);
    take(L.sched, q.gu ? (size_t)kTcMaxRoute * 4 : 0, 16);
    take(L.srow, q.gu ? (size_t)kTcMaxRoute * 4 : 0, 16);
    const int mg = q.dn ? q.max_groups : 0;
    take(L.hfrag, (size_t)mg * L.Smax * 256, 16);
    take(L.hcin, (size_t)mg * (Fm / q.group) * 4, 16);
    take(L.htmp, (size_t)mg * (Fm / 8) * 4, 16);
    take(L.dpart, (size_t)mg * L.nrb_max * L.PF * 64, 16);
    take(L.yc, (size_t)mg * L.nrb_max * 64, 16);
    take(L.qe, (size_t)mg * 4, 16);
    take(L.hrow, (size_t)mg * 4, 16);
    take(L.yrow, q.dn ? (size_t)q.rows * 4 : 0, 16);
    take(L.cand, q.route ? (size_t)kTcWarps * 32 * 12 + 64 * 4 : 0, 16);
    take(L.route, q.route ? (size_t)4 * 32 * 4 : 0, 16);
    take(L.misc, 16 + 8 * 64 + 4 * kTcWarps, 16);
    L.total = o;
    return L;
}

// Small values: the abort flag, sigma of x and 2^(133 - sigma), row maxima
// and sigmas of staged H rows; the warps' ring parities follow.
struct Misc {
    int abort;
    int xsigma;
    float post;
    int pad;
    int mx[64];
    int sigma[64];
};
__device__ __forceinline__ Misc* misc(char* sm, const DecSmem& L) {
    return reinterpret_cast<Misc*>(sm + L.misc);
}
__device__ __forceinline__ int* ring_par(char* sm, const DecSmem& L) {
    return reinterpret_cast<int*>(sm + L.misc + sizeof(Misc));
}

// Per-warp ring barriers, parities, the abort flag and the tensor maps, once
// per CTA.
__device__ __forceinline__ void ring_setup(char* sm, const DecSmem& L, const CUtensorMap* tm0,
                                           const CUtensorMap* tm1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        const uint32_t bars = smem_u32(sm + L.bars) + (uint32_t)(warp * L.R * 8);
        for (int p = 0; p < L.R; ++p) mbar_init(bars + 8 * p, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        ring_par(sm, L)[warp] = 0;
        if (warp == 0) {
            misc(sm, L)->abort = 0;
            if (tm0) prefetch_tmap(tm0);
            if (tm1) prefetch_tmap(tm1);
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- staging
// Stage `nrows` bf16 rows as activation fragments, the whole CTA.  Row r
// starts at base + (rowidx ? rowidx[r] : r) * ld and has K0 (r = 0) or K1
// (r > 0) elements.  Destinations: frag + r * fstride uint4 laid out
// [span][word i][lane t]; accumulator starts cin + r * cstride (one per
// group); sigma[r].  tmp: scratch of tstride floats per row; mx: nrows ints.
// Each pass is flattened over all rows.  coh: the rows were written earlier
// by this kernel and are read through L2.
template <int G>
__device__ __noinline__ void stage_rows(const uint16_t* base, int64_t ld, const int* rowidx,
                                        int nrows, int K0, int K1, uint4* frag, int fstride,
                                        float* cin, int cstride, int* sigma, float* tmp,
                                        int tstride, int* mx, bool coh) {
    constexpr int NG = 128 / G, WPG = G / 32, SPG = G / 8;  // slots (8 elements) per group
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int n0 = K0 / 8, n1 = K1 / 8;
    const int total = n0 + (nrows - 1) * n1;
    auto slot = [&](int idx, int& r, int& sl) {
        if (idx < n0) {
            r = 0;
            sl = idx;
        } else {
            r = 1 + (idx - n0) / n1;
            sl = idx - n0 - (r - 1) * n1;
        }
    };
    auto ld16 = [&](int r, int sl) {
        const int s = sl >> 4, i = (sl >> 2) & 3, t = sl & 3;
        const int j = i / WPG, ii = i % WPG;
        const uint4* p = reinterpret_cast<const uint4*>(
            base + (int64_t)(rowidx ? rowidx[r] : r) * ld + 128 * s + j * G + t * (G / 4) + 8 * ii);
        return coh ? __ldcg(p) : __ldg(p);
    };
    for (int r = tid; r < nrows; r += nthr) mx[r] = 0;
    __syncthreads();
    // pass 1: largest |value| of each row
#pragma unroll 1
    for (int idx = tid; idx < total; idx += nthr) {
        int r, sl;
        slot(idx, r, sl);
        const uint4 v = ld16(r, sl);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        int m = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            m = max(m, (int)((u[w] << 16) & 0x7FFFFFFFu));
            m = max(m, (int)(u[w] & 0x7FFF0000u));
        }
        if (m) atomicMax(mx + r, m);
    }
    __syncthreads();
    for (int r = tid; r < nrows; r += nthr) sigma[r] = row_sigma(mx[r]);
    __syncthreads();
    // pass 2: permuted, scaled fragments; 8-element partial sums in K order
#pragma unroll 1
    for (int idx = tid; idx < total; idx += nthr) {
        int r, sl;
        slot(idx, r, sl);
        const uint4 v = ld16(r, sl);
        const int s = sl >> 4, i = (sl >> 2) & 3, t = sl & 3;
        const int j = i / WPG, ii = i % WPG;
        const int sg = sigma[r];
        const float f0 = ldexpf(1.0f, sg), f1 = ldexpf(1.0f, sg - 4);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        float x[8];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            x[2 * w] = __uint_as_float(u[w] << 16);
            x[2 * w + 1] = __uint_as_float(u[w] & 0xFFFF0000u);
        }
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += x[w];
        // elements (0, 4) and (2, 6) against nibbles in bits 0-3, (1, 5) and
        // (3, 7) against bits 4-7
        uint4 o;
        o.x = (uint32_t)float_to_bf16_bits(x[0] * f0) | ((uint32_t)float_to_bf16_bits(x[4] * f0) << 16);
        o.y = (uint32_t)float_to_bf16_bits(x[1] * f1) | ((uint32_t)float_to_bf16_bits(x[5] * f1) << 16);
        o.z = (uint32_t)float_to_bf16_bits(x[2] * f0) | ((uint32_t)float_to_bf16_bits(x[6] * f0) << 16);
        o.w = (uint32_t)float_to_bf16_bits(x[3] * f1) | ((uint32_t)float_to_bf16_bits(x[7] * f1) << 16);
        frag[r * fstride + (s * 4 + i) * 4 + t] = o;
        // slot position inside its group, in K order
        tmp[r * tstride + (s * NG + j) * SPG + t * WPG + ii] = sum;
    }
    __syncthreads();
    // pass 3: accumulator starts, -8 * sum(group) * 2^(sigma - 133)
    const int g0 = K0 / G, g1 = K1 / G;
    const int gtotal = g0 + (nrows - 1) * g1;
    for (int idx = tid; idx < gtotal; idx += nthr) {
        int r, gi;
        if (idx < g0) {
            r = 0;
            gi = idx;
        } else {
            r = 1 + (idx - g0) / g1;
            gi = idx - g0 - (r - 1) * g1;
        }
        float sum = 0.f;
        for (int p = 0; p < SPG; ++p) sum += tmp[r * tstride + gi * SPG + p];
        cin[r * cstride + gi] = -ldexpf(sum, sigma[r] - 130);
    }
    __syncthreads();
}

template <int G>
__device__ __forceinline__ void stage_x(const uint16_t* x, int d, char* sm, const DecSmem& L) {
    Misc* m = misc(sm, L);
    stage_rows<G>(x, 0, nullptr, 1, d, d, reinterpret_cast<uint4*>(sm + L.xfrag), 0,
                  reinterpret_cast<float*>(sm + L.xcin), 0, &m->xsigma,
                  reinterpret_cast<float*>(sm + L.xtmp), 0, m->mx, false);
    if (threadIdx.x == 0) m->post = ldexpf(1.0f, 133 - m->xsigma);
    __syncthreads();
}

// ---------------------------------------------------------------- gate+up
struct TcGuArgs {
    CUtensorMap tm_r;  // routed experts' gate+up nibbles, box {128, 8, 2, 1, 1}
    CUtensorMap tm_s;  // the shared expert's
    const uint16_t* x;
    int d, T, k, F, Fs;
    const int32_t* offsets;
    const int32_t* sched;
    const __half* s_r;
    const __half* s_sh;
    uint16_t* H;
    int ldh;
    int n_route_max;
    const int32_t* n_active;
    WsHeader* hdr;
    int max_rb;  // row blocks a CTA holds (shared-memory tables)
};

__device__ __forceinline__ int tile_row(int g) { return (g >> 1) | ((g & 1) << 2); }

// A warp's gate+up units of a phase: span pair `pair` of the row blocks
// rbs, rbs + wpp, ...  (P = d / 256 pairs, wpp = 16 / P warps per pair).
struct GuWarp {
    int pair, rbs, wpp, n;
};
__device__ __forceinline__ GuWarp gu_warp(int P, int nrb) {
    GuWarp w;
    const int warp = threadIdx.x >> 5;
    w.wpp = kTcWarps / P;
    w.pair = warp % P;
    w.rbs = warp / P;
    w.n = (warp < P * w.wpp && w.rbs < nrb) ? (nrb - w.rbs + w.wpp - 1) / w.wpp : 0;
    return w;
}

// Row blocks [rb0, rb0 + nrb) of the shared expert (shared) or of the routed
// list (group y = rb / (F / 8) in schedule order, expert sched[y]).
template <int G>
__device__ __forceinline__ void gu_tables(const TcGuArgs& a, bool shared, int64_t rb0, int nrb,
                                          char* sm, const DecSmem& L) {
    const int ng = a.d / G, nfb = (shared ? a.Fs : a.F) / 8;
    int2* coord = reinterpret_cast<int2*>(sm + L.coord);
    int64_t* soff = reinterpret_cast<int64_t*>(sm + L.soff);
    const int* ssched = reinterpret_cast<const int*>(sm + L.sched);
    for (int i = threadIdx.x; i < nrb; i += blockDim.x) {
        const int64_t rb = rb0 + i;
        const int y = (int)(rb / nfb), fb = (int)(rb - (int64_t)y * nfb);
        const int e = shared ? 0 : ssched[y];
        coord[i] = make_int2(fb, e);
        soff[i] = (shared ? 0 : (int64_t)e * 2 * a.F * ng) + (int64_t)fb * 8 * ng;
    }
    __syncthreads();
}

// Request unit i of the warp into ring slot `slot`: the weight tile by TMA
// (lane 0), each lane's two rows' scales by cp.async.
template <int G>
__device__ __forceinline__ void gu_issue(const TcGuArgs& a, bool shared, char* sm, const DecSmem& L,
                                         const GuWarp& W, int i, int slot) {
    constexpr int NG = 128 / G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, rr = tile_row(lane >> 2);
    const int rbl = W.rbs + i * W.wpp;
    const int2 c = reinterpret_cast<const int2*>(sm + L.coord)[rbl];
    const int64_t so = reinterpret_cast<const int64_t*>(sm + L.soff)[rbl];
    const uint64_t pol = l2_evict_first();
    if (lane == 0) {
        const uint32_t bar = smem_u32(sm + L.bars) + (uint32_t)((warp * L.R + slot) * 8);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(bar, kTile);
        tma_load_5d_hint(smem_u32(sm + L.wring) + (uint32_t)((warp * L.R + slot) * kTile),
                         shared ? &a.tm_s : &a.tm_r, 128 * W.pair, 0, 0, c.x, c.y, bar, pol);
    }
    const int ng = a.d / G;
    const __half* s0 = (shared ? a.s_sh : a.s_r) + so + (int64_t)rr * ng + 2 * NG * W.pair;
    const int64_t ds = (int64_t)(shared ? a.Fs : a.F) * ng;  // gate row -> up row
    const uint32_t sdst = smem_u32(sm + L.sring) + (uint32_t)(((warp * L.R + slot) * 32 + lane) * 8 * NG);
    cp_async_ca<4 * NG>(sdst, s0);
    cp_async_ca<4 * NG>(sdst + 4 * NG, s0 + ds);
    cp_commit();
}

template <int G>
__device__ __forceinline__ void gu_prologue(const TcGuArgs& a, bool shared, int nrb, char* sm,
                                            const DecSmem& L) {
    const GuWarp W = gu_warp(L.P, nrb);
    for (int i = 0; i < W.n && i < L.R; ++i) gu_issue<G>(a, shared, sm, L, W, i, i);
}

// Lane t's words of one 128-byte tile row (swizzled: chunk c at c ^ rr), the
// bytes tc_mma expects: per span and group, G / 8 bytes at group offset
// t * G / 8.
template <int G>
__device__ __forceinline__ void read_tile_row(uint32_t row, int rr, int t, uint32_t* w) {
    constexpr int NG = 128 / G, PB = G / 8, WPG = G / 32;
#pragma unroll
    for (int sp = 0; sp < 2; ++sp)
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int byte = 64 * sp + j * (G / 2) + t * PB;
            const uint32_t addr = row + ((((byte >> 4) ^ rr) << 4) | (byte & 15));
            uint32_t* d = w + 4 * sp + j * WPG;
            if constexpr (PB == 16) {
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                             : "r"(addr));
            } else if constexpr (PB == 8) {
                asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(d[0]), "=r"(d[1]) : "r"(addr));
            } else {
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(d[0]) : "r"(addr));
            }
        }
}

// Wait until the ring slot of unit i (of n) has its cp.async copies: the
// R - 1 most recent groups may still be in flight while later units follow.
__device__ __forceinline__ void ring_wait_copies(int i, int n, int R) {
    if (n - i > R - 1) {
        if (R == 4)
            cp_wait<3>();
        else
            cp_wait<2>();
    } else {
        cp_wait<0>();
    }
}

// Consume the warp's units of the phase (the first min(R, n) already
// requested), refilling each slot as soon as it has been read.
template <int G>
__device__ __noinline__ void gu_consume(const TcGuArgs& a, bool shared, int nrb, char* sm,
                                        const DecSmem& L) {
    constexpr int NG = 128 / G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const GuWarp W = gu_warp(L.P, nrb);
    if (W.n == 0) return;
    const int rr = tile_row(g);
    volatile int* abort_flag = &misc(sm, L)->abort;
    const uint32_t frag = smem_u32(sm + L.xfrag);
    const float* cin = reinterpret_cast<const float*>(sm + L.xcin) + 2 * NG * W.pair;
    float* part = reinterpret_cast<float*>(sm + L.gpart);
    int* parw = ring_par(sm, L) + warp;
    uint32_t par = (uint32_t)*parw;
    for (int i = 0; i < W.n; ++i) {
        const int slot = i % L.R;
        const uint32_t bar = smem_u32(sm + L.bars) + (uint32_t)((warp * L.R + slot) * 8);
        if (!mbar_wait(bar, (par >> slot) & 1u, abort_flag, a.hdr)) break;
        par ^= 1u << slot;
        ring_wait_copies(i, W.n, L.R);
        const uint32_t tile = smem_u32(sm + L.wring) + (uint32_t)((warp * L.R + slot) * kTile);
        TcUnit<G> U;
        read_tile_row<G>(tile + rr * 128, rr, t, U.w0);
        read_tile_row<G>(tile + 1024 + rr * 128, rr, t, U.w1);
        const uint32_t ssrc = smem_u32(sm + L.sring) + (uint32_t)(((warp * L.R + slot) * 32 + lane) * 8 * NG);
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(U.s0[q]) : "r"(ssrc + 4 * q));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(U.s1[q]) : "r"(ssrc + 4 * NG + 4 * q));
        }
        float pg = 0.f, pu = 0.f;
        tc_mma<G>(U, frag, W.pair, t, cin, pg, pu);
        if (t == 0) {
            float* pp = part + ((W.rbs + i * W.wpp) * L.P + W.pair) * 16;
            pp[g] = pg;
            pp[8 + g] = pu;
        }
        __syncwarp();  // every lane has read the slot
        if (i + L.R < W.n) gu_issue<G>(a, shared, sm, L, W, i + L.R, slot);
    }
    *parw = (int)par;
}

// Sum the partials over the pairs in order, SwiGLU, one bf16 rounding; part
// slot g holds weight row f0 + tile_row(g).  H row of a routed group: srow.
template <int G>
__device__ __noinline__ void gu_reduce(const TcGuArgs& a, bool shared, int64_t rb0, int nrb, char* sm,
                                       const DecSmem& L) {
    __syncthreads();
    const float* part = reinterpret_cast<const float*>(sm + L.gpart);
    const int* srow = reinterpret_cast<const int*>(sm + L.srow);
    const int nfb = (shared ? a.Fs : a.F) / 8;
    const float ps = misc(sm, L)->post;
    for (int i = threadIdx.x; i < nrb * 8; i += blockDim.x) {
        const int rbl = i >> 3, gg = i & 7;
        float sg = 0.f, su = 0.f;
        for (int q = 0; q < L.P; ++q) {
            sg += part[(rbl * L.P + q) * 16 + gg];
            su += part[(rbl * L.P + q) * 16 + 8 + gg];
        }
        sg *= ps;
        su *= ps;
        const int64_t rb = rb0 + rbl;
        const int y = (int)(rb / nfb);
        const int f = (int)(rb - (int64_t)y * nfb) * 8 + tile_row(gg);
        const int hr = shared ? a.T * a.k : srow[y];
        a.H[(int64_t)hr * a.ldh + f] = float_to_bf16_bits(swiglu_f32(sg, su));
    }
    __syncthreads();
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) gateup_tc_kernel(const __grid_constant__ TcGuArgs a) {
    extern __shared__ uint8_t gu_raw[];
    char* sm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(gu_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_nact;
    DecDims q{a.d, a.F, a.Fs, G, a.max_rb, 0, 0, 0, true, false, false};
    const DecSmem L = dec_smem(q);
    ring_setup(sm, L, &a.tm_s, &a.tm_r);
    const int Gr = gridDim.x, b = blockIdx.x;
    {   // the shared expert depends on x alone: it runs before the wait for the router
        const int R = a.Fs / 8;
        const int lo = (int)((int64_t)b * R / Gr), hi = (int)((int64_t)(b + 1) * R / Gr);
        gu_tables<G>(a, true, lo, hi - lo, sm, L);
        gu_prologue<G>(a, true, hi - lo, sm, L);
        stage_x<G>(a.x, a.d, sm, L);
        gu_consume<G>(a, true, hi - lo, sm, L);
        gu_reduce<G>(a, true, lo, hi - lo, sm, L);
    }
    pdl_wait();
    pdl_trigger();  // dependents launch once the routing is complete
    // the routing into shared memory: the schedule, then each group's H row
    int* ssched = reinterpret_cast<int*>(sm + L.sched);
    int* srow = reinterpret_cast<int*>(sm + L.srow);
    for (int y = threadIdx.x; y < a.n_route_max; y += blockDim.x) {
        const int e = ld_cg_i32(a.sched + y);
        ssched[y] = e;
        srow[y] = ld_cg_i32(a.offsets + e);
    }
    if (threadIdx.x < 32) {
        int n;
        if (a.n_active) {
            n = ld_cg_i32(a.n_active);
        } else {
            n = 0;
            for (int y0 = 0; y0 < a.n_route_max; y0 += 32) {
                const int y = y0 + threadIdx.x;
                bool act = false;
                if (y < a.n_route_max) {
                    const int e = ld_cg_i32(a.sched + y);
                    act = ld_cg_i32(a.offsets + e + 1) > ld_cg_i32(a.offsets + e);
                }
                n += __popc(__ballot_sync(0xffffffffu, act));
            }
        }
        if (threadIdx.x == 0) s_nact = min(n, a.n_route_max);
    }
    __syncthreads();
    const int64_t R = (int64_t)s_nact * (a.F / 8);
    const int64_t lo = (int64_t)b * R / Gr, hi = (int64_t)(b + 1) * R / Gr;
    gu_tables<G>(a, false, lo, (int)(hi - lo), sm, L);
    gu_prologue<G>(a, false, (int)(hi - lo), sm, L);
    gu_consume<G>(a, false, (int)(hi - lo), sm, L);
    gu_reduce<G>(a, false, lo, (int)(hi - lo), sm, L);
}

// ---------------------------------------------------------------- down
struct TcDnArgs {
    const uint16_t* H;
    int ldh;
    int d, T, k, F, Fs;
    const int32_t* offsets;
    const int32_t* sched;
    const uint8_t* q_r;
    const __half* s_r;
    const uint8_t* q_sh;
    const __half* s_sh;
    float* Y;                  // per-row output when out is null
    int n_route_max;
    const int32_t* n_active;
    const float* topk_w;       // fused combine when out is non-null
    const int32_t* pos;
    const uint16_t* residual;  // nullable; may alias out
    uint16_t* out;
    int max_groups;            // 1 + routed groups, the tables' capacity
    int max_ch;                // output channels of a CTA, at most
};

// A warp's down units: 16-channel block rb and span pair `pair` of the groups
// ys, ys + wpc, ...  Combos (block, pair): nc = nrb * PF; warp w takes combo
// w % nc (16 / nc warps per combo).  A group narrower than the pair has no
// unit there.
struct DnWarp {
    int c_lo, c_hi, nrb, nc, wpc, rb, pair, ys, n;
};
__device__ __forceinline__ DnWarp dn_warp(const TcDnArgs& a, const DecSmem& L, int ngr) {
    DnWarp W;
    const int warp = threadIdx.x >> 5;
    const int Gr = gridDim.x, b = blockIdx.x;
    W.c_lo = (int)((int64_t)b * a.d / Gr);
    W.c_hi = (int)((int64_t)(b + 1) * a.d / Gr);
    W.nrb = (W.c_hi - W.c_lo + 15) / 16;
    W.nc = W.nrb * L.PF;
    W.wpc = kTcWarps / W.nc;
    const int combo = warp % W.nc;
    W.rb = combo / L.PF;
    W.pair = combo % L.PF;
    W.ys = warp / W.nc;
    W.n = (warp < W.nc * W.wpc && W.ys < ngr) ? (ngr - W.ys + W.wpc - 1) / W.wpc : 0;
    return W;
}

// Request unit i (group ys + i * wpc) into ring slot `slot`: each lane copies
// the pieces of its two rows it will read, and their scales (cp.async; a
// masked row or a group without this pair copies nothing).
template <int G>
__device__ __forceinline__ void dn_issue(const TcDnArgs& a, char* sm, const DecSmem& L,
                                         const DnWarp& W, int i, int slot) {
    constexpr int NG = 128 / G, PB = G / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int y = W.ys + i * W.wpc;
    const int e = reinterpret_cast<const int*>(sm + L.qe)[y];
    const int K = e < 0 ? a.Fs : a.F;
    const uint64_t pol = l2_evict_first();
    if (256 * W.pair < K) {
        const int64_t rowb = K / 2;
        const int ng = K / G;
        const uint8_t* qb = (e < 0 ? a.q_sh : a.q_r + (int64_t)e * a.d * rowb) + 128 * W.pair;
        const __half* sb = (e < 0 ? a.s_sh : a.s_r + (int64_t)e * a.d * ng) + 2 * NG * W.pair;
        const uint32_t wdst = smem_u32(sm + L.wring) + (uint32_t)((warp * L.R + slot) * kTile);
        const uint32_t sdst = smem_u32(sm + L.sring) + (uint32_t)(((warp * L.R + slot) * 32 + lane) * 8 * NG);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int c = W.c_lo + 16 * W.rb + g + 8 * r;
            if (c >= W.c_hi) continue;
            const uint8_t* row = qb + c * rowb;
#pragma unroll
            for (int sp = 0; sp < 2; ++sp)
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    const int piece = (r * 2 + sp) * NG + j;
                    cp_async<PB>(wdst + (uint32_t)((piece * 32 + lane) * PB),
                                 row + 64 * sp + j * (G / 2) + t * PB, pol);
                }
            cp_async_ca<4 * NG>(sdst + 4 * NG * r, sb + (int64_t)c * ng);
        }
    }
    cp_commit();
}

template <int G>
__device__ __forceinline__ void dn_prologue(const TcDnArgs& a, int ngr, char* sm, const DecSmem& L) {
    const DnWarp W = dn_warp(a, L, ngr);
    for (int i = 0; i < W.n && i < L.R; ++i) dn_issue<G>(a, sm, L, W, i, i);
}

// Consume the warp's units (the first min(R, n) already requested; H staged),
// refilling each slot once read.
template <int G>
__device__ __noinline__ void dn_consume(const TcDnArgs& a, int ngr, char* sm, const DecSmem& L) {
    constexpr int NG = 128 / G, PB = G / 8, WPG = G / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const DnWarp W = dn_warp(a, L, ngr);
    const int Fm = a.F > a.Fs ? a.F : a.Fs;
    const uint32_t hfrag = smem_u32(sm + L.hfrag);
    const float* hcin = reinterpret_cast<const float*>(sm + L.hcin);
    float* part = reinterpret_cast<float*>(sm + L.dpart);
    const int* qe = reinterpret_cast<const int*>(sm + L.qe);
    for (int i = 0; i < W.n; ++i) {
        const int slot = i % L.R;
        ring_wait_copies(i, W.n, L.R);
        const int y = W.ys + i * W.wpc;
        const int K = qe[y] < 0 ? a.Fs : a.F;
        if (256 * W.pair < K) {
            const uint32_t wsrc = smem_u32(sm + L.wring) + (uint32_t)((warp * L.R + slot) * kTile);
            const uint32_t ssrc = smem_u32(sm + L.sring) + (uint32_t)(((warp * L.R + slot) * 32 + lane) * 8 * NG);
            TcUnit<G> U;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                uint32_t* w = r ? U.w1 : U.w0;
                uint32_t* s = r ? U.s1 : U.s0;
                const bool live = W.c_lo + 16 * W.rb + g + 8 * r < W.c_hi;
#pragma unroll
                for (int sp = 0; sp < 2; ++sp)
#pragma unroll
                    for (int j = 0; j < NG; ++j) {
                        const int piece = (r * 2 + sp) * NG + j;
                        const uint32_t addr = wsrc + (uint32_t)((piece * 32 + lane) * PB);
                        uint32_t* dd = w + 4 * sp + j * WPG;
                        if constexpr (PB == 16) {
                            const uint4 v = lds_v4(addr);
                            dd[0] = v.x;
                            dd[1] = v.y;
                            dd[2] = v.z;
                            dd[3] = v.w;
                        } else if constexpr (PB == 8) {
                            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(dd[0]), "=r"(dd[1]) : "r"(addr));
                        } else {
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(dd[0]) : "r"(addr));
                        }
                        if (!live)
#pragma unroll
                            for (int z = 0; z < WPG; ++z) dd[z] = 0u;
                    }
#pragma unroll
                for (int q = 0; q < NG; ++q) {
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(s[q]) : "r"(ssrc + 4 * NG * r + 4 * q));
                    if (!live) s[q] = 0u;
                }
            }
            float p0 = 0.f, p1 = 0.f;
            tc_mma<G>(U, hfrag + (uint32_t)(y * L.Smax * 256), W.pair, t,
                      hcin + y * (Fm / G) + 2 * NG * W.pair, p0, p1);
            if (t == 0) {
                float* pp = part + ((y * L.nrb_max + W.rb) * L.PF + W.pair) * 16;
                pp[g] = p0;
                pp[8 + g] = p1;
            }
        }
        __syncwarp();  // every lane has read the slot
        if (i + L.R < W.n) dn_issue<G>(a, sm, L, W, i + L.R, slot);
    }
}

// Each group's channel values (pairs summed in order, rescaled), then Y rows
// or the fused combine in the order of moe_combine_shared: routed slots
// j = 0..k-1, then the shared expert, then the residual.  coh: topk_w / pos
// were written earlier by this kernel.
__device__ __noinline__ void dn_finish(const TcDnArgs& a, int ngr, char* sm, const DecSmem& L,
                                       bool coh) {
    __syncthreads();
    const float* part = reinterpret_cast<const float*>(sm + L.dpart);
    float* yc = reinterpret_cast<float*>(sm + L.yc);
    const int* hrow = reinterpret_cast<const int*>(sm + L.hrow);
    const int* yrow = reinterpret_cast<const int*>(sm + L.yrow);
    const int* sigma = misc(sm, L)->sigma;
    const int Gr = gridDim.x, b = blockIdx.x;
    const int c_lo = (int)((int64_t)b * a.d / Gr), c_hi = (int)((int64_t)(b + 1) * a.d / Gr);
    const int nch = c_hi - c_lo;
    for (int i = threadIdx.x; i < ngr * nch; i += blockDim.x) {
        const int y = i / nch, c = i - y * nch;
        const int cb = c >> 4, r = c & 15;
        const int py = (y == 0 ? a.Fs : a.F) / 256;
        float v = 0.f;
        for (int q = 0; q < py; ++q) v += part[((y * L.nrb_max + cb) * L.PF + q) * 16 + r];
        v *= ldexpf(1.0f, 133 - sigma[y]);
        if (a.out)
            yc[y * L.nrb_max * 16 + c] = v;
        else
            a.Y[(int64_t)hrow[y] * a.d + c_lo + c] = v;
    }
    if (!a.out) return;
    __syncthreads();
    for (int c = threadIdx.x; c < nch; c += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < a.k; ++j) {
            const int p = coh ? __ldcg(a.pos + j) : __ldg(a.pos + j);
            const float w = coh ? __ldcg(a.topk_w + j) : __ldg(a.topk_w + j);
            acc = fmaf(w, yc[yrow[p] * L.nrb_max * 16 + c], acc);
        }
        acc += yc[c];
        if (a.residual) acc = __uint_as_float((uint32_t)a.residual[c_lo + c] << 16) + acc;
        a.out[c_lo + c] = float_to_bf16_bits(acc);
    }
}

template <int G>
__device__ __forceinline__ void stage_h(const TcDnArgs& a, int ngr, char* sm, const DecSmem& L, bool coh) {
    const int Fm = a.F > a.Fs ? a.F : a.Fs;
    Misc* m = misc(sm, L);
    stage_rows<G>(a.H, a.ldh, reinterpret_cast<const int*>(sm + L.hrow), ngr, a.Fs, a.F,
                  reinterpret_cast<uint4*>(sm + L.hfrag), L.Smax * 16, reinterpret_cast<float*>(sm + L.hcin),
                  Fm / G, m->sigma, reinterpret_cast<float*>(sm + L.htmp), Fm / 8, m->mx, coh);
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) down_tc_kernel(const TcDnArgs a) {
    extern __shared__ uint8_t dn_raw[];
    char* sm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(dn_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_nact;
    const int rows = a.T * a.k + a.T;
    DecDims q{a.d, a.F, a.Fs, G, 0, a.max_groups, a.max_ch, rows, false, true, false};
    const DecSmem L = dec_smem(q);
    int* qe = reinterpret_cast<int*>(sm + L.qe);
    int* hrow = reinterpret_cast<int*>(sm + L.hrow);
    int* yrow = reinterpret_cast<int*>(sm + L.yrow);
    pdl_trigger();
    if (threadIdx.x < 32) {  // the routing is complete when this kernel starts
        int n;
        if (a.n_active) {
            n = ld_cg_i32(a.n_active);
        } else {
            n = 0;
            for (int y0 = 0; y0 < a.n_route_max; y0 += 32) {
                const int y = y0 + threadIdx.x;
                bool act = false;
                if (y < a.n_route_max) {
                    const int e = ld_cg_i32(a.sched + y);
                    act = ld_cg_i32(a.offsets + e + 1) > ld_cg_i32(a.offsets + e);
                }
                n += __popc(__ballot_sync(0xffffffffu, act));
            }
        }
        if (threadIdx.x == 0) s_nact = min(n, a.max_groups - 1);
    }
    __syncthreads();
    const int ngr = 1 + s_nact;
    for (int y = threadIdx.x; y < ngr; y += blockDim.x) {
        const int e = y == 0 ? -1 : ld_cg_i32(a.sched + y - 1);
        qe[y] = e;
        hrow[y] = e < 0 ? a.T * a.k : ld_cg_i32(a.offsets + e);
    }
    for (int r = threadIdx.x; r < rows; r += blockDim.x) yrow[r] = 0;
    __syncthreads();
    for (int y = threadIdx.x; y < ngr; y += blockDim.x) yrow[hrow[y]] = y;
    dn_prologue<G>(a, ngr, sm, L);
    pdl_wait();  // H is written by the gate+up kernel
    stage_h<G>(a, ngr, sm, L, false);
    dn_consume<G>(a, ngr, sm, L);
    dn_finish(a, ngr, sm, L, false);
}

// ---------------------------------------------------------------------------
// The whole single-token step in one launch: router, descriptors, gate+up
// SwiGLU (routed and shared) and down with the fused combine.
//
// With three kernels the step's time went mostly to hand-offs: the router's
// top-k ran in its last CTA after a grid-wide arrival count, the gate+up
// CTAs could not start beside the router's CTAs, and the down kernel waited
// for the slowest gate+up CTA before staging H.  Here one persistent CTA per
// SM (a cooperative launch, so every CTA is resident) runs:
//   1. the shared expert's first gate+up tiles and this CTA's router-weight
//      chunks are requested first (they depend on x alone); x is staged and
//      the split-K logit partials computed while they are in flight;
//   2. grid barrier; every CTA then reads all logit partials and takes the
//      top-k itself: the selection is deterministic, so every CTA holds the
//      same routing with no further exchange (CTA 0 writes the descriptor
//      outputs);
//   3. the routed gate+up tiles; a warp done with its tiles requests its
//      first down-projection units into its ring;
//   4. grid barrier (every H row written); the down units, the per-group
//      channel sums and the combine, as in the separate kernels.
// The arithmetic of every step is that of the separate router, gate+up and
// down kernels, so the results are bit-identical to the step-by-step calls.
struct StepArgs {
    TcGuArgs gu;
    TcDnArgs dn;  // dn.topk_w / dn.pos are the outputs written by this kernel
    const float* W_r;
    const float* bias;
    int E, ksplit;
    float* partial;  // router logit partials [ksplit][E]
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* pos;
    int32_t* sched;
};

// Grid-wide barrier on a 64-bit arrival counter in the workspace header
// (done[2..3]).  Every CTA is resident (cooperative launch).  The counter only
// grows: a launch adds 2 * G (two barriers of G CTAs), so with c0 the value a
// CTA reads at kernel start (before its first arrival; fewer than G arrivals
// of this launch can precede it), base = c0 - c0 % (2G) and barrier j (1, 2)
// opens when the counter reaches base + j * G.  An arrival is one release
// add, the wait an acquire poll: about one L2 round trip after the last
// arrival.  A wait that gives up records kErrWaitTimeout and raises the CTA's
// abort flag (the counter is then out of step: zero the workspace again).
__device__ __forceinline__ unsigned long long* barrier_count(WsHeader* h) {
    return reinterpret_cast<unsigned long long*>(&h->done[2]);
}
__device__ __forceinline__ unsigned long long barrier_base(WsHeader* h) {
    unsigned long long c;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(c) : "l"(barrier_count(h)) : "memory");
    return c - c % (2ull * gridDim.x);
}
__device__ __noinline__ void grid_sync(WsHeader* h, unsigned long long target, volatile int* abort_flag) {
    __syncthreads();
    if (threadIdx.x == 0 && !*abort_flag) {
        unsigned long long* cnt = barrier_count(h);
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
        if (v < target) {
            const uint64_t t0 = globaltimer();
            for (uint32_t i = 1;; ++i) {
                asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
                if (v >= target) break;
                if ((i & 63u) == 0 && globaltimer() - t0 > kWaitNs) {
                    *abort_flag = 1;
                    record_error(h, kErrWaitTimeout);
                    break;
                }
            }
        }
    }
    __syncthreads();
}

// Split-K logit partials of this CTA's units (e, kc): a warp's first unit's
// W_r chunk was copied into buf + warp * 2 KB; the arithmetic of
// router_gemv_warp for one token.
__device__ __noinline__ void router_partials(const StepArgs& a, const char* buf) {
    const TcGuArgs& gu = a.gu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = gu.d, E = a.E, kchunk = d / a.ksplit, nvec = kchunk / 128;
    const int U = E * a.ksplit, Gr = gridDim.x, b = blockIdx.x;
    const int u0 = (int)((int64_t)b * U / Gr), u1 = (int)((int64_t)(b + 1) * U / Gr);
    for (int u = u0 + warp, it = 0; u < u1; u += kTcWarps, ++it) {
        const int e = u / a.ksplit, kc = u - e * a.ksplit;
        float4 wv[4];
        if (it == 0) {
            const float4* src = reinterpret_cast<const float4*>(buf + warp * 2048);
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] = i < nvec ? src[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {  // a CTA with more units than warps: the rest from global memory
#pragma unroll
            for (int i = 0; i < 4; ++i)
                wv[i] = i < nvec ? __ldg(reinterpret_cast<const float4*>(a.W_r + (int64_t)e * d + kc * kchunk) + lane + 32 * i)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const uint2* xr = reinterpret_cast<const uint2*>(gu.x + kc * kchunk);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < nvec) {
                const uint2 xv = __ldg(xr + lane + 32 * i);
                acc = fmaf(bf16_lo(xv.x), wv[i].x, acc);
                acc = fmaf(bf16_hi(xv.x), wv[i].y, acc);
                acc = fmaf(bf16_lo(xv.y), wv[i].z, acc);
                acc = fmaf(bf16_hi(xv.y), wv[i].w, acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) a.partial[(int64_t)kc * E + e] = acc;
    }
}

// The routing of the single token, identically in every CTA: keys, top-k by
// warp bitonic sorts and candidate ranks, weights normalised by the selected
// scores in selection order (the arithmetic of router_topk_warp), then the
// chosen ids ascending with their slots (descriptor row r is the r-th
// smallest id).  CTA 0 writes the outputs.
__device__ __noinline__ void route_token(const StepArgs& a, char* sm, const DecSmem& L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int E = a.E, k = a.gu.k;
    float* ck = reinterpret_cast<float*>(sm + L.cand);
    int* ce = reinterpret_cast<int*>(ck + kTcWarps * 32);
    float* cs = reinterpret_cast<float*>(ce + kTcWarps * 32);
    int* sel_e = reinterpret_cast<int*>(cs + kTcWarps * 32);
    float* sel_s = reinterpret_cast<float*>(sel_e + 32);
    int* r_sorted = reinterpret_cast<int*>(sm + L.route);
    const int nc = min(k + 1, 32);
    const int nw = (E + 31) / 32;  // warps holding experts
    if (warp < nw) {
        float key = -INFINITY, sc = 0.f;
        int ee = 0x7fffffff;
        if (tid < E) {
            const float l = router_logit(a.partial, a.ksplit, 1, E, 0, tid);
            sc = 1.0f / (1.0f + expf(-l));
            key = sc + __ldg(a.bias + tid);
            if (key != key) key = -INFINITY;
            ee = tid;
        }
        warp_bitonic<true>(key, ee, sc, lane);
        if (lane < nc) {
            ck[warp * nc + lane] = key;
            ce[warp * nc + lane] = ee;
            cs[warp * nc + lane] = sc;
        }
    }
    __syncthreads();
    const int ncand = nc * nw;
    if (tid < ncand) {
        const float key = ck[tid];
        const int e = ce[tid];
        if (e < E) {
            int rank = 0;
#pragma unroll 4
            for (int j = 0; j < ncand; ++j) {
                const int e2 = ce[j];
                rank += e2 < E && router_better(ck[j], e2, key, e);
            }
            if (rank < k) {
                sel_e[rank] = e;
                sel_s[rank] = cs[tid];
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += sel_s[r];
        int e = 0x7fffffff;
        float slot = 0.f;
        if (lane < k) {
            e = sel_e[lane];
            const float w = __fdiv_rn(sel_s[lane], sum);
            slot = (float)lane;
            if (blockIdx.x == 0) {
                a.topk_idx[lane] = e;
                a.topk_w[lane] = w;
            }
        }
        float dummy = 0.f;
        warp_bitonic<false>(dummy, e, slot, lane);
        if (lane < k) {
            const int j = (int)slot;
            r_sorted[lane] = e;
            if (blockIdx.x == 0) {
                a.perm[lane] = j;
                a.pos[j] = lane;
                a.sched[lane] = e;
            }
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {  // the remaining descriptor outputs
        for (int e = tid; e < E; e += blockDim.x) {
            int lb = 0;  // chosen ids below e
            while (lb < k && r_sorted[lb] < e) ++lb;
            const bool chosen = lb < k && r_sorted[lb] == e;
            a.counts[e] = chosen ? 1 : 0;
            a.offsets[e] = lb;
            if (!chosen) a.sched[k + (e - lb)] = e;
        }
        if (tid == 0) {
            a.offsets[E] = k;
            a.gu.hdr->n_active = k;
        }
    }
    // gate+up groups: the chosen experts ascending, H row y; down groups: the
    // shared expert (H row k), then the chosen experts
    int* ssched = reinterpret_cast<int*>(sm + L.sched);
    int* srow = reinterpret_cast<int*>(sm + L.srow);
    int* qe = reinterpret_cast<int*>(sm + L.qe);
    int* hrow = reinterpret_cast<int*>(sm + L.hrow);
    int* yrow = reinterpret_cast<int*>(sm + L.yrow);
    if (tid < k) {
        ssched[tid] = r_sorted[tid];
        srow[tid] = tid;
        qe[1 + tid] = r_sorted[tid];
        hrow[1 + tid] = tid;
        yrow[tid] = 1 + tid;
    }
    if (tid == 0) {
        qe[0] = -1;
        hrow[0] = k;
        yrow[k] = 0;
    }
    __syncthreads();
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) decode_step_kernel(const __grid_constant__ StepArgs a) {
    extern __shared__ uint8_t st_raw[];
    char* sm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(st_raw) + 1023) & ~uintptr_t(1023));
    const TcGuArgs& gu = a.gu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = gu.k, d = gu.d;
    const int Gr = gridDim.x, b = blockIdx.x;
    DecDims q{d, gu.F, gu.Fs, G, gu.max_rb, 1 + k, a.dn.max_ch, k + 1, true, true, true};
    const DecSmem L = dec_smem(q);
    __shared__ unsigned long long s_base;
    if (threadIdx.x == 0) s_base = barrier_base(gu.hdr);
    ring_setup(sm, L, &gu.tm_s, &gu.tm_r);
    volatile int* abort_flag = &misc(sm, L)->abort;

    // 1. the shared expert's first gate+up tiles, then this CTA's router
    //    weight chunks (a warp's first unit, kchunk floats, into the down
    //    phase's work area, unused until barrier 2), then x
    const int R = gu.Fs / 8;
    const int lo = (int)((int64_t)b * R / Gr), hi = (int)((int64_t)(b + 1) * R / Gr);
    gu_tables<G>(gu, true, lo, hi - lo, sm, L);
    gu_prologue<G>(gu, true, hi - lo, sm, L);
    char* wbuf = sm + L.hfrag;
    {
        const int kchunk = d / a.ksplit, U = a.E * a.ksplit;
        const int u = (int)((int64_t)b * U / Gr) + warp;
        if (u < (int)((int64_t)(b + 1) * U / Gr)) {
            const int e = u / a.ksplit, kc = u - e * a.ksplit;
            const float* src = a.W_r + (int64_t)e * d + kc * kchunk;
            const uint64_t pol = l2_evict_first();
            for (int i = lane; i < kchunk / 4; i += 32)
                cp_async<16>(smem_u32(wbuf + warp * 2048 + 16 * i), src + 4 * i, pol);
        }
        cp_commit();
    }
    stage_x<G>(gu.x, d, sm, L);
    cp_wait<0>();
    __syncwarp();
    router_partials(a, wbuf);
    gu_consume<G>(gu, true, hi - lo, sm, L);
    gu_reduce<G>(gu, true, lo, hi - lo, sm, L);

    // 2. every CTA's partials are written; the routing, identically in every CTA
    grid_sync(gu.hdr, s_base + Gr, abort_flag);
    route_token(a, sm, L);

    // 3. the routed gate+up; a warp through its tiles requests its first down units
    {
        const int64_t Rr = (int64_t)k * (gu.F / 8);
        const int64_t rlo = (int64_t)b * Rr / Gr, rhi = (int64_t)(b + 1) * Rr / Gr;
        gu_tables<G>(gu, false, rlo, (int)(rhi - rlo), sm, L);
        gu_prologue<G>(gu, false, (int)(rhi - rlo), sm, L);
        gu_consume<G>(gu, false, (int)(rhi - rlo), sm, L);
        dn_prologue<G>(a.dn, k + 1, sm, L);
        gu_reduce<G>(gu, false, rlo, (int)(rhi - rlo), sm, L);
    }

    // 4. every H row is written; the down projection and the combine
    grid_sync(gu.hdr, s_base + 2ull * Gr, abort_flag);
    stage_h<G>(a.dn, k + 1, sm, L, true);
    dn_consume<G>(a.dn, k + 1, sm, L);
    dn_finish(a.dn, k + 1, sm, L, true);
}

// ---------------------------------------------------------------- host side
template <typename Kern, typename Args>
cudaError_t launch_tc(Kern kern, int grid, size_t smem, bool pdl, bool coop, cudaStream_t st,
                      const Args& args) {
    cudaError_t err = ensure_dynamic_smem((const void*)kern, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (coop) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (pdl || coop) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

constexpr size_t kTcMaxSmem = 227 * 1024;

int gu_max_rb(const moe_dims_t& d, int grid) {
    const int64_t routed = (int64_t)std::min(d.E, d.T * d.k) * (d.F / 8);
    const int64_t shared = d.F_s / 8;
    return (int)((std::max(routed, shared) + grid - 1) / grid);
}
int dn_grid(const moe_dims_t& d) { return std::min(sm_count(), d.d / 8); }
int dn_max_ch(const moe_dims_t& d, int grid) { return (d.d + grid - 1) / grid; }
int dn_max_groups(const moe_dims_t& d) { return 1 + std::min(d.E, d.T * d.k); }

DecDims gu_dims(const moe_dims_t& d) {
    return DecDims{d.d, d.F, d.F_s, d.group, gu_max_rb(d, sm_count()), 0, 0, 0, true, false, false};
}
DecDims dn_dims(const moe_dims_t& d) {
    return DecDims{d.d, d.F, d.F_s, d.group, 0, dn_max_groups(d), dn_max_ch(d, dn_grid(d)),
                   d.T * d.k + d.T, false, true, false};
}
DecDims step_dims(const moe_dims_t& d) {
    const int grid = sm_count();
    return DecDims{d.d, d.F, d.F_s, d.group, gu_max_rb(d, grid), 1 + d.k, dn_max_ch(d, grid),
                   d.k + 1, true, true, true};
}

bool make_gu_map(CUtensorMap* m, const void* q, int d, int Fg, int experts) {
    // {d/2 bytes, 8 rows, gate/up, row blocks of 8, experts}: one box = 8 gate
    // rows and their 8 up rows, 128 bytes of K each
    const uint64_t rowb = d / 2;
    const cuuint64_t dims[5] = {rowb, 8, 2, (cuuint64_t)Fg / 8, (cuuint64_t)experts};
    const cuuint64_t strides[4] = {rowb, (cuuint64_t)Fg * rowb, 8 * rowb, 2 * (cuuint64_t)Fg * rowb};
    const cuuint32_t box[5] = {128, 8, 2, 1, 1};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 5, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

void fill_gu(TcGuArgs& g, const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
             const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H, const int32_t* n_active,
             WsHeader* hdr) {
    g.x = x;
    g.d = d.d;
    g.T = d.T;
    g.k = d.k;
    g.F = d.F;
    g.Fs = d.F_s;
    g.offsets = offsets;
    g.sched = sched;
    g.s_r = reinterpret_cast<const __half*>(Wgu.s);
    g.s_sh = reinterpret_cast<const __half*>(Wgu_s.s);
    g.H = H;
    g.ldh = std::max(d.F, d.F_s);
    g.n_route_max = std::min(d.E, d.T * d.k);
    g.n_active = n_active;
    g.hdr = hdr;
    g.max_rb = gu_max_rb(d, sm_count());
}

void fill_dn(TcDnArgs& n, const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
             const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y, const int32_t* n_active,
             const float* topk_w, const int32_t* pos, const uint16_t* residual, uint16_t* out,
             int grid) {
    n.H = H;
    n.ldh = std::max(d.F, d.F_s);
    n.d = d.d;
    n.T = d.T;
    n.k = d.k;
    n.F = d.F;
    n.Fs = d.F_s;
    n.offsets = offsets;
    n.sched = sched;
    n.q_r = Wd.q;
    n.s_r = reinterpret_cast<const __half*>(Wd.s);
    n.q_sh = Wd_s.q;
    n.s_sh = reinterpret_cast<const __half*>(Wd_s.s);
    n.Y = Y;
    n.n_route_max = std::min(d.E, d.T * d.k);
    n.n_active = n_active;
    n.topk_w = topk_w;
    n.pos = pos;
    n.residual = residual;
    n.out = out;
    n.max_groups = dn_max_groups(d);
    n.max_ch = dn_max_ch(d, grid);
}

size_t smem_of(const DecDims& q) { return dec_smem(q).total + 1024; }  // + alignment slack

}  // namespace

bool tc_decode_supported(const moe_dims_t& d) {
    if (d.T != 1 || d.k > 32 || std::min(d.E, d.T * d.k) > kTcMaxRoute || sm_count() <= 0)
        return false;
    // whole span pairs (256 K elements) everywhere; one pair per warp at most
    if (d.d % 256 || d.F % 256 || d.F_s % 256 || d.d > 4096 || std::max(d.F, d.F_s) > 8192)
        return false;
    if (dn_max_ch(d, dn_grid(d)) > 32) return false;
    return smem_of(gu_dims(d)) <= kTcMaxSmem && smem_of(dn_dims(d)) <= kTcMaxSmem;
}

bool tc_weights_ok(moe_w4_t a, moe_w4_t b) {
    // 16-byte aligned bytes and scales (vector and cp.async copies)
    auto ok = [](moe_w4_t w) {
        return reinterpret_cast<uintptr_t>(w.q) % 16 == 0 && reinterpret_cast<uintptr_t>(w.s) % 16 == 0;
    };
    return ok(a) && ok(b);
}

cudaError_t launch_gateup_tc(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H,
                             const int32_t* n_active, WsHeader* hdr, bool pdl, cudaStream_t st) {
    TcGuArgs a;
    memset(&a, 0, sizeof(a));
    if (!make_gu_map(&a.tm_r, Wgu.q, d.d, d.F, d.E) || !make_gu_map(&a.tm_s, Wgu_s.q, d.d, d.F_s, 1))
        return cudaErrorInvalidValue;
    fill_gu(a, x, d, offsets, sched, Wgu, Wgu_s, H, n_active, hdr);
    const size_t smem = smem_of(gu_dims(d));
    const int grid = sm_count();
    switch (d.group) {
        case 32: return launch_tc(gateup_tc_kernel<32>, grid, smem, pdl, false, st, a);
        case 64: return launch_tc(gateup_tc_kernel<64>, grid, smem, pdl, false, st, a);
        default: return launch_tc(gateup_tc_kernel<128>, grid, smem, pdl, false, st, a);
    }
}

cudaError_t launch_down_tc(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                           const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                           const int32_t* n_active, const float* topk_w, const int32_t* pos,
                           const uint16_t* residual, uint16_t* out, bool pdl, cudaStream_t st) {
    TcDnArgs a;
    memset(&a, 0, sizeof(a));
    const int grid = dn_grid(d);
    fill_dn(a, H, d, offsets, sched, Wd, Wd_s, Y, n_active, topk_w, pos, residual, out, grid);
    const size_t smem = smem_of(dn_dims(d));
    switch (d.group) {
        case 32: return launch_tc(down_tc_kernel<32>, grid, smem, pdl, false, st, a);
        case 64: return launch_tc(down_tc_kernel<64>, grid, smem, pdl, false, st, a);
        default: return launch_tc(down_tc_kernel<128>, grid, smem, pdl, false, st, a);
    }
}

bool step_supported(const moe_dims_t& d) {
    // one expert per thread for the routing, k + 1 candidates per warp; the
    // router weight chunks (16 warps x at most 2 KB) are staged in the H area
    if (!tc_decode_supported(d) || d.E > kTcThreads || d.k + 1 > 32) return false;
    const int ks = (d.d % 512 == 0) ? d.d / 512 : d.d / 256;
    if ((d.d / ks) * 4 > 2048) return false;
    const DecSmem L = dec_smem(step_dims(d));
    if (L.total + 1024 > kTcMaxSmem) return false;
    if ((size_t)kTcWarps * 2048 > L.qe - L.hfrag) return false;  // the down work area
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return false;
    return true;
}

cudaError_t launch_decode_step(const uint16_t* x, const float* W_r, const float* bias,
                               const moe_dims_t& d, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                               int32_t* sched, float* logits, int ksplit, moe_w4_t Wgu, moe_w4_t Wd,
                               moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* H, const uint16_t* residual,
                               uint16_t* out, WsHeader* hdr, cudaStream_t st) {
    StepArgs a;
    memset(&a, 0, sizeof(a));
    const int grid = sm_count();
    if (!make_gu_map(&a.gu.tm_r, Wgu.q, d.d, d.F, d.E) ||
        !make_gu_map(&a.gu.tm_s, Wgu_s.q, d.d, d.F_s, 1))
        return cudaErrorInvalidValue;
    fill_gu(a.gu, x, d, offsets, sched, Wgu, Wgu_s, H, nullptr, hdr);
    a.gu.n_route_max = d.k;
    fill_dn(a.dn, H, d, offsets, sched, Wd, Wd_s, nullptr, nullptr, topk_w, pos, residual, out, grid);
    a.dn.max_groups = 1 + d.k;
    a.dn.n_route_max = d.k;
    a.W_r = W_r;
    a.bias = bias;
    a.E = d.E;
    a.ksplit = ksplit;
    a.partial = logits;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.pos = pos;
    a.sched = sched;
    const size_t smem = smem_of(step_dims(d));
    switch (d.group) {
        case 32: return launch_tc(decode_step_kernel<32>, grid, smem, false, true, st, a);
        case 64: return launch_tc(decode_step_kernel<64>, grid, smem, false, true, st, a);
        default: return launch_tc(decode_step_kernel<128>, grid, smem, false, true, st, a);
    }
}

}  // namespace moe
