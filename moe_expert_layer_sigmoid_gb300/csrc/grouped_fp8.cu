// W8A8 expert projections: a persistent grouped fp8 GEMM on the tcgen05
// tensor cores (kind::f8f6f4, E4M3 x E4M3, fp32 accumulators in TMEM), with
// the kernels that quantise its operands.
//
// The pages' GB10 work adds W4A8 and W8A8 grouped MoE paths next to the W4A16
// one, W8A8 with near-lossless fp8 weights and unchanged argmax
// (thewafflehaus/FFAI PR #72, Nemotron-H section), and quantises FP8
// projections with one scale per weight channel and one per activation row,
// folded in after the GEMM (same PR, the per-channel FP8 commit).  On GB10
// fp8 activations measured slower than W4A16 at tiny-expert shapes; on
// sm_103a the fp8 tensor rate is twice the bf16 one and, with per-row scales,
// the kernel needs no dequantisation and no per-group epilogue: the whole K
// accumulates in TMEM and the scales are applied once per tile.
//
// Numerics: E4M3 codes (round to nearest even, saturate to +-448); a weight row
// w has s_w = absmax / 448 and codes e4m3(w / s_w); an activation row x (a
// token's bf16 x for gate+up, an H row for down) has a = absmax / 448 and codes
// e4m3(x / a), both divisions in fp32.  Each product of two codes is exact; a
// projection is v = (acc * a) * s_w with acc the fp32 sum over K.
//
// Tiles come from the descriptors, as on the W4A16 grouped path but with up to
// 256 tokens: M = 128 weight rows (gate+up: 64 gate rows and their 64 up rows
// interleaved in blocks of 16, so a gate row and its up row are 16 lanes apart
// in one warp; down: 128 output channels), N = up to 256 tokens of one expert,
// K in stages of 128 bytes.  Per stage one TMA box of weight codes (128 x 128
// B) and one of activation codes (32, 64, 128 or 256 rows x 128 B, the
// smallest that holds the tile's tokens), both with 128-byte swizzle, the UMMA
// K-major canonical layout; four MMAs of K = 32 per stage.  The kernel is
// bound by the bytes each SM has in flight over their latency, so 256-token
// tiles (twice the flops per weight byte of 128-token ones) go faster.
//
// Warp roles (14 warps, one CTA per SM): warp 0 TMA producer; warp 1 allocates
// TMEM and issues the MMAs; warps 2-13 the epilogue, three per TMEM lane quarter
// (each reads the 32 lanes of its quarter; the warp of part p takes the
// 32-column chunks p, p + 3, ...).  Two 256-column accumulators let the
// epilogue of one tile overlap the MMAs of the next.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include "tma.cuh"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kF8Warps = 14;
constexpr int kF8EpiPerQuarter = (kF8Warps - 2) / 4;
constexpr int kF8Threads = kF8Warps * 32;
constexpr int kF8EpiWarp0 = 2;
constexpr int kF8Stages = 4;
constexpr int kF8K = 128;                    // K bytes (= elements) per stage
constexpr int kF8Tok = 256;                  // tokens (N) per tile at most
constexpr int kF8ABytes = 128 * kF8K;        // weight codes of a stage
constexpr int kF8BBytes = kF8Tok * kF8K;     // activation codes of a stage
constexpr int kF8Acc = 2;                    // accumulator buffers in TMEM
constexpr int kF8TmemCols = kF8Acc * kF8Tok;

constexpr int kF8OffA = 0;
constexpr int kF8OffB = kF8OffA + kF8Stages * kF8ABytes;
constexpr int kF8OffBar = kF8OffB + kF8Stages * kF8BBytes;
// FULL[stages], EMPTY[stages], AFULL[acc], AEMPTY[acc], TD (committed by the MMA
// thread after an abort, to wait for its MMAs in flight before TMEM is freed)
constexpr int kF8BarFull = 0, kF8BarEmpty = kF8Stages, kF8BarAFull = 2 * kF8Stages,
              kF8BarAEmpty = kF8BarAFull + kF8Acc, kF8BarTd = kF8BarAEmpty + kF8Acc,
              kF8NumBars = kF8BarTd + 1;
constexpr int kF8OffMisc = kF8OffBar + kF8NumBars * 8;
constexpr int kF8Smem = kF8OffMisc + 16 + 1024;  // + alignment slack
static_assert(kF8Smem <= 227 * 1024, "shared memory budget");

enum F8Mode : int { kF8GateUp = 0, kF8Down = 1 };

struct F8Params {
    CUtensorMap tm_b;        // activation codes [rows][K] bytes, box {128, 128}
    CUtensorMap tm_b32;      // box {128, 32}: tiles of at most 32 tokens
    CUtensorMap tm_b64;      // box {128, 64}: tiles of 33-64 tokens
    CUtensorMap tm_b256;     // box {128, 256}: tiles of 129-256 tokens
    CUtensorMap tm_a;        // routed weight codes (gate+up 5D, down 2D)
    CUtensorMap tm_a_sh;     // shared-expert weight codes, same boxes
    const float* s_routed;   // weight row scales [E * rows_per_expert]
    const float* s_shared;   // [rows_shared]
    const float* a_rows;     // activation row scales [T*k + T]
    const int4* tiles;
    WsHeader* hdr;
    void* out;               // H (bf16) or Y (fp32)
    int64_t ld_out;          // row stride of out, elements
    int64_t rows;            // activation / output rows, T*k + T
    int max_tiles;           // capacity of the tile list
    int mode;
    int T, d, k, E, F, Fs;
};

// Activation rows a stage loads for a tile: the smallest box of 32, 64 or 128
// rows holding its npad tokens (the MMA reads npad rows).
__device__ __forceinline__ int f8_box_rows(int n) {
    const int npad = (n + 15) & ~15;
    return npad <= 32 ? 32 : npad <= 64 ? 64 : npad <= 128 ? 128 : 256;
}

// A tile the descriptors could have written: a group id in [-1, E), 1..128
// tokens inside the activation rows, a weight band inside the group's rows.
// Every role skips an invalid tile the same way (and the producer records it),
// so no access leaves its tensor and the pipeline stays in step.
__device__ __forceinline__ bool tile_ok(const F8Params& p, int4 t) {
    const int grp = t.x, row0 = t.y, n = t.z, band = t.w;
    const int nbands = p.mode == kF8GateUp ? (grp >= 0 ? p.F : p.Fs) / 64 : p.d / 128;
    return grp >= -1 && grp < p.E && n >= 1 && n <= kF8Tok && row0 >= 0 &&
           (int64_t)row0 + n <= p.rows && band >= 0 && band < nbands;
}

__global__ void __launch_bounds__(kF8Threads, 1)
grouped_w8a8_kernel(const __grid_constant__ F8Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF8OffBar);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kF8OffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kF8OffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kF8Stages; ++s) {
            mbar_init(bar(kF8BarFull + s), 1);
            mbar_init(bar(kF8BarEmpty + s), 1);
        }
        for (int b = 0; b < kF8Acc; ++b) {
            mbar_init(bar(kF8BarAFull + b), 1);
            mbar_init(bar(kF8BarAEmpty + b), kF8Warps - kF8EpiWarp0);
        }
        mbar_init(bar(kF8BarTd), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tm_a);
        prefetch_tmap(&p.tm_a_sh);
        prefetch_tmap(&p.tm_b);
        prefetch_tmap(&p.tm_b32);
        prefetch_tmap(&p.tm_b64);
        prefetch_tmap(&p.tm_b256);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kF8TmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_tiles = min(*reinterpret_cast<volatile int*>(&p.hdr->n_tiles[p.mode]), p.max_tiles);
    const int grid = gridDim.x;
    const bool gateup = p.mode == kF8GateUp;

    auto tile_K = [&](int grp) { return gateup ? p.d : (grp >= 0 ? p.F : p.Fs); };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            // test hook: CTA 0 of a gate+up launch skips the copies of one stage
            const int64_t withheld =
                (gateup && blockIdx.x == 0)
                    ? (int64_t)*reinterpret_cast<volatile int32_t*>(&p.hdr->withhold_stage) - 1
                    : -1;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += grid) {
                const int4 t = __ldg(p.tiles + tile);
                if (!tile_ok(p, t)) {
                    record_error(p.hdr, kErrBadTile);
                    continue;
                }
                const int grp = t.x, row0 = t.y, band = t.w;
                const CUtensorMap* tma = grp >= 0 ? &p.tm_a : &p.tm_a_sh;
                const int brows = f8_box_rows(t.z);
                const CUtensorMap* tmb = brows == 32    ? &p.tm_b32
                                         : brows == 64  ? &p.tm_b64
                                         : brows == 128 ? &p.tm_b
                                                        : &p.tm_b256;
                const int nks = tile_K(grp) / kF8K;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = it % kF8Stages;
                    const uint32_t ph = (it / kF8Stages) & 1;
                    if (!mbar_wait(bar(kF8BarEmpty + s), ph ^ 1, abort_flag, p.hdr)) {
                        ok = false;
                        break;
                    }
                    if ((int64_t)it == withheld) continue;  // its FULL phase never completes
                    mbar_expect_tx(bar(kF8BarFull + s), (uint32_t)(kF8ABytes + brows * kF8K));
                    const uint32_t adst = sbase + kF8OffA + s * kF8ABytes;
                    if (gateup)  // rows m = 32 * blk + 16 * gu + i
                        tma_load_5d(adst, tma, ks * kF8K, 0, 0, 4 * band, grp >= 0 ? grp : 0,
                                    bar(kF8BarFull + s));
                    else
                        tma_load_2d(adst, tma, ks * kF8K, (grp >= 0 ? grp * p.d : 0) + 128 * band,
                                    bar(kF8BarFull + s));
                    tma_load_2d(sbase + kF8OffB + s * kF8BBytes, tmb, ks * kF8K, row0,
                                bar(kF8BarFull + s));
                }
            }
            // do not leave with copies in flight: wait (bounded, whatever the abort flag)
            // for the stages issued last; without an abort their phases are complete
            for (uint32_t j = (it >= kF8Stages ? it - kF8Stages : 0); j < it; ++j)
                if ((int64_t)j != withheld)
                    mbar_drain(bar(kF8BarFull + j % kF8Stages), (j / kF8Stages) & 1, p.hdr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            int64_t last = -1;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += grid) {
                const int4 t = __ldg(p.tiles + tile);
                if (!tile_ok(p, t)) continue;
                const int npad = (t.z + 15) & ~15;
                const uint32_t idesc = idesc_e4m3(128, npad);
                const int b = tc % kF8Acc;
                if (!mbar_wait(bar(kF8BarAEmpty + b), ((tc / kF8Acc) & 1) ^ 1, abort_flag, p.hdr)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + (uint32_t)(b * kF8Tok);
                const int nks = tile_K(t.x) / kF8K;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = it % kF8Stages;
                    if (!mbar_wait(bar(kF8BarFull + s), (it / kF8Stages) & 1, abort_flag, p.hdr)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(sbase + kF8OffA + s * kF8ABytes);
                    const uint64_t bd = smem_desc_sw128(sbase + kF8OffB + s * kF8BBytes);
#pragma unroll
                    for (int kk = 0; kk < kF8K / 32; ++kk)  // 32 bytes = 2 address units per step
                        mma_ss_f8(dcol, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc,
                                  (ks | kk) ? 1u : 0u);
                    mma_commit(bar(kF8BarEmpty + s));
                    last = it;
                }
                if (!ok) break;
                mma_commit(bar(kF8BarAFull + b));
                ++tc;
            }
            // the MMAs are done before the CTA frees TMEM: a commit of its own, waited
            // for whatever the abort flag
            (void)last;
            mma_commit(bar(kF8BarTd));
            mbar_drain(bar(kF8BarTd), 0, p.hdr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // After a failed wait every epilogue warp keeps walking the tiles
        // (skipping the work), so no warp waits on a barrier the others left.
        const int q = warp & 3;
        const int part = (warp - kF8EpiWarp0) >> 2;  // which 32-column chunks of a tile
        const int m = q * 32 + lane;  // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int gu = (m >> 4) & 1;                     // gate+up: gate (0) or up (1) row
        const int f_local = (m >> 5) * 16 + (m & 15);    // gate+up: row pair within the band
        const bool lo = (lane & 16) == 0;
        bool ok = true;
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += grid) {
            const int4 t = __ldg(p.tiles + tile);
            if (!tile_ok(p, t)) continue;
            const int grp = t.x, row0 = t.y, n = t.z, band = t.w;
            const int b = tc % kF8Acc;
            if (ok && !mbar_wait(bar(kF8BarAFull + b), (tc / kF8Acc) & 1, abort_flag, p.hdr)) ok = false;
            if (ok) {
                tc_fence_after();
                float s_w;
                int col;  // gate+up: f; down: output channel
                if (gateup) {
                    col = 64 * band + f_local;
                    s_w = grp >= 0 ? __ldg(p.s_routed + (int64_t)grp * 2 * p.F + gu * p.F + col)
                                   : __ldg(p.s_shared + gu * p.Fs + col);
                } else {
                    col = 128 * band + m;
                    s_w = grp >= 0 ? __ldg(p.s_routed + (int64_t)grp * p.d + col)
                                   : __ldg(p.s_shared + col);
                }
                const int npad = (n + 15) & ~15;
                for (int c0 = 32 * part; c0 < npad; c0 += 32 * kF8EpiPerQuarter) {
                    uint32_t v[32];
                    tmem_ld_x32(tmem + lane_base + (uint32_t)(b * kF8Tok + c0), v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    const float a_mine = c0 + lane < n ? __ldg(p.a_rows + row0 + c0 + lane) : 0.f;
                    if (gateup) {
                        // lane i holds gate row f, lane i ^ 16 the up row of the same f.
                        // Step j finishes token c0 + j on the gate lanes and c0 + j + 16 on
                        // the up lanes: each lane sends the value its partner needs
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float a_lo = __shfl_sync(0xffffffffu, a_mine, j);
                            const float a_hi = __shfl_sync(0xffffffffu, a_mine, j + 16);
                            const float v_lo = (__uint_as_float(v[j]) * a_lo) * s_w;
                            const float v_hi = (__uint_as_float(v[j + 16]) * a_hi) * s_w;
                            const float other = __shfl_xor_sync(0xffffffffu, lo ? v_hi : v_lo, 16);
                            const float gv = lo ? v_lo : other;
                            const float uv = lo ? other : v_hi;
                            const int nn = c0 + j + (lo ? 0 : 16);
                            if (nn < n)
                                reinterpret_cast<uint16_t*>(p.out)[(int64_t)(row0 + nn) * p.ld_out + col] =
                                    float_to_bf16_bits(swiglu_f32(gv, uv));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float aj = __shfl_sync(0xffffffffu, a_mine, j);
                            const float val = (__uint_as_float(v[j]) * aj) * s_w;
                            const int nn = c0 + j;
                            if (nn < n)
                                reinterpret_cast<float*>(p.out)[(int64_t)(row0 + nn) * p.ld_out + col] = val;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kF8BarAEmpty + b));
            ++tc;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kF8TmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- quantisers
// E4M3 codes of two fp32 values (round to nearest even, saturate to +-448).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// One warp per row: scale = absmax / 448 (fp32 division), codes e4m3(v / scale).
// Row r of the output reads source row src_row(r) of `src` (row stride ld,
// `cols` valid columns, a multiple of 8).  bf16 or fp32 source.
template <typename Src>
__device__ __forceinline__ void load8(const Src* p, float* v);
template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, float* v) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename Src>
__device__ __forceinline__ void quant_row(const Src* src, int cols, uint8_t* dst, float* scale,
                                          int lane) {
    float amax = 0.f;
    for (int c = 8 * lane; c < cols; c += 256) {
        float v[8];
        load8<Src>(src + c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = __fdiv_rn(amax, 448.0f);
    if (lane == 0) *scale = sc;
    for (int c = 8 * lane; c < cols; c += 256) {
        float v[8];
        load8<Src>(src + c, v);
        uint2 o = make_uint2(0u, 0u);
        if (sc != 0.f) {
            o.x = e4m3x2(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc)) |
                  (e4m3x2(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc)) << 16);
            o.y = e4m3x2(__fdiv_rn(v[4], sc), __fdiv_rn(v[5], sc)) |
                  (e4m3x2(__fdiv_rn(v[6], sc), __fdiv_rn(v[7], sc)) << 16);
        }
        *reinterpret_cast<uint2*>(dst + c) = o;
    }
}

// Gate+up operand in descriptor order, from each token's codes: row r < T*k is
// slot perm[r]'s token, row T*k + t token t.  One warp per row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_codes_kernel(const uint8_t* __restrict__ xt,
                                                           const float* __restrict__ xta,
                                                           const int32_t* __restrict__ perm,
                                                           int T, int k, int d,
                                                           uint8_t* __restrict__ xq,
                                                           float* __restrict__ a) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t slots = (int64_t)T * k;
    if (r >= slots + T) return;
    const int64_t t = r < slots ? __ldg(perm + r) / k : r - slots;
    const uint4* src = reinterpret_cast<const uint4*>(xt + t * d);
    uint4* dst = reinterpret_cast<uint4*>(xq + r * d);
    for (int c = threadIdx.x & 31; c < d / 16; c += 32) dst[c] = __ldg(src + c);
    if ((threadIdx.x & 31) == 0) a[r] = __ldg(xta + t);
}

// Down operand: H rows [T*k + T][ld] (routed rows F columns, shared rows F_s).
__global__ void __launch_bounds__(256) quant_h_kernel(const uint16_t* __restrict__ H, int64_t rows,
                                                      int64_t slots, int ld, int F, int Fs,
                                                      uint8_t* __restrict__ hq,
                                                      float* __restrict__ a) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    quant_row<uint16_t>(H + r * ld, r < slots ? F : Fs, hq + r * ld, a + r, threadIdx.x & 31);
}

// Plain rows (weights, or any activation rows): [rows][K] -> codes, scales.
template <typename Src>
__global__ void __launch_bounds__(256) quant_rows_kernel(const Src* __restrict__ w, int64_t rows,
                                                         int64_t K, uint8_t* __restrict__ q,
                                                         float* __restrict__ s) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    quant_row<Src>(w + r * K, (int)K, q + r * K, s + r, threadIdx.x & 31);
}

// ---------------------------------------------------------------- host side
bool make_codes_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_rows = 128) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)kF8K, box_rows};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 2, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// Gate+up codes [experts][2Fg][d] read as {128 B of K, 16 rows, gate/up, 16-row
// blocks, expert}: one box holds 64 gate rows and their 64 up rows.
bool make_gateup_codes_map(CUtensorMap* m, const void* base, uint64_t d, uint64_t Fg,
                           uint64_t experts) {
    const cuuint64_t dims[5] = {d, 16, 2, Fg / 16, experts};
    const cuuint64_t strides[4] = {d, Fg * d, 16 * d, 2 * Fg * d};
    const cuuint32_t box[5] = {(cuuint32_t)kF8K, 16, 2, 4, 1};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 5, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_f8(F8Params& prm, cudaStream_t st) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t err = ensure_dynamic_smem((const void*)grouped_w8a8_kernel, kF8Smem);
    if (err != cudaSuccess) return err;
    grouped_w8a8_kernel<<<sms, kF8Threads, kF8Smem, st>>>(prm);
    return cudaGetLastError();
}

}  // namespace

bool w8a8_supported(const moe_dims_t& d) {
    return d.d % kF8K == 0 && d.F % kF8K == 0 && d.F_s % kF8K == 0 && d.F % 64 == 0 &&
           d.F_s % 64 == 0;
}

cudaError_t launch_quant_rows_fp8(const void* src, bool bf16, int64_t rows, int64_t K, uint8_t* q,
                                  float* s, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (bf16)
        quant_rows_kernel<uint16_t><<<blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src), rows,
                                                            K, q, s);
    else
        quant_rows_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(src), rows, K,
                                                         q, s);
    return cudaGetLastError();
}

cudaError_t launch_gateup_w8a8(const uint16_t* x, const moe_dims_t& d, const int32_t* perm,
                               moe_w8_t Wgu, moe_w8_t Wgu_s, uint16_t* H, WsHeader* hdr,
                               const int4* tiles, int64_t max_tiles, uint8_t* xq, float* a,
                               uint8_t* xt, float* xta, cudaStream_t st) {
    const int64_t rows = (int64_t)d.T * d.k + d.T;
    cudaError_t err = launch_quant_rows_fp8(x, true, d.T, d.d, xt, xta, st);
    if (err != cudaSuccess) return err;
    gather_codes_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(xt, xta, perm, d.T, d.k, d.d,
                                                                    xq, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    F8Params prm;
    memset(&prm, 0, sizeof(prm));
    if (!make_codes_map(&prm.tm_b, xq, d.d, rows, d.d) ||
        !make_codes_map(&prm.tm_b32, xq, d.d, rows, d.d, 32) ||
        !make_codes_map(&prm.tm_b64, xq, d.d, rows, d.d, 64) ||
        !make_codes_map(&prm.tm_b256, xq, d.d, rows, d.d, 256) ||
        !make_gateup_codes_map(&prm.tm_a, Wgu.q, d.d, d.F, d.E) ||
        !make_gateup_codes_map(&prm.tm_a_sh, Wgu_s.q, d.d, d.F_s, 1))
        return cudaErrorInvalidValue;
    prm.s_routed = Wgu.s;
    prm.s_shared = Wgu_s.s;
    prm.a_rows = a;
    prm.tiles = tiles;
    prm.hdr = hdr;
    prm.out = H;
    prm.ld_out = std::max(d.F, d.F_s);
    prm.rows = rows;
    prm.max_tiles = (int)max_tiles;
    prm.mode = kF8GateUp;
    prm.T = d.T; prm.d = d.d; prm.k = d.k; prm.E = d.E; prm.F = d.F; prm.Fs = d.F_s;
    return launch_f8(prm, st);
}

cudaError_t launch_down_w8a8(const uint16_t* H, const moe_dims_t& d, moe_w8_t Wd, moe_w8_t Wd_s,
                             float* Y, WsHeader* hdr, const int4* tiles, int64_t max_tiles,
                             uint8_t* hq, float* a, cudaStream_t st) {
    const int64_t slots = (int64_t)d.T * d.k, rows = slots + d.T;
    const int Fmax = std::max(d.F, d.F_s);
    quant_h_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(H, rows, slots, Fmax, d.F, d.F_s,
                                                               hq, a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    F8Params prm;
    memset(&prm, 0, sizeof(prm));
    if (!make_codes_map(&prm.tm_b, hq, Fmax, rows, Fmax) ||
        !make_codes_map(&prm.tm_b32, hq, Fmax, rows, Fmax, 32) ||
        !make_codes_map(&prm.tm_b64, hq, Fmax, rows, Fmax, 64) ||
        !make_codes_map(&prm.tm_b256, hq, Fmax, rows, Fmax, 256) ||
        !make_codes_map(&prm.tm_a, Wd.q, d.F, (uint64_t)d.E * d.d, d.F) ||
        !make_codes_map(&prm.tm_a_sh, Wd_s.q, d.F_s, (uint64_t)d.d, d.F_s))
        return cudaErrorInvalidValue;
    prm.s_routed = Wd.s;
    prm.s_shared = Wd_s.s;
    prm.a_rows = a;
    prm.tiles = tiles;
    prm.hdr = hdr;
    prm.out = Y;
    prm.ld_out = d.d;
    prm.rows = rows;
    prm.max_tiles = (int)max_tiles;
    prm.mode = kF8Down;
    prm.T = d.T; prm.d = d.d; prm.k = d.k; prm.E = d.E; prm.F = d.F; prm.Fs = d.F_s;
    return launch_f8(prm, st);
}

}  // namespace moe
