// Prefill-side expert projections: a persistent grouped W4A16 GEMM on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA staging).
//
// The pages' prefill MoE runs the experts as a grouped GEMM over on-device
// descriptors, gate and up stacked per expert, largest expert first and with
// N-banded CTA order so CTAs that share a weight band run together and reuse
// it in L2 (thewafflehaus/butter PR #69, commit "feat(laguna): batched prefill
// with tensor-core projections, fused MoE, CTA scheduling"); activations are
// read through the router-sorted token index instead of a separate gather pass
// (thewafflehaus/FFAI PR #72, Nemotron CUTLASS MoE commit).  Their kernels are
// mma.sync code for GB10; this one is written for sm_103a.
//
// Shape of one tile: M = 128 weight rows (swap-AB: weights take the M slot),
// N = up to 128 tokens of one expert (rounded up to 16), K = the full
// contraction in stages of 128.  Gate+up tiles hold 64 gate rows and the 64
// matching up rows, so SwiGLU is finished inside the tile.
//
// Warp roles (14 warps, one CTA per SM):
//   warp 0      TMA producer: per stage, the int4 weight tile (64B swizzle) and
//               the activation rows, gathered four rows per tile::gather4 load
//               (128B swizzle, the UMMA K-major canonical layout)
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16, A from
//               TMEM, B from shared memory, fp32 accumulator in TMEM
//   warps 2-5   dequantisers: int4 -> bf16 integers (exact), tcgen05.st to TMEM
//   warps 6-13  epilogue: per quantisation group, read the group's partial
//               sums from TMEM and accumulate s * partial in fp32 registers;
//               at the end of a tile apply SwiGLU (gate+up) or store Y (down)
//
// Numerics: each group's partial sum is sum_k x_k * q_k with exact bf16
// products and fp32 accumulation; multiplying by the fp16 scale s in fp32
// gives sum_k x_k * (q_k * s), the dequantised product, without rounding the
// weights.  TMEM: A stages at columns [0, 256), two 128-column accumulators at
// [256, 512).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kKStage = 128;                    // K elements per stage
constexpr int kTokTile = 128;                   // max tokens (N) per tile
constexpr int kBStageBytes = 2 * kTokTile * 128;  // two 64-wide K blocks, 128 B per row
constexpr int kAStageBytes = 128 * 64;          // 128 rows x 64 bytes of nibbles
constexpr int kUStride = 129;                   // padded row stride of the up-row buffer (floats)
constexpr int kMaxGroupsPerRow = 32;            // scale prefetch capacity (K / group)
constexpr int kTmemCols = 512;
constexpr int kTmemD = 256;                     // first accumulator column

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffB = 0;
constexpr int kOffA = kOffB + kStages * kBStageBytes;
constexpr int kOffU = kOffA + kStages * kAStageBytes;
constexpr int kOffSc = kOffU + 64 * kUStride * 4;
constexpr int kOffBar = kOffSc + 2 * 128 * kMaxGroupsPerRow * 2;
constexpr int kNumBars = 4 * kStages + 4;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: a wait that long means something broke

enum Mode : int { kGateUp = 0, kDown = 1 };

struct GroupedParams {
    CUtensorMap tm_b;       // activations (x or H), bf16, box {64, 1}, 128B swizzle
    CUtensorMap tm_a;       // routed int4 weights, uint8 rows
    CUtensorMap tm_a_sh;    // shared-expert int4 weights
    const __half* s_routed; // [E * rows_per_expert][K / group]
    const __half* s_shared; // [rows_shared][K_shared / group]
    const int32_t* perm;
    const int4* tiles;
    WsHeader* hdr;
    void* out;              // H (bf16) or Y (fp32)
    int64_t ld_out;         // row stride of out, elements
    int mode;
    int T, d, k, F, Fs, group;
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after kWaitNs (or once another warp gave up), records
// the failure in the workspace header and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          WsHeader* hdr) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) {
                *abort_flag = 1;
                record_error(hdr, kErrWaitTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int x, int y0,
                                            int y1, int y2, int y3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// UMMA shared-memory descriptor: K-major operand, 128B swizzle, 8-row groups
// 1024 B apart (SBO), descriptor version 1 (sm_100 family).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset
    d |= (uint64_t)1 << 46;                   // version
    d |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- int4 -> bf16
// One 32-bit word holds elements 0..7 (element 2j in the low nibble of byte
// j).  Produces four bf16x2 registers {e_2j, e_2j+1} holding the exact
// integers q in [-8, 7]: each nibble becomes 128 + (q + 8) through the bf16
// exponent pattern 0x43xx, then one packed fma subtracts 136.
__device__ __forceinline__ void nib8_to_bf16x2(uint32_t w, uint32_t* out) {
    const uint32_t w4 = w >> 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t r, t, q;
        const uint32_t sel = (uint32_t)j | ((uint32_t)(4 + j) << 8);
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(w4), "r"(sel));
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(t) : "r"(r), "r"(0x000F000Fu), "r"(0x43084308u));
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(t), "r"(0x3F803F80u), "r"(0xC308C308u));
        out[j] = q;
    }
}

// ---------------------------------------------------------------- TMEM copies
__device__ __forceinline__ void tmem_st_x64(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
        "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
        "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]),
        "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]),
        "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]),
        "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]),
        "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
        "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ---------------------------------------------------------------- tile decoding
struct TileInfo {
    int grp;    // expert id, -1 for the shared expert
    int row0;   // first row of H / Y for this tile
    int n;      // tokens in the tile
    int band;   // weight band index
    int npad;   // n rounded up to 16
    int K;      // contraction length
};

__device__ __forceinline__ TileInfo decode_tile(const GroupedParams& p, int4 t) {
    TileInfo ti;
    ti.grp = t.x;
    ti.row0 = t.y;
    ti.n = t.z;
    ti.band = t.w;
    ti.npad = (t.z + 15) & ~15;
    ti.K = p.mode == kGateUp ? p.d : (t.x >= 0 ? p.F : p.Fs);
    return ti;
}

// The scales of a tile's 128 weight rows form one contiguous block (down: 128
// rows) or two (gate+up: 64 gate rows, 64 up rows) of rows x (K / group)
// fp16 values.  Each block starts on a 16-byte boundary (a multiple of 64 rows).
__device__ __forceinline__ const __half* scale_block(const GroupedParams& p, const TileInfo& ti,
                                                     int blk) {
    const int ng = ti.K / p.group;
    int64_t row;
    if (p.mode == kGateUp) {
        const int Fg = ti.grp >= 0 ? p.F : p.Fs;
        const int local = blk == 0 ? 64 * ti.band : Fg + 64 * ti.band;
        row = ti.grp >= 0 ? (int64_t)ti.grp * 2 * p.F + local : local;
    } else {
        const int local = 128 * ti.band;
        row = ti.grp >= 0 ? (int64_t)ti.grp * p.d + local : local;
    }
    return (ti.grp >= 0 ? p.s_routed : p.s_shared) + row * ng;
}

// Loads the tile's scales as 16-byte words: word u (of 16 * ng) is returned in
// v[u / 128] for thread t = u % 128 of the 128 loading threads.
constexpr int kScaleWordsPerThread = kMaxGroupsPerRow * 16 / 128;  // 4

__device__ __forceinline__ void load_scales(const GroupedParams& p, const TileInfo& ti, int t,
                                            uint4* v) {
    const int ng = ti.K / p.group;
    const int words = 16 * ng;  // 128 rows x ng halves / 8
    const int per_blk = p.mode == kGateUp ? 8 * ng : 16 * ng;
#pragma unroll
    for (int i = 0; i < kScaleWordsPerThread; ++i) {
        const int u = t + 128 * i;
        if (u < words) {
            const int blk = u / per_blk, w = u - blk * per_blk;
            v[i] = __ldg(reinterpret_cast<const uint4*>(scale_block(p, ti, blk)) + w);
        }
    }
}

// Stores them to shared memory as [128 rows][ng] halves.
__device__ __forceinline__ void store_scales(__half* dst, int ng, int t, const uint4* v) {
#pragma unroll
    for (int i = 0; i < kScaleWordsPerThread; ++i) {
        const int u = t + 128 * i;
        if (u < 16 * ng) reinterpret_cast<uint4*>(dst)[u] = v[i];
    }
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 1) grouped_w4a16_kernel(const __grid_constant__ GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    // barrier indices
    const int FULL = 0, EMPTY = kStages, AREADY = 2 * kStages, AFREE = 3 * kStages,
              DFULL = 4 * kStages, DEMPTY = 4 * kStages + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1 + 4);
            mbar_init(bar(AREADY + s), 4);
            mbar_init(bar(AFREE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(DFULL + b), 1);
            mbar_init(bar(DEMPTY + b), 8);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_tiles = *reinterpret_cast<volatile int*>(&p.hdr->n_tiles[p.mode]);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            const TileInfo ti = decode_tile(p, __ldg(p.tiles + tile));
            int rows[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * lane + r;
                const int src = i < ti.n ? i : 0;
                if (p.mode == kGateUp)
                    rows[r] = ti.grp >= 0 ? __ldg(p.perm + ti.row0 + src) / p.k
                                          : ti.row0 - p.T * p.k + src;
                else
                    rows[r] = ti.row0 + src;
            }
            const CUtensorMap* tma = ti.grp >= 0 ? &p.tm_a : &p.tm_a_sh;
            int arow0, arow1 = 0;
            if (p.mode == kGateUp) {
                const int Fg = ti.grp >= 0 ? p.F : p.Fs;
                const int base = ti.grp >= 0 ? ti.grp * 2 * p.F : 0;
                arow0 = base + 64 * ti.band;
                arow1 = base + Fg + 64 * ti.band;
            } else {
                arow0 = (ti.grp >= 0 ? ti.grp * p.d : 0) + 128 * ti.band;
            }
            const uint32_t bytes = (uint32_t)kAStageBytes + (uint32_t)ti.npad * 256u;
            const int nks = ti.K / kKStage;
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(bar(EMPTY + s), ph ^ 1, abort_flag, p.hdr)) { ok = false; break; }
                if (lane == 0) mbar_expect_tx(bar(FULL + s), bytes);
                __syncwarp();
                const uint32_t bdst = sbase + kOffB + s * kBStageBytes;
                if (4 * lane < ti.npad) {
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
                        tma_gather4(bdst + kb * (kTokTile * 128) + 4 * lane * 128, &p.tm_b,
                                    ks * kKStage + kb * 64, rows[0], rows[1], rows[2], rows[3],
                                    bar(FULL + s));
                }
                if (lane == 0) {
                    const uint32_t adst = sbase + kOffA + s * kAStageBytes;
                    tma_load_2d(adst, tma, ks * 64, arow0, bar(FULL + s));
                    if (p.mode == kGateUp) tma_load_2d(adst + 64 * 64, tma, ks * 64, arow1, bar(FULL + s));
                }
            }
        }
        // do not leave with copies in flight: wait until every issued stage has landed
        if (!ok) {
            for (uint32_t j = (it >= kStages ? it - kStages : 0); j < it; ++j)
                mbar_wait(bar(FULL + j % kStages), (j / kStages) & 1, abort_flag, p.hdr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, gi = 0;
            bool ok = true;
            const int kk_per_group = p.group / 16;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const TileInfo ti = decode_tile(p, __ldg(p.tiles + tile));
                const uint32_t idesc = idesc_bf16(128, ti.npad);
                const int nks = ti.K / kKStage;
                for (int ks = 0; ks < nks && ok; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(bar(FULL + s), ph, abort_flag, p.hdr) ||
                        !mbar_wait(bar(AREADY + s), ph, abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t bstage = sbase + kOffB + s * kBStageBytes;
                    for (int gg = 0; gg < kKStage / p.group; ++gg, ++gi) {
                        const int b = gi & 1;
                        if (!mbar_wait(bar(DEMPTY + b), ((gi >> 1) & 1) ^ 1, abort_flag, p.hdr)) { ok = false; break; }
                        tc_fence_after();
                        for (int kk = 0; kk < kk_per_group; ++kk) {
                            const int kg = gg * kk_per_group + kk;  // 16-wide K step within the stage
                            const uint32_t a_addr = tmem + (uint32_t)(s * 64 + kg * 8);
                            const uint64_t bdesc =
                                smem_desc_sw128(bstage + (kg >> 2) * (kTokTile * 128) + (kg & 3) * 32);
                            mma_ts(tmem + kTmemD + b * 128, a_addr, bdesc, idesc, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(DFULL + b));
                    }
                    if (!ok) break;
                    mma_commit(bar(EMPTY + s));
                    mma_commit(bar(AFREE + s));
                }
            }
            // the last commit has landed before the CTA can exit
            if (ok && it > 0)
                mbar_wait(bar(AFREE + (it - 1) % kStages), ((it - 1) / kStages) & 1, abort_flag, p.hdr);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ dequantisers
        const int q = warp & 3;
        const int m = q * 32 + lane;  // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            const TileInfo ti = decode_tile(p, __ldg(p.tiles + tile));
            const int nks = ti.K / kKStage;
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(bar(FULL + s), ph, abort_flag, p.hdr)) { ok = false; break; }
                const uint8_t* arow = smem + kOffA + s * kAStageBytes + m * 64;
                uint4 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[c] = *reinterpret_cast<const uint4*>(arow + ((c ^ ((m >> 1) & 3)) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(EMPTY + s));
                uint32_t r[64];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    nib8_to_bf16x2(v[c].x, r + 16 * c + 0);
                    nib8_to_bf16x2(v[c].y, r + 16 * c + 4);
                    nib8_to_bf16x2(v[c].z, r + 16 * c + 8);
                    nib8_to_bf16x2(v[c].w, r + 16 * c + 12);
                }
                if (!mbar_wait(bar(AFREE + s), ph ^ 1, abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
                tmem_st_x64(tmem + lane_base + (uint32_t)(s * 64), r);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(AREADY + s));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // After a failed wait every epilogue warp keeps walking the same tiles
        // (skipping the work) so the named barriers stay matched.
        const int q = warp & 3;
        const int half = (warp - 6) >> 2;
        const int m = q * 32 + lane;
        const int col0 = half * 64;
        const int t128 = threadIdx.x - 6 * 32 - half * 128;  // 0..127 within the half
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        __half* sc = reinterpret_cast<__half*>(smem + kOffSc);  // [2][128 * kMaxGroupsPerRow]
        float* U = reinterpret_cast<float*>(smem + kOffU);        // [64][kUStride]
        uint32_t gi = 0;
        bool ok = true;
        int tile = blockIdx.x;
        if (tile < n_tiles && half == 0) {  // scales of the first tile
            const TileInfo ti = decode_tile(p, __ldg(p.tiles + tile));
            uint4 v[kScaleWordsPerThread];
            load_scales(p, ti, t128, v);
            store_scales(sc, ti.K / p.group, t128, v);
        }
        epi_bar();
        for (int tc = 0; tile < n_tiles; tile += gridDim.x, ++tc) {
            const TileInfo ti = decode_tile(p, __ldg(p.tiles + tile));
            const int ngroups = ti.K / p.group;
            const __half* scur = sc + (tc & 1) * 128 * kMaxGroupsPerRow + m * ngroups;
            // prefetch the next tile's scales into registers
            uint4 nxt[kScaleWordsPerThread];
            const int next = tile + gridDim.x;
            TileInfo tn = ti;
            if (next < n_tiles) tn = decode_tile(p, __ldg(p.tiles + next));
            if (next < n_tiles && half == 0) load_scales(p, tn, t128, nxt);
            float acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0.f;
            for (int g = 0; g < ngroups; ++g, ++gi) {
                const int b = gi & 1;
                if (ok && !mbar_wait(bar(DFULL + b), (gi >> 1) & 1, abort_flag, p.hdr)) ok = false;
                if (!ok) continue;
                tc_fence_after();
                const float s = __half2float(scur[g]);
                const uint32_t dcol = tmem + lane_base + (uint32_t)(kTmemD + b * 128 + col0);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (col0 + 32 * c < ti.npad) {
                        uint32_t v[32];
                        tmem_ld_x32(dcol + 32 * c, v);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            acc[32 * c + j] = fmaf(s, __uint_as_float(v[j]), acc[32 * c + j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(DEMPTY + b));
            }
            if (p.mode == kGateUp) {
                if (ok && m >= 64) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) U[(m - 64) * kUStride + col0 + j] = acc[j];
                }
                epi_bar();
                if (ok && m < 64) {
                    uint16_t* H = reinterpret_cast<uint16_t*>(p.out);
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const int nn = col0 + j;
                        if (nn < ti.n) {
                            const float gv = acc[j];
                            const float uv = U[m * kUStride + nn];
                            const float h = gv / (1.0f + expf(-gv)) * uv;
                            H[(int64_t)(ti.row0 + nn) * p.ld_out + 64 * ti.band + m] = float_to_bf16_bits(h);
                        }
                    }
                }
            } else if (ok) {
                float* Y = reinterpret_cast<float*>(p.out);
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int nn = col0 + j;
                    if (nn < ti.n) Y[(int64_t)(ti.row0 + nn) * p.ld_out + 128 * ti.band + m] = acc[j];
                }
            }
            // publish the next tile's scales: the other buffer is free, every
            // epilogue thread has finished the previous tile
            if (next < n_tiles && half == 0)
                store_scales(sc + ((tc + 1) & 1) * 128 * kMaxGroupsPerRow, tn.K / p.group, t128, nxt);
            epi_bar();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!counts[dev]) cudaDeviceGetAttribute(&counts[dev], cudaDevAttrMultiProcessorCount, dev);
    return counts[dev];
}

cudaError_t launch(GroupedParams& prm, cudaStream_t st) {
    cudaError_t err = ensure_dynamic_smem((const void*)grouped_w4a16_kernel, kSmemBytes);
    if (err != cudaSuccess) return err;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    grouped_w4a16_kernel<<<sms, kThreads, kSmemBytes, st>>>(prm);
    return cudaGetLastError();
}

}  // namespace

bool grouped_supported(const moe_dims_t& d) {
    const int Fmax = std::max(d.F, d.F_s);
    return d.d % kKStage == 0 && d.F % kKStage == 0 && d.F_s % kKStage == 0 &&
           d.d / d.group <= kMaxGroupsPerRow && Fmax / d.group <= kMaxGroupsPerRow &&
           d.F % 64 == 0 && d.F_s % 64 == 0 && d.d % 128 == 0 && d.group % 16 == 0 &&
           kKStage % d.group == 0;
}

cudaError_t launch_gateup_grouped(const uint16_t* x, const moe_dims_t& d, const int32_t* perm,
                                  moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H, WsHeader* hdr,
                                  const int4* tiles, cudaStream_t st) {
    GroupedParams prm;
    memset(&prm, 0, sizeof(prm));
    const int Fmax = std::max(d.F, d.F_s);
    if (!make_map(&prm.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, d.d, d.T, (uint64_t)d.d * 2, 64, 1,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&prm.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wgu.q, d.d / 2, (uint64_t)d.E * 2 * d.F,
                  d.d / 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&prm.tm_a_sh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wgu_s.q, d.d / 2,
                  (uint64_t)2 * d.F_s, d.d / 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    prm.s_routed = reinterpret_cast<const __half*>(Wgu.s);
    prm.s_shared = reinterpret_cast<const __half*>(Wgu_s.s);
    prm.perm = perm;
    prm.tiles = tiles;
    prm.hdr = hdr;
    prm.out = H;
    prm.ld_out = Fmax;
    prm.mode = kGateUp;
    prm.T = d.T; prm.d = d.d; prm.k = d.k; prm.F = d.F; prm.Fs = d.F_s; prm.group = d.group;
    return launch(prm, st);
}

cudaError_t launch_down_grouped(const uint16_t* H, const moe_dims_t& d, moe_w4_t Wd,
                                moe_w4_t Wd_s, float* Y, WsHeader* hdr, const int4* tiles,
                                cudaStream_t st) {
    GroupedParams prm;
    memset(&prm, 0, sizeof(prm));
    const int Fmax = std::max(d.F, d.F_s);
    const uint64_t rows = (uint64_t)d.T * d.k + d.T;
    if (!make_map(&prm.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, H, Fmax, rows, (uint64_t)Fmax * 2, 64, 1,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&prm.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wd.q, d.F / 2, (uint64_t)d.E * d.d,
                  d.F / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&prm.tm_a_sh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wd_s.q, d.F_s / 2, (uint64_t)d.d,
                  d.F_s / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    prm.s_routed = reinterpret_cast<const __half*>(Wd.s);
    prm.s_shared = reinterpret_cast<const __half*>(Wd_s.s);
    prm.perm = nullptr;
    prm.tiles = tiles;
    prm.hdr = hdr;
    prm.out = Y;
    prm.ld_out = d.d;
    prm.mode = kDown;
    prm.T = d.T; prm.d = d.d; prm.k = d.k; prm.F = d.F; prm.Fs = d.F_s; prm.group = d.group;
    return launch(prm, st);
}

}  // namespace moe
