// Prefill-side expert projections: a persistent grouped W4A16 GEMM on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA staging).
//
// The pages' prefill MoE runs the experts as a grouped GEMM over on-device
// descriptors, gate and up stacked per expert, largest expert first and with
// N-banded CTA order so CTAs that share a weight band run together and reuse
// it in L2 (thewafflehaus/butter PR #69, commit "feat(laguna): batched prefill
// with tensor-core projections, fused MoE, CTA scheduling").  Their kernels are
// mma.sync code for GB10; this one is written for sm_103a.
//
// Shape of one tile: M = 128 weight rows (swap-AB: weights take the M slot),
// N = up to 192 tokens of one expert (rounded up to 16), K = the full
// contraction in stages of 128.  192 is the widest N for which two A stages and two
// accumulators fit in the 512 TMEM columns; against 128-token tiles it cuts the
// MMA instructions per flop by a third, and the dequantisation passes over each
// weight tile (one per token tile) by up to a third.  A gate+up tile holds 64
// gate rows and the 64 matching up rows, interleaved in blocks of 16 (gate
// f..f+15, up f..f+15, ...), so a gate row and its up row sit 16 lanes apart in
// the same warp and SwiGLU is finished with one shuffle.
//
// Activation rows are read as plain TMA boxes of up to 192 rows: the down
// projection reads H, whose rows are already grouped by expert; gate+up reads x
// gathered once into that same row order (gather_rows_kernel), which replaces
// per-row gathers inside the GEMM that the TMA unit serves slowly.
//
// Warp roles (20 warps, one CTA per SM; setmaxnreg moves registers from the
// control and dequantiser warpgroups to the epilogue's):
//   warp 0      TMA producer: per tile the fp16 scale block (bulk copy), per
//               stage the int4 weight tile (64B swizzle) and the activation
//               tile (128B swizzle, the UMMA K-major canonical layout)
//   warps 1-2   MMA issuers (warp 1 also allocates TMEM): tcgen05.mma
//               kind::f16, A from TMEM, B from shared memory, fp32 accumulator
//               in TMEM; even quantisation groups on warp 1, odd on warp 2
//   warp 3      idle
//   warps 4-7   dequantisers, one per TMEM lane quarter, the stage's full K:
//               int4 -> bf16 integers (exact), tcgen05.st to TMEM
//   warps 8-19  epilogue, three per lane quarter (warp part p takes the
//               32-column blocks p and p + 3): per group, read the group's
//               partial sums from TMEM and accumulate s * partial in fp32
//               registers (packed f32x2 FMAs); at the end of a tile apply
//               SwiGLU (gate+up) or store Y (down)
// Launches of at most 64 tokens use the other layout (Layout<2>): warps 4-11
// dequantise (two per quarter, half of a stage's K each), warps 12-19 are the
// epilogue (two per quarter, 32 columns each), and TMEM holds three 64-column
// accumulators instead of two 192-column ones.
//
// With many tokens per tile the per-group drain of the accumulators is the loop
// that sets the stage period (MMA -> commit -> epilogue reads -> accumulator
// free -> next MMA), so the epilogue gets three warps per quarter (two TMEM
// round trips per group and warp instead of three) and the dequantisers, which
// convert before they wait for their TMEM slot, one.  With few tokens the
// conversion, paid per stage whatever the token count, sets it.  Two MMA
// issuers on two schedulers hide each other's barrier and commit latency; each
// TMEM A slot is used by every second stage, so splitting the stages by parity
// gives every AREADY barrier a single waiter that consumes its phases in order
// (a parity wait cannot tell phase k from phase k - 2).
//
// Numerics: each group's partial sum is sum_k x_k * q_k with exact bf16
// products and fp32 accumulation; multiplying by the fp16 scale s in fp32
// gives sum_k x_k * (q_k * s), the dequantised product, without rounding the
// weights.  TMEM: two A stages at columns [0, 128), then two 192-column
// accumulators (three 64-column ones in the small-tile layout), so the MMAs
// can run one (two) groups ahead of the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tma.cuh"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kWarps = 20;  // control warpgroup + dequantisers + epilogue
constexpr int kThreads = kWarps * 32;
constexpr int kDequantWarp0 = 4;
constexpr int kStages = 3;                        // shared-memory pipeline depth
constexpr int kAStagesT = 2;                      // A operand stages in TMEM
constexpr int kMaxDBufs = 3;                      // accumulator buffers in TMEM, at most
static_assert(kAStagesT < kStages, "dequant reuses the stage barrier of the MMA it waits for");
constexpr int kKStage = 128;                      // K elements per stage
constexpr int kTokTile = 192;                     // max tokens (N) per tile
constexpr int kBStageBytes = 2 * kTokTile * 128;  // two 64-wide K blocks, 128 B per row
constexpr int kAStageBytes = 128 * 64;            // 128 rows x 64 bytes of nibbles
constexpr int kMaxGroupsPerRow = 32;              // scale buffer capacity (K / group)
constexpr int kScBytes = 128 * kMaxGroupsPerRow * 2;
constexpr int kTmemCols = 512;
constexpr int kTmemD = kAStagesT * 64;            // first accumulator column
static_assert(kTokTile == kTileN, "the descriptors' tile lists use kTileN tokens per tile");

// Warp layouts after the control warpgroup (warps 0-3), both 20 warps:
//   DQ = 1: one dequantiser and three epilogue warps per TMEM lane quarter
//           (tiles of many tokens: the accumulator drain sets the stage period)
//   DQ = 2: two dequantisers and two epilogue warps per quarter and three
//           64-column accumulators (tiles of at most 64 tokens: the fixed
//           per-stage conversion and the drain latency set it, and the third
//           accumulator lets the MMAs run two groups ahead of the drain)
// Registers per thread after setmaxnreg: control, dequantisers, epilogue.  Their
// sum over the CTA must not exceed what the launch holds (checked on the host
// before every launch: a setmaxnreg.inc that cannot be served would wait forever).
template <int DQ>
struct Layout {
    static constexpr int kDqPerQuarter = DQ;
    static constexpr int kEpiPerQuarter = DQ == 1 ? 3 : 2;
    static constexpr int kDequantWarps = 4 * kDqPerQuarter;
    static constexpr int kEpilogueWarp0 = kDequantWarp0 + kDequantWarps;
    static constexpr int kEpilogueWarps = 4 * kEpiPerQuarter;
    static constexpr int kDBufs = DQ == 1 ? 2 : 3;          // accumulator buffers in TMEM
    static constexpr int kAccCols = DQ == 1 ? kTokTile : 64;  // tokens one accumulator holds
    static constexpr int kRegCtl = 40, kRegDq = DQ == 1 ? 80 : 56, kRegEpi = DQ == 1 ? 120 : 160;
    static constexpr int kRegBudget =
        128 * (kRegCtl + kDqPerQuarter * kRegDq + kEpiPerQuarter * kRegEpi);
    static_assert(kEpilogueWarp0 + kEpilogueWarps == 20, "20 warps per CTA");
    static_assert(kDBufs <= kMaxDBufs, "barrier arrays");
    static_assert(kTmemD + kDBufs * kAccCols <= 512, "A stages and accumulators exceed the TMEM columns");
    static_assert(kRegBudget <= 65536, "register split exceeds the register file");
};

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffB = 0;
constexpr int kOffA = kOffB + kStages * kBStageBytes;
constexpr int kOffSc = kOffA + kStages * kAStageBytes;
constexpr int kOffBar = kOffSc + 2 * kScBytes;
// barriers: FULL[kStages], EMPTY[kStages], AREADY[kAStagesT], DFULL[kMaxDBufs], DEMPTY[kMaxDBufs],
// SCFULL[2], SCEMPTY[2]
// EMPTY[s] completes when the MMAs of smem stage s are done and the dequant
// warps have read its int4 tile; it also tells the dequant warps that the
// TMEM A stage those MMAs read is free again.
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarAReady = 2 * kStages,
              kBarDFull = kBarAReady + kAStagesT,
              kBarDEmpty = kBarDFull + kMaxDBufs, kBarScFull = kBarDEmpty + kMaxDBufs,
              kBarScEmpty = kBarScFull + 2, kBarTd = kBarScEmpty + 2, kNumBars = kBarTd + 2;
// TD[2]: one per MMA issuer, committed after an abort so the issuer can wait for
// its MMAs in flight before the CTA frees TMEM.
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");


enum Mode : int { kGateUp = 0, kDown = 1 };

struct GroupedParams {
    CUtensorMap tm_b;        // activation rows (gathered x or H), bf16, box {64, 192}, 128B swizzle
    CUtensorMap tm_b32;      // the same rows, box {64, 32}: tiles of at most 32 tokens
    CUtensorMap tm_b64;      // box {64, 64}: tiles of 33-64 tokens
    CUtensorMap tm_b128;     // box {64, 128}: tiles of 65-128 tokens
    CUtensorMap tm_a;        // routed int4 weights, uint8 rows; gate+up box {64, 16}, down {64, 128}
    CUtensorMap tm_a_sh;     // shared-expert int4 weights, same boxes
    const __half* s_routed;  // [E * rows_per_expert][K / group]
    const __half* s_shared;  // [rows_shared][K_shared / group]
    const int4* tiles;
    WsHeader* hdr;
    void* out;               // H (bf16) or Y (fp32)
    int64_t ld_out;          // row stride of out, elements
    int mode;
    int T, d, k, F, Fs, group;
};

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

// Same word, pairs (j, j + 4) instead: out[j] = {e_j, e_j+4}, one shift and one
// lop3 per pair (no byte permute).  The contraction is unchanged if the other
// operand stores each 8-element block in the matching order (x0, x4, x1, x5,
// x2, x6, x3, x7), which gather_rows_kernel does for the gate+up activations.
__device__ __forceinline__ void nib8_to_bf16x2_paired(uint32_t w, uint32_t* out) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t t, q;
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(t) : "r"(w >> (4 * j)), "r"(0x000F000Fu), "r"(0x43084308u));
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(t), "r"(0x3F803F80u), "r"(0xC308C308u));
        out[j] = q;
    }
}

// ---------------------------------------------------------------- tiles
struct TileInfo {
    int grp;    // expert id, -1 for the shared expert
    int row0;   // first row of the activation / output rows of this tile
    int n;      // tokens in the tile
    int band;   // weight band index
    int npad;   // n rounded up to 16
    int K;      // contraction length
    int ng;     // quantisation groups along K
};

template <int G, int MODE>
__device__ __forceinline__ TileInfo decode_tile(const GroupedParams& p, int4 t) {
    TileInfo ti;
    ti.grp = t.x;
    ti.row0 = t.y;
    ti.n = t.z;
    ti.band = t.w;
    ti.npad = (t.z + 15) & ~15;
    ti.K = MODE == kGateUp ? p.d : (t.x >= 0 ? p.F : p.Fs);
    ti.ng = ti.K / G;
    return ti;
}

// Activation rows one stage loads for a tile: the smallest box of 32, 64, 128 or
// 192 rows that holds its npad tokens (the MMA reads npad rows; smaller boxes
// keep small-token tiles from moving 192 rows per stage).
__device__ __forceinline__ int b_box_rows(int npad) {
    return npad <= 32 ? 32 : npad <= 64 ? 64 : npad <= 128 ? 128 : 192;
}

__device__ __forceinline__ int4 load_tile(const GroupedParams& p, int tile, int n_tiles) {
    return tile < n_tiles ? __ldg(p.tiles + tile) : make_int4(0, 0, 1, 0);
}

// First weight row (within the routed or shared weight tensor) of the tile's
// block of rows: gate+up block (gu, blk) = 16 rows; down = the 128 rows.
template <int MODE>
__device__ __forceinline__ int weight_row(const GroupedParams& p, const TileInfo& ti, int gu,
                                          int blk) {
    if (MODE == kGateUp) {
        const int Fg = ti.grp >= 0 ? p.F : p.Fs;
        const int base = ti.grp >= 0 ? ti.grp * 2 * p.F : 0;
        return base + gu * Fg + 64 * ti.band + 16 * blk;
    }
    return (ti.grp >= 0 ? ti.grp * p.d : 0) + 128 * ti.band;
}

// ---------------------------------------------------------------- the kernel
// G: quantisation group size along K; MODE: kGateUp or kDown; DQ: the warp layout
// (Layout).  One instantiation each, so each gets its own register allocation.
template <int G, int MODE, int DQ>
__global__ void __launch_bounds__(kThreads, 1)
grouped_w4a16_kernel(const __grid_constant__ GroupedParams p) {
    using L = Layout<DQ>;
    constexpr int kDqPerQuarter = L::kDqPerQuarter, kEpiPerQuarter = L::kEpiPerQuarter;
    constexpr int kDequantWarps = L::kDequantWarps, kEpilogueWarp0 = L::kEpilogueWarp0;
    constexpr int kEpilogueWarps = L::kEpilogueWarps;
    constexpr int kRegCtl = L::kRegCtl, kRegDq = L::kRegDq, kRegEpi = L::kRegEpi;
    constexpr int kDBufs = L::kDBufs, kAccCols = L::kAccCols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarFull + s), 1);
            // the MMA commit(s) of the stage (both issuers when it holds two or more
            // groups) + the dequant warps
            mbar_init(bar(kBarEmpty + s), (kKStage / G >= 2 ? 2 : 1) + kDequantWarps);
        }
        for (int a = 0; a < kAStagesT; ++a) mbar_init(bar(kBarAReady + a), kDequantWarps);
        for (int b = 0; b < kDBufs; ++b) {
            mbar_init(bar(kBarDFull + b), 1);
            mbar_init(bar(kBarDEmpty + b), kEpilogueWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarScFull + b), 1);
            mbar_init(bar(kBarScEmpty + b), kEpilogueWarps);
            mbar_init(bar(kBarTd + b), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_a_sh)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_b)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_b32)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_b64)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_b128)) : "memory");
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
    const int n_tiles = *reinterpret_cast<volatile int*>(&p.hdr->n_tiles[MODE]);
    const int grid = gridDim.x;

    if (warp < kDequantWarp0) {
        // each warpgroup changes its register count inside its own branch
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegCtl));
        if (warp == 0) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                uint32_t it = 0;
                bool ok = true;
                int tc = 0, sc_issued = 0;
                // test hook: CTA 0 of a gate+up launch skips the copies of one stage
                const int64_t withheld =
                    (MODE == kGateUp && blockIdx.x == 0)
                        ? (int64_t)*reinterpret_cast<volatile int32_t*>(&p.hdr->withhold_stage) - 1
                        : -1;
                int4 cur = load_tile(p, blockIdx.x, n_tiles);
                for (int tile = blockIdx.x; tile < n_tiles && ok; tile += grid, ++tc) {
                    const int4 nxt = load_tile(p, tile + grid, n_tiles);  // one tile ahead
                    const TileInfo ti = decode_tile<G, MODE>(p, cur);
                    // the tile's scale block(s)
                    const int sb = tc & 1;
                    if (!mbar_wait(bar(kBarScEmpty + sb), ((tc >> 1) & 1) ^ 1, abort_flag, p.hdr)) {
                        ok = false;
                        break;
                    }
                    const __half* sbase_g = ti.grp >= 0 ? p.s_routed : p.s_shared;
                    const uint32_t scdst = sbase + kOffSc + sb * kScBytes;
                    if (MODE == kGateUp) {
                        const uint32_t blk_bytes = 64u * ti.ng * 2u;
                        mbar_expect_tx(bar(kBarScFull + sb), 2 * blk_bytes);
                        bulk_load(scdst, sbase_g + (int64_t)weight_row<MODE>(p, ti, 0, 0) * ti.ng, blk_bytes,
                                  bar(kBarScFull + sb));
                        bulk_load(scdst + blk_bytes, sbase_g + (int64_t)weight_row<MODE>(p, ti, 1, 0) * ti.ng,
                                  blk_bytes, bar(kBarScFull + sb));
                    } else {
                        const uint32_t bytes = 128u * ti.ng * 2u;
                        mbar_expect_tx(bar(kBarScFull + sb), bytes);
                        bulk_load(scdst, sbase_g + (int64_t)weight_row<MODE>(p, ti, 0, 0) * ti.ng, bytes,
                                  bar(kBarScFull + sb));
                    }
                    ++sc_issued;
                    const CUtensorMap* tma = ti.grp >= 0 ? &p.tm_a : &p.tm_a_sh;
                    const int nks = ti.K / kKStage;
                    for (int ks = 0; ks < nks; ++ks, ++it) {
                        const int s = it % kStages;
                        const uint32_t ph = (it / kStages) & 1;
                        if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1, abort_flag, p.hdr)) { ok = false; break; }
                        if ((int64_t)it == withheld) continue;  // its FULL phase never completes
                        const int brows = b_box_rows(ti.npad);
                        mbar_expect_tx(bar(kBarFull + s), (uint32_t)(kAStageBytes + brows * 256));
                        // one box each: the weight tile and both 64-wide K blocks of the activations
                        const uint32_t adst = sbase + kOffA + s * kAStageBytes;
                        if (MODE == kGateUp)  // rows m = 32*blk + 16*gu + i (gate/up interleaved)
                            tma_load_5d(adst, tma, ks * 64, 0, 0, 4 * ti.band, ti.grp >= 0 ? ti.grp : 0,
                                        bar(kBarFull + s));
                        else
                            tma_load_2d(adst, tma, ks * 64, weight_row<MODE>(p, ti, 0, 0), bar(kBarFull + s));
                        tma_load_3d(sbase + kOffB + s * kBStageBytes,
                                    brows == 32    ? &p.tm_b32
                                    : brows == 64  ? &p.tm_b64
                                    : brows == 128 ? &p.tm_b128
                                                   : &p.tm_b,
                                    0, ti.row0, 2 * ks,
                                    bar(kBarFull + s));
                    }
                    cur = nxt;
                }
                // do not leave with copies in flight: wait (bounded, whatever the abort
                // flag) for the stages and scale blocks issued last.  In a run that did
                // not abort their phases are complete and each test passes at once.
                for (uint32_t j = (it >= kStages ? it - kStages : 0); j < it; ++j)
                    if ((int64_t)j != withheld)
                        mbar_drain(bar(kBarFull + j % kStages), (j / kStages) & 1, p.hdr);
                for (int t = sc_issued > 2 ? sc_issued - 2 : 0; t < sc_issued; ++t)
                    mbar_drain(bar(kBarScFull + (t & 1)), (t >> 1) & 1, p.hdr);
            }
            __syncwarp();
        } else if (warp == 1 || warp == 2) {
            // ------------------------------------------------------------ MMA issuers
            // Two issuers on two schedulers: group gi (its own accumulator buffer
            // gi % kDBufs, fresh at its first K step) is issued by warp 1 + (gi & 1).
            // One issuing thread spent most of each stage on barrier and commit
            // latency next to the dequantiser and epilogue warps of its scheduler.
            const uint32_t me = (uint32_t)(warp - 1);
            if (lane == 0) {
                uint32_t it = 0, gi = 0;
                int64_t last = -1;  // last stage this issuer committed
                bool ok = true;
                int4 cur = load_tile(p, blockIdx.x, n_tiles);
                for (int tile = blockIdx.x; tile < n_tiles && ok; tile += grid) {
                    const int4 nxt = load_tile(p, tile + grid, n_tiles);
                    const TileInfo ti = decode_tile<G, MODE>(p, cur);
                    const uint32_t idesc = idesc_bf16(128, ti.npad);
                    // 16-byte units between the stage's two 64-wide K blocks of B
                    const int kb_units = b_box_rows(ti.npad) * 8;
                    const int nks = ti.K / kKStage;
                    for (int ks = 0; ks < nks && ok; ++ks, ++it) {
                        const int s = it % kStages;
                        const int ta = it % kAStagesT;
                        const uint32_t tph = (it / kAStagesT) & 1;
                        constexpr int kGroups = kKStage / G;
                        if (kGroups == 1 && (gi & 1) != me) {  // the other issuer's stage
                            ++gi;
                            continue;
                        }
                        // AREADY completes only after every dequantiser warp has seen FULL for
                        // this stage (A and B land on the same barrier), so it also orders the
                        // B tile before the MMAs
                        if (!mbar_wait(bar(kBarAReady + ta), tph, abort_flag, p.hdr)) { ok = false; break; }
                        tc_fence_after();
                        // descriptor of the stage's B tile; K steps add (kg/4) K blocks (box rows x
                        // 128 B each) + (kg%4)*32 B, in units of 16 bytes
                        const uint64_t bdesc0 = smem_desc_sw128(sbase + kOffB + s * kBStageBytes);
                        const uint32_t a0 = tmem + (uint32_t)(ta * 64);
    #pragma unroll
                        for (int gg = 0; gg < kGroups; ++gg, ++gi) {
                            if ((gi & 1) != me) continue;
                            const int b = gi % kDBufs;
                            if (!mbar_wait(bar(kBarDEmpty + b), ((gi / kDBufs) & 1) ^ 1, abort_flag, p.hdr)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t dcol = tmem + (uint32_t)(kTmemD + b * kAccCols);
    #pragma unroll
                            for (int kk = 0; kk < G / 16; ++kk) {
                                const int kg = gg * (G / 16) + kk;  // 16-wide K step within the stage
                                mma_ts(dcol, a0 + (uint32_t)(kg * 8),
                                       bdesc0 + (uint64_t)((kg >> 2) * kb_units + (kg & 3) * 2), idesc,
                                       kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar(kBarDFull + b));
                        }
                        if (!ok) break;
                        mma_commit(bar(kBarEmpty + s));
                        last = it;
                    }
                    cur = nxt;
                }
                // this issuer's MMAs are done before the CTA frees TMEM: a commit of its
                // own, waited for whatever the abort flag
                (void)last;
                mma_commit(bar(kBarTd + me));
                mbar_drain(bar(kBarTd + me), 0, p.hdr);
            }
            __syncwarp();
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------------ dequantisers
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegDq));
        const int q = warp & 3;
        const int h = (warp - kDequantWarp0) >> 2;  // which part of the stage's K
        constexpr int kChunks = 4 / kDqPerQuarter;  // 16-byte chunks (32 K each) per warp
        const int m = q * 32 + lane;  // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        int4 cur = load_tile(p, blockIdx.x, n_tiles);
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += grid) {
            const int4 nxt = load_tile(p, tile + grid, n_tiles);
            const TileInfo ti = decode_tile<G, MODE>(p, cur);
            const int nks = ti.K / kKStage;
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(bar(kBarFull + s), ph, abort_flag, p.hdr)) { ok = false; break; }
                // row m of the int4 tile: 64 bytes, 16-byte chunks 64B-swizzled by the TMA;
                // this warp's part is chunks kChunks * h .. kChunks * h + kChunks - 1
                const uint8_t* arow = smem + kOffA + s * kAStageBytes + m * 64;
                uint4 v[kChunks];
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    v[c] = *reinterpret_cast<const uint4*>(arow + (((kChunks * h + c) ^ ((m >> 1) & 3)) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarEmpty + s));
                uint32_t r[16 * kChunks];
                if (MODE == kGateUp) {  // activations stored block-permuted
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        nib8_to_bf16x2_paired(v[c].x, r + 16 * c + 0);
                        nib8_to_bf16x2_paired(v[c].y, r + 16 * c + 4);
                        nib8_to_bf16x2_paired(v[c].z, r + 16 * c + 8);
                        nib8_to_bf16x2_paired(v[c].w, r + 16 * c + 12);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        nib8_to_bf16x2(v[c].x, r + 16 * c + 0);
                        nib8_to_bf16x2(v[c].y, r + 16 * c + 4);
                        nib8_to_bf16x2(v[c].z, r + 16 * c + 8);
                        nib8_to_bf16x2(v[c].w, r + 16 * c + 12);
                    }
                }
                const int ta = it % kAStagesT;
                if (it >= kAStagesT) {  // TMEM stage ta is free once the MMAs of stage it - kAStagesT are done
                    const uint32_t j = it - kAStagesT;
                    if (!mbar_wait(bar(kBarEmpty + j % kStages), (j / kStages) & 1, abort_flag, p.hdr)) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
#pragma unroll
                for (int c2 = 0; c2 < kChunks / 2; ++c2)
                    tmem_st_x32(tmem + lane_base + (uint32_t)(ta * 64 + 32 * (h * kChunks / 2 + c2)), r + 32 * c2);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAReady + ta));
            }
            cur = nxt;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegEpi));
        // After a failed wait every epilogue warp keeps walking the same tiles
        // (skipping the work), so no warp waits on a barrier the others left.
        const int q = warp & 3;
        const int part = (warp - kEpilogueWarp0) >> 2;  // which of the quarter's epilogue warps
        const int m = q * 32 + lane;
        // the 32-column blocks part, part + kEpiPerQuarter, ..., so every warp of a
        // quarter has work whenever a tile holds more than 32 * (kEpiPerQuarter - 1)
        // tokens: acc[j] is column col(j)
        constexpr int kEpiCols = kAccCols / kEpiPerQuarter;
        static_assert(kEpiCols % 32 == 0, "whole 32-column blocks per epilogue warp");
        auto col = [&](int j) { return 32 * (kEpiPerQuarter * (j >> 5) + part) + (j & 31); };
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        // gate+up: row m is gate (gu = 0) or up (gu = 1) row f_local of the band
        const int gu = (m >> 4) & 1;
        const int f_local = (m >> 5) * 16 + (m & 15);
        uint32_t gi = 0;
        bool ok = true;
        int tc = 0;
        int4 cur = load_tile(p, blockIdx.x, n_tiles);
        for (int tile = blockIdx.x; tile < n_tiles; tile += grid, ++tc) {
            const int4 nxt = load_tile(p, tile + grid, n_tiles);
            const TileInfo ti = decode_tile<G, MODE>(p, cur);
            const int sb = tc & 1;
            if (ok && !mbar_wait(bar(kBarScFull + sb), (tc >> 1) & 1, abort_flag, p.hdr)) ok = false;
            const __half* sc = reinterpret_cast<const __half*>(smem + kOffSc + sb * kScBytes);
            const __half* srow = MODE == kGateUp ? sc + (gu * 64 + f_local) * ti.ng : sc + m * ti.ng;
            float acc[kEpiCols];
#pragma unroll
            for (int j = 0; j < kEpiCols; ++j) acc[j] = 0.f;
            for (int g = 0; g < ti.ng; ++g, ++gi) {
                const int b = gi % kDBufs;
                if (ok && !mbar_wait(bar(kBarDFull + b), (gi / kDBufs) & 1, abort_flag, p.hdr)) ok = false;
                if (!ok) continue;
                tc_fence_after();
                const float s = __half2float(srow[g]);
                const uint32_t dcol = tmem + lane_base + (uint32_t)(kTmemD + b * kAccCols);
                // the accumulator is released as soon as the warp's last block of it is
                // in registers, before that block's FMAs
#pragma unroll
                for (int blk = 0; blk < kEpiCols / 32; ++blk) {
                    const int c0 = 32 * (kEpiPerQuarter * blk + part);
                    const bool last = blk == kEpiCols / 32 - 1 || c0 + 32 * kEpiPerQuarter >= ti.npad;
                    uint32_t v[32];
                    if (c0 < ti.npad) {
                        tmem_ld_x32(dcol + (uint32_t)c0, v);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    }
                    if (last) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kBarDEmpty + b));
                    }
                    if (c0 < ti.npad) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2)
                            ffma2(acc[32 * blk + j], acc[32 * blk + j + 1], s, __uint_as_float(v[j]),
                                  __uint_as_float(v[j + 1]));
                    }
                    if (last) break;
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(bar(kBarScEmpty + sb));
            if (MODE == kGateUp) {
                // lane i holds gate row f, lane i ^ 16 the up row of the same f.  Step j
                // finishes column col(j) on the gate lanes and column col(j + kEpiCols / 2)
                // on the up lanes: each lane sends the value its partner needs, so every
                // lane computes one SwiGLU per step
                uint16_t* H = reinterpret_cast<uint16_t*>(p.out) + 64 * ti.band + f_local;
                const bool lo = (lane & 16) == 0;
#pragma unroll
                for (int j = 0; j < kEpiCols / 2; ++j) {
                    const float mine = lo ? acc[j] : acc[j + kEpiCols / 2];
                    const float other = __shfl_xor_sync(0xffffffffu, lo ? acc[j + kEpiCols / 2] : acc[j], 16);
                    const float gv = lo ? mine : other;
                    const float uv = lo ? other : mine;
                    const int nn = col(lo ? j : j + kEpiCols / 2);
                    if (ok && nn < ti.n)
                        H[(int64_t)(ti.row0 + nn) * p.ld_out] = float_to_bf16_bits(swiglu_f32(gv, uv));
                }
            } else if (ok) {
                float* Y = reinterpret_cast<float*>(p.out);
#pragma unroll
                for (int j = 0; j < kEpiCols; ++j) {
                    const int nn = col(j);
                    if (nn < ti.n) Y[(int64_t)(ti.row0 + nn) * p.ld_out + 128 * ti.band + m] = acc[j];
                }
            }
            cur = nxt;
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

// Gate+up activation rows in descriptor order: xs[r] = x[perm[r] / k] for the
// T*k routed rows, then xs[T*k + t] = x[t] for the shared expert.  Each
// 8-element block is stored as (x0, x4, x1, x5, x2, x6, x3, x7), the order of
// the dequantiser's weight pairs (nib8_to_bf16x2_paired).  One warp per row,
// 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int T,
                                                          int k, int d, uint16_t* __restrict__ xs) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t slots = (int64_t)T * k;
    if (r >= slots + T) return;
    const int64_t t = r < slots ? __ldg(perm + r) / k : r - slots;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    uint4* dst = reinterpret_cast<uint4*>(xs + r * d);
    for (int c = threadIdx.x & 31; c < d / 8; c += 32) {
        const uint4 v = __ldg(src + c);
        uint4 o;
        o.x = __byte_perm(v.x, v.z, 0x5410);
        o.y = __byte_perm(v.x, v.z, 0x7632);
        o.z = __byte_perm(v.y, v.w, 0x5410);
        o.w = __byte_perm(v.y, v.w, 0x7632);
        dst[c] = o;
    }
}

// ---------------------------------------------------------------- host side
}  // namespace

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

// General tiled map (rank <= 5); strides[i] is the byte stride of dim i + 1.
bool make_map_nd(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                 CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// Activation rows [rows][cols] bf16 read as {64 elements, box_rows rows, 2 K
// blocks}: one box fills both 64-wide K blocks of a stage.
bool make_act_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                  uint32_t box_rows) {
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 3, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_act_maps(GroupedParams& prm, const void* base, uint64_t cols, uint64_t rows) {
    return make_act_map(&prm.tm_b, base, cols, rows, kTokTile) &&
           make_act_map(&prm.tm_b128, base, cols, rows, 128) &&
           make_act_map(&prm.tm_b32, base, cols, rows, 32) &&
           make_act_map(&prm.tm_b64, base, cols, rows, 64);
}

// Gate+up int4 weights of `experts` experts ([experts][2Fg][d/2] bytes) read as
// {64 bytes of K, 16 rows, gate/up, 16-row blocks, expert}: one box holds 64
// gate rows and their 64 up rows interleaved in blocks of 16.
bool make_gateup_map(CUtensorMap* m, const void* base, uint64_t d, uint64_t Fg, uint64_t experts) {
    const uint64_t rb = d / 2;
    const cuuint64_t dims[5] = {rb, 16, 2, Fg / 16, experts};
    const cuuint64_t strides[4] = {rb, Fg * rb, 16 * rb, 2 * Fg * rb};
    const cuuint32_t box[5] = {64, 16, 2, 4, 1};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 5, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_64B);
}

// 2D row-major tensor [outer][inner] with rows row_bytes apart.
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

template <int G, int MODE, int DQ>
cudaError_t launch_gm(GroupedParams& prm, int sms, cudaStream_t st) {
    cudaError_t err = ensure_dynamic_smem((const void*)grouped_w4a16_kernel<G, MODE, DQ>, kSmemBytes);
    if (err != cudaSuccess) return err;
    // the warpgroups' setmaxnreg targets must fit in the registers the launch holds
    static int launch_regs = -1;
    if (launch_regs < 0) {
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, grouped_w4a16_kernel<G, MODE, DQ>);
        if (err != cudaSuccess) return err;
        launch_regs = fa.numRegs;
    }
    if (launch_regs * kThreads < Layout<DQ>::kRegBudget) return cudaErrorInvalidConfiguration;
    grouped_w4a16_kernel<G, MODE, DQ><<<sms, kThreads, kSmemBytes, st>>>(prm);
    return cudaGetLastError();
}

// A launch of at most 64 tokens has tiles of at most 64 tokens (kTileN >= 64): it
// takes the layout with two dequantisers per quarter; larger ones the layout
// with three epilogue warps per quarter.
constexpr int kSmallTileT = 64;

template <int G>
cudaError_t launch_g(GroupedParams& prm, int sms, cudaStream_t st) {
    if (prm.T <= kSmallTileT)
        return prm.mode == kGateUp ? launch_gm<G, kGateUp, 2>(prm, sms, st)
                                   : launch_gm<G, kDown, 2>(prm, sms, st);
    return prm.mode == kGateUp ? launch_gm<G, kGateUp, 1>(prm, sms, st)
                               : launch_gm<G, kDown, 1>(prm, sms, st);
}

cudaError_t launch(GroupedParams& prm, cudaStream_t st) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    switch (prm.group) {
        case 32: return launch_g<32>(prm, sms, st);
        case 64: return launch_g<64>(prm, sms, st);
        case 128: return launch_g<128>(prm, sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool grouped_supported(const moe_dims_t& d) {
    const int Fmax = std::max(d.F, d.F_s);
    return d.d % kKStage == 0 && d.F % kKStage == 0 && d.F_s % kKStage == 0 &&
           d.d / d.group <= kMaxGroupsPerRow && Fmax / d.group <= kMaxGroupsPerRow &&
           d.F % 64 == 0 && d.F_s % 64 == 0 && d.group % 16 == 0 && kKStage % d.group == 0;
}

cudaError_t launch_gateup_grouped(const uint16_t* x, const moe_dims_t& d, const int32_t* perm,
                                  moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H, WsHeader* hdr,
                                  const int4* tiles, uint16_t* xs, cudaStream_t st) {
    const int64_t rows = (int64_t)d.T * d.k + d.T;
    gather_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(x, perm, d.T, d.k, d.d, xs);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    GroupedParams prm;
    memset(&prm, 0, sizeof(prm));
    const int Fmax = std::max(d.F, d.F_s);
    if (!make_act_maps(prm, xs, d.d, rows) ||
        !make_gateup_map(&prm.tm_a, Wgu.q, d.d, d.F, d.E) ||
        !make_gateup_map(&prm.tm_a_sh, Wgu_s.q, d.d, d.F_s, 1))
        return cudaErrorInvalidValue;
    prm.s_routed = reinterpret_cast<const __half*>(Wgu.s);
    prm.s_shared = reinterpret_cast<const __half*>(Wgu_s.s);
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
    if (!make_act_maps(prm, H, Fmax, rows) ||
        !make_map(&prm.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wd.q, d.F / 2, (uint64_t)d.E * d.d,
                  d.F / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&prm.tm_a_sh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wd_s.q, d.F_s / 2, (uint64_t)d.d,
                  d.F_s / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    prm.s_routed = reinterpret_cast<const __half*>(Wd.s);
    prm.s_shared = reinterpret_cast<const __half*>(Wd_s.s);
    prm.tiles = tiles;
    prm.hdr = hdr;
    prm.out = Y;
    prm.ld_out = d.d;
    prm.mode = kDown;
    prm.T = d.T; prm.d = d.d; prm.k = d.k; prm.F = d.F; prm.Fs = d.F_s; prm.group = d.group;
    return launch(prm, st);
}

}  // namespace moe
