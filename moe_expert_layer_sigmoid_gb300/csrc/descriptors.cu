// On-device expert descriptors.
//
// The prefill MoE runs its experts as a grouped GEMM over descriptors built on
// the device (thewafflehaus/butter PR #69, commit "feat(laguna): batched
// prefill with tensor-core projections, fused MoE, CTA scheduling"); the
// descriptor form here follows the Nemotron W4A16 MoE commit of
// thewafflehaus/FFAI PR #72: CSR offsets with E + 1 entries and a
// router-sorted token index, built without any host round trip so the layer
// stays graph-capturable.
//
//   counts[e]  slots routed to expert e
//   offsets    exclusive scan of counts, E + 1 entries
//   perm[r]    slot id t*k + j of row r; rows sorted by (expert, token)
//   pos[s]     row of slot s (inverse of perm)
//   sched[i]   experts by count, largest first, ties to the lower id
//
// The sort is a stable counting sort over blocks of 1024 slots: per-block
// expert histograms, their sums and per-block prefixes (one thread per
// expert), one CTA per expert for its offset, schedule rank and tiles, and a
// placement pass in which every block writes its slots at
//   offsets[e] + (earlier blocks' slots of e) + (earlier slots of e in this block),
// the last term from warp-range prefixes and a match within each 32-slot
// chunk.  Nothing depends on the order in which atomics land, so the result
// is bit-reproducible.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kDescSlots = 1024;   // slots per block of the counting sort
constexpr int kDescThreads = 256;  // 8 warps of 128 slots each

// Per-block expert histogram: hist[b][e] = slots of block b routed to e.
__global__ void __launch_bounds__(kDescThreads)
desc_hist(const int32_t* __restrict__ topk_idx, int64_t nslots, int E, int32_t* __restrict__ hist,
          WsHeader* hdr) {
    extern __shared__ int h_smem[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h_smem[e] = 0;
    __syncthreads();
    const int64_t s0 = (int64_t)blockIdx.x * kDescSlots;
    for (int i = threadIdx.x; i < kDescSlots; i += blockDim.x) {
        const int64_t s = s0 + i;
        if (s >= nslots) break;
        const int e = __ldg(topk_idx + s);
        if (e < 0 || e >= E) {
            record_error(hdr, kErrBadExpertId);
            continue;
        }
        atomicAdd(h_smem + e, 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = h_smem[e];
}

// counts[e] = sum over blocks; hist[b][e] becomes the exclusive prefix over blocks.
__global__ void desc_counts(int32_t* __restrict__ hist, int nblk, int E, int32_t* __restrict__ counts) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
        const int c = hist[(int64_t)b * E + e];
        hist[(int64_t)b * E + e] = run;
        run += c;
    }
    counts[e] = run;
}

// Stable placement of block b's slots: perm[row] = slot, pos[slot] = row.
__global__ void __launch_bounds__(kDescThreads)
desc_place(const int32_t* __restrict__ topk_idx, int64_t nslots, int E,
           const int32_t* __restrict__ offsets, const int32_t* __restrict__ blkoff,
           int32_t* __restrict__ perm, int32_t* __restrict__ pos) {
    extern __shared__ int w_smem[];  // [8 warps][E]: slots of e in earlier warp ranges, then running
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = kDescThreads / 32, kRange = kDescSlots / kWarps;
    const int64_t s0 = (int64_t)blockIdx.x * kDescSlots + warp * kRange;
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) w_smem[i] = 0;
    __syncthreads();
    int* mine = w_smem + warp * E;
    for (int c = 0; c < kRange; c += 32) {  // warp range histogram
        const int64_t s = s0 + c + lane;
        const int e = s < nslots ? __ldg(topk_idx + s) : -1;
        if (e >= 0 && e < E) atomicAdd(mine + e, 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {  // exclusive prefix over the warps
        int run = offsets[e] + blkoff[(int64_t)blockIdx.x * E + e];
        for (int w = 0; w < kWarps; ++w) {
            const int c = w_smem[w * E + e];
            w_smem[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int c = 0; c < kRange; c += 32) {
        const int64_t s = s0 + c + lane;
        const int e = s < nslots ? __ldg(topk_idx + s) : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned grp = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok) {
            const int r = mine[e] + __popc(grp & lt);
            perm[r] = (int32_t)s;
            pos[s] = r;
        }
        __syncwarp();
        if (ok && (grp & lt) == 0) mine[e] += __popc(grp);  // the group's first lane
        __syncwarp();
    }
}

constexpr int kScatterThreads = 256;

// Tile schedule of the grouped tcgen05 kernels.  A token tile is up to tn (192
// for the W4A16 kernel, 256 for the W8A8 kernel) consecutive rows of one group (routed expert or the shared expert); a tile
// pairs it with one weight band (gate+up: 64 gate rows and their 64 up rows;
// down: 128 output channels).  Groups run largest first: the shared expert,
// then the routed experts in schedule order.  Within a group the order is
// N-banded, band-major then token tiles, so CTAs running neighbouring tiles
// read the same weight band (L2 reuse); with MOE_FLAG_NO_SCHED groups go in
// expert-id order and tiles token-tile-major.
struct TileGeom {
    int T, k, nb_gu_routed, nb_gu_shared, nb_dn, tn;
    bool sched;
    int64_t max_tiles;
};

__device__ __forceinline__ void write_group_tiles(int4* tiles, int list, int64_t base, int grp,
                                                  int row0, int count, int nb, bool banded, int tn,
                                                  int64_t max_tiles, WsHeader* hdr) {
    const int ntt = (count + tn - 1) / tn;
    for (int i = threadIdx.x; i < ntt * nb; i += blockDim.x) {
        const int band = banded ? i / ntt : i % nb;
        const int tt = banded ? i % ntt : i / nb;
        const int64_t idx = base + i;
        if (idx >= max_tiles) {
            record_error(hdr, kErrBadTile);
            continue;
        }
        tiles[list * max_tiles + idx] =
            make_int4(grp, row0 + tn * tt, min(tn, count - tn * tt), band);
    }
}

__global__ void __launch_bounds__(kScatterThreads)
desc_plan(int64_t nslots, int E, const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
          int32_t* __restrict__ sched, WsHeader* hdr, int4* __restrict__ tiles, TileGeom tg) {
    __shared__ int red[6][kScatterThreads / 32];
    const bool shared_cta = blockIdx.x == E;  // the last CTA schedules the shared expert
    const int e = shared_cta ? 0 : blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int my_count = counts[e];
    // off: rows before e; rank: schedule position; tt_before: token tiles of the
    // routed groups scheduled before e; tt_all: token tiles of every routed group
    int off = 0, rank = 0, active = 0, total = 0, tt_before = 0, tt_all = 0;
    for (int e2 = tid; e2 < E; e2 += kScatterThreads) {
        const int c2 = counts[e2];
        const bool before = c2 > my_count || (c2 == my_count && e2 < e);
        const int ntt2 = (c2 + tg.tn - 1) / tg.tn;
        if (e2 < e) off += c2;
        if (before) ++rank;
        if (tg.sched ? before : e2 < e) tt_before += ntt2;
        tt_all += ntt2;
        active += (c2 > 0);
        total += c2;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        rank += __shfl_xor_sync(0xffffffffu, rank, o);
        active += __shfl_xor_sync(0xffffffffu, active, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
        tt_before += __shfl_xor_sync(0xffffffffu, tt_before, o);
        tt_all += __shfl_xor_sync(0xffffffffu, tt_all, o);
    }
    if (lane == 0) {
        red[0][warp] = off;
        red[1][warp] = rank;
        red[2][warp] = active;
        red[3][warp] = tt_before;
        red[4][warp] = tt_all;
        red[5][warp] = total;
    }
    __syncthreads();
    if (tid == 0) {
        int o = 0, r = 0, a = 0, tt = 0, tb = 0, ta = 0;
        for (int w = 0; w < kScatterThreads / 32; ++w) {
            o += red[0][w];
            r += red[1][w];
            a += red[2][w];
            tt += red[5][w];
            tb += red[3][w];
            ta += red[4][w];
        }
        red[0][0] = o;
        red[3][0] = tb;
        red[4][0] = ta;
        if (!shared_cta) {
            offsets[e] = o;
            sched[r] = e;
            if (e == E - 1) offsets[E] = o + my_count;
            if (e == 0) {
                if (hdr) hdr->n_active = a;
                if ((int64_t)tt != nslots) record_error(hdr, kErrCountMismatch);
            }
        }
    }
    __syncthreads();
    const int base_row = red[0][0];
    const int ntt_sh = (tg.T + tg.tn - 1) / tg.tn;
    if (shared_cta) {
        const int row0 = (int)nslots;
        write_group_tiles(tiles, 0, 0, -1, row0, tg.T, tg.nb_gu_shared, tg.sched, tg.tn, tg.max_tiles,
                          hdr);
        write_group_tiles(tiles, 1, 0, -1, row0, tg.T, tg.nb_dn, tg.sched, tg.tn, tg.max_tiles, hdr);
        if (tid == 0 && hdr) {
            const int ta = red[4][0];
            hdr->n_tiles[0] = ntt_sh * tg.nb_gu_shared + ta * tg.nb_gu_routed;
            hdr->n_tiles[1] = (ntt_sh + ta) * tg.nb_dn;
        }
        return;
    }
    if (my_count > 0) {
        const int tb = red[3][0];
        write_group_tiles(tiles, 0, (int64_t)ntt_sh * tg.nb_gu_shared + (int64_t)tb * tg.nb_gu_routed,
                          e, base_row, my_count, tg.nb_gu_routed, tg.sched, tg.tn, tg.max_tiles, hdr);
        write_group_tiles(tiles, 1, (int64_t)(ntt_sh + tb) * tg.nb_dn, e, base_row, my_count,
                          tg.nb_dn, tg.sched, tg.tn, tg.max_tiles, hdr);
    }
}

}  // namespace

int desc_blocks(int64_t nslots) { return (int)((nslots + kDescSlots - 1) / kDescSlots); }

cudaError_t launch_descriptors(const int32_t* topk_idx, const moe_dims_t& d, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched,
                               WsHeader* hdr, int4* tiles, int64_t max_tiles, int32_t* hist,
                               cudaStream_t st, int tile_n) {
    const int64_t nslots = (int64_t)d.T * d.k;
    const int nblk = desc_blocks(nslots);
    const size_t hist_smem = sizeof(int) * (size_t)d.E;
    const size_t place_smem = sizeof(int) * (size_t)(kDescThreads / 32) * d.E;
    cudaError_t err = ensure_dynamic_smem((const void*)desc_place, place_smem);
    if (err != cudaSuccess) return err;
    if (nblk > 0) {
        desc_hist<<<nblk, kDescThreads, hist_smem, st>>>(topk_idx, nslots, d.E, hist, hdr);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    desc_counts<<<(d.E + 255) / 256, 256, 0, st>>>(hist, nblk, d.E, counts);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    TileGeom tg;
    tg.T = d.T;
    tg.k = d.k;
    tg.nb_gu_routed = d.F / 64;
    tg.nb_gu_shared = d.F_s / 64;
    tg.nb_dn = d.d / 128;
    tg.sched = !(d.flags & MOE_FLAG_NO_SCHED);
    tg.max_tiles = max_tiles;
    tg.tn = tile_n;
    desc_plan<<<d.E + 1, kScatterThreads, 0, st>>>(nslots, d.E, counts, offsets, sched, hdr, tiles, tg);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (nblk > 0) {
        desc_place<<<nblk, kDescThreads, place_smem, st>>>(topk_idx, nslots, d.E, offsets, hist,
                                                            perm, pos);
        err = cudaGetLastError();
    }
    return err;
}

}  // namespace moe
