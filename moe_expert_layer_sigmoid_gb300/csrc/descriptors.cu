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
// The sort is a stable counting sort: a count pass, then one CTA per expert
// that computes its offset and its schedule rank from the counts and
// compacts that expert's slots in slot order.  Nothing depends on the order in
// which atomics land, so the result is bit-reproducible.
#include "common.cuh"

namespace moe {
namespace {

__global__ void desc_count(const int32_t* __restrict__ topk_idx, int64_t nslots, int E,
                           int32_t* __restrict__ counts, WsHeader* hdr) {
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < nslots;
         s += (int64_t)gridDim.x * blockDim.x) {
        const int e = topk_idx[s];
        if (e < 0 || e >= E) {
            record_error(hdr, kErrBadExpertId);
            continue;
        }
        atomicAdd(counts + e, 1);
    }
}

constexpr int kScatterThreads = 256;

// Tile schedule of the grouped tcgen05 kernels.  A token tile is up to 128
// consecutive rows of one group (routed expert or the shared expert); a tile
// pairs it with one weight band (gate+up: 64 gate rows and their 64 up rows;
// down: 128 output channels).  Groups run largest first: the shared expert,
// then the routed experts in schedule order.  Within a group the order is
// N-banded, band-major then token tiles, so CTAs running neighbouring tiles
// read the same weight band (L2 reuse); with MOE_FLAG_NO_SCHED groups go in
// expert-id order and tiles token-tile-major.
struct TileGeom {
    int T, k, nb_gu_routed, nb_gu_shared, nb_dn;
    bool sched;
    int64_t max_tiles;
};

__device__ __forceinline__ void write_group_tiles(int4* tiles, int list, int64_t base, int grp,
                                                  int row0, int count, int nb, bool banded,
                                                  int64_t max_tiles, WsHeader* hdr) {
    const int ntt = (count + 127) / 128;
    for (int i = threadIdx.x; i < ntt * nb; i += blockDim.x) {
        const int band = banded ? i / ntt : i % nb;
        const int tt = banded ? i % ntt : i / nb;
        const int64_t idx = base + i;
        if (idx >= max_tiles) {
            record_error(hdr, kErrBadTile);
            continue;
        }
        tiles[list * max_tiles + idx] =
            make_int4(grp, row0 + 128 * tt, min(128, count - 128 * tt), band);
    }
}

__global__ void __launch_bounds__(kScatterThreads)
desc_scatter(const int32_t* __restrict__ topk_idx, int64_t nslots, int E,
             const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ perm, int32_t* __restrict__ pos, int32_t* __restrict__ sched,
             WsHeader* hdr, int4* __restrict__ tiles, TileGeom tg) {
    __shared__ int red[6][kScatterThreads / 32];
    __shared__ int warp_tot[kScatterThreads / 32];
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
        const int ntt2 = (c2 + 127) / 128;
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
    const int ntt_sh = (tg.T + 127) / 128;
    if (shared_cta) {
        const int row0 = (int)nslots;
        write_group_tiles(tiles, 0, 0, -1, row0, tg.T, tg.nb_gu_shared, tg.sched, tg.max_tiles, hdr);
        write_group_tiles(tiles, 1, 0, -1, row0, tg.T, tg.nb_dn, tg.sched, tg.max_tiles, hdr);
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
                          e, base_row, my_count, tg.nb_gu_routed, tg.sched, tg.max_tiles, hdr);
        write_group_tiles(tiles, 1, (int64_t)(ntt_sh + tb) * tg.nb_dn, e, base_row, my_count,
                          tg.nb_dn, tg.sched, tg.max_tiles, hdr);
    }
    if (my_count == 0) return;
    int running = 0;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t b = 0; b < nslots; b += kScatterThreads) {
        const int64_t s = b + tid;
        const bool hit = s < nslots && topk_idx[s] == e;
        const unsigned ball = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) warp_tot[warp] = __popc(ball);
        __syncthreads();
        int before = running, blk = 0;
        for (int w = 0; w < kScatterThreads / 32; ++w) {
            if (w < warp) before += warp_tot[w];
            blk += warp_tot[w];
        }
        if (hit) {
            const int r = base_row + before + __popc(ball & lt_mask);
            perm[r] = (int32_t)s;
            pos[s] = r;
        }
        running += blk;
        __syncthreads();
        if (running >= my_count) break;
    }
}

}  // namespace

cudaError_t launch_descriptors(const int32_t* topk_idx, const moe_dims_t& d, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched,
                               WsHeader* hdr, int4* tiles, int64_t max_tiles, cudaStream_t st) {
    const int64_t nslots = (int64_t)d.T * d.k;
    cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)d.E, st);
    if (err != cudaSuccess) return err;
    const int threads = 256;
    int blocks = (int)((nslots + threads - 1) / threads);
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    desc_count<<<blocks, threads, 0, st>>>(topk_idx, nslots, d.E, counts, hdr);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    TileGeom tg;
    tg.T = d.T;
    tg.k = d.k;
    tg.nb_gu_routed = d.F / 64;
    tg.nb_gu_shared = d.F_s / 64;
    tg.nb_dn = d.d / 128;
    tg.sched = !(d.flags & MOE_FLAG_NO_SCHED);
    tg.max_tiles = max_tiles;
    desc_scatter<<<d.E + 1, kScatterThreads, 0, st>>>(topk_idx, nslots, d.E, counts, offsets,
                                                      perm, pos, sched, hdr, tiles, tg);
    return cudaGetLastError();
}

}  // namespace moe
