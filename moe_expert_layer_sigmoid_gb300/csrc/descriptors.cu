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

__global__ void __launch_bounds__(kScatterThreads)
desc_scatter(const int32_t* __restrict__ topk_idx, int64_t nslots, int E,
             const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ perm, int32_t* __restrict__ pos, int32_t* __restrict__ sched,
             WsHeader* hdr) {
    __shared__ int red[4][kScatterThreads / 32];
    __shared__ int warp_tot[kScatterThreads / 32];
    const int e = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int my_count = counts[e];
    int off = 0, rank = 0, active = 0, total = 0;
    for (int e2 = tid; e2 < E; e2 += kScatterThreads) {
        const int c2 = counts[e2];
        if (e2 < e) off += c2;
        if (c2 > my_count || (c2 == my_count && e2 < e)) ++rank;
        active += (c2 > 0);
        total += c2;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        rank += __shfl_xor_sync(0xffffffffu, rank, o);
        active += __shfl_xor_sync(0xffffffffu, active, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if (lane == 0) {
        red[0][warp] = off;
        red[1][warp] = rank;
        red[2][warp] = active;
        red[3][warp] = total;
    }
    __syncthreads();
    if (tid == 0) {
        int o = 0, r = 0, a = 0, tt = 0;
        for (int w = 0; w < kScatterThreads / 32; ++w) {
            o += red[0][w];
            r += red[1][w];
            a += red[2][w];
            tt += red[3][w];
        }
        red[0][0] = o;
        offsets[e] = o;
        sched[r] = e;
        if (e == E - 1) offsets[E] = o + my_count;
        if (e == 0) {
            if (hdr) hdr->n_active = a;
            if ((int64_t)tt != nslots) record_error(hdr, kErrCountMismatch);
        }
    }
    __syncthreads();
    const int base_row = red[0][0];
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
    (void)tiles;
    (void)max_tiles;
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
    desc_scatter<<<d.E, kScatterThreads, 0, st>>>(topk_idx, nslots, d.E, counts, offsets, perm,
                                                  pos, sched, hdr);
    return cudaGetLastError();
}

}  // namespace moe
