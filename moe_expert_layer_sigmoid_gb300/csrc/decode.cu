// Decode-side routing (T <= 64) in one launch.
//
// The pages' decode step keeps the whole MoE layer on the device and replays
// it as a CUDA graph (thewafflehaus/butter PR #69, commit "feat(laguna):
// Laguna-S-2.1 decode on the CUDA engine"); the descriptors are built by one
// device kernel, not a host round trip (thewafflehaus/FFAI PR #72, Nemotron
// W4A16 MoE commit).  At T = 1 every one of those steps is a few microseconds
// of latency, so here the router logits, the top-k and the descriptors are one
// kernel:
//
//   1. every CTA computes split-K logit partials (router_gemv_warp);
//   2. the last CTA to finish (completion counter in the workspace header,
//      reset by that CTA) takes the top-k of each token and builds counts,
//      offsets, perm, pos, sched and n_active with the same definitions as
//      moe_build_descriptors (stable by token, schedule by count then id);

#include "router_dev.cuh"

namespace moe {
namespace {

constexpr int kMaxDecodeK = 32;
constexpr int kRouterThreads = 256;
constexpr int kRankTopkMaxT = 8;     // T up to this: rank-count top-k over the whole CTA
constexpr int kRankTopkKeys = 2048;  // keys held at once by the rank-count top-k

struct DecodeRouterArgs {
    const uint16_t* x;
    const float* W_r;
    const float* bias;
    int T, d, E, k, kchunk;
    float* partial;
    int32_t* topk_idx;
    float* topk_w;
    float* margin;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* pos;
    int32_t* sched;
    WsHeader* hdr;
};

// Block-wide exclusive scan of one int per thread (kRouterThreads threads).
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();  // s_warp is reused across calls
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kRouterThreads / 32; ++w) {
        const int t = s_warp[w];
        if (w < warp) before += t;
        all += t;
    }
    *total = all;
    return before + incl - v;
}

// Top-k of tokens t0 .. t0 + G - 1 by rank counting, the whole CTA: P = 256 / G
// threads per token, each holding experts j, j + P, ...  The rank of expert e
// is the number of experts whose key beats e's (a larger key, or an equal key
// and a lower id), so the experts of rank < k are exactly the k rounds of
// arg-max that router_topk_warp takes, in the same order.  A NaN key ranks as
// -inf.  Writes topk_idx / topk_w (normalised by the selected scores summed in
// selection order), margin, and s_idx for the descriptors.
__device__ __forceinline__ void topk_rank_block(const DecodeRouterArgs& a, int ksplit, int t0,
                                                int G, float* s_key, float* s_sc, int* s_sel_e,
                                                float* s_sel_s, float* s_gap, int32_t* s_idx) {
    const int E = a.E, k = a.k, T = a.T;
    const int Ep = (E + 3) & ~3;  // key row stride: 16-byte rows, padded with -inf
    const int P = kRouterThreads / G;
    const int g = threadIdx.x / P, j = threadIdx.x - g * P;
    const int t = t0 + g;
    const bool live = g < G && t < T;
    if (live) {
        for (int e = j; e < E; e += P) {
            const float l = router_logit(a.partial, ksplit, T, E, t, e);
            const float sc = 1.0f / (1.0f + expf(-l));
            float key = sc + __ldg(a.bias + e);
            if (key != key) key = -INFINITY;
            s_key[g * Ep + e] = key;
            s_sc[g * Ep + e] = sc;
        }
        if (j < Ep - E) s_key[g * Ep + E + j] = -INFINITY;
    }
    __syncthreads();
    if (live) {
        const float* kk = s_key + g * Ep;
        for (int e = j; e < E; e += P) {
            const float key = kk[e];
            // experts below e win ties, the others must be strictly larger
            int rank = 0;
            int e2 = 0;
            for (; e2 + 4 <= e; e2 += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(kk + e2);
                rank += (k4.x >= key) + (k4.y >= key) + (k4.z >= key) + (k4.w >= key);
            }
            for (; e2 < e; ++e2) rank += kk[e2] >= key;
            for (++e2; e2 < E && (e2 & 3); ++e2) rank += kk[e2] > key;
#pragma unroll 4
            for (; e2 < E; e2 += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(kk + e2);
                rank += (k4.x > key) + (k4.y > key) + (k4.z > key) + (k4.w > key);
            }
            if (rank < k) {
                s_sel_e[g * kMaxDecodeK + rank] = e;
                s_sel_s[g * kMaxDecodeK + rank] = s_sc[g * Ep + e];
            }
            if (rank == k - 1) s_gap[2 * g] = key;
            if (rank == k) s_gap[2 * g + 1] = key;
        }
    }
    __syncthreads();
    if (live && j < k) {
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += s_sel_s[g * kMaxDecodeK + r];
        const int e = s_sel_e[g * kMaxDecodeK + j];
        a.topk_idx[(int64_t)t * k + j] = e;
        a.topk_w[(int64_t)t * k + j] = __fdiv_rn(s_sel_s[g * kMaxDecodeK + j], sum);
        s_idx[t * k + j] = e;
        if (a.margin && j == 0) a.margin[t] = k < E ? s_gap[2 * g] - s_gap[2 * g + 1] : INFINITY;
    }
    __syncthreads();
}

// Single token, E <= 256: one expert per thread.  Each warp sorts its 32 keys
// and keeps its best k + 1 as candidates; a candidate's rank among all
// candidates is its rank among all experts (an expert outside its warp's best
// k + 1 has rank above k).  The descriptors of one token follow directly:
// the k chosen experts have one row each, in id order.
__device__ __forceinline__ void decode_route_one(const DecodeRouterArgs& a, int ksplit,
                                                 float* s_ckey, float* s_cs, int32_t* s_ce,
                                                 int* s_sel_e, float* s_sel_s, float* s_gap) {
    const int E = a.E, k = a.k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = min(k + 1, 32);  // candidates per warp
    {
        const int e = tid;
        float key = -INFINITY, sc = 0.f;
        int ee = 0x7fffffff;
        if (e < E) {
            const float l = router_logit(a.partial, ksplit, 1, E, 0, e);
            sc = 1.0f / (1.0f + expf(-l));
            key = sc + __ldg(a.bias + e);
            if (key != key) key = -INFINITY;
            ee = e;
        }
        warp_bitonic<true>(key, ee, sc, lane);
        if (lane < nc) {
            s_ckey[warp * nc + lane] = key;
            s_ce[warp * nc + lane] = ee;
            s_cs[warp * nc + lane] = sc;
        }
    }
    __syncthreads();
    const int ncand = nc * (kRouterThreads / 32);
    if (tid < ncand) {
        const float key = s_ckey[tid];
        const int e = s_ce[tid];
        if (e < E) {
            int rank = 0;
            for (int j = 0; j < ncand; ++j) {
                const int e2 = s_ce[j];
                rank += e2 < E && router_better(s_ckey[j], e2, key, e);
            }
            if (rank < k) {
                s_sel_e[rank] = e;
                s_sel_s[rank] = s_cs[tid];
            }
            if (rank == k - 1) s_gap[0] = key;
            if (rank == k) s_gap[1] = key;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // outputs of the selection, then the chosen ids sorted ascending with
        // their slots: row r of the descriptors is the r-th smallest id
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += s_sel_s[r];
        int e = 0x7fffffff;
        float slot = 0.f;
        if (lane < k) {
            e = s_sel_e[lane];
            a.topk_idx[lane] = e;
            a.topk_w[lane] = __fdiv_rn(s_sel_s[lane], sum);
            slot = (float)lane;
        }
        if (a.margin && lane == 0) a.margin[0] = k < E ? s_gap[0] - s_gap[1] : INFINITY;
        float dummy = 0.f;
        warp_bitonic<false>(dummy, e, slot, lane);
        if (lane < k) {
            const int j = (int)slot;
            a.perm[lane] = j;
            a.pos[j] = lane;
            a.sched[lane] = e;
            s_ce[lane] = e;  // sorted ids for the per-expert pass
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouterThreads) {
        int lb = 0;  // chosen ids below e
        while (lb < k && s_ce[lb] < e) ++lb;
        const bool chosen = lb < k && s_ce[lb] == e;
        a.counts[e] = chosen ? 1 : 0;
        a.offsets[e] = lb;
        if (!chosen) a.sched[k + (e - lb)] = e;
    }
    if (tid == 0) {
        a.offsets[E] = k;
        a.hdr->n_active = k;
    }
}

template <int NV>
__global__ void __launch_bounds__(kRouterThreads) router_decode_kernel(const DecodeRouterArgs a) {
    __shared__ int32_t s_idx[kMaxDecodeT * kMaxDecodeK];
    __shared__ int32_t s_cnt[kMaxExperts];
    __shared__ int32_t s_cur[kMaxExperts];
    __shared__ int32_t s_act[kMaxExperts];
    __shared__ int s_warp[kRouterThreads / 32];
    __shared__ int s_last;
    __shared__ __align__(16) float s_key[kRankTopkKeys];
    __shared__ float s_sc[kRankTopkKeys];
    __shared__ int s_sel_e[kRankTopkMaxT * kMaxDecodeK];
    __shared__ float s_sel_s[kRankTopkMaxT * kMaxDecodeK];
    __shared__ float s_gap[2 * kRankTopkMaxT];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nblk = gridDim.x * gridDim.y;
    const int T = a.T, E = a.E, k = a.k;

    pdl_trigger();  // the expert kernels may start; they wait for this grid before reading it

    {
        const int e = blockIdx.x * 8 + warp;
        if (e < E) router_gemv_warp(a.x, a.W_r, T, a.d, E, e, blockIdx.y, a.kchunk, a.partial, lane);
    }

    // last-CTA election
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&a.hdr->done[0], 1) == nblk - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) a.hdr->done[0] = 0;  // every CTA has arrived: ready for the next launch

    if (T == 1 && E <= kRouterThreads) {
        decode_route_one(a, gridDim.y, s_key, s_sc, s_act, s_sel_e, s_sel_s, s_gap);
        return;
    }

    // ---- top-k: few tokens by rank counting over the whole CTA, more tokens
    // one warp per token
    const int G = min(kRankTopkMaxT, kRankTopkKeys / ((E + 3) & ~3));
    if (T <= G) {
        topk_rank_block(a, gridDim.y, 0, T, s_key, s_sc, s_sel_e, s_sel_s, s_gap, s_idx);
    } else {
        for (int t = warp; t < T; t += kRouterThreads / 32) {
            int sel;
            router_topk_warp<NV>(a.partial, gridDim.y, a.bias, T, E, k, t, lane, a.topk_idx,
                                 a.topk_w, a.margin, &sel);
            if (lane < k) s_idx[t * k + lane] = sel;
        }
    }
    for (int e = tid; e < E; e += kRouterThreads) s_cnt[e] = 0;
    __syncthreads();

    // ---- counts (a selection outside [0, E) can only come from non-finite scores)
    const int nslots = T * k;
    for (int s = tid; s < nslots; s += kRouterThreads) {
        const int e = s_idx[s];
        if (e >= 0 && e < E)
            atomicAdd(&s_cnt[e], 1);
        else
            record_error(a.hdr, kErrBadExpertId);
    }
    __syncthreads();

    // ---- offsets (exclusive scan of counts) and the active list in id order;
    // thread tid owns experts [tid * per, (tid + 1) * per)
    const int per = (E + kRouterThreads - 1) / kRouterThreads;
    const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
    int my_rows = 0, my_act = 0;
    for (int e = e_lo; e < e_hi; ++e) {
        my_rows += s_cnt[e];
        my_act += s_cnt[e] > 0;
    }
    int rows_total, n_act;
    int row = block_excl_scan(my_rows, &rows_total, s_warp);
    int act = block_excl_scan(my_act, &n_act, s_warp);
    const int act_lo = act;
    for (int e = e_lo; e < e_hi; ++e) {
        const int c = s_cnt[e];
        a.counts[e] = c;
        a.offsets[e] = row;
        s_cur[e] = row;
        row += c;
        if (c > 0) s_act[act++] = e;
    }
    if (tid == 0) {
        a.offsets[E] = rows_total;
        a.hdr->n_active = n_act;
        if (rows_total != nslots) record_error(a.hdr, kErrCountMismatch);
    }
    __syncthreads();

    // ---- schedule: active experts by count (largest first, ties to the lower
    // id), then the idle experts in id order
    for (int i = tid; i < n_act; i += kRouterThreads) {
        const int e = s_act[i], c = s_cnt[e];
        int rank = 0;
        for (int j = 0; j < n_act; ++j) {
            const int e2 = s_act[j], c2 = s_cnt[e2];
            rank += (c2 > c) || (c2 == c && e2 < e);
        }
        a.sched[rank] = e;
    }
    {
        int idle_before = e_lo - act_lo;  // idle experts with a lower id
        for (int e = e_lo; e < e_hi; ++e)
            if (s_cnt[e] == 0) a.sched[n_act + idle_before++] = e;
    }

    // ---- perm / pos: rows of an expert in token order (a token's k experts
    // are distinct, so the k lanes of one token never share a cursor)
    if (warp == 0) {
        for (int t = 0; t < T; ++t) {
            if (lane < k) {
                const int s = t * k + lane;
                const int e = s_idx[s];
                if (e >= 0 && e < E) {
                    const int r = s_cur[e]++;
                    a.perm[r] = s;
                    a.pos[s] = r;
                } else {
                    a.pos[s] = nslots;  // the shared row: keeps the combine in bounds
                }
            }
            __syncwarp();
        }
    }
}

}  // namespace

cudaError_t launch_router_decode(const uint16_t* x, const float* W_r, const float* bias,
                                 const moe_dims_t& d, int32_t* topk_idx, float* topk_w,
                                 float* margin, float* logits, int ksplit, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched,
                                 WsHeader* hdr, cudaStream_t st) {
    if (d.T > kMaxDecodeT || d.k > kMaxDecodeK || d.E > kMaxExperts) return cudaErrorInvalidValue;
    DecodeRouterArgs a;
    a.x = x;
    a.W_r = W_r;
    a.bias = bias;
    a.T = d.T;
    a.d = d.d;
    a.E = d.E;
    a.k = d.k;
    a.kchunk = d.d / ksplit;
    a.partial = logits;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.margin = margin;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.pos = pos;
    a.sched = sched;
    a.hdr = hdr;
    dim3 grid((d.E + 7) / 8, ksplit);
    if (d.E <= 256)
        router_decode_kernel<8><<<grid, kRouterThreads, 0, st>>>(a);
    else if (d.E <= 512)
        router_decode_kernel<16><<<grid, kRouterThreads, 0, st>>>(a);
    else
        router_decode_kernel<32><<<grid, kRouterThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
