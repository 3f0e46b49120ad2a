// extern "C" entry points of libmoe.so: argument validation, workspace
// layout, path dispatch.  Every entry point validates on the host, then
// enqueues kernels on the caller's stream; none allocates or synchronises
// (moe_check_device_status excepted).
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace moe {

WsLayout ws_layout(const moe_dims_t& d) {
    WsLayout L{};
    const int64_t T = d.T, E = d.E, k = d.k;
    const int64_t slots = T * k;
    const int64_t rows = slots + T;
    const int64_t Fmax = std::max(d.F, d.F_s);
    L.router_ksplit = (d.d % 512 == 0) ? d.d / 512 : d.d / 256;
    L.router_ksplit_large = router_ksplit_large(d);
    const int64_t ks = T <= kRouterSmallT ? L.router_ksplit : L.router_ksplit_large;
    // tile lists: one entry per (group, 128-row weight band, token tile of up to kTileN)
    const int64_t groups = std::min<int64_t>(E, slots) + 1;
    const int64_t tok_tiles = (slots + kTileN - 1) / kTileN + groups + (T + kTileN - 1) / kTileN;
    const int64_t bands = (std::max<int64_t>(d.d, 2 * Fmax) + kTileM - 1) / kTileM;
    L.max_tiles = tok_tiles * bands;

    size_t off = 0;
    L.header = off;
    off += align256(sizeof(WsHeader));
    L.logits = off;
    off += align256(sizeof(float) * (size_t)(ks * T * E));
    L.tiles = off;
    off += align256(sizeof(int4) * (size_t)(2 * L.max_tiles));
    L.xs = off;
    off += align256(sizeof(uint16_t) * (size_t)(rows * d.d));
    L.hist = off;
    off += align256(sizeof(int32_t) * (size_t)desc_blocks(slots) * (size_t)E);
    L.wr_planes = off;
    if (T > kRouterSmallT && router_tc_supported(d)) off += align256(sizeof(uint16_t) * 3 * (size_t)E * d.d);
    L.step_bytes = off;

    L.topk_idx = off;
    off += align256(sizeof(int32_t) * (size_t)slots);
    L.topk_w = off;
    off += align256(sizeof(float) * (size_t)slots);
    L.counts = off;
    off += align256(sizeof(int32_t) * (size_t)E);
    L.offsets = off;
    off += align256(sizeof(int32_t) * (size_t)(E + 1));
    L.perm = off;
    off += align256(sizeof(int32_t) * (size_t)slots);
    L.pos = off;
    off += align256(sizeof(int32_t) * (size_t)slots);
    L.sched = off;
    off += align256(sizeof(int32_t) * (size_t)E);
    L.H = off;
    off += align256(sizeof(uint16_t) * (size_t)(rows * Fmax));
    L.Y = off;
    off += align256(sizeof(float) * (size_t)(rows * d.d));
    L.x_stage = off;
    off += align256(sizeof(uint16_t) * (size_t)(T * d.d));
    L.out_stage = off;
    off += align256(sizeof(uint16_t) * (size_t)(T * d.d));
    L.layer_bytes = off;
    L.w8_xa = off;
    off += align256(sizeof(float) * (size_t)rows);
    L.w8_hq = off;
    off += align256((size_t)(rows * Fmax));
    L.w8_ha = off;
    off += align256(sizeof(float) * (size_t)rows);
    L.w8_xt = off;
    off += align256((size_t)(T * d.d));
    L.w8_xta = off;
    off += align256(sizeof(float) * (size_t)T);
    L.w8a8_bytes = off;
    return L;
}

int sm_count() {
    // cached per device; host threads may race to fill an entry with the same value
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (!n && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        counts[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    // per (kernel, device) once; a small table is enough for the handful of kernels
    static std::mutex mu;
    static const void* seen_k[64];
    static int seen_dev[64];
    static size_t seen_bytes[64];
    static int n_seen = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_seen; ++i)
        if (seen_k[i] == kernel && seen_dev[i] == dev && seen_bytes[i] >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err != cudaSuccess) return err;
    if (n_seen < 64) {
        seen_k[n_seen] = kernel;
        seen_dev[n_seen] = dev;
        seen_bytes[n_seen] = bytes;
        ++n_seen;
    }
    return cudaSuccess;
}

// Quantisation groups the layer kernels take.
bool group_ok(int g) { return g == 32 || g == 64 || g == 128; }

// Shape validation shared by every entry point that takes moe_dims_t.
moe_status_t check_dims(const moe_dims_t* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->d <= 0 || d->E <= 0 || d->k <= 0 || d->F <= 0 || d->F_s <= 0 ||
        d->group <= 0)
        return MOE_ERR_INVALID_ARG;
    if (d->k > d->E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)d->T * (d->k + 1) >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (!group_ok(d->group)) return MOE_ERR_UNSUPPORTED;
    if (d->d % 256 || d->F % 128 || d->F_s % 128) return MOE_ERR_UNSUPPORTED;
    if (d->d % d->group || d->F % d->group || d->F_s % d->group) return MOE_ERR_UNSUPPORTED;
    if (d->k > 32 || d->E > 1024) return MOE_ERR_UNSUPPORTED;
    // Weight-row indices are 32-bit (the grouped kernel's TMA row coordinates):
    // the routed gate+up tensor has E * 2F rows, the down tensor E * d.
    if ((int64_t)d->E * 2 * d->F >= (int64_t)1 << 31 || (int64_t)d->E * d->d >= (int64_t)1 << 31)
        return MOE_ERR_UNSUPPORTED;
    if ((d->flags & MOE_FLAG_FORCE_GEMV) && (d->flags & MOE_FLAG_FORCE_GROUPED))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Activation and fp32 buffers are read or written with vector accesses of up
// to 16 bytes; 16-byte alignment (what any device allocation gives) is
// required, so a misaligned pointer is an argument error, never a fault.
bool act_ok(const void* p) { return p && reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace moe

using namespace moe;

namespace {

moe_status_t map_err(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

__global__ void set_waits_kernel(WsHeader* hdr, unsigned long long wait_ns, int withhold_stage) {
    hdr->wait_ns = wait_ns;
    hdr->withhold_stage = withhold_stage;
}

moe_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) % 256) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// q is read with 16-byte loads, s with 2-byte loads.
bool w4_ok(moe_w4_t w) {
    return w.q && w.s && reinterpret_cast<uintptr_t>(w.q) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(w.s) % 2 == 0;
}

// q is read by the TMA unit (16-byte aligned base), s with 4-byte loads.
bool w8_ok(moe_w8_t w) {
    return w.q && w.s && reinterpret_cast<uintptr_t>(w.q) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(w.s) % 4 == 0;
}

template <typename T>
T* ws_at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Expert path: CUDA-core GEMV for small T (or when forced), the tcgen05
// grouped kernel otherwise.  A shape only one of them covers runs there; a
// forced path that does not cover the shape reports UNSUPPORTED.
enum class Path { kGemv, kGrouped, kUnsupported };

Path expert_path(const moe_dims_t& d) {
    const bool gemv = gemv_supported(d), grouped = grouped_supported(d);
    if (d.flags & MOE_FLAG_FORCE_GEMV) return gemv ? Path::kGemv : Path::kUnsupported;
    if (d.flags & MOE_FLAG_FORCE_GROUPED) return grouped ? Path::kGrouped : Path::kUnsupported;
    if (grouped && (d.T > kGemvMaxT || !gemv)) return Path::kGrouped;
    return gemv ? Path::kGemv : Path::kUnsupported;
}

moe_status_t gateup_impl(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                         const int32_t* perm, const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s,
                         uint16_t* H, void* ws, cudaStream_t st) {
    const WsLayout L = ws_layout(d);
    WsHeader* hdr = ws_at<WsHeader>(ws, L.header);
    switch (expert_path(d)) {
        case Path::kGemv:
            if ((d.flags & MOE_FLAG_DECODE_MMA) && tc_decode_supported(d) && tc_weights_ok(Wgu, Wgu_s))
                return map_err(launch_gateup_tc(x, d, offsets, sched, Wgu, Wgu_s, H, nullptr, hdr,
                                                false, st));
            return map_err(launch_gateup_gemv(x, d, offsets, perm, sched, Wgu, Wgu_s, H, nullptr,
                                              hdr, false, st));
        case Path::kGrouped:
            return map_err(launch_gateup_grouped(x, d, perm, Wgu, Wgu_s, H, hdr,
                                                 ws_at<int4>(ws, L.tiles), ws_at<uint16_t>(ws, L.xs),
                                                 st));
        default: return MOE_ERR_UNSUPPORTED;
    }
}

moe_status_t down_impl(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                       const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y, void* ws,
                       cudaStream_t st) {
    const WsLayout L = ws_layout(d);
    WsHeader* hdr = ws_at<WsHeader>(ws, L.header);
    switch (expert_path(d)) {
        case Path::kGemv:
            if ((d.flags & MOE_FLAG_DECODE_MMA) && tc_decode_supported(d) && tc_weights_ok(Wd, Wd_s))
                return map_err(launch_down_tc(H, d, offsets, sched, Wd, Wd_s, Y, nullptr, nullptr,
                                              nullptr, nullptr, nullptr, false, st));
            return map_err(launch_down_gemv(H, d, offsets, sched, Wd, Wd_s, Y, nullptr, nullptr,
                                            nullptr, nullptr, nullptr, hdr, false, st));
        case Path::kGrouped:
            return map_err(launch_down_grouped(H, d, Wd, Wd_s, Y, hdr,
                                               ws_at<int4>(ws, L.tiles) + L.max_tiles, st));
        default: return MOE_ERR_UNSUPPORTED;
    }
}

// The whole layer; `residual` null for the plain output.
moe_status_t layer_forward(const uint16_t* x, const float* W_r, const float* bias,
                           const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd, moe_w4_t Wgu_s,
                           moe_w4_t Wd_s, const uint16_t* residual, uint16_t* out, void* ws,
                           size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.layer_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(x) || !act_ok(W_r) || !bias || !act_ok(out) || !w4_ok(Wgu) || !w4_ok(Wd) ||
        !w4_ok(Wgu_s) || !w4_ok(Wd_s))
        return MOE_ERR_INVALID_ARG;
    const moe_dims_t& d = *dims;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* topk_idx = ws_at<int32_t>(ws, L.topk_idx);
    float* topk_w = ws_at<float>(ws, L.topk_w);
    int32_t* counts = ws_at<int32_t>(ws, L.counts);
    int32_t* offsets = ws_at<int32_t>(ws, L.offsets);
    int32_t* perm = ws_at<int32_t>(ws, L.perm);
    int32_t* pos = ws_at<int32_t>(ws, L.pos);
    int32_t* sched = ws_at<int32_t>(ws, L.sched);
    uint16_t* H = ws_at<uint16_t>(ws, L.H);
    float* Y = ws_at<float>(ws, L.Y);
    WsHeader* hdr = ws_at<WsHeader>(ws, L.header);
    const Path path = expert_path(d);
    if (path == Path::kUnsupported) return MOE_ERR_UNSUPPORTED;
    cudaError_t e;
    const bool tc_w = (d.flags & MOE_FLAG_DECODE_MMA) && tc_weights_ok(Wgu, Wgu_s) &&
                      tc_weights_ok(Wd, Wd_s);
    if (path == Path::kGemv && d.T == 1 && tc_w && step_supported(d)) {
        // the single-token step in one cooperative launch
        return map_err(launch_decode_step(x, W_r, bias, d, topk_idx, topk_w, counts, offsets, perm,
                                          pos, sched, ws_at<float>(ws, L.logits), L.router_ksplit,
                                          Wgu, Wd, Wgu_s, Wd_s, H, residual, out, hdr, s));
    }
    if (path == Path::kGemv) {
        // decode chain: fused router + descriptors, then the two GEMVs with the
        // combine fused into the down kernel; each waits on its predecessor
        // through programmatic dependent launch
        if (d.T <= kMaxDecodeT) {
            e = launch_router_decode(x, W_r, bias, d, topk_idx, topk_w, nullptr,
                                     ws_at<float>(ws, L.logits), L.router_ksplit, counts, offsets,
                                     perm, pos, sched, hdr, s);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
        } else {
            e = launch_router(x, W_r, bias, d, topk_idx, topk_w, nullptr,
                              ws_at<float>(ws, L.logits), L.router_ksplit, L.router_ksplit_large,
                              ws_at<uint16_t>(ws, L.wr_planes), hdr, s);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            e = launch_descriptors(topk_idx, d, counts, offsets, perm, pos, sched, hdr,
                                   ws_at<int4>(ws, L.tiles), L.max_tiles,
                                   ws_at<int32_t>(ws, L.hist), s);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
        }
        if (tc_w && tc_decode_supported(d)) {
            e = launch_gateup_tc(x, d, offsets, sched, Wgu, Wgu_s, H, &hdr->n_active, hdr, true, s);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            return map_err(launch_down_tc(H, d, offsets, sched, Wd, Wd_s, Y, &hdr->n_active,
                                          topk_w, pos, residual, out, true, s));
        }
        e = launch_gateup_gemv(x, d, offsets, perm, sched, Wgu, Wgu_s, H, &hdr->n_active, hdr,
                               true, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        return map_err(launch_down_gemv(H, d, offsets, sched, Wd, Wd_s, Y, &hdr->n_active, topk_w,
                                        pos, residual, out, hdr, true, s));
    }
    e = launch_router(x, W_r, bias, d, topk_idx, topk_w, nullptr, ws_at<float>(ws, L.logits),
                      L.router_ksplit, L.router_ksplit_large, ws_at<uint16_t>(ws, L.wr_planes), hdr,
                      s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_descriptors(topk_idx, d, counts, offsets, perm, pos, sched, hdr,
                           ws_at<int4>(ws, L.tiles), L.max_tiles, ws_at<int32_t>(ws, L.hist), s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if ((st = gateup_impl(x, d, offsets, perm, sched, Wgu, Wgu_s, H, ws, s)) != MOE_OK) return st;
    if ((st = down_impl(H, d, offsets, sched, Wd, Wd_s, Y, ws, s)) != MOE_OK) return st;
    return map_err(launch_combine(Y, topk_w, pos, d, residual, out, s));
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer or inconsistent size";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape outside the supported set";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a device-side check tripped";
    }
    return "unknown moe_status_t";
}

size_t moe_pack_w4_bytes(int64_t rows, int64_t K, int32_t group, size_t* scale_bytes) {
    if (scale_bytes) *scale_bytes = 0;
    if (rows < 0 || K <= 0 || group <= 0 || K % group) return 0;
    if (!(group == 8 || group == 16 || group_ok(group))) return 0;
    if (scale_bytes) *scale_bytes = (size_t)rows * (size_t)(K / group) * sizeof(uint16_t);
    return (size_t)rows * (size_t)(K / 2);
}

moe_status_t moe_pack_w4(const float* w, int64_t rows, int64_t K, int32_t group, uint8_t* q,
                         uint16_t* s, void* stream) {
    if (rows < 0 || K <= 0 || group <= 0) return MOE_ERR_INVALID_ARG;
    if (!(group == 8 || group == 16 || group_ok(group))) return MOE_ERR_UNSUPPORTED;
    if (K % group) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !s) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(w) % 16 || reinterpret_cast<uintptr_t>(q) % 4 ||
        reinterpret_cast<uintptr_t>(s) % 2)
        return MOE_ERR_INVALID_ARG;
    return map_err(launch_pack_w4(w, rows, K, group, q, s, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_import_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, int32_t group,
                                  float* w_scratch, uint8_t* q, uint16_t* s, void* stream) {
    if (rows < 0 || K <= 0 || group <= 0) return MOE_ERR_INVALID_ARG;
    if (!(group == 8 || group == 16 || group_ok(group))) return MOE_ERR_UNSUPPORTED;
    if (K % 32 || K % group) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !act_ok(w_scratch) || !q || !s) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) % 4 || reinterpret_cast<uintptr_t>(s) % 2)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (group <= 32)  // each group inside one block: s = d, q = n - 8, exact
        return map_err(launch_import_q4_direct(blocks, rows, K, group, w_scratch, q, s, st));
    if (launch_decode_q4_blocks(blocks, rows, K, w_scratch, st) != cudaSuccess) return MOE_ERR_CUDA;
    return map_err(launch_pack_w4(w_scratch, rows, K, group, q, s, st));
}

size_t moe_workspace_bytes(const moe_dims_t* dims) {
    if (check_dims(dims) != MOE_OK) return 0;
    return ws_layout(*dims).step_bytes;
}

size_t moe_layer_workspace_bytes(const moe_dims_t* dims) {
    if (check_dims(dims) != MOE_OK) return 0;
    return ws_layout(*dims).layer_bytes;
}

moe_status_t moe_router_topk(const uint16_t* x, const float* W_r, const float* bias,
                             const moe_dims_t* dims, int32_t* topk_idx, float* topk_w,
                             float* margin, void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.step_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(x) || !act_ok(W_r) || !bias || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    return map_err(launch_router(x, W_r, bias, *dims, topk_idx, topk_w, margin,
                                 ws_at<float>(ws, L.logits), L.router_ksplit,
                                 L.router_ksplit_large, ws_at<uint16_t>(ws, L.wr_planes),
                                 ws_at<WsHeader>(ws, L.header), static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_build_descriptors(const int32_t* topk_idx, const moe_dims_t* dims,
                                   int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                                   int32_t* sched, void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.step_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!topk_idx || !counts || !offsets || !perm || !pos || !sched) return MOE_ERR_INVALID_ARG;
    return map_err(launch_descriptors(topk_idx, *dims, counts, offsets, perm, pos, sched,
                                      ws_at<WsHeader>(ws, L.header), ws_at<int4>(ws, L.tiles),
                                      L.max_tiles, ws_at<int32_t>(ws, L.hist),
                                      static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_gateup_swiglu_w4a16(const uint16_t* x, const moe_dims_t* dims,
                                     const int32_t* offsets, const int32_t* perm,
                                     const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s,
                                     uint16_t* H, void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.step_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(x) || !offsets || !perm || !sched || !act_ok(H) || !w4_ok(Wgu) || !w4_ok(Wgu_s))
        return MOE_ERR_INVALID_ARG;
    return gateup_impl(x, *dims, offsets, perm, sched, Wgu, Wgu_s, H, ws,
                       static_cast<cudaStream_t>(stream));
}

moe_status_t moe_down_w4a16(const uint16_t* H, const moe_dims_t* dims, const int32_t* offsets,
                            const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y, void* ws,
                            size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.step_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(H) || !offsets || !sched || !act_ok(Y) || !w4_ok(Wd) || !w4_ok(Wd_s))
        return MOE_ERR_INVALID_ARG;
    return down_impl(H, *dims, offsets, sched, Wd, Wd_s, Y, ws, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_down_combine_w4a16(const uint16_t* H, const moe_dims_t* dims,
                                    const int32_t* offsets, const int32_t* sched,
                                    const float* topk_w, const int32_t* pos, moe_w4_t Wd,
                                    moe_w4_t Wd_s, const uint16_t* residual, uint16_t* out,
                                    void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.layer_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(H) || !offsets || !sched || !topk_w || !pos || !act_ok(out) || !w4_ok(Wd) ||
        !w4_ok(Wd_s) || (residual && !act_ok(residual)))
        return MOE_ERR_INVALID_ARG;
    const moe_dims_t& d = *dims;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* Y = ws_at<float>(ws, L.Y);
    WsHeader* hdr = ws_at<WsHeader>(ws, L.header);
    switch (expert_path(d)) {
        case Path::kGemv:
            if ((d.flags & MOE_FLAG_DECODE_MMA) && tc_decode_supported(d) && tc_weights_ok(Wd, Wd_s))
                return map_err(launch_down_tc(H, d, offsets, sched, Wd, Wd_s, Y, nullptr, topk_w,
                                              pos, residual, out, false, s));
            return map_err(launch_down_gemv(H, d, offsets, sched, Wd, Wd_s, Y, nullptr, topk_w, pos,
                                            residual, out, hdr, false, s));
        case Path::kGrouped:
            if ((st = down_impl(H, d, offsets, sched, Wd, Wd_s, Y, ws, s)) != MOE_OK) return st;
            return map_err(launch_combine(Y, topk_w, pos, d, residual, out, s));
        default: return MOE_ERR_UNSUPPORTED;
    }
}

moe_status_t moe_combine_shared(const float* Y, const float* topk_w, const int32_t* pos,
                                const moe_dims_t* dims, uint16_t* out, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(Y) || !topk_w || !pos || !act_ok(out)) return MOE_ERR_INVALID_ARG;
    return map_err(launch_combine(Y, topk_w, pos, *dims, nullptr, out,
                                  static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine_shared_residual(const float* Y, const float* topk_w, const int32_t* pos,
                                         const moe_dims_t* dims, const uint16_t* residual,
                                         uint16_t* out, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(Y) || !topk_w || !pos || !act_ok(residual) || !act_ok(out))
        return MOE_ERR_INVALID_ARG;
    return map_err(launch_combine(Y, topk_w, pos, *dims, residual, out,
                                  static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward(const uint16_t* x, const float* W_r, const float* bias,
                               const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                               moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* out, void* ws,
                               size_t ws_bytes, void* stream) {
    return layer_forward(x, W_r, bias, dims, Wgu, Wd, Wgu_s, Wd_s, nullptr, out, ws, ws_bytes,
                         stream);
}

moe_status_t moe_layer_forward_residual(const uint16_t* x, const float* W_r, const float* bias,
                                        const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                                        moe_w4_t Wgu_s, moe_w4_t Wd_s, const uint16_t* residual,
                                        uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
    if (dims && dims->T > 0 && (!act_ok(residual) || !act_ok(out))) return MOE_ERR_INVALID_ARG;
    return layer_forward(x, W_r, bias, dims, Wgu, Wd, Wgu_s, Wd_s, residual, out, ws, ws_bytes,
                         stream);
}

moe_status_t moe_pack_w8(const float* w, int64_t rows, int64_t K, uint8_t* q, float* s,
                         void* stream) {
    if (rows < 0 || K <= 0 || K % 8) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!act_ok(w) || !q || !s || reinterpret_cast<uintptr_t>(q) % 8 ||
        reinterpret_cast<uintptr_t>(s) % 4)
        return MOE_ERR_INVALID_ARG;
    return map_err(launch_quant_rows_fp8(w, false, rows, K, q, s, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quant_rows_fp8(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q, float* a,
                                void* stream) {
    if (rows < 0 || K <= 0 || K % 8) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!act_ok(x) || !q || !a || reinterpret_cast<uintptr_t>(q) % 8 ||
        reinterpret_cast<uintptr_t>(a) % 4)
        return MOE_ERR_INVALID_ARG;
    return map_err(launch_quant_rows_fp8(x, true, rows, K, q, a, static_cast<cudaStream_t>(stream)));
}

size_t moe_layer_workspace_bytes_w8a8(const moe_dims_t* dims) {
    if (check_dims(dims) != MOE_OK || !w8a8_supported(*dims)) return 0;
    return ws_layout(*dims).w8a8_bytes;
}

moe_status_t moe_gateup_swiglu_w8a8(const uint16_t* x, const moe_dims_t* dims,
                                    const int32_t* perm, moe_w8_t Wgu, moe_w8_t Wgu_s,
                                    uint16_t* H, void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    if (!w8a8_supported(*dims)) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.w8a8_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(x) || !perm || !act_ok(H) || !w8_ok(Wgu) || !w8_ok(Wgu_s))
        return MOE_ERR_INVALID_ARG;
    return map_err(launch_gateup_w8a8(x, *dims, perm, Wgu, Wgu_s, H, ws_at<WsHeader>(ws, L.header),
                                      ws_at<int4>(ws, L.tiles), L.max_tiles,
                                      ws_at<uint8_t>(ws, L.xs), ws_at<float>(ws, L.w8_xa),
                                      ws_at<uint8_t>(ws, L.w8_xt), ws_at<float>(ws, L.w8_xta),
                                      static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_down_w8a8(const uint16_t* H, const moe_dims_t* dims, moe_w8_t Wd, moe_w8_t Wd_s,
                           float* Y, void* ws, size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    if (!w8a8_supported(*dims)) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.w8a8_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(H) || !act_ok(Y) || !w8_ok(Wd) || !w8_ok(Wd_s)) return MOE_ERR_INVALID_ARG;
    return map_err(launch_down_w8a8(H, *dims, Wd, Wd_s, Y, ws_at<WsHeader>(ws, L.header),
                                    ws_at<int4>(ws, L.tiles) + L.max_tiles, L.max_tiles,
                                    ws_at<uint8_t>(ws, L.w8_hq), ws_at<float>(ws, L.w8_ha),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward_w8a8(const uint16_t* x, const float* W_r, const float* bias,
                                    const moe_dims_t* dims, moe_w8_t Wgu, moe_w8_t Wd,
                                    moe_w8_t Wgu_s, moe_w8_t Wd_s, uint16_t* out, void* ws,
                                    size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    if (!w8a8_supported(*dims)) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.w8a8_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!act_ok(x) || !act_ok(W_r) || !bias || !act_ok(out) || !w8_ok(Wgu) || !w8_ok(Wd) ||
        !w8_ok(Wgu_s) || !w8_ok(Wd_s))
        return MOE_ERR_INVALID_ARG;
    const moe_dims_t& d = *dims;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* topk_idx = ws_at<int32_t>(ws, L.topk_idx);
    float* topk_w = ws_at<float>(ws, L.topk_w);
    int32_t* pos = ws_at<int32_t>(ws, L.pos);
    int32_t* perm = ws_at<int32_t>(ws, L.perm);
    uint16_t* H = ws_at<uint16_t>(ws, L.H);
    float* Y = ws_at<float>(ws, L.Y);
    WsHeader* hdr = ws_at<WsHeader>(ws, L.header);
    const int4* tiles = ws_at<int4>(ws, L.tiles);
    cudaError_t e = launch_router(x, W_r, bias, d, topk_idx, topk_w, nullptr,
                                  ws_at<float>(ws, L.logits), L.router_ksplit,
                                  L.router_ksplit_large, ws_at<uint16_t>(ws, L.wr_planes), hdr, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // 256-token tiles: the fp8 kernel goes faster with more flops per weight byte
    e = launch_descriptors(topk_idx, d, ws_at<int32_t>(ws, L.counts), ws_at<int32_t>(ws, L.offsets),
                           perm, pos, ws_at<int32_t>(ws, L.sched), hdr, ws_at<int4>(ws, L.tiles),
                           L.max_tiles, ws_at<int32_t>(ws, L.hist), s, 256);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_gateup_w8a8(x, d, perm, Wgu, Wgu_s, H, hdr, tiles, L.max_tiles,
                           ws_at<uint8_t>(ws, L.xs), ws_at<float>(ws, L.w8_xa),
                           ws_at<uint8_t>(ws, L.w8_xt), ws_at<float>(ws, L.w8_xta), s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_down_w8a8(H, d, Wd, Wd_s, Y, hdr, tiles + L.max_tiles, L.max_tiles,
                         ws_at<uint8_t>(ws, L.w8_hq), ws_at<float>(ws, L.w8_ha), s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return map_err(launch_combine(Y, topk_w, pos, d, nullptr, out, s));
}

moe_status_t moe_layer_forward_host(const uint16_t* x_host, const float* W_r, const float* bias,
                                    const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                                    moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* out_host, void* ws,
                                    size_t ws_bytes, void* stream) {
    moe_status_t st = check_dims(dims);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(*dims);
    if ((st = check_ws(ws, ws_bytes, L.layer_bytes)) != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = sizeof(uint16_t) * (size_t)dims->T * dims->d;
    uint16_t* xd = ws_at<uint16_t>(ws, L.x_stage);
    uint16_t* od = ws_at<uint16_t>(ws, L.out_stage);
    if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = moe_layer_forward(xd, W_r, bias, dims, Wgu, Wd, Wgu_s, Wd_s, od, ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
    if (cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t moe_debug_set_waits(void* ws, size_t ws_bytes, uint64_t wait_ns,
                                 int32_t withhold_stage, void* stream) {
    if (!ws || ws_bytes < sizeof(WsHeader) || reinterpret_cast<uintptr_t>(ws) % 256)
        return MOE_ERR_WORKSPACE;
    if (withhold_stage < 0) return MOE_ERR_INVALID_ARG;
    set_waits_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<WsHeader*>(ws), (unsigned long long)wait_ns, withhold_stage);
    return map_err(cudaGetLastError());
}

moe_status_t moe_check_device_status(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    int32_t flags = 0;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    if (cudaMemcpy(&flags, &hdr->error_flags, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (flags) {
        const int32_t zero = 0;
        if (cudaMemcpy(&hdr->error_flags, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_ERR_DEVICE_CHECK;
    }
    return MOE_OK;
}

}  // extern "C"
