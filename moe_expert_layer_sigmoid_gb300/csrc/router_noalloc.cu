// moe_router_topk_noalloc: the router for callers that cannot allocate device
// memory at call time, so cannot size and pass a workspace.  Two kinds of
// caller need this: a host framework that owns every device allocation through
// its own pool and forbids side allocations, and a serving process that has
// reserved all of HBM for weights and caches at start-up.
//
// The router's only scratch is its fp32 logit partials.  Here they live in a
// file-scope device array of fixed size, so the call needs no workspace and
// allocates nothing.  Every GPU that loads libmoe.so holds the array until the
// process exits.
//
// Host code must not pass the array's name to a kernel: on the host that name
// is a stand-in symbol, not a device address.  On each device the first call
// looks up the array's device address with cudaGetSymbolAddress, with that
// device current, and caches it.  Under lazy module loading (the runtime's
// default) that lookup is what loads this file's module, so the array is
// allocated by the first call on each device: callers that reserve all of HBM
// make one call per device first, or set CUDA_MODULE_LOADING=EAGER.  The
// address is the current device's, so the caller's stream must belong to it.
#include <mutex>

#include "common.cuh"

namespace {

// 1 Mi floats = 4 MiB of logit partials: [ksplit][T][E] fp32.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_router_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_router_scratch on the current device (set up on first use).
cudaError_t scratch_on_current_device(float** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_router_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_router_topk_noalloc(const uint16_t* x, const float* W_r,
                                                const float* bias, const moe_dims_t* dims,
                                                int32_t* topk_idx, float* topk_w, float* margin,
                                                void* stream) {
    moe_status_t st = moe::check_dims(dims);
    if (st != MOE_OK) return st;
    const moe::WsLayout L = moe::ws_layout(*dims);
    const int ks = dims->T <= moe::kRouterSmallT ? L.router_ksplit : 1;
    const int64_t need = (int64_t)ks * dims->T * dims->E;
    if (need > (int64_t)kScratchFloats) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
    if (dims->T == 0) return MOE_OK;
    if (!moe::act_ok(x) || !moe::act_ok(W_r) || !bias || !topk_idx || !topk_w)
        return MOE_ERR_INVALID_ARG;
    float* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // The logits kernel writes every partial that the top-k kernel reads within
    // this call, so leftovers of an earlier call never leak into the result.
    cudaError_t err = moe::launch_router(x, W_r, bias, *dims, topk_idx, topk_w, margin, scratch,
                                         L.router_ksplit, 1, nullptr, nullptr,
                                         static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
