// Internal definitions shared by the CUDA translation units of libmoe.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device check flags, recorded in the workspace header instead of trapping.
enum : int32_t {
    kErrBadExpertId = 1 << 0,    // a topk id outside [0, E)
    kErrCountMismatch = 1 << 1,  // descriptor counts do not add up to T*k
    kErrWaitTimeout = 1 << 2,    // a bounded spin-wait gave up
    kErrBadTile = 1 << 3,        // a tile index outside its bounds
};

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
    int32_t error_flags;   // OR of kErr* bits; cleared by moe_check_device_status
    int32_t n_active;      // routed experts with count > 0 (written by the descriptors)
    int32_t n_tiles[2];    // grouped-GEMM tile counts: [0] gate+up, [1] down
    int32_t done[4];       // arrival counters; [0]: CTAs of router_decode_kernel (the last resets it);
                           // [2..3]: the single-launch step's 64-bit grid-barrier arrival count
    // test hook (moe_debug_set_waits); both 0 in normal use
    uint64_t wait_ns;       // limit of every bounded mbarrier wait (0: the 2 s default)
    int32_t withhold_stage; // s > 0: the gate+up grouped kernel's CTA 0 skips the copies of
                            // its s-th pipeline stage, so the stage's consumers time out
    int32_t pad[53];
};
static_assert(sizeof(WsHeader) == 256, "header size");

__device__ __forceinline__ void record_error(WsHeader* h, int32_t bit) {
    if (h) atomicOr(&h->error_flags, bit);
}

// ---------------------------------------------------------------------------
// Workspace layout.  Offsets are 256-byte aligned.
struct WsLayout {
    // per-step workspace (moe_workspace_bytes)
    size_t header;        // WsHeader
    size_t logits;        // fp32 [ksplit][T][E] router logit partials
    size_t tiles;         // int4 tile descriptors of the grouped kernels
    size_t xs;            // bf16 [T*k + T][d] gathered activation rows (grouped path)
    size_t hist;          // int32 [desc_blocks(T*k)][E] descriptor-sort histograms
    size_t wr_planes;     // bf16 [3][E][d] router weight planes (tensor-core router, T > 64)
    size_t step_bytes;
    // whole-layer workspace (moe_layer_workspace_bytes) adds the intermediates
    size_t topk_idx, topk_w, counts, offsets, perm, pos, sched, H, Y, x_stage, out_stage;
    size_t layer_bytes;
    // W8A8 layer (moe_layer_workspace_bytes_w8a8) adds the fp8 operands; the
    // gate+up codes [T*k + T][d] reuse the xs region
    size_t w8_xa, w8_hq, w8_ha;  // x row scales, H codes [T*k + T][max(F, F_s)], H row scales
    size_t w8_xt, w8_xta;        // each token's x codes [T][d] and scale [T]
    size_t w8a8_bytes;
    int router_ksplit;    // K split of the small-T router
    int router_ksplit_large;  // K split of the large-T router
    int64_t max_tiles;    // capacity of each tile list
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Router tiling: T <= kRouterSmallT uses the split-K GEMV form.
constexpr int kRouterSmallT = 64;

// GEMV (decode) expert path by default for T <= kGemvMaxT, from a sweep of the
// layer time over T on both forced paths at the decode shapes (GB300): the
// CUDA-core GEMV took 35.7 / 77.0 / 107.1 / 141.8 us at T = 1 / 2 / 3 / 4 (its
// multi-token form is FMA-bound, ~36 us per token), the grouped tensor-core
// kernel 95.6 / 97.7 / 104.8 / 114.5 us; the flags can force either.  One pass of
// the GEMV's loads covers rows of up to kGemvMaxD (gate+up) / kGemvMaxF (down).
constexpr int kGemvMaxT = 2;
constexpr int kGemvMaxD = 4096;
constexpr int kGemvMaxF = 2048;

// Single-token expert projections on the warp-level tensor cores
// (decode_tc.cu); taken for T == 1 on the GEMV path when the shapes fit.
bool tc_decode_supported(const moe_dims_t& d);
bool tc_weights_ok(moe_w4_t a, moe_w4_t b);  // 16-byte aligned bytes and scales
cudaError_t launch_gateup_tc(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H,
                             const int32_t* n_active, WsHeader* hdr, bool pdl, cudaStream_t st);
cudaError_t launch_down_tc(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                           const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                           const int32_t* n_active, const float* topk_w, const int32_t* pos,
                           const uint16_t* residual, uint16_t* out, bool pdl, cudaStream_t st);

// The whole single-token step in one cooperative launch (decode_tc.cu):
// router, descriptors, both projections and the combine.
bool step_supported(const moe_dims_t& d);
cudaError_t launch_decode_step(const uint16_t* x, const float* W_r, const float* bias,
                               const moe_dims_t& d, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                               int32_t* sched, float* logits, int ksplit, moe_w4_t Wgu, moe_w4_t Wd,
                               moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* H, const uint16_t* residual,
                               uint16_t* out, WsHeader* hdr, cudaStream_t st);

// Fused decode router (decode.cu) limits.
constexpr int kMaxDecodeT = 64;
constexpr int kMaxExperts = 1024;

// Grouped-GEMM tile geometry (weight rows x tokens).
constexpr int kTileM = 128;
constexpr int kTileN = 192;

WsLayout ws_layout(const moe_dims_t& d);

// Host-side argument checks shared by the entry points (abi.cu).
moe_status_t check_dims(const moe_dims_t* d);
bool act_ok(const void* p);  // non-null and 16-byte aligned

// ---------------------------------------------------------------------------
// Launchers (defined in the .cu files).  All enqueue on `st` and return the
// cudaGetLastError of the launch.
cudaError_t launch_pack_w4(const float* w, int64_t rows, int64_t K, int group, uint8_t* q,
                           uint16_t* s, cudaStream_t st);
// GGUF-style Q4 blocks [rows][K/32][18 B] -> fp32 w [rows][K] (K % 32 == 0).
cudaError_t launch_decode_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, float* w,
                                    cudaStream_t st);
// GGUF-style Q4 blocks straight to the packed format for group <= 32 (s = d,
// q = n - 8, exact), also writing the decoded fp32 weights to w.
cudaError_t launch_import_q4_direct(const uint8_t* blocks, int64_t rows, int64_t K, int group,
                                    float* w, uint8_t* q, uint16_t* s, cudaStream_t st);

// Router: logits as split-K partials (ksplit slices for T <= kRouterSmallT,
// ksplit_large above it), then the top-k.  Above kRouterSmallT the logits run
// on the tensor cores (router_tc.cu) when `planes` (workspace for the bf16
// split of W_r) is given and the shape allows, else as an fp32 SGEMM.
int router_ksplit_large(const moe_dims_t& d);
cudaError_t launch_router(const uint16_t* x, const float* W_r, const float* bias,
                          const moe_dims_t& d, int32_t* topk_idx, float* topk_w, float* margin,
                          float* logits, int ksplit, int ksplit_large, uint16_t* planes,
                          WsHeader* hdr, cudaStream_t st);
bool router_tc_supported(const moe_dims_t& d);
int router_tc_ksplit(const moe_dims_t& d);
cudaError_t launch_router_logits_tc(const uint16_t* x, const float* W_r, const moe_dims_t& d,
                                    uint16_t* planes, float* logits, int ks, WsHeader* hdr,
                                    cudaStream_t st);

// `hist` is workspace of desc_blocks(T * k) * E int32 (per-block histograms).
int desc_blocks(int64_t nslots);
// `tile_n`: tokens per tile of the tile lists (192; 256 for the W8A8 kernel).
cudaError_t launch_descriptors(const int32_t* topk_idx, const moe_dims_t& d, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched,
                               WsHeader* hdr, int4* tiles, int64_t max_tiles, int32_t* hist,
                               cudaStream_t st, int tile_n = kTileN);

// Decode expert GEMVs (experts_gemv.cu).  `n_active` is the count of routed
// groups with rows (the workspace header's, written by the fused router) or
// null, in which case the kernels count them from offsets and sched.  `pdl`
// launches with programmatic stream serialisation: the kernel's prologue
// overlaps the previous kernel, and it waits for it before reading its
// outputs.  With `out` non-null the down kernel also does the combine (plus
// `residual` when that is non-null; `out` may alias it).
bool gemv_supported(const moe_dims_t& d);
cudaError_t launch_gateup_gemv(const uint16_t* x, const moe_dims_t& d, const int32_t* offsets,
                               const int32_t* perm, const int32_t* sched, moe_w4_t Wgu,
                               moe_w4_t Wgu_s, uint16_t* H, const int32_t* n_active,
                               WsHeader* hdr, bool pdl, cudaStream_t st);

cudaError_t launch_down_gemv(const uint16_t* H, const moe_dims_t& d, const int32_t* offsets,
                             const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y,
                             const int32_t* n_active, const float* topk_w, const int32_t* pos,
                             const uint16_t* residual, uint16_t* out, WsHeader* hdr, bool pdl,
                             cudaStream_t st);

// Fused decode router: logits, top-k and descriptors in one launch (T <= 64).
cudaError_t launch_router_decode(const uint16_t* x, const float* W_r, const float* bias,
                                 const moe_dims_t& d, int32_t* topk_idx, float* topk_w,
                                 float* margin, float* logits, int ksplit, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched,
                                 WsHeader* hdr, cudaStream_t st);

// Grouped tcgen05 path (prefill).  `tiles` is the tile schedule that
// launch_descriptors wrote into the workspace (two lists of max_tiles each).
bool grouped_supported(const moe_dims_t& d);
// `xs` is workspace for the gate+up activation rows gathered into descriptor
// order, [T*k + T][d] bf16.
cudaError_t launch_gateup_grouped(const uint16_t* x, const moe_dims_t& d, const int32_t* perm,
                                  moe_w4_t Wgu, moe_w4_t Wgu_s, uint16_t* H, WsHeader* hdr,
                                  const int4* tiles, uint16_t* xs, cudaStream_t st);
cudaError_t launch_down_grouped(const uint16_t* H, const moe_dims_t& d, moe_w4_t Wd,
                                moe_w4_t Wd_s, float* Y, WsHeader* hdr, const int4* tiles,
                                cudaStream_t st);

// W8A8 grouped path (grouped_fp8.cu).  The gate+up launch quantises the
// gathered token rows into xq / a, the down launch the H rows into hq / a.
bool w8a8_supported(const moe_dims_t& d);
cudaError_t launch_quant_rows_fp8(const void* src, bool bf16, int64_t rows, int64_t K, uint8_t* q,
                                  float* s, cudaStream_t st);
// The gate+up launch quantises each token's x once (xt, xta: [T][d], [T]), then
// copies the codes into descriptor order (xq, a).
cudaError_t launch_gateup_w8a8(const uint16_t* x, const moe_dims_t& d, const int32_t* perm,
                               moe_w8_t Wgu, moe_w8_t Wgu_s, uint16_t* H, WsHeader* hdr,
                               const int4* tiles, int64_t max_tiles, uint8_t* xq, float* a,
                               uint8_t* xt, float* xta, cudaStream_t st);
cudaError_t launch_down_w8a8(const uint16_t* H, const moe_dims_t& d, moe_w8_t Wd, moe_w8_t Wd_s,
                             float* Y, WsHeader* hdr, const int4* tiles, int64_t max_tiles,
                             uint8_t* hq, float* a, cudaStream_t st);

// `residual` (nullable, bf16 [T][d]) is added to the routed + shared sum
// before the bf16 rounding; `out` may alias it.
cudaError_t launch_combine(const float* Y, const float* topk_w, const int32_t* pos,
                           const moe_dims_t& d, const uint16_t* residual, uint16_t* out,
                           cudaStream_t st);

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Raise a kernel's dynamic shared-memory limit when `bytes` exceeds the 48 KB
// default (once per kernel and device; safe to call during stream capture).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// ---------------------------------------------------------------------------
// Small device helpers.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) {
    return __uint_as_float(pair & 0xFFFF0000u);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

// SwiGLU of one gate / up pair in fp32: silu(g) * u with silu(g) = g / (1 + e^-g).
// The exponential and the division are the hardware approximations (__expf,
// __fdividef): a few fp32 ulp from the correctly rounded forms, far below the
// bf16 rounding that H gets next.  Every expert path uses this one form.
// Limits: g -> -inf gives -0 (e^-g = inf), g -> +inf gives g * u.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// a0 += s * v0, a1 += s * v1 as one packed f32x2 FMA (sm_100 family); each
// lane rounds exactly as fmaf, so results match the scalar form bit for bit.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float s, float v0, float v1) {
    asm("{\n .reg .b64 acc, vv, ss;\n mov.b64 acc, {%0, %1};\n mov.b64 vv, {%2, %3};\n"
        " mov.b64 ss, {%4, %4};\n fma.rn.f32x2 acc, ss, vv, acc;\n mov.b64 {%0, %1}, acc;\n}"
        : "+f"(a0), "+f"(a1)
        : "f"(v0), "f"(v1), "f"(s));
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait until the previous kernel has completed and its writes are
// visible.  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


}  // namespace moe
