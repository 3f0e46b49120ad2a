/*
 * moe.h -- C ABI of libmoe.so, the GB300 (sm_103a) routed MoE FFN layer.
 *
 * The layer (thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1
 * decode on the CUDA engine"): a sigmoid top-k router with a score-correction
 * bias, routed experts with int4 weights and fused gate+up SwiGLU, a down
 * projection, and a weighted combine plus an always-on shared expert.  The
 * prefill form (same page, commit "feat(laguna): batched prefill with
 * tensor-core projections, fused MoE, CTA scheduling") runs the experts as a
 * grouped GEMM driven by on-device descriptors, largest expert first, with
 * N-banded tile order for weight reuse in L2.
 *
 * Conventions shared by every call
 *  - Pointers marked (device) are CUDA device memory owned by the caller; the
 *    library allocates nothing, frees nothing and keeps no pointer after a
 *    call returns.  Pointers marked (host) are host memory; pinned memory is
 *    needed for the copies to overlap.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    is asynchronous on that stream and performs no host synchronisation and
 *    no host read of device data, so a sequence of calls can be captured into
 *    a CUDA graph.  moe_check_device_status is the one exception (it syncs).
 *  - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 *  - Alignment: x, W_r, H, Y, out and residual must be 16-byte aligned (they
 *    are accessed with vector loads and stores; any device allocation is),
 *    packed weights q 16-byte and scales 2-byte aligned, the workspace
 *    256-byte aligned.  A misaligned pointer is MOE_ERR_INVALID_ARG (the
 *    workspace: MOE_ERR_WORKSPACE), never a device fault.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned synchronously; nothing is enqueued in that case.  A failed
 *    launch returns MOE_ERR_CUDA.  Device-side consistency checks (an expert
 *    id out of range, inconsistent counts) set a flag in the workspace instead
 *    of trapping; moe_check_device_status reads it.
 *  - T = 0 is valid: the call validates the other arguments, returns MOE_OK
 *    and enqueues nothing.
 *  - Determinism: every call is deterministic, always: the same inputs on the
 *    same flags and shapes give the same bits, run after run.  No kernel uses
 *    floating-point atomics or an order that depends on timing; every sum is
 *    taken in a fixed order.  So there is no switch for it (the pages' MoE
 *    keeps a deterministic scatter-add for the same reason).  Different paths
 *    (flags, or T on either side of the path crossover) sum in different
 *    orders and may differ in the last bits.
 *
 * Numerics (the reading of the layer statement this library implements)
 *  - int4 weights: per row, per group of `group` consecutive K elements,
 *    s = fp16(absmax / 7) (absmax/7 evaluated in fp32, then rounded to fp16),
 *    q = clamp(rint(w / s), -8, 7) (w/s in fp32, ties to even), s = 0 gives
 *    q = 0.  Packed layout [rows][K/2] bytes: byte j holds element 2j in bits
 *    0-3 and element 2j+1 in bits 4-7, two's complement.  Scales are fp16
 *    [rows][K/group].  The dequantised weight is q * s, exactly.
 *  - Router: l = x . W_r[e] (fp32 accumulate), s = sigmoid(l); the k experts
 *    with the largest s + bias[e] are selected (ties to the lower id, listed
 *    in descending order); combine weights w_j = s_j / sum_j s_j.  The bias
 *    takes part in the selection only.
 *  - Expert e on token t: g = x . w^_gate[f], u = x . w^_up[f] (fp32
 *    accumulate), H = bf16(silu(g) * u); Y = H . w^_down[c] (fp32 accumulate).
 *  - out[t] = bf16( sum_j w_tj * Y[pos(t, j)] + Y[shared row of t] ),
 *    accumulated in fp32 in the order j = 0..k-1, then the shared expert.
 *    The _residual forms add a bf16 residual row r[t] to that finished fp32
 *    sum before the one rounding: out[t] = bf16( r[t] + (routed + shared) ).
 *
 * Row numbering of the expert intermediates H [rows][F] and Y [rows][d]:
 * rows 0..T*k-1 are the routed slots in descriptor order (expert ascending,
 * token ascending within an expert; row r belongs to slot perm[r]); rows
 * T*k..T*k+T-1 are the shared expert's rows for tokens 0..T-1.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, negative or
                                 inconsistent size                                */
    MOE_ERR_UNSUPPORTED = 2,  /* valid, but outside the shapes the kernels handle */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required       */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or a kernel launch failed    */
    MOE_ERR_DEVICE_CHECK = 5  /* a device-side consistency check tripped          */
} moe_status_t;

/* Layer dimensions.  Supported: d % 256 == 0, F % 128 == 0, F_s % 128 == 0,
   group in {32, 64, 128} dividing d, F and F_s, 1 <= k <= min(E, 32),
   1 <= E <= 1024, 0 <= T, T * (k + 1) < 2^31, and E * 2F < 2^31 and
   E * d < 2^31 (the routed weight tensors' row counts). */
typedef struct {
    int32_t T;      /* tokens in the batch                      */
    int32_t d;      /* model width                              */
    int32_t E;      /* routed experts                           */
    int32_t k;      /* experts selected per token               */
    int32_t F;      /* routed expert FFN width                  */
    int32_t F_s;    /* shared expert FFN width                  */
    int32_t group;  /* int4 quantisation group along K          */
    uint32_t flags; /* MOE_FLAG_* below                         */
} moe_dims_t;

/* Path selection and scheduling switches (dims.flags). */
#define MOE_FLAG_FORCE_GEMV 0x1u    /* run the experts on the CUDA-core GEMV path     */
#define MOE_FLAG_FORCE_GROUPED 0x2u /* run the experts on the tcgen05 grouped path    */
#define MOE_FLAG_NO_SCHED 0x4u      /* grouped path: expert-id order, no N-banding     */
#define MOE_FLAG_DECODE_MMA 0x8u    /* T = 1 on the GEMV path: the warp-level tensor-core
                                       projections (one cooperative launch for the whole
                                       layer) instead of the CUDA-core GEMVs              */

/* Packed int4 weights: q [rows][K/2] bytes, s [rows][K/group] fp16 (device);
   q 16-byte aligned, s 2-byte aligned (MOE_ERR_INVALID_ARG otherwise). */
typedef struct {
    const uint8_t* q;
    const uint16_t* s;
} moe_w4_t;

/* fp8 weights of the W8A8 variant: q [rows][K] E4M3 codes, s fp32 [rows]
   (one scale per row); q 16-byte and s 4-byte aligned. */
typedef struct {
    const uint8_t* q;
    const float* s;
} moe_w8_t;

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status_t status);

/* ----------------------------------------------------------------------------
 * moe_pack_w4 -- quantise fp32 weights to the packed int4 format above.
 * Source: the Q4 re-quantised expert weights of thewafflehaus/butter PR #69
 * (commit "feat(laguna): Laguna-S-2.1 decode on the CUDA engine"; weights are
 * re-quantised at load).  Load-time, not on the per-token path.
 *   w    (device) fp32 [rows][K], row-major
 *   q    (device) out: uint8 [rows][K/2]
 *   s    (device) out: fp16 bits [rows][K/group]
 * Requires K % group == 0, group in {8, 16, 32, 64, 128} (the layer calls take
 * 32, 64 or 128), rows >= 0, w 16-byte aligned.  Weights must be finite.
 * Returns MOE_ERR_UNSUPPORTED for other group sizes.
 */
moe_status_t moe_pack_w4(const float* w, int64_t rows, int64_t K, int32_t group, uint8_t* q,
                         uint16_t* s, void* stream);

/* moe_pack_w4_bytes -- sizes of moe_pack_w4's outputs for these arguments:
 * returns the packed bytes (rows * K/2) and writes the scale bytes
 * (rows * K/group * 2) to *scale_bytes when that is non-null.  Host only, no
 * CUDA call.  Returns 0 (and writes 0) for arguments moe_pack_w4 rejects. */
size_t moe_pack_w4_bytes(int64_t rows, int64_t K, int32_t group, size_t* scale_bytes);

/* moe_import_q4_blocks -- load-time import of GGUF-style Q4 blocks into the
 * packed int4 format above.  Source: the Q4 re-quantised weight load straight
 * from GGUF of thewafflehaus/butter PR #69 (commit "feat(laguna): Laguna-S-2.1
 * decode on the CUDA engine").  Block format (the GGUF Q4 block): 32 weights
 * in 18 bytes, an fp16 scale d (little-endian) and then 16 bytes whose byte i
 * holds the 4-bit code n of weight i in bits 0-3 and of weight i + 16 in bits
 * 4-7; the weight is (n - 8) * d.  With group <= 32 every quantisation group
 * lies inside one block and the import is exact: s = d (its fp16 bits, sign
 * included) and q = n - 8.  With group 64 or 128 a group spans blocks with
 * different scales, so the import decodes every block exactly to fp32 in
 * w_scratch and then quantises w_scratch as moe_pack_w4 does (s = absmax / 7
 * per group; lossy wherever a group's blocks do not share one scale grid).
 * Either way w_scratch is left holding the decoded weights.
 *   blocks    (device) uint8 [rows][K/32][18], row-major, any alignment
 *   w_scratch (device) out: fp32 [rows][K], 16-byte aligned (left holding the
 *             decoded weights)
 *   q, s      (device) out: as moe_pack_w4 (q 4-byte, s 2-byte aligned)
 * Requires K % 32 == 0 and K % group == 0, group as for moe_pack_w4.
 */
moe_status_t moe_import_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, int32_t group,
                                  float* w_scratch, uint8_t* q, uint16_t* s, void* stream);

/* Bytes of workspace the per-step calls below need for these dimensions
   (the same number serves every call; 0 on invalid dims). */
size_t moe_workspace_bytes(const moe_dims_t* dims);

/* ----------------------------------------------------------------------------
 * moe_router_topk -- sigmoid router with score-correction bias, top-k.
 * Source: the Laguna MoE router (sigmoid scores, ten experts per token, a
 * correction bias added to the scores for the choice), thewafflehaus/butter
 * PR #69, commit "feat(laguna): Laguna-S-2.1 decode on the CUDA engine".
 *   x        (device) bf16 [T][d]
 *   W_r      (device) fp32 [E][d]
 *   bias     (device) fp32 [E]
 *   topk_idx (device) out: int32 [T][k], descending s + bias
 *   topk_w   (device) out: fp32 [T][k], s_j / sum_j s_j
 *   margin   (device) out, nullable: fp32 [T], (k-th largest s + bias) minus
 *            ((k+1)-th largest), +inf when k == E
 *   ws       (device) workspace of moe_workspace_bytes(dims) bytes
 */
moe_status_t moe_router_topk(const uint16_t* x, const float* W_r, const float* bias,
                             const moe_dims_t* dims, int32_t* topk_idx, float* topk_w,
                             float* margin, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------
 * moe_router_topk_noalloc -- moe_router_topk without a workspace, for callers
 * that cannot allocate device memory when they call the router.  Examples: a
 * host framework that owns every device allocation through its own pool and
 * forbids side allocations; a serving process that reserved all of HBM for
 * weights and caches at start-up.  The pages have no counterpart: this is a
 * library convenience, not part of the layer they describe.
 *
 * Arguments and results are those of moe_router_topk, minus ws/ws_bytes; the
 * caller still passes x, W_r, bias and the output buffers.  The router's
 * scratch (its fp32 logit partials) lives in a fixed 4 MiB device array inside
 * libmoe.so.  Every GPU that loads the library holds that array until the
 * process exits.  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *  - Limit: the partials need ksplit * T * E * 4 bytes, where ksplit = d / 512
 *    (d / 256 when d % 512 != 0) for T <= 64 and 1 above.  Anything beyond
 *    4 MiB returns MOE_ERR_UNSUPPORTED before launching.  For E = 256 that is
 *    T <= 64 in the decode form (at d <= 16384) and T <= 4096 above it.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it.  With
 *    lazy module loading (CUDA_MODULE_LOADING=LAZY, the default of current CUDA
 *    runtimes) that lookup is also what loads the array's module, so the 4 MiB
 *    are allocated on the device by that first call, not when the library is
 *    loaded.  A caller that reserves all of HBM must therefore make one call on
 *    each device first (a T = 1 call is enough), or run with
 *    CUDA_MODULE_LOADING=EAGER so that the array is allocated when the library
 *    loads.  Make the first call before any stream capture too.
 *  - Devices: the cached address belongs to the current device (cudaGetDevice)
 *    at the time of the call, so `stream` must be a stream of that device.
 *  - Sharing: every call uses the same array.  The call writes every partial
 *    it reads, so nothing needs clearing between calls.  Calls that overlap on
 *    the GPU (concurrent streams, or several host threads on one device)
 *    race on the array: serialise them.
 */
moe_status_t moe_router_topk_noalloc(const uint16_t* x, const float* W_r, const float* bias,
                                     const moe_dims_t* dims, int32_t* topk_idx, float* topk_w,
                                     float* margin, void* stream);

/* ----------------------------------------------------------------------------
 * moe_build_descriptors -- on-device expert descriptors (counting sort).
 * Source: the prefill MoE's expert descriptors, built on the device,
 * thewafflehaus/butter PR #69, commit "feat(laguna): batched prefill with
 * tensor-core projections, fused MoE, CTA scheduling"; CSR offsets with one
 * entry per expert plus one and a router-sorted token index, thewafflehaus/
 * FFAI PR #72 (Nemotron W4A16 Marlin MoE commit).
 *   topk_idx (device) int32 [T][k], every id in [0, E)
 *   counts   (device) out: int32 [E], slots per expert
 *   offsets  (device) out: int32 [E+1], exclusive scan of counts
 *   perm     (device) out: int32 [T*k], slot ids t*k+j sorted by (expert, token)
 *   pos      (device) out: int32 [T*k], pos[perm[r]] = r
 *   sched    (device) out: int32 [E], experts by count, largest first, ties to
 *            the lower id
 *   ws       (device) workspace; also receives the tile schedule that
 *            moe_gateup_swiglu_w4a16 and moe_down_w4a16 read, so pass the same
 *            workspace to them for this batch.
 * An id outside [0, E) sets the device check flag (see moe_check_device_status)
 * and the slot is dropped from the descriptors.
 */
moe_status_t moe_build_descriptors(const int32_t* topk_idx, const moe_dims_t* dims,
                                   int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                                   int32_t* sched, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------
 * moe_gateup_swiglu_w4a16 -- fused gate+up projection with SwiGLU, every
 * selected expert plus the shared expert, reading x through perm (gather on
 * read).  Source: the fused gate+up MoE projection, with the shared expert
 * run through the same gathered kernel, thewafflehaus/butter PR #69, commit
 * "feat(laguna): Laguna-S-2.1 decode on the CUDA engine"; gate and up stacked
 * per expert in the prefill path, commit "feat(laguna): batched prefill with
 * tensor-core projections, fused MoE, CTA scheduling".
 *   x        (device) bf16 [T][d]
 *   offsets, perm, sched (device) from moe_build_descriptors
 *   Wgu      routed gate+up, q [E][2F][d/2], s [E][2F][d/group]; rows 0..F-1
 *            of each expert are the gate, rows F..2F-1 the up projection
 *   Wgu_s    shared gate+up, q [2F_s][d/2], s [2F_s][d/group]
 *   H        (device) out: bf16 [T*k + T][max(F, F_s)] (row stride max(F, F_s))
 *   ws       the workspace moe_build_descriptors filled for this batch
 * T <= 2 runs a CUDA-core GEMV, larger T the tcgen05 grouped kernel; the
 * flags can force either (the GEMV needs d <= 4096 and max(F, F_s) <= 2048,
 * the grouped kernel d, F, F_s multiples of 128 and at most 32 quantisation
 * groups per row; a forced path that does not cover the shape returns
 * MOE_ERR_UNSUPPORTED).
 */
moe_status_t moe_gateup_swiglu_w4a16(const uint16_t* x, const moe_dims_t* dims,
                                     const int32_t* offsets, const int32_t* perm,
                                     const int32_t* sched, moe_w4_t Wgu, moe_w4_t Wgu_s,
                                     uint16_t* H, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------
 * moe_down_w4a16 -- down projection of every row of H (routed rows with their
 * expert's down weights, the shared rows with the shared expert's).  Sources:
 * the gathered Q4 down GEMV of the decode step, thewafflehaus/butter PR #69,
 * commit "feat(laguna): Laguna-S-2.1 decode on the CUDA engine"; the
 * per-expert down projection of the W4A16 grouped MoE, thewafflehaus/FFAI
 * PR #72, Nemotron W4A16 Marlin MoE commit.  H rows are already grouped by
 * expert (descriptor order), so no gather is needed and perm is not an
 * argument.
 *   H        (device) bf16 [T*k + T][max(F, F_s)]
 *   offsets, sched (device) from moe_build_descriptors
 *   Wd       routed down, q [E][d][F/2], s [E][d][F/group]
 *   Wd_s     shared down, q [d][F_s/2], s [d][F_s/group]
 *   Y        (device) out: fp32 [T*k + T][d]
 *   ws       the workspace moe_build_descriptors filled for this batch
 */
moe_status_t moe_down_w4a16(const uint16_t* H, const moe_dims_t* dims, const int32_t* offsets,
                            const int32_t* sched, moe_w4_t Wd, moe_w4_t Wd_s, float* Y, void* ws,
                            size_t ws_bytes, void* stream);

/* moe_down_combine_w4a16 -- the down projection with the weighted combine
 * fused in (the deterministic scatter-add of the same FFAI commit, here a
 * fixed-order per-token sum instead of atomics):
 *   out[t] = bf16( [float(residual[t]) +] (sum_j topk_w[t][j] * Y[pos[t*k+j]]
 *                                           + Y[T*k + t]) ),
 * the same value and summation order as moe_down_w4a16 followed by
 * moe_combine_shared (or moe_combine_shared_residual), without the caller's Y.
 * On the GEMV path (T <= 2 by default) the combine runs inside the down
 * kernel and Y stays in L2; on the grouped path it is the down launch and a
 * combine launch, Y in the workspace.
 *   topk_w   (device) fp32 [T][k], from moe_router_topk
 *   pos      (device) int32 [T*k], from moe_build_descriptors
 *   residual (device) bf16 [T][d], 16-byte aligned, or NULL; may be out
 *   out      (device) out: bf16 [T][d], 16-byte aligned
 *   ws       a workspace of moe_layer_workspace_bytes(dims), the one
 *            moe_build_descriptors filled for this batch (Y lives in it)
 */
moe_status_t moe_down_combine_w4a16(const uint16_t* H, const moe_dims_t* dims,
                                    const int32_t* offsets, const int32_t* sched,
                                    const float* topk_w, const int32_t* pos, moe_w4_t Wd,
                                    moe_w4_t Wd_s, const uint16_t* residual, uint16_t* out,
                                    void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------
 * moe_combine_shared -- weighted combine of the routed rows plus the shared
 * row, fixed summation order (deterministic).  Source: the deterministic
 * scatter-add and the residual + routed + shared add of thewafflehaus/FFAI
 * PR #72 (Nemotron commits "ffai_add3" and W4A16 Marlin MoE).
 *   Y        (device) fp32 [T*k + T][d]
 *   topk_w   (device) fp32 [T][k]
 *   pos      (device) int32 [T*k]
 *   out      (device) out: bf16 [T][d]
 */
moe_status_t moe_combine_shared(const float* Y, const float* topk_w, const int32_t* pos,
                                const moe_dims_t* dims, uint16_t* out, void* stream);

/* moe_combine_shared_residual -- moe_combine_shared plus a residual row in
 * the same launch (thewafflehaus/FFAI PR #72, Nemotron commit "ffai_add3":
 * residual + routed accumulator + shared output in one kernel, the routed and
 * shared terms summed first):
 *   out[t] = bf16( float(residual[t]) + (sum_j topk_w[t][j] * Y[pos[t*k+j]]
 *                                        + Y[T*k + t]) ),
 * the bracket summed in fp32 in the order of moe_combine_shared, one rounding.
 *   residual (device) bf16 [T][d], 16-byte aligned; may be the same buffer
 *            as out (in-place residual update)
 *   out      (device) out: bf16 [T][d], 16-byte aligned
 * MOE_ERR_INVALID_ARG for a null or misaligned residual or out.
 */
moe_status_t moe_combine_shared_residual(const float* Y, const float* topk_w, const int32_t* pos,
                                         const moe_dims_t* dims, const uint16_t* residual,
                                         uint16_t* out, void* stream);

/* ----------------------------------------------------------------------------
 * moe_layer_forward -- the whole layer in one call: router, descriptors,
 * gate+up SwiGLU, down, combine, with the intermediates in the workspace.
 * Same arguments as the calls above; ws must hold moe_layer_workspace_bytes
 * and be zero-filled before its first use (the single-launch decode router
 * keeps a completion counter in it, which every call leaves at zero).
 * On the GEMV path (T <= 2 by default) the call is three launches chained by
 * programmatic dependent launch: the router with the top-k and descriptors in
 * its last CTA, gate+up, and down with the combine fused in; otherwise the
 * router, descriptors, grouped gate+up and down, and combine.
 * Graph-capturable.
 */
size_t moe_layer_workspace_bytes(const moe_dims_t* dims);
moe_status_t moe_layer_forward(const uint16_t* x, const float* W_r, const float* bias,
                               const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                               moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* out, void* ws,
                               size_t ws_bytes, void* stream);

/* moe_layer_forward_residual -- moe_layer_forward with the residual add of
 * moe_combine_shared_residual folded into the layer's last kernel (the
 * combine, or on the GEMV path the down kernel's fused combine): out =
 * bf16(residual + (routed + shared)).  residual and out are bf16 [T][d],
 * 16-byte aligned; out may be the residual buffer (in-place update), not x.
 * Same workspace and launches as moe_layer_forward. */
moe_status_t moe_layer_forward_residual(const uint16_t* x, const float* W_r, const float* bias,
                                        const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                                        moe_w4_t Wgu_s, moe_w4_t Wd_s, const uint16_t* residual,
                                        uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* moe_layer_forward_host -- as moe_layer_forward, but x_host is read from
 * host memory and the output is written to out_host: the call enqueues the
 * host-to-device copy of x, the layer and the device-to-host copy of out on
 * `stream` and returns without waiting (the caller synchronises the stream
 * before reading out_host).  Both host buffers should be pinned.  The device
 * staging buffers for x and out are part of moe_layer_workspace_bytes. */
moe_status_t moe_layer_forward_host(const uint16_t* x_host, const float* W_r, const float* bias,
                                    const moe_dims_t* dims, moe_w4_t Wgu, moe_w4_t Wd,
                                    moe_w4_t Wgu_s, moe_w4_t Wd_s, uint16_t* out_host, void* ws,
                                    size_t ws_bytes, void* stream);

/* moe_check_device_status -- synchronises `stream`, reads and clears the
 * device check flag in `ws`.  Returns MOE_ERR_DEVICE_CHECK if a kernel
 * recorded an inconsistency since the last check, MOE_ERR_CUDA if the stream
 * reported an error, MOE_OK otherwise.  For tests and debugging; it is the one
 * call that blocks the host. */
moe_status_t moe_check_device_status(void* ws, size_t ws_bytes, void* stream);

/* moe_debug_set_waits -- test hook for the bounded waits.  Every mbarrier wait
 * in the grouped kernels gives up after a limit (2 s by default), records a
 * wait timeout in the workspace header (moe_check_device_status then returns
 * MOE_ERR_DEVICE_CHECK) and ends its kernel in order: the other roles leave at
 * their next wait, the copy and MMA issuers wait (bounded) for their own work
 * in flight, TMEM is freed.  This
 * call stores, in the workspace header (stream-ordered, graph-capturable):
 *   wait_ns         the limit of every such wait using this workspace (0: the
 *                   default);
 *   withhold_stage  s > 0: in every later gate+up launch on the grouped path
 *                   (W4A16 and W8A8), CTA 0 skips the copies of its s-th
 *                   pipeline stage, so that stage's consumers wait until the
 *                   limit; 0: off.
 * No memory access changes.  A call with (0, 0) restores normal operation; the
 * workspace stays usable (moe_check_device_status clears the flag). */
moe_status_t moe_debug_set_waits(void* ws, size_t ws_bytes, uint64_t wait_ns,
                                 int32_t withhold_stage, void* stream);

/* ============================================================================
 * W8A8 variant: fp8 (E4M3) weights and activations on the tcgen05 fp8 tensor
 * cores.  Source: the W8A8 grouped MoE of thewafflehaus/FFAI PR #72
 * (Nemotron-H section: fp8 activations x fp8 weights, argmax unchanged), with
 * the scale recipe of the same PR's per-channel FP8 commit (one weight scale
 * per output channel, one activation scale per token row, folded in after the
 * GEMM).  Numerics:
 *  - E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits, no infinities,
 *    largest finite 448; conversions round to nearest even and saturate.
 *  - a weight row w: s = absmax(w) / 448 (fp32), codes e4m3(w / s) (fp32
 *    division); an all-zero row has s = 0 and codes 0.  Activation rows
 *    (each token's x for gate+up, each H row for down) the same way, scale a.
 *  - a projection is (acc * a) * s, acc = sum over K of code products in fp32
 *    (each product exact); SwiGLU, H = bf16, routing, the shared expert and
 *    the combine as in the W4A16 layer.
 * The router and descriptors are the W4A16 layer's; the experts always run
 * on the grouped tensor-core kernel (any T).
 * ========================================================================= */

/* moe_pack_w8 -- fp32 weights [rows][K] (device) to E4M3 codes q [rows][K]
 * and fp32 row scales s [rows] (device).  K % 8 == 0; w 16-byte, q 8-byte and
 * s 4-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Routed gate+up weights
 * are one call on [E*2F][d] (rows 0..F-1 of each expert the gate), down on
 * [E*d][F]; the shared expert's [2F_s][d] and [d][F_s]. */
moe_status_t moe_pack_w8(const float* w, int64_t rows, int64_t K, uint8_t* q, float* s,
                         void* stream);

/* moe_quant_rows_fp8 -- bf16 rows [rows][K] (device) to E4M3 codes
 * [rows][K] and fp32 row scales [rows] (device), the activation quantisation
 * the layer applies.  K % 8 == 0; x 16-byte, q 8-byte, a 4-byte aligned. */
moe_status_t moe_quant_rows_fp8(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                float* a, void* stream);

/* Workspace of moe_layer_forward_w8a8 and of the two W8A8 step calls below
   (0 for unsupported dims). */
size_t moe_layer_workspace_bytes_w8a8(const moe_dims_t* dims);

/* The W8A8 expert projections as separate calls, after moe_router_topk and
 * moe_build_descriptors on a workspace of moe_layer_workspace_bytes_w8a8:
 *   moe_gateup_swiglu_w8a8: quantises each gathered token row (perm order,
 *     then the shared rows) and runs gate+up with SwiGLU into H, bf16
 *     [T*k + T][max(F, F_s)], as moe_gateup_swiglu_w4a16;
 *   moe_down_w8a8: quantises each H row and writes Y, fp32 [T*k + T][d], as
 *     moe_down_w4a16.
 * Then moe_combine_shared (or its residual form) gives the layer output. */
moe_status_t moe_gateup_swiglu_w8a8(const uint16_t* x, const moe_dims_t* dims,
                                    const int32_t* perm, moe_w8_t Wgu, moe_w8_t Wgu_s,
                                    uint16_t* H, void* ws, size_t ws_bytes, void* stream);
moe_status_t moe_down_w8a8(const uint16_t* H, const moe_dims_t* dims, moe_w8_t Wd, moe_w8_t Wd_s,
                           float* Y, void* ws, size_t ws_bytes, void* stream);

/* moe_layer_forward_w8a8 -- the whole layer with W8A8 experts.  Arguments as
 * moe_layer_forward, the weights in moe_pack_w8's format.  Needs d, F, F_s
 * multiples of 128 (MOE_ERR_UNSUPPORTED otherwise). */
moe_status_t moe_layer_forward_w8a8(const uint16_t* x, const float* W_r, const float* bias,
                                    const moe_dims_t* dims, moe_w8_t Wgu, moe_w8_t Wd,
                                    moe_w8_t Wgu_s, moe_w8_t Wd_s, uint16_t* out, void* ws,
                                    size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
