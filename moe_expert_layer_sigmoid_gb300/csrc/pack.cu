// int4 weight packing (load-time).
//
// The Laguna expert weights are 4-bit, re-quantised when the model is loaded
// (thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1 decode on
// the CUDA engine").  Format: per row, per group of `group` consecutive K
// elements, s = fp16(absmax / 7) and q = clamp(rint(w / s), -8, 7); byte j of a
// row holds element 2j in bits 0-3 and element 2j+1 in bits 4-7.
#include "common.cuh"

namespace moe {
namespace {

// One thread per (row, group).  Reads `group` floats with 16-byte loads and
// writes group/8 32-bit words of nibbles plus one fp16 scale.
template <int G>
__global__ void __launch_bounds__(256) pack_w4_kernel(const float* __restrict__ w, int64_t rows,
                                                      int64_t K, uint8_t* __restrict__ q,
                                                      __half* __restrict__ s) {
    const int64_t ngroups = K / G;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= rows * ngroups) return;
    const int64_t r = gid / ngroups;
    const int64_t g = gid - r * ngroups;
    const float4* src = reinterpret_cast<const float4*>(w + r * K + g * G);

    float amax = 0.0f;
#pragma unroll 8
    for (int i = 0; i < G / 4; ++i) {
        float4 v = __ldg(src + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
    const float sf = __half2float(sh);

    uint32_t* dst = reinterpret_cast<uint32_t*>(q + r * (K / 2) + g * (G / 2));
#pragma unroll 4
    for (int i = 0; i < G / 8; ++i) {
        float4 a = __ldg(src + 2 * i), b = __ldg(src + 2 * i + 1);
        float e[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int qi = 0;
            if (sf != 0.0f) {
                float t = rintf(__fdiv_rn(e[j], sf));
                t = fminf(fmaxf(t, -8.0f), 7.0f);
                qi = (int)t;
            }
            word |= ((uint32_t)qi & 0xFu) << (4 * j);
        }
        dst[i] = word;
    }
    s[gid] = sh;
}

// GGUF-style Q4 blocks -> fp32 rows (load-time import; the weights are read
// from GGUF and re-quantised at load in the same commit).  A block is 18
// bytes: an fp16 scale d (little-endian) and 16 bytes whose byte i holds the
// code n of weight i in bits 0-3 and of weight i + 16 in bits 4-7; the
// weight is (n - 8) * d, exact in fp32.  One thread per block; blocks are
// row-major, so block b covers w[32 b .. 32 b + 31].  Bytes are read one at a
// time: a block is only 2-byte aligned.
__global__ void __launch_bounds__(256) q4_blocks_decode_kernel(const uint8_t* __restrict__ blocks,
                                                               int64_t nblocks,
                                                               float* __restrict__ w) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* blk = blocks + b * 18;
    const float d = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
    float* out = w + b * 32;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int byte = blk[2 + i];
        out[i] = (float)((byte & 15) - 8) * d;
        out[i + 16] = (float)((byte >> 4) - 8) * d;
    }
}

// Groups of at most 32 lie inside one block, so the block is already in the
// canonical form: s = d (its fp16 bits), q = n - 8, whose two's-complement
// nibble is n ^ 8.  One thread per block: 16 packed bytes (element 2j low),
// 32 / G scales, and the decoded fp32 weights for w_scratch.
template <int G>
__global__ void __launch_bounds__(256) q4_blocks_direct_kernel(const uint8_t* __restrict__ blocks,
                                                               int64_t nblocks, float* __restrict__ w,
                                                               uint8_t* __restrict__ q,
                                                               uint16_t* __restrict__ s) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* blk = blocks + b * 18;
    const uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    const float d = __half2float(__ushort_as_half(dbits));
    uint8_t n[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int byte = blk[2 + i];
        n[i] = (uint8_t)(byte & 15);
        n[i + 16] = (uint8_t)(byte >> 4);
    }
    uint8_t* qo = q + b * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) qo[j] = (uint8_t)((n[2 * j] ^ 8) | ((n[2 * j + 1] ^ 8) << 4));
#pragma unroll
    for (int i = 0; i < 32 / G; ++i) s[b * (32 / G) + i] = dbits;
    float* out = w + b * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = (float)((int)n[i] - 8) * d;
}

}  // namespace

cudaError_t launch_import_q4_direct(const uint8_t* blocks, int64_t rows, int64_t K, int group,
                                    float* w, uint8_t* q, uint16_t* s, cudaStream_t st) {
    const int64_t nblocks = rows * (K / 32);
    if (nblocks == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned grid = (unsigned)((nblocks + threads - 1) / threads);
    switch (group) {
        case 8: q4_blocks_direct_kernel<8><<<grid, threads, 0, st>>>(blocks, nblocks, w, q, s); break;
        case 16: q4_blocks_direct_kernel<16><<<grid, threads, 0, st>>>(blocks, nblocks, w, q, s); break;
        case 32: q4_blocks_direct_kernel<32><<<grid, threads, 0, st>>>(blocks, nblocks, w, q, s); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, float* w,
                                    cudaStream_t st) {
    const int64_t nblocks = rows * (K / 32);
    if (nblocks == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned grid = (unsigned)((nblocks + threads - 1) / threads);
    q4_blocks_decode_kernel<<<grid, threads, 0, st>>>(blocks, nblocks, w);
    return cudaGetLastError();
}

cudaError_t launch_pack_w4(const float* w, int64_t rows, int64_t K, int group, uint8_t* q,
                           uint16_t* s, cudaStream_t st) {
    const int64_t n = rows * (K / group);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    __half* sh = reinterpret_cast<__half*>(s);
    switch (group) {
        case 8: pack_w4_kernel<8><<<blocks, threads, 0, st>>>(w, rows, K, q, sh); break;
        case 16: pack_w4_kernel<16><<<blocks, threads, 0, st>>>(w, rows, K, q, sh); break;
        case 32: pack_w4_kernel<32><<<blocks, threads, 0, st>>>(w, rows, K, q, sh); break;
        case 64: pack_w4_kernel<64><<<blocks, threads, 0, st>>>(w, rows, K, q, sh); break;
        case 128: pack_w4_kernel<128><<<blocks, threads, 0, st>>>(w, rows, K, q, sh); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace moe
