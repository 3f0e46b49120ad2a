/*
 * Seeded synthetic inputs for the routed MoE FFN layer.
 *
 * This file only draws random numbers; it holds none of the layer's arithmetic.
 * Both the CPU oracle (through the test suite) and the CUDA path (through the
 * tests and the benchmark) take their inputs from here, so the two sides see
 * bit-identical x, router weights, biases and fp32 expert weights.
 *
 * Generator: a counter-based stream.  Element i of tensor `tid` under `seed`
 * is a pure function of (seed, tid, i):
 *   key   = mix64(seed * phi + mix64(tid + c0))
 *   h(i)  = mix64(key + (i + 1) * phi)
 *   U(i)  = ((h(i) >> 11) + 0.5) * 2^-53            uniform on (0, 1)
 *   N(2m)   = sqrt(-2 ln U(2m)) * cos(2 pi U(2m+1))  Box & Muller (1958); both
 *   N(2m+1) = sqrt(-2 ln U(2m)) * sin(2 pi U(2m+1))  outputs of the pair are used
 * mix64 is the 64-bit finaliser of SplitMix64 (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014), phi = 2^64 / golden ratio.
 * Everything is evaluated in double; a value is converted to fp32 (and, for
 * activations, to bf16 by round-to-nearest-even) only at the end.
 */
#include <math.h>
#include <stdint.h>

#define GEN_PHI 0x9E3779B97F4A7C15ULL
#define GEN_C0 0x632BE59BD9B4E019ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t tensor_key(uint64_t seed, uint64_t tid) {
    return mix64(seed * GEN_PHI + mix64(tid + GEN_C0));
}

static double unit_open(uint64_t key, uint64_t i) {
    uint64_t h = mix64(key + (i + 1) * GEN_PHI);
    return ((double)(h >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* The Box-Muller pair m: out[0] = N(2m), out[1] = N(2m+1). */
static void normal_pair(uint64_t key, uint64_t m, double out[2]) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = unit_open(key, 2 * m);
    double u2 = unit_open(key, 2 * m + 1);
    double r = sqrt(-2.0 * log(u1));
    out[0] = r * cos(two_pi * u2);
    out[1] = r * sin(two_pi * u2);
}

/* Calls emit(j, N(start + j)) for j in [0, n). */
#define FOR_EACH_NORMAL(key, start, n, BODY)                       \
    do {                                                           \
        uint64_t i_ = (start), end_ = (start) + (n);               \
        double p_[2];                                              \
        while (i_ < end_) {                                        \
            normal_pair((key), i_ / 2, p_);                        \
            for (int h_ = (int)(i_ & 1); h_ < 2 && i_ < end_; ++h_, ++i_) { \
                const uint64_t j = i_ - (start);                   \
                const double v = p_[h_];                           \
                BODY;                                              \
            }                                                      \
        }                                                          \
    } while (0)

/* bf16 bit pattern of a finite fp32 value, round to nearest even. */
static uint16_t f32_to_bf16_bits(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* out[j] = (float)(std * N(start + j)), j in [0, n). */
void gen_normal_f32(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, double std,
                    float* out) {
    uint64_t key = tensor_key(seed, tid);
    FOR_EACH_NORMAL(key, start, n, out[j] = (float)(std * v));
}

/* out[j] = bf16 bits of (float)(std * N(start + j)). */
void gen_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, double std,
                     uint16_t* out) {
    uint64_t key = tensor_key(seed, tid);
    FOR_EACH_NORMAL(key, start, n, out[j] = f32_to_bf16_bits((float)(std * v)));
}

/* A seeded permutation of 0..n-1 (Fisher & Yates, Durstenfeld's in-place form). */
void gen_permutation(uint64_t seed, uint64_t tid, int32_t n, int32_t* perm) {
    uint64_t key = tensor_key(seed, tid);
    for (int32_t i = 0; i < n; ++i) perm[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        int32_t j = (int32_t)(unit_open(key, (uint64_t)i) * (double)(i + 1));
        if (j > i) j = i;
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}

/*
 * Skewed correction bias: b_e = scale * ln p(r_e), where r_e = 1 + pi(e) is
 * expert e's rank under a seeded permutation pi and p(r) = r^-s / sum_r' r'^-s
 * is the Zipf(s) law over E ranks.
 */
void gen_zipf_bias(uint64_t seed, uint64_t tid, int32_t E, double s, double scale,
                   int32_t* perm_scratch, float* out) {
    gen_permutation(seed, tid, E, perm_scratch);
    double z = 0.0;
    for (int32_t r = 1; r <= E; ++r) z += pow((double)r, -s);
    for (int32_t e = 0; e < E; ++e) {
        double r = (double)(1 + perm_scratch[e]);
        out[e] = (float)(scale * log(pow(r, -s) / z));
    }
}
