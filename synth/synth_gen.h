/*
 * synth_gen.h - counter-based seeded generator for the synthetic GDN workloads.
 *
 * Harness code shared by the oracle tests and the CUDA path's tests/benchmarks.
 * It draws inputs only: it contains none of the Gated DeltaNet arithmetic.
 *
 * Every value is a pure function of (seed, stream, element index), so any
 * slice (a tail of a prefix, one head, one probe) can be regenerated alone and
 * comes out bit-identical.  The same inline functions are compiled for the
 * host (gcc, -ffp-contract=off) and for the GPU (nvcc, explicit _rn
 * intrinsics), and only IEEE-exact operations are used (integer ops, +, *, /,
 * sqrt in fp64, RNE narrowing), so both builds give the same bits.
 *
 * Hash: Chris Wellons' published "lowbias32" 32-bit integer finaliser.
 * Normal variates: Irwin-Hall sum of four 24-bit uniforms, centred and scaled
 * to unit variance (an exact-arithmetic stand-in for N(0,1); bounded by
 * 2*sqrt(3)).
 */
#ifndef SYNTH_GEN_H
#define SYNTH_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

/* stream identifiers: each input tensor draws from its own stream */
enum {
    SYN_STREAM_Q = 1,
    SYN_STREAM_K = 2,
    SYN_STREAM_V = 3,
    SYN_STREAM_ALPHA = 4,
    SYN_STREAM_BETA = 5,
    SYN_STREAM_STATE = 6,
    SYN_STREAM_AUX = 7
};

SYN_FN uint32_t syn_hash32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

SYN_FN uint32_t syn_key(uint64_t seed, uint32_t stream) {
    uint32_t s = syn_hash32((uint32_t)seed ^ syn_hash32((uint32_t)(seed >> 32) + 0x3c6ef372U));
    return syn_hash32(s ^ (stream * 0x9e3779b9U));
}

/* 24-bit uniform integer for element idx of a keyed stream */
SYN_FN uint32_t syn_bits24(uint32_t key, uint64_t idx) {
    uint32_t h = syn_hash32(key ^ (uint32_t)idx);
    h = syn_hash32(h ^ (uint32_t)(idx >> 32) ^ 0x68e31da4U);
    return h >> 8;
}

/* uniform in [0,1) with 2^-24 resolution (exact in fp32 and fp64) */
SYN_FN double syn_uniform(uint32_t key, uint64_t idx) {
    return (double)syn_bits24(key, idx) * (1.0 / 16777216.0);
}

/* Irwin-Hall(4) normal: mean 0, variance 1.  The four-term sum is exact in
 * fp64 (26 significant bits); the centring is exact; one rounding in the scale. */
SYN_FN double syn_normal(uint32_t key, uint64_t idx) {
    double s = (double)syn_bits24(key, 4 * idx) + (double)syn_bits24(key, 4 * idx + 1) +
               (double)syn_bits24(key, 4 * idx + 2) + (double)syn_bits24(key, 4 * idx + 3);
    double c = s * (1.0 / 16777216.0) - 2.0;
#if defined(__CUDA_ARCH__)
    return __dmul_rn(c, 1.7320508075688772);
#else
    return c * 1.7320508075688772;
#endif
}

/* fp32 -> bf16 bits, round to nearest even (inputs are finite here) */
SYN_FN uint16_t syn_f32_to_bf16_bits(float f) {
    union { float f; uint32_t u; } c;
    c.f = f;
    uint32_t lsb = (c.u >> 16) & 1U;
    uint32_t r = c.u + 0x7fffU + lsb;
    return (uint16_t)(r >> 16);
}

#endif /* SYNTH_GEN_H */
