/*
 * synth_lib.cu - host and GPU fill routines for the seeded synthetic inputs.
 *
 * Harness code (not part of the scan library).  The host routines are plain
 * loops; the GPU routines run the same inline functions from synth_gen.h in
 * one thread per row, so a tensor generated on either side has the same bits.
 * Element index convention: a [T, H, d] stream element (t, h, e) has index
 * (t*H + h)*d + e, with t the absolute row of the packed token stream.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "synth_gen.h"

#define SYN_API extern "C" __attribute__((visibility("default")))

enum { SYN_F32 = 0, SYN_BF16 = 1 };

/* sum of squares of one row in the fixed pairwise-tree order (d a power of 2) */
static __host__ __device__ double row_sumsq(uint32_t key, uint64_t base, int d) {
    double stack[24];
    int sp = 0;
    for (int e = 0; e < d; ++e) {
        double x = syn_normal(key, base + (uint64_t)e);
#if defined(__CUDA_ARCH__)
        double v = __dmul_rn(x, x);
#else
        double v = x * x;
#endif
        unsigned m = (unsigned)e;
        while (m & 1U) {
#if defined(__CUDA_ARCH__)
            v = __dadd_rn(stack[--sp], v);
#else
            v = stack[--sp] + v;
#endif
            m >>= 1;
        }
        stack[sp++] = v;
    }
    return stack[0];
}

static __host__ __device__ void write_row(void* out, int dtype, uint64_t out_off, uint32_t key,
                                          uint64_t base, int d, int normalize) {
    double nrm = 1.0;
    if (normalize) {
#if defined(__CUDA_ARCH__)
        nrm = __dsqrt_rn(row_sumsq(key, base, d));
#else
        nrm = sqrt(row_sumsq(key, base, d));
#endif
    }
    for (int e = 0; e < d; ++e) {
        double x = syn_normal(key, base + (uint64_t)e);
        double y = x;
        if (normalize) {
#if defined(__CUDA_ARCH__)
            y = __ddiv_rn(x, nrm);
#else
            y = x / nrm;
#endif
        }
#if defined(__CUDA_ARCH__)
        float f = __double2float_rn(y);
#else
        float f = (float)y;
#endif
        if (dtype == SYN_F32)
            ((float*)out)[out_off + e] = f;
        else
            ((uint16_t*)out)[out_off + e] = syn_f32_to_bf16_bits(f);
    }
}

static int check_rows(int64_t t0, int64_t t1, int32_t H, int32_t h0, int32_t h1, int32_t d, int dtype) {
    if (t0 < 0 || t1 < t0 || H <= 0 || h0 < 0 || h1 < h0 || h1 > H) return 1;
    if (d <= 0 || d > (1 << 20) || (d & (d - 1)) != 0) return 1;
    if (dtype != SYN_F32 && dtype != SYN_BF16) return 1;
    return 0;
}

/* out[(t-t0), (h-h0), e] for t in [t0,t1), h in [h0,h1): unit-norm rows when
 * normalize != 0 (q, k), raw normals otherwise (v). */
SYN_API int syn_fill_rows_host(void* out, int dtype, uint64_t seed, uint32_t stream, int64_t t0,
                               int64_t t1, int32_t H, int32_t h0, int32_t h1, int32_t d,
                               int normalize) {
    if (check_rows(t0, t1, H, h0, h1, d, dtype) || (!out && t1 > t0 && h1 > h0)) return 1;
    uint32_t key = syn_key(seed, stream);
    int64_t nh = h1 - h0;
    for (int64_t t = t0; t < t1; ++t)
        for (int32_t h = h0; h < h1; ++h) {
            uint64_t base = ((uint64_t)t * (uint64_t)H + (uint64_t)h) * (uint64_t)d;
            uint64_t off = ((uint64_t)(t - t0) * (uint64_t)nh + (uint64_t)(h - h0)) * (uint64_t)d;
            write_row(out, dtype, off, key, base, d, normalize);
        }
    return 0;
}

static __global__ void fill_rows_kernel(void* out, int dtype, uint32_t key, int64_t t0,
                                        int64_t nrows, int32_t H, int32_t h0, int32_t nh,
                                        int32_t d, int normalize) {
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= nrows) return;
    int64_t tt = r / nh;
    int32_t hh = (int32_t)(r - tt * nh);
    uint64_t base = ((uint64_t)(t0 + tt) * (uint64_t)H + (uint64_t)(h0 + hh)) * (uint64_t)d;
    write_row(out, dtype, (uint64_t)r * (uint64_t)d, key, base, d, normalize);
}

SYN_API int syn_fill_rows_dev(void* out, int dtype, uint64_t seed, uint32_t stream, int64_t t0,
                              int64_t t1, int32_t H, int32_t h0, int32_t h1, int32_t d,
                              int normalize, void* cuda_stream) {
    if (check_rows(t0, t1, H, h0, h1, d, dtype)) return 1;
    int64_t nrows = (t1 - t0) * (int64_t)(h1 - h0);
    if (nrows == 0) return 0;
    if (!out) return 1;
    int threads = 128;
    int64_t blocks = (nrows + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return 1;
    fill_rows_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)cuda_stream>>>(
        out, dtype, syn_key(seed, stream), t0, nrows, H, h0, h1 - h0, d, normalize);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

/* out[i] = scale * normal(idx0 + i), fp32, i in [0, n) */
SYN_API int syn_fill_normal_host(float* out, uint64_t seed, uint32_t stream, uint64_t idx0,
                                 int64_t n, double scale) {
    if (n < 0 || (!out && n > 0)) return 1;
    uint32_t key = syn_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(scale * syn_normal(key, idx0 + (uint64_t)i));
    return 0;
}

static __global__ void fill_normal_kernel(float* out, uint32_t key, uint64_t idx0, int64_t n,
                                          double scale) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    out[i] = __double2float_rn(__dmul_rn(scale, syn_normal(key, idx0 + (uint64_t)i)));
}

SYN_API int syn_fill_normal_dev(float* out, uint64_t seed, uint32_t stream, uint64_t idx0,
                                int64_t n, double scale, void* cuda_stream) {
    if (n < 0) return 1;
    if (n == 0) return 0;
    if (!out) return 1;
    int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return 1;
    fill_normal_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)cuda_stream>>>(
        out, syn_key(seed, stream), idx0, n, scale);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

/* Gates for (t, h) in [t0,t1) x [h0,h1), written [(t-t0), (h-h0)] fp32.
 * alpha = a_lo + (a_hi - a_lo) * U, rounded once to fp32.
 * beta: kind 0 -> U[0,1) (exact), kind 1 -> sigmoid(normal) rounded to fp32. */
SYN_API int syn_fill_gates_host(float* alpha, float* beta, uint64_t seed, int64_t t0, int64_t t1,
                                int32_t H, int32_t h0, int32_t h1, double a_lo, double a_hi,
                                int beta_kind) {
    if (t0 < 0 || t1 < t0 || H <= 0 || h0 < 0 || h1 < h0 || h1 > H) return 1;
    if (beta_kind != 0 && beta_kind != 1) return 1;
    if ((t1 > t0 && h1 > h0) && (!alpha || !beta)) return 1;
    uint32_t ka = syn_key(seed, SYN_STREAM_ALPHA), kb = syn_key(seed, SYN_STREAM_BETA);
    int64_t nh = h1 - h0;
    for (int64_t t = t0; t < t1; ++t)
        for (int32_t h = h0; h < h1; ++h) {
            uint64_t idx = (uint64_t)t * (uint64_t)H + (uint64_t)h;
            int64_t o = (t - t0) * nh + (h - h0);
            alpha[o] = (float)(a_lo + (a_hi - a_lo) * syn_uniform(ka, idx));
            if (beta_kind == 0)
                beta[o] = (float)syn_uniform(kb, idx);
            else
                beta[o] = (float)(1.0 / (1.0 + exp(-syn_normal(kb, idx))));
        }
    return 0;
}

/* Integer draws in [lo, hi] (inclusive) for request lengths and probe depths. */
SYN_API int syn_fill_int_host(int64_t* out, uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n,
                              int64_t lo, int64_t hi) {
    if (n < 0 || hi < lo || (!out && n > 0)) return 1;
    uint32_t key = syn_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1;
    for (int64_t i = 0; i < n; ++i) {
        uint64_t a = syn_bits24(key, 2 * (idx0 + (uint64_t)i));
        uint64_t b = syn_bits24(key, 2 * (idx0 + (uint64_t)i) + 1);
        uint64_t r = (a << 24) | b; /* 48 random bits */
        out[i] = lo + (int64_t)(r % span);
    }
    return 0;
}
