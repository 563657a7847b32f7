// gdn_chunk.cuh - chunkwise (WY / UT-transform) form of the Gated DeltaNet scan on
// the tensor cores, for d_k = d_v = 128 and bf16 q/k/v.
//
// The recurrence of the notes page "Tail-Replay: Escaping the Curse of Linear
// Attention in Prefix Caching for Hybrid LLMs" (section 2.3, equation (1), state
// S in R^{d_v x d_k}, key operator applied from the right) is regrouped over a
// chunk of C tokens with state S_0 before the chunk.  With u_t the value written
// at token t (S_t = alpha_t S_{t-1} + u_t k_t^T, u_t = beta_t (v_t - alpha_t S_{t-1} k_t))
// and gamma_t = alpha_1 ... alpha_t inside the chunk:
//     (I + L) U = diag(beta) V - diag(beta gamma) K S_0^T,
//         L[t][s] = beta_t (gamma_t / gamma_s) (k_t . k_s) for s < t,
//     U = U~ - W S_0^T,  W = T diag(beta gamma) K,  U~ = T diag(beta) V,  T = (I + L)^-1,
//     O = diag(gamma) Q S_0^T + P U,   P[t][s] = (gamma_t / gamma_s) (q_t . k_s) for s <= t,
//     S_C = gamma_C S_0 + (diag(gamma_C / gamma) U)^T K.
// This is the same recurrence regrouped; every token's output and every chunk-end
// state follow exactly.  Chunk boundaries fall every 64 tokens from the job start
// and at every checkpoint position, so checkpoint states are chunk-end states.
//
// GB300 mapping (one CTA = one (job, head), 8 warps):
//  * k, q, v chunk tiles arrive by TMA (128-byte swizzle, double buffered).
//  * All products run on the tensor cores (mma.sync bf16 -> fp32).  q, k, v are
//    exact in bf16; every other operand (T, W, P, U, S) is split into two bf16
//    halves x = hi + lo and the product is hi*hi + hi*lo + lo*hi, fp32 accumulated.
//  * Warp w owns state rows 16w..16w+15 as fp32 mma accumulators for the whole
//    job; their fragments double as the S_0^T operand, and movmatrix transposes U
//    in registers, so the state never leaves the register file between chunks.
//  * T is formed by blocked forward substitution in fp32 on the CUDA cores.
#pragma once

#include "gdn_kernel.cuh"

namespace gdn {
namespace chunk {

constexpr int C = 64;        // tokens per chunk
constexpr int D = 128;       // d_k = d_v
constexpr int NWARP = 8;
constexpr int NTHREADS = NWARP * 32;

// ---- shared-memory layout (bytes) ----
constexpr int kTileBytes = C * D * 2;                    // one bf16 [64][128] tile (two 64-column halves)
constexpr int kInBytes = 3 * kTileBytes;                 // K, Q, V
constexpr int kLdH = 72;                                 // bf16 row stride of [64][64] operands
constexpr int kLdW = 136;                                // bf16 / fp32 row stride of [64][128] operands
constexpr int kLdB = 24;                                 // bf16 row stride of [16][16] diagonal blocks
constexpr int kLdD = 17;                                 // fp32 row stride of [16][16] diagonal blocks
constexpr int kBlk = 16 * kLdB * 2;                      // bytes of one bf16 [16][24] block
constexpr int OFF_IN = 0;                                // 2 x kInBytes, 1024-aligned
constexpr int OFF_W = OFF_IN + 2 * kInBytes;             // bf16 -W: hi, lo [64][136]
constexpr int OFF_UT = OFF_W + 2 * C * kLdW * 2;         // fp32 U~ [64][136]
constexpr int OFF_P = OFF_UT + C * kLdW * 4;             // bf16 P: hi, lo [64][72]
constexpr int OFF_L = OFF_P + 2 * C * kLdH * 2;          // bf16 L: hi, lo [64][72]
constexpr int OFF_TB = OFF_L + 2 * C * kLdH * 2;         // bf16 diagonal inverses: 3 kinds x hi/lo x 4 blocks
constexpr int OFF_LD = OFF_TB + 3 * 2 * 4 * kBlk;        // fp32 diagonal blocks of L: 4 x [16][17]
constexpr int OFF_SC = OFF_LD + 4 * 16 * kLdD * 4;       // fp32 per-token scalars: g, ginv, bg, b, dC
constexpr int OFF_BAR = OFF_SC + 5 * C * 4;              // 2 mbarriers
constexpr int kSmemBytes = OFF_BAR + 64 + 1024;          // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

// ---- fragment helpers (mma.sync m16n8k16, row.col, bf16 -> f32) ----
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t trans8x8(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// bf16x2 (low half = a) of the rounded pair, and of the rounding remainders
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// byte offset of (row, col) in a TMA 128-byte-swizzled [64][128] bf16 tile
// stored as two 64-column halves of [64 rows][128 bytes]; col multiple of 8
__device__ __forceinline__ uint32_t swz(int row, int col) {
    const int half = col >> 6;
    const int chunk16 = (col & 63) >> 3;
    return (uint32_t)(half * (C * 128) + row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

struct Pos {   // chunk schedule cursor
    int begin, len;
};

// ------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------
template <bool OUT_BF16, bool READOUT>
__global__ void __launch_bounds__(NTHREADS, 1) gdn_chunk_kernel(const __grid_constant__ Params p) {
    using OutT = typename std::conditional<OUT_BF16, __nv_bfloat16, float>::type;
    extern __shared__ unsigned char smem_raw[];
    // aligned by pointer arithmetic on the shared array (not through an integer), so that the compiler keeps
    // its address space and plain C++ accesses below compile to shared-memory loads and stores
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    float* sc_g = reinterpret_cast<float*>(smem + OFF_SC);
    float* sc_ginv = sc_g + C;
    float* sc_bg = sc_ginv + C;
    float* sc_b = sc_bg + C;
    float* sc_dC = sc_b + C;
    float* Ld = reinterpret_cast<float*>(smem + OFF_LD);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c4 = lane & 3;     // mma fragment coordinates
    const int job_idx = blockIdx.x / p.H;
    const int h = blockIdx.x - job_idx * p.H;
    const int H = p.H;
    const Job& job = p.jobs[job_idx];
    const int64_t tok_begin = job.tok_begin;
    const int len = job.len;
    const int ck_begin = job.ck_begin, ck_end = job.ck_begin + job.ck_count;
    void* const o_job = job.o;
    const uint64_t limit = p.wait_limit_ns;
    const size_t head_state = (size_t)h * D * D;

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }

    // state slab: rows 16*warp + g (+8), columns 8j + 2c4 (+1) for j = 0..15
    float S[16][4];
    {
        const float* s0 = job.s0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
            if (s0) {
                const float* base = s0 + head_state + (size_t)(16 * warp + g) * D + 8 * j + 2 * c4;
                a = __ldg(reinterpret_cast<const float2*>(base));
                b = __ldg(reinterpret_cast<const float2*>(base + 8 * D));
            }
            S[j][0] = a.x; S[j][1] = a.y; S[j][2] = b.x; S[j][3] = b.y;
        }
    }
    __syncthreads();

    // chunk schedule: 64-token steps from the job start, split at checkpoints
    auto next_chunk = [&](int pos, int& ck) -> Pos {
        int end = pos + C < len ? pos + C : len;
        while (ck < ck_end && p.ckpts[ck].pos <= pos) ++ck;
        if (ck < ck_end && p.ckpts[ck].pos < end) end = p.ckpts[ck].pos;
        return Pos{pos, end - pos};
    };
    auto issue = [&](int buf, int pos) {
        // executed by thread 0
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&bar[buf], (uint32_t)kInBytes);
        unsigned char* dst = smem + OFF_IN + buf * kInBytes;
        const int t0 = (int)(tok_begin + pos);
        tma_load_3d(dst + 0 * kTileBytes, &p.tm_k, 0, h, t0, &bar[buf]);
        tma_load_3d(dst + 0 * kTileBytes + C * 128, &p.tm_k, 64, h, t0, &bar[buf]);
        tma_load_3d(dst + 1 * kTileBytes, &p.tm_q, 0, h, t0, &bar[buf]);
        tma_load_3d(dst + 1 * kTileBytes + C * 128, &p.tm_q, 64, h, t0, &bar[buf]);
        tma_load_3d(dst + 2 * kTileBytes, &p.tm_v, 0, h, t0, &bar[buf]);
        tma_load_3d(dst + 2 * kTileBytes + C * 128, &p.tm_v, 64, h, t0, &bar[buf]);
    };

    // gates of one chunk, held by warp 0: tokens lane and lane + 32 (alpha = 1, beta = 0 past the end)
    auto load_gates = [&](Pos c, float& a0, float& a1, float& b0, float& b1) {
        a0 = a1 = 1.f;
        b0 = b1 = 0.f;
        const size_t gbase = (size_t)(tok_begin + c.begin) * (size_t)H + (size_t)h;
        if (lane < c.len) {
            a0 = __ldg(p.alpha + gbase + (size_t)lane * H);
            b0 = __ldg(p.beta + gbase + (size_t)lane * H);
        }
        if (lane + 32 < c.len) {
            a1 = __ldg(p.alpha + gbase + (size_t)(lane + 32) * H);
            b1 = __ldg(p.beta + gbase + (size_t)(lane + 32) * H);
        }
    };

    bool ok = true;
    int ck_sched = ck_begin;     // cursor for the schedule
    int ck_dump = ck_begin;      // cursor for dumps
    Pos cur = next_chunk(0, ck_sched);
    int chunk_no = 0;            // chunks consumed
    int issued = 0;              // chunks whose copies were issued (uniform across threads)
    const bool may_issue0 = p.stall_after < 0 || p.stall_after > 0;   // testing hook (see Params)
    if (len > 0 && may_issue0 && threadIdx.x == 0) issue(0, 0);
    if (len > 0 && may_issue0) issued = 1;
    float ga0 = 1.f, ga1 = 1.f, gb0 = 0.f, gb1 = 0.f;
    if (len > 0 && warp == 0) load_gates(cur, ga0, ga1, gb0, gb1);

    while (len > 0 && cur.begin < len) {
        const int buf = chunk_no & 1;
        const Pos nxt = (cur.begin + cur.len < len) ? next_chunk(cur.begin + cur.len, ck_sched) : Pos{len, 0};
        const bool may_issue = nxt.len > 0 && issued == chunk_no + 1 && (p.stall_after < 0 || issued < p.stall_after);
        if (may_issue && threadIdx.x == 0) issue(buf ^ 1, nxt.begin);
        if (may_issue) ++issued;
        const int clen = cur.len;
        const uint32_t inK = sbase + OFF_IN + buf * kInBytes;
        const uint32_t inQ = inK + kTileBytes;
        const uint32_t inV = inK + 2 * kTileBytes;

        // ---- gates: gamma (prefix product), scalars; the next chunk's gates are prefetched ----
        if (warp == 0) {
            float a0 = ga0, a1 = ga1, b0 = gb0, b1 = gb1;
            if (nxt.len > 0) load_gates(nxt, ga0, ga1, gb0, gb1);
            float g0 = a0, g1 = a1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float x0 = __shfl_up_sync(0xffffffffu, g0, off);
                const float x1 = __shfl_up_sync(0xffffffffu, g1, off);
                if (lane >= off) {
                    g0 *= x0;
                    g1 *= x1;
                }
            }
            g1 *= __shfl_sync(0xffffffffu, g0, 31);
            const float gC = __shfl_sync(0xffffffffu, clen > 32 ? g1 : g0, (clen - 1) & 31);
            sc_g[lane] = g0;
            sc_g[lane + 32] = g1;
            sc_ginv[lane] = __frcp_rn(g0);
            sc_ginv[lane + 32] = __frcp_rn(g1);
            sc_bg[lane] = b0 * g0;
            sc_bg[lane + 32] = b1 * g1;
            sc_b[lane] = b0;
            sc_b[lane + 32] = b1;
            sc_dC[lane] = lane < clen ? __fdiv_rn(gC, g0) : 0.f;
            sc_dC[lane + 32] = lane + 32 < clen ? __fdiv_rn(gC, g1) : 0.f;
        }
        // ---- wait for the chunk's tiles; zero the rows past the chunk ----
        {
            bool w_ok = true;
            if (!mbar_try_wait(&bar[buf], (uint32_t)((chunk_no >> 1) & 1))) {
                const uint64_t t0 = global_ns();
                while (!(w_ok = mbar_try_wait(&bar[buf], (uint32_t)((chunk_no >> 1) & 1))))
                    if (global_ns() - t0 > limit) break;
            }
            ok = __syncthreads_and(w_ok) != 0;
            if (!ok) break;
            if (clen < C) {
                // whole 128-byte rows: the swizzle permutes within a row only
                for (int i = threadIdx.x; i < 3 * 2 * (C - clen) * 8; i += NTHREADS) {
                    const int seg = i & 7, rowi = (i >> 3) % (C - clen), part = (i >> 3) / (C - clen);
                    const int tensor = part >> 1, half = part & 1;
                    uint4* d = reinterpret_cast<uint4*>(smem + OFF_IN + buf * kInBytes + tensor * kTileBytes +
                                                        half * C * 128 + (clen + rowi) * 128 + seg * 16);
                    *d = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            __syncthreads();
        }

        // ---- A = K K^T -> L (bf16 hi/lo; diagonal blocks also fp32), P = mask(gamma ratio) (Q K^T) ----
        {
            const int mt = warp >> 1, nbase = 32 * (warp & 1);
            float accA[4][4], accP[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) accA[j][e] = accP[j][e] = 0.f;
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                uint32_t ak[4], aq[4];
                const int arow = 16 * mt + (lane & 15), acol = 16 * kt + 8 * (lane >> 4);
                ldsm_x4(inK + swz(arow, acol), ak);
                ldsm_x4(inQ + swz(arow, acol), aq);
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    uint32_t b[4];
                    const int brow = nbase + 16 * jp + 8 * (lane >> 4) + (lane & 7);
                    const int bcol = 16 * kt + 8 * ((lane >> 3) & 1);
                    ldsm_x4(inK + swz(brow, bcol), b);
                    mma(accA[2 * jp], ak, b[0], b[1]);
                    mma(accA[2 * jp + 1], ak, b[2], b[3]);
                    mma(accP[2 * jp], aq, b[0], b[1]);
                    mma(accP[2 * jp + 1], aq, b[2], b[3]);
                }
            }
            __nv_bfloat16* Phi = reinterpret_cast<__nv_bfloat16*>(smem + OFF_P);
            __nv_bfloat16* Plo = Phi + C * kLdH;
            __nv_bfloat16* Lhi = reinterpret_cast<__nv_bfloat16*>(smem + OFF_L);
            __nv_bfloat16* Llo = Lhi + C * kLdH;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = nbase + 8 * j + 2 * c4;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = 16 * mt + g + 8 * hh;
                    const float gt = sc_g[t], bt = sc_b[t];
                    const float r0 = gt * sc_ginv[s], r1 = gt * sc_ginv[s + 1];
                    const float l0 = s < t ? bt * r0 * accA[j][2 * hh] : 0.f;
                    const float l1 = s + 1 < t ? bt * r1 * accA[j][2 * hh + 1] : 0.f;
                    uint32_t hi, lo;
                    split2(l0, l1, hi, lo);
                    *reinterpret_cast<uint32_t*>(Lhi + t * kLdH + s) = hi;
                    *reinterpret_cast<uint32_t*>(Llo + t * kLdH + s) = lo;
                    if ((t >> 4) == (s >> 4)) {   // diagonal block: keep fp32 for the inversion
                        float* d = Ld + (t >> 4) * 16 * kLdD + (t & 15) * kLdD + (s & 15);
                        d[0] = l0;
                        d[1] = l1;
                    }
                    const float q0 = s <= t ? r0 * accP[j][2 * hh] : 0.f;
                    const float q1 = s + 1 <= t ? r1 * accP[j][2 * hh + 1] : 0.f;
                    split2(q0, q1, hi, lo);
                    *reinterpret_cast<uint32_t*>(Phi + t * kLdH + s) = hi;
                    *reinterpret_cast<uint32_t*>(Plo + t * kLdH + s) = lo;
                }
            }
        }
        __syncthreads();

        // ---- inverses of the 16x16 diagonal blocks of (I + L), fp32 forward substitution;
        //      stored as bf16 hi/lo in three column scalings: 1, beta*gamma, beta ----
        if (warp < 4 && lane < 16) {
            const int b = warp, j = lane;
            const float* Lb = Ld + b * 16 * kLdD;
            float x[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float v = (t == j) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < t; ++s2) v = fmaf(-Lb[t * kLdD + s2], x[s2], v);
                x[t] = v;
            }
            const float f1 = sc_bg[16 * b + j], f2 = sc_b[16 * b + j];
            __nv_bfloat16* TB = reinterpret_cast<__nv_bfloat16*>(smem + OFF_TB) + b * (kBlk / 2);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float y[3] = {x[t], x[t] * f1, x[t] * f2};
#pragma unroll
                for (int kind = 0; kind < 3; ++kind) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(y[kind]);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(y[kind] - __bfloat162float(hi));
                    TB[(2 * kind) * 4 * (kBlk / 2) + t * kLdB + j] = hi;
                    TB[(2 * kind + 1) * 4 * (kBlk / 2) + t * kLdB + j] = lo;
                }
            }
        }
        __syncthreads();

        // ---- blocked forward substitution (I + L) X = diag(f) R on the tensor cores:
        //      warps 0-3: X = W, R = K, f = beta gamma; warps 4-7: X = U~, R = V, f = beta.
        //      Warp w owns 32 columns of X; block i: X_i = T_ii diag(f_i) R_i - T_ii sum_k<i L_ik X_k ----
        {
            const bool isW = warp < 4;
            const int cbase = 32 * (warp & 3);
            const uint32_t R = isW ? inK : inV;
            const uint32_t TB = sbase + OFF_TB;
            const uint32_t Tplain_h = TB, Tplain_l = TB + 4 * kBlk;
            const uint32_t Tsc_h = TB + (isW ? 2 : 4) * 4 * kBlk, Tsc_l = Tsc_h + 4 * kBlk;
            const uint32_t Lh = sbase + OFF_L, Ll = Lh + C * kLdH * 2;
            float X[4][4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float Y[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) Y[nt][e] = X[i][nt][e] = 0.f;
                // Y = sum_{k<i} L_ik X_k
#pragma unroll
                for (int k = 0; k < i; ++k) {
                    uint32_t lh[4], ll[4];
                    const uint32_t aoff = (uint32_t)(((16 * i + (lane & 15)) * kLdH + 16 * k + 8 * (lane >> 4)) * 2);
                    ldsm_x4(Lh + aoff, lh);
                    ldsm_x4(Ll + aoff, ll);
                    uint32_t bh[4][2], bl[4][2];
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        uint32_t h0, l0, h1, l1;
                        split2(X[k][nt][0], X[k][nt][1], h0, l0);
                        split2(X[k][nt][2], X[k][nt][3], h1, l1);
                        bh[nt][0] = trans8x8(h0);
                        bh[nt][1] = trans8x8(h1);
                        bl[nt][0] = trans8x8(l0);
                        bl[nt][1] = trans8x8(l1);
                    }
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) mma(Y[nt], lh, bh[nt][0], bh[nt][1]);
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) mma(Y[nt], lh, bl[nt][0], bl[nt][1]);
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) mma(Y[nt], ll, bh[nt][0], bh[nt][1]);
                }
                // X_i = (T_ii diag(f_i)) R_i - T_ii Y
                {
                    uint32_t th[4], tl[4], sh[4], sl[4];
                    const uint32_t boff = (uint32_t)(i * kBlk + ((lane & 15) * kLdB + 8 * (lane >> 4)) * 2);
                    ldsm_x4(Tsc_h + boff, sh);
                    ldsm_x4(Tsc_l + boff, sl);
                    ldsm_x4(Tplain_h + boff, th);
                    ldsm_x4(Tplain_l + boff, tl);
                    uint32_t rb[2][4];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int brow = 16 * i + (lane & 7) + 8 * ((lane >> 3) & 1);
                        const int bcol = cbase + 16 * jj + 8 * (lane >> 4);
                        ldsm_x4_t(R + swz(brow, bcol), rb[jj]);
                    }
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) mma(X[i][nt], sh, rb[nt >> 1][2 * (nt & 1)], rb[nt >> 1][2 * (nt & 1) + 1]);
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) mma(X[i][nt], sl, rb[nt >> 1][2 * (nt & 1)], rb[nt >> 1][2 * (nt & 1) + 1]);
                    if (i > 0) {
                        uint32_t yh[4][2], yl[4][2];
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            uint32_t h0, l0, h1, l1;
                            split2(-Y[nt][0], -Y[nt][1], h0, l0);
                            split2(-Y[nt][2], -Y[nt][3], h1, l1);
                            yh[nt][0] = trans8x8(h0);
                            yh[nt][1] = trans8x8(h1);
                            yl[nt][0] = trans8x8(l0);
                            yl[nt][1] = trans8x8(l1);
                        }
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) mma(X[i][nt], th, yh[nt][0], yh[nt][1]);
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) mma(X[i][nt], th, yl[nt][0], yl[nt][1]);
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) mma(X[i][nt], tl, yh[nt][0], yh[nt][1]);
                    }
                }
            }
            // W (negated, bf16 hi/lo) or U~ (fp32) to shared memory
            if (isW) {
                __nv_bfloat16* Wh = reinterpret_cast<__nv_bfloat16*>(smem + OFF_W);
                __nv_bfloat16* Wl = Wh + C * kLdW;
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int t = 16 * i + g + 8 * hh, col = cbase + 8 * nt + 2 * c4;
                            uint32_t hi, lo;
                            split2(-X[i][nt][2 * hh], -X[i][nt][2 * hh + 1], hi, lo);
                            *reinterpret_cast<uint32_t*>(Wh + t * kLdW + col) = hi;
                            *reinterpret_cast<uint32_t*>(Wl + t * kLdW + col) = lo;
                        }
            } else {
                float* Ut = reinterpret_cast<float*>(smem + OFF_UT);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int t = 16 * i + g + 8 * hh, col = cbase + 8 * nt + 2 * c4;
                            *reinterpret_cast<float2*>(Ut + t * kLdW + col) =
                                make_float2(X[i][nt][2 * hh], X[i][nt][2 * hh + 1]);
                        }
            }
        }
        __syncthreads();
        // U starts from U~ (this warp's 16 dv columns)
        float U[4][2][4];
        {
            const float* Ut = reinterpret_cast<const float*>(smem + OFF_UT);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float2 u = *reinterpret_cast<const float2*>(
                            Ut + (16 * mt + g + 8 * hh) * kLdW + 16 * warp + 8 * nt + 2 * c4);
                        U[mt][nt][2 * hh] = u.x;
                        U[mt][nt][2 * hh + 1] = u.y;
                    }
        }

        // ---- U += (-W) S_0^T and O = Q S_0^T over the state columns (dk) ----
        float O[4][2][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) O[mt][nt][e] = 0.f;
        {
            const uint32_t Wh = sbase + OFF_W, Wl = Wh + C * kLdW * 2;
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                // S_0^T operand for dk 16kt..16kt+15 and this warp's 16 rows (two n-tiles)
                uint32_t sh[2][2], sl[2][2];
                split2(S[2 * kt][0], S[2 * kt][1], sh[0][0], sl[0][0]);
                split2(S[2 * kt + 1][0], S[2 * kt + 1][1], sh[0][1], sl[0][1]);
                split2(S[2 * kt][2], S[2 * kt][3], sh[1][0], sl[1][0]);
                split2(S[2 * kt + 1][2], S[2 * kt + 1][3], sh[1][1], sl[1][1]);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    uint32_t wh[4], wl[4], aq[4];
                    const uint32_t aoff = (uint32_t)(((16 * mt + (lane & 15)) * kLdW + 16 * kt + 8 * (lane >> 4)) * 2);
                    ldsm_x4(Wh + aoff, wh);
                    ldsm_x4(Wl + aoff, wl);
                    if (READOUT) ldsm_x4(inQ + swz(16 * mt + (lane & 15), 16 * kt + 8 * (lane >> 4)), aq);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        mma(U[mt][nt], wh, sh[nt][0], sh[nt][1]);
                        if (READOUT) mma(O[mt][nt], aq, sh[nt][0], sh[nt][1]);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        mma(U[mt][nt], wh, sl[nt][0], sl[nt][1]);
                        if (READOUT) mma(O[mt][nt], aq, sl[nt][0], sl[nt][1]);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) mma(U[mt][nt], wl, sh[nt][0], sh[nt][1]);
                }
            }
        }

        // ---- O = diag(gamma) O + P U ; write the readout ----
        if (READOUT) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float gt = sc_g[16 * mt + g + 8 * hh];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        O[mt][nt][2 * hh] *= gt;
                        O[mt][nt][2 * hh + 1] *= gt;
                    }
                }
            const uint32_t Ph = sbase + OFF_P, Pl = Ph + C * kLdH * 2;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                // U (tokens 16kt.., this warp's dv) as the B operand: transpose 8x8 blocks
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    uint32_t h0, l0, h1, l1;
                    split2(U[kt][nt][0], U[kt][nt][1], h0, l0);
                    split2(U[kt][nt][2], U[kt][nt][3], h1, l1);
                    bh[nt][0] = trans8x8(h0);
                    bh[nt][1] = trans8x8(h1);
                    bl[nt][0] = trans8x8(l0);
                    bl[nt][1] = trans8x8(l1);
                }
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    uint32_t ph[4], pl[4];
                    const uint32_t aoff = (uint32_t)(((16 * mt + (lane & 15)) * kLdH + 16 * kt + 8 * (lane >> 4)) * 2);
                    ldsm_x4(Ph + aoff, ph);
                    ldsm_x4(Pl + aoff, pl);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) mma(O[mt][nt], ph, bh[nt][0], bh[nt][1]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) mma(O[mt][nt], ph, bl[nt][0], bl[nt][1]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) mma(O[mt][nt], pl, bh[nt][0], bh[nt][1]);
                }
            }
            if (o_job != nullptr) {
                OutT* obase = reinterpret_cast<OutT*>(o_job) + (size_t)h * D + 16 * warp + 2 * c4;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int t = 16 * mt + g + 8 * hh;
                        if (t < clen) {
                            OutT* orow = obase + (size_t)(cur.begin + t) * (size_t)H * D;
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                if constexpr (OUT_BF16)
                                    *reinterpret_cast<uint32_t*>(orow + 8 * nt) =
                                        pack_bf16(O[mt][nt][2 * hh], O[mt][nt][2 * hh + 1]);
                                else
                                    *reinterpret_cast<float2*>(orow + 8 * nt) =
                                        make_float2(O[mt][nt][2 * hh], O[mt][nt][2 * hh + 1]);
                            }
                        }
                    }
            }
        }

        // ---- S = gamma_C S + (diag(gamma_C / gamma) U)^T K ----
        {
            const float gC = sc_g[clen - 1];
#pragma unroll
            for (int j = 0; j < 16; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] *= gC;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const float d0 = sc_dC[16 * kt + g], d1 = sc_dC[16 * kt + g + 8];
                uint32_t ah[4], al[4];
                {
                    uint32_t h00, l00, h01, l01, h10, l10, h11, l11;
                    split2(U[kt][0][0] * d0, U[kt][0][1] * d0, h00, l00);   // tokens 0-7,  dv 0-7
                    split2(U[kt][1][0] * d0, U[kt][1][1] * d0, h01, l01);   // tokens 0-7,  dv 8-15
                    split2(U[kt][0][2] * d1, U[kt][0][3] * d1, h10, l10);   // tokens 8-15, dv 0-7
                    split2(U[kt][1][2] * d1, U[kt][1][3] * d1, h11, l11);   // tokens 8-15, dv 8-15
                    ah[0] = trans8x8(h00); ah[1] = trans8x8(h01); ah[2] = trans8x8(h10); ah[3] = trans8x8(h11);
                    al[0] = trans8x8(l00); al[1] = trans8x8(l01); al[2] = trans8x8(l10); al[3] = trans8x8(l11);
                }
                uint32_t b[8][4];
#pragma unroll
                for (int jp = 0; jp < 8; ++jp) {
                    const int brow = 16 * kt + (lane & 7) + 8 * ((lane >> 3) & 1);
                    const int bcol = 16 * jp + 8 * (lane >> 4);
                    ldsm_x4_t(inK + swz(brow, bcol), b[jp]);
                }
#pragma unroll
                for (int jp = 0; jp < 8; ++jp) {
                    mma(S[2 * jp], ah, b[jp][0], b[jp][1]);
                    mma(S[2 * jp + 1], ah, b[jp][2], b[jp][3]);
                }
#pragma unroll
                for (int jp = 0; jp < 8; ++jp) {
                    mma(S[2 * jp], al, b[jp][0], b[jp][1]);
                    mma(S[2 * jp + 1], al, b[jp][2], b[jp][3]);
                }
            }
        }

        // ---- checkpoint dump at the chunk end ----
        const int chunk_end = cur.begin + clen;
        while (ck_dump < ck_end && p.ckpts[ck_dump].pos < chunk_end) ++ck_dump;
        if (ck_dump < ck_end && p.ckpts[ck_dump].pos == chunk_end) {
            float* dst = p.ckpt_states + (size_t)p.ckpts[ck_dump].slot * (size_t)H * D * D + head_state;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float* base = dst + (size_t)(16 * warp + g) * D + 8 * j + 2 * c4;
                *reinterpret_cast<float2*>(base) = make_float2(S[j][0], S[j][1]);
                *reinterpret_cast<float2*>(base + 8 * D) = make_float2(S[j][2], S[j][3]);
            }
        }
        __syncthreads();   // all reads of this chunk's buffers are done
        cur = nxt;
        ++chunk_no;
    }

    if (!ok) {
        // drain: never leave with a copy in flight into this CTA's shared memory
        if (threadIdx.x == 0) {
            for (int cc = chunk_no; cc < issued; ++cc) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&bar[cc & 1], (uint32_t)((cc >> 1) & 1)))
                    if (global_ns() - t0 > (limit > kDrainLimitNs ? limit : kDrainLimitNs)) break;
            }
            atomicOr(p.status, STATUS_TIMEOUT);
        }
        return;
    }
    float* fin = job.s_final;
    if (fin) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float* base = fin + head_state + (size_t)(16 * warp + g) * D + 8 * j + 2 * c4;
            *reinterpret_cast<float2*>(base) = make_float2(S[j][0], S[j][1]);
            *reinterpret_cast<float2*>(base + 8 * D) = make_float2(S[j][2], S[j][3]);
        }
    }
}

template <bool OUT_BF16, bool READOUT>
cudaError_t launch_chunk(const Params& p, int grid, cudaStream_t stream) {
    auto kern = gdn_chunk_kernel<OUT_BF16, READOUT>;
    static std::atomic<int> optin[kMaxOptinDevices];
    cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), kSmemBytes, optin);
    if (e != cudaSuccess) return e;
    kern<<<grid, NTHREADS, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace chunk
}  // namespace gdn
