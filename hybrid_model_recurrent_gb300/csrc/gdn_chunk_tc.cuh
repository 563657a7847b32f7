// gdn_chunk_tc.cuh - chunkwise (WY / UT-transform) Gated DeltaNet scan on the 5th-generation
// tensor cores (tcgen05 + TMEM), for d_k = d_v = 128 and bf16 q/k/v.
//
// The recurrence of the notes page "Tail-Replay: Escaping the Curse of Linear Attention in
// Prefix Caching for Hybrid LLMs" (section 2.3, equation (1): S in R^{d_v x d_k}, key operator
// from the right), S_t = alpha_t S_{t-1} + u_t k_t^T with u_t = beta_t (v_t - alpha_t S_{t-1} k_t),
// regrouped over a chunk of n <= 64 tokens (gamma_t = alpha_1 ... alpha_t within the chunk):
//
//   (I + L) U = diag(beta) V - diag(beta gamma) K S_0^T,  L[t][s] = beta_t (gamma_t/gamma_s) k_t.k_s, s < t
//   U^T = U~^T - S_0 W^T,  W = T diag(beta gamma) K,  U~ = T diag(beta) V,  T = (I + L)^-1
//   o_t = gamma_t S_0 q_t + sum_{s<=t} (gamma_t/gamma_s) (q_t.k_s) u_s
//   S_n = gamma_n S_0 + sum_s (gamma_n/gamma_s) u_s k_s^T
//
// Every product is one tcgen05.mma with M = 128: the state rows (d_v) or the stacked [K; Q] rows.
// The state lives in TMEM as S = sigma St for the whole job.  With sigma_n = sigma_0 gamma_n and
// U''_s = c_s u_s, c_s = 1/(sigma_0 gamma_s), the update is St_n = St_0 + U''^T K (the accumulator
// is never rescaled per chunk) and the readout is o_t = gamma_t (S_0 Q^T)[:, t] + (U''^T P''^T)[:, t]
// with P''[t][s] = sigma_0 gamma_t (q_t.k_s).  What keeps every factor finite:
//   * a chunk ends before the token at which gamma would fall below 2^-32, so gamma_s >= 2^-32;
//   * a chunk of one token with alpha < 2^-32 first scales St to alpha_1 S_0 (sigma -> 1) and then
//     takes c = 1 and P'' = q.k, so no factor exceeds 1;
//   * sigma is folded into St (St <- sigma St, sigma <- 1) when it falls below 2^-40, at every
//     checkpoint and at the end, so checkpoints are plain states and a resume from one repeats
//     the full run's arithmetic bit for bit.
// Chunk ends depend only on the checkpoint list and on the gates after the previous chunk end,
// which the full run and a resume see alike.
//
// Operands that are not exact in bf16 (T diag(.), W, U'', P'', S_0) are split x = hi + lo into two
// bf16 halves and multiplied as hi*hi + hi*lo + lo*hi (or hi*x + lo*x against the exact q, k, v),
// accumulated in fp32 in TMEM.
//
// TMEM (512 columns x 128 lanes of 32 bit):
//   [0,128) St   [128,192) U^T   [192,256) S_0 Q^T   [256,320) G, then U''^T P''^T   [320,384) W^T
//   [384,448) S_0 hi (bf16 pairs)   [448,512) S_0 lo
// Thread 0 issues the TMA copies and the MMAs; warp w reaches TMEM lanes 32(w%4)..+31, and warps
// w and w+4 split the columns.
#pragma once

#include "gdn_kernel.cuh"

namespace gdn {
namespace tc {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 256;

struct Pos {   // chunk schedule cursor
    int begin, len;
};

// ---- shared memory (bytes); swizzled operand tiles are 1024-aligned ----
constexpr int OFF_IN = 0;              // 2 x 32 KB: [K;Q] as two 64-column blocks of [128 rows][128 B]
constexpr int OFF_V = 65536;           // 16 KB: V as two 64-column blocks of [64 rows][128 B]
constexpr int OFF_T1H = 81920;         // [64 t][64 s] bf16 (T diag(beta gamma)) hi
constexpr int OFF_T1L = 90112;         //   lo
constexpr int OFF_T2H = 98304;         // (T diag(beta)) hi
constexpr int OFF_T2L = 106496;        //   lo
constexpr int OFF_PH = 114688;         // [64 t][64 s] P'' hi
constexpr int OFF_PL = 122880;         //   lo
constexpr int OFF_WH = 131072;         // [128 dk][64 t] -W^T hi (MN-major B operand)
constexpr int OFF_WL = 147456;         //   lo
constexpr int OFF_UH = 163840;         // [128 dv][64 t] U''^T hi (K-major A operand)
constexpr int OFF_UL = 180224;         //   lo
constexpr int OFF_LF = 196608;         // fp32 [64][68]: L, then T in place
constexpr int OFF_LD = 214016;         // fp32 4 x [16][17]: diagonal blocks of L
constexpr int OFF_Y = 218368;          // fp32 [32][33] scratch
constexpr int OFF_SC = 222592;         // fp32 per-token scalars: g, ginv, bg, b, c, pscale (6 x 64)
constexpr int OFF_BAR = 224128;        // mbarriers, TMEM address, chunk schedule
constexpr int kSmemBytes = OFF_BAR + 128 + 1024;
constexpr int kLdF = 68;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(OFF_SC + 6 * C * 4 <= OFF_BAR, "scalar area");
static_assert(OFF_Y + 32 * 33 * 4 <= OFF_SC, "scratch area");

constexpr uint32_t T_S = 0, T_U = 128, T_O = 192, T_G = 256, T_W = 320, T_SH = 384, T_SL = 448;
constexpr float kGammaFloor = 0x1p-32f;   // smallest in-chunk decay product
constexpr float kSigmaFloor = 0x1p-40f;   // fold the running scale into the state below this

// ---- tcgen05 / descriptor helpers ----
// shared-memory matrix descriptor: start, leading / stride byte offsets, version 1, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// instruction descriptor of kind::f16: D fp32, A and B bf16, M = 128; a_mn / b_mn: the operand is
// stored with M (or N) contiguous instead of K
__host__ __device__ constexpr uint32_t idesc(int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,"
        "%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
        "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
        "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
        "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31]));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// byte offset of element (row, col) in a 128-byte-swizzled [rows][64] bf16 block (1024-aligned base)
__device__ __forceinline__ uint32_t sw128(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) & 7) << 4) + (col & 7) * 2);
}
// x = hi + lo for a pair, both halves packed as bf16x2 (first element in the low half)
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(hv);
    const __nv_bfloat162 lv = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&hv);
    lo = *reinterpret_cast<const uint32_t*>(&lv);
}
// columns c0..c0+31 (c0 % 8 == 0) of `row`, split and stored to two swizzled [rows][64] tiles
__device__ __forceinline__ void st_split32(unsigned char* th, unsigned char* tl, int row, int c0, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_pair(v[8 * q + 2 * e], v[8 * q + 2 * e + 1], hw[e], lw[e]);
        *reinterpret_cast<uint4*>(th + sw128(row, c0 + 8 * q)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(tl + sw128(row, c0 + 8 * q)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

// ------------------------------------------------------------------------------------
// the kernel: one CTA = one (job, head)
// ------------------------------------------------------------------------------------
template <bool OUT_BF16, bool READOUT>
__global__ void __launch_bounds__(NTHREADS, 1) gdn_chunk_tc_kernel(const __grid_constant__ Params p) {
    using OutT = typename std::conditional<OUT_BF16, __nv_bfloat16, float>::type;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    uint64_t* bar_in = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // [2]: K/Q buffers
    uint64_t* bar_v = bar_in + 2;                                       // V buffer
    uint64_t* bar_mma = bar_in + 3;                                     // tcgen05.commit
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 64);
    int* sh_sched = reinterpret_cast<int*>(smem + OFF_BAR + 72);        // n, single, next begin, next len
    float* sc_g = reinterpret_cast<float*>(smem + OFF_SC);
    float* sc_ginv = sc_g + C;
    float* sc_bg = sc_ginv + C;
    float* sc_b = sc_bg + C;
    float* sc_c = sc_b + C;
    float* sc_p = sc_c + C;
    float* Lf = reinterpret_cast<float*>(smem + OFF_LF);
    float* Ld = reinterpret_cast<float*>(smem + OFF_LD);
    float* Yb = reinterpret_cast<float*>(smem + OFF_Y);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3;                 // TMEM lane quarter of this warp
    const int row = 32 * lq + lane;          // TMEM lane = accumulator row
    const int half = warp >> 2;              // column half handled by this warp
    const int job_idx = blockIdx.x / p.H;
    const int h = blockIdx.x - job_idx * p.H;
    const int H = p.H;
    const Job& job = p.jobs[job_idx];
    const int64_t tok_begin = job.tok_begin;
    const int len = job.len;
    const int ck_end = job.ck_begin + job.ck_count;
    const int64_t o_row0 = job.o_row_begin;
    const bool rd = READOUT && o_row0 >= 0;
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = limit > kDrainLimitNs ? limit : kDrainLimitNs;
    const size_t head_state = (size_t)h * D * D;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        mbar_init(&bar_in[0], 1);
        mbar_init(&bar_in[1], 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t trow = tbase + ((uint32_t)(32 * lq) << 16);   // this warp's lane quarter

    // ---- initial state into TMEM: St = S_0, sigma = 1 ----
    {
        const float* s0 = job.s0;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            const int c0 = 64 * half + 32 * cb;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s0) x = __ldg(reinterpret_cast<const float4*>(s0 + head_state + (size_t)row * D + c0 + i));
                v[i] = x.x;
                v[i + 1] = x.y;
                v[i + 2] = x.z;
                v[i + 3] = x.w;
            }
            tmem_st32(trow + T_S + c0, v);
        }
        tmem_st_wait();
    }

    auto issue_kq = [&](int buf, int pos) {   // thread 0
        proxy_fence();
        mbar_arrive_expect_tx(&bar_in[buf], 4u * 8192u);
        unsigned char* dst = smem + OFF_IN + buf * 32768;
        const int t0 = (int)(tok_begin + pos);
        tma_load_3d(dst + 0, &p.tm_k, 0, h, t0, &bar_in[buf]);
        tma_load_3d(dst + 8192, &p.tm_q, 0, h, t0, &bar_in[buf]);
        tma_load_3d(dst + 16384, &p.tm_k, 64, h, t0, &bar_in[buf]);
        tma_load_3d(dst + 16384 + 8192, &p.tm_q, 64, h, t0, &bar_in[buf]);
    };
    auto issue_v = [&](int pos) {   // thread 0
        proxy_fence();
        mbar_arrive_expect_tx(bar_v, 2u * 8192u);
        const int t0 = (int)(tok_begin + pos);
        tma_load_3d(smem + OFF_V, &p.tm_v, 0, h, t0, bar_v);
        tma_load_3d(smem + OFF_V + 8192, &p.tm_v, 64, h, t0, bar_v);
    };
    // 64-token window from pos, cut at the next checkpoint and at the end of the job
    auto next_window = [&](int pos, int& ck) -> Pos {
        int end = pos + C < len ? pos + C : len;
        while (ck < ck_end && p.ckpts[ck].pos <= pos) ++ck;
        if (ck < ck_end && p.ckpts[ck].pos < end) end = p.ckpts[ck].pos;
        return Pos{pos, end - pos};
    };
    // bounded wait by every thread; the block agrees on the outcome
    auto block_wait = [&](uint64_t* b, uint32_t parity) -> bool {
        bool w = mbar_try_wait(b, parity);
        if (!w) {
            const uint64_t t0 = global_ns();
            while (!(w = mbar_try_wait(b, parity)))
                if (global_ns() - t0 > limit) break;
        }
        return __syncthreads_and(w) != 0;
    };
    // gates of a window, held by warp 0: tokens lane and lane + 32 (alpha = 1, beta = 0 past it)
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
    auto prefix = [&](float a0, float a1, float& g0, float& g1) {   // warp 0: inclusive products
        g0 = a0;
        g1 = a1;
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
    };

    bool ok = true;
    bool mma_pending = false;
    int ck_sched = job.ck_begin;   // schedule cursor (advanced by warp 0 only)
    int ck_dump = job.ck_begin;
    Pos cur = next_window(0, ck_sched);
    int chunk_no = 0, kq_issued = 0, v_issued = 0;
    uint32_t mma_phase = 0;
    float sigma = 1.f;   // S = sigma St (the same in every thread)
    float ga0 = 1.f, ga1 = 1.f, gb0 = 0.f, gb1 = 0.f;
    const bool stall_on = p.stall_after >= 0;   // testing hook: stop issuing copies after stall_after chunks
    if (len > 0) {
        if (!stall_on || p.stall_after > 0) {
            if (tid == 0) {
                issue_kq(0, 0);
                issue_v(0);
            }
            kq_issued = 1;
            v_issued = 1;
        }
        if (warp == 0) load_gates(cur, ga0, ga1, gb0, gb1);
    }

    auto mma_wait = [&]() -> bool {
        const bool r = block_wait(bar_mma, mma_phase & 1);
        ++mma_phase;
        tc_fence_after();
        return r;
    };

    while (len > 0 && cur.begin < len) {
        const int buf = chunk_no & 1;
        const uint32_t inKQ = sbase + OFF_IN + buf * 32768;
        const uint32_t inV = sbase + OFF_V;
        const float sigma0 = sigma;

        // ---- gates: gamma, the cut where gamma < 2^-32, per-token scalars; next window's gates ----
        if (warp == 0) {
            float a0 = ga0, a1 = ga1, b0 = gb0, b1 = gb1;
            float g0, g1;
            prefix(a0, a1, g0, g1);
            const unsigned m0 = __ballot_sync(0xffffffffu, g0 < kGammaFloor);
            const unsigned m1 = __ballot_sync(0xffffffffu, g1 < kGammaFloor);
            const int first = m0 ? __ffs(m0) - 1 : (m1 ? 31 + __ffs(m1) : C);
            int n = cur.len;
            if (first < n) {
                n = first > 0 ? first : 1;
                if (lane >= n) {
                    a0 = 1.f;
                    b0 = 0.f;
                }
                if (lane + 32 >= n) {
                    a1 = 1.f;
                    b1 = 0.f;
                }
                prefix(a0, a1, g0, g1);
            }
            const bool single = n == 1 && __shfl_sync(0xffffffffu, g0, 0) < kGammaFloor;
            const Pos nx = (cur.begin + n < len) ? next_window(cur.begin + n, ck_sched) : Pos{len, 0};
            if (nx.len > 0) load_gates(nx, ga0, ga1, gb0, gb1);
            sc_g[lane] = g0;
            sc_g[lane + 32] = g1;
            sc_ginv[lane] = __frcp_rn(g0);
            sc_ginv[lane + 32] = __frcp_rn(g1);
            sc_bg[lane] = b0 * g0;
            sc_bg[lane + 32] = b1 * g1;
            sc_b[lane] = b0;
            sc_b[lane + 32] = b1;
            sc_c[lane] = lane < n ? (single ? 1.f : __frcp_rn(sigma0 * g0)) : 0.f;
            sc_c[lane + 32] = lane + 32 < n ? __frcp_rn(sigma0 * g1) : 0.f;
            sc_p[lane] = single ? 1.f : sigma0 * g0;
            sc_p[lane + 32] = sigma0 * g1;
            if (lane == 0) {
                sh_sched[0] = n;
                sh_sched[1] = single ? 1 : 0;
                sh_sched[2] = nx.begin;
                sh_sched[3] = nx.len;
            }
        }
        // ---- wait for this chunk's K, Q, V ----
        if (!block_wait(&bar_in[buf], (uint32_t)((chunk_no >> 1) & 1))) { ok = false; break; }
        if (!block_wait(bar_v, (uint32_t)(chunk_no & 1))) { ok = false; break; }
        const int clen = sh_sched[0];
        const bool single = sh_sched[1] != 0;
        const Pos nxt = Pos{sh_sched[2], sh_sched[3]};
        // zero the tile rows past the chunk (whole 128-byte rows: the swizzle stays within a row)
        if (clen < C) {
            const int nz = C - clen;
            for (int i = tid; i < 6 * nz * 8; i += NTHREADS) {
                const int seg = i & 7, rz = (i >> 3) % nz, part = (i >> 3) / nz;   // part 0-3: [K;Q], 4-5: V
                unsigned char* base = part < 4 ? smem + OFF_IN + buf * 32768 + (part >> 1) * 16384 + (part & 1) * 8192
                                               : smem + OFF_V + (part - 4) * 8192;
                *reinterpret_cast<uint4*>(base + (clen + rz) * 128 + seg * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            proxy_fence();
            __syncthreads();
        }

        // ---- G = [K; Q] K^T ----
        const bool issue_next_kq = nxt.len > 0 && kq_issued == chunk_no + 1 && (!stall_on || kq_issued < p.stall_after);
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc(64, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_ss(tbase + T_G, sdesc(inKQ + off, 16, 1024), sdesc(inKQ + off, 16, 1024), id, kk > 0);
            }
            umma_commit(bar_mma);
            // the other K/Q buffer was last read by the previous chunk's MMAs, which have completed
            if (issue_next_kq) issue_kq(buf ^ 1, nxt.begin);
        }
        if (issue_next_kq) ++kq_issued;
        mma_pending = true;
        if (!mma_wait()) { ok = false; break; }
        mma_pending = false;

        // ---- L (fp32, zero on and above the diagonal) and P'' = pscale_t mask(q_t.k_s) (bf16 hi/lo) ----
        {
            float v[32];
            tmem_ld32(trow + T_G + 32 * half, v);
            const int s0 = 32 * half;
            if (row < 64) {
                const int t = row;
                const float f = sc_bg[t];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = s0 + j;
                    const float l = s < t ? f * sc_ginv[s] * v[j] : 0.f;
                    Lf[t * kLdF + s] = l;
                    if ((s >> 4) == (t >> 4)) Ld[(t >> 4) * 16 * 17 + (t & 15) * 17 + (s & 15)] = l;
                }
            } else if (rd) {
                const int t = row - 64;
                const float ps = sc_p[t];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (s0 + j <= t) ? ps * v[j] : 0.f;
                st_split32(smem + OFF_PH, smem + OFF_PL, t, s0, v);
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + L)^-1 in place over Lf: 16x16 diagonal inverses, then a two-level merge ----
        if (warp < 4 && lane < 16) {
            const int b = warp, j = lane;
            const float* Lb = Ld + b * 16 * 17;
            float x[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float vv = (t == j) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < t; ++s2) vv = fmaf(-Lb[t * 17 + s2], x[s2], vv);
                x[t] = vv;
            }
#pragma unroll
            for (int t = 0; t < 16; ++t) Lf[(16 * b + t) * kLdF + 16 * b + j] = x[t];
        }
        __syncthreads();
        {   // T_10 = -T_11 L_10 T_00 (threads 0-127) and T_32 = -T_33 L_32 T_22 (threads 128-255)
            const int grp = tid >> 7, tg = tid & 127;
            const int jb = 2 * grp, ib = jb + 1;
            const int r = tg >> 3, c = 2 * (tg & 7);
            float* Y = Yb + grp * 16 * 17;
            float y0 = 0.f, y1 = 0.f;
            const float* Lr = Lf + (16 * ib + r) * kLdF + 16 * jb;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float l = Lr[m];
                const float2 tv = *reinterpret_cast<const float2*>(Lf + (16 * jb + m) * kLdF + 16 * jb + c);
                y0 = fmaf(l, tv.x, y0);
                y1 = fmaf(l, tv.y, y1);
            }
            Y[r * 17 + c] = y0;
            Y[r * 17 + c + 1] = y1;
            asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory");
            float x0 = 0.f, x1 = 0.f;
            const float* Ti = Lf + (16 * ib + r) * kLdF + 16 * ib;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float tv = Ti[m];
                x0 = fmaf(tv, Y[m * 17 + c], x0);
                x1 = fmaf(tv, Y[m * 17 + c + 1], x1);
            }
            Lf[(16 * ib + r) * kLdF + 16 * jb + c] = -x0;
            Lf[(16 * ib + r) * kLdF + 16 * jb + c + 1] = -x1;
        }
        __syncthreads();
        {   // T_BA = -T_BB (L_BA T_AA) for the lower-left 32x32 block
            const int r = tid >> 3, c = 4 * (tid & 7);
            float y[4] = {0.f, 0.f, 0.f, 0.f};
            const float* Lr = Lf + (32 + r) * kLdF;
#pragma unroll 8
            for (int m = 0; m < 32; ++m) {
                const float l = Lr[m];
                const float4 tv = *reinterpret_cast<const float4*>(Lf + m * kLdF + c);
                y[0] = fmaf(l, tv.x, y[0]);
                y[1] = fmaf(l, tv.y, y[1]);
                y[2] = fmaf(l, tv.z, y[2]);
                y[3] = fmaf(l, tv.w, y[3]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) Yb[r * 33 + c + e] = y[e];
            __syncthreads();
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            const float* Tr = Lf + (32 + r) * kLdF + 32;
#pragma unroll 8
            for (int m = 0; m < 32; ++m) {
                const float tv = Tr[m];
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] = fmaf(tv, Yb[m * 33 + c + e], x[e]);
            }
            *reinterpret_cast<float4*>(Lf + (32 + r) * kLdF + c) = make_float4(-x[0], -x[1], -x[2], -x[3]);
        }
        __syncthreads();
        // ---- T1 = T diag(beta gamma), T2 = T diag(beta) as bf16 hi/lo, K-major [t][s] ----
        {
            const int t = tid >> 2, s0 = 16 * (tid & 3);
            float x1[16], x2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float tv = Lf[t * kLdF + s0 + j];
                x1[j] = tv * sc_bg[s0 + j];
                x2[j] = tv * sc_b[s0 + j];
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    split_pair(x1[8 * q + 2 * e], x1[8 * q + 2 * e + 1], ah[e], al[e]);
                    split_pair(x2[8 * q + 2 * e], x2[8 * q + 2 * e + 1], bh[e], bl[e]);
                }
                const uint32_t o = sw128(t, s0 + 8 * q);
                *reinterpret_cast<uint4*>(smem + OFF_T1H + o) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T1L + o) = make_uint4(al[0], al[1], al[2], al[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T2H + o) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T2L + o) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
            }
        }
        proxy_fence();
        tc_fence_before();
        __syncthreads();

        // ---- W^T = K^T T1^T, U~^T = V^T T2^T (into the U^T accumulator) ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc(64, true, false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ak = sdesc(inKQ + ks * 2048, 16384, 1024);   // K^T: MN-major, d_k blocks 16 KB apart
                const uint64_t av = sdesc(inV + ks * 2048, 8192, 1024);     // V^T: MN-major, d_v blocks 8 KB apart
                umma_ss(tbase + T_W, ak, sdesc(sbase + OFF_T1H + ks * 32, 16, 1024), id, ks > 0);
                umma_ss(tbase + T_W, ak, sdesc(sbase + OFF_T1L + ks * 32, 16, 1024), id, 1);
                umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2H + ks * 32, 16, 1024), id, ks > 0);
                umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2L + ks * 32, 16, 1024), id, 1);
            }
            umma_commit(bar_mma);
        }
        mma_pending = true;
        // ---- meanwhile: S_0 = sigma_0 St as bf16 hi/lo pairs in TMEM (the A operand); a single
        //      small-alpha token first takes St to alpha_1 S_0 ----
        {
            const float pre = sigma0 * sc_g[0];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int c0 = 64 * half + 32 * cb;
                float v[32];
                tmem_ld32(trow + T_S + c0, v);
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) split_pair(sigma0 * v[2 * e], sigma0 * v[2 * e + 1], hw[e], lw[e]);
                tmem_st16(trow + T_SH + c0 / 2, hw);
                tmem_st16(trow + T_SL + c0 / 2, lw);
                if (single) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= pre;
                    tmem_st32(trow + T_S + c0, v);
                }
            }
            tmem_st_wait();
        }
        if (!mma_wait()) { ok = false; break; }
        mma_pending = false;
        // the V buffer is free again: fetch the next chunk's V
        const bool issue_next_v = nxt.len > 0 && v_issued == chunk_no + 1 && (!stall_on || v_issued < p.stall_after);
        if (issue_next_v && tid == 0) issue_v(nxt.begin);
        if (issue_next_v) ++v_issued;
        // ---- -W^T as the MN-major B operand [d_k][t] ----
        {
            float v[32];
            tmem_ld32(trow + T_W + 32 * half, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = -v[j];
            st_split32(smem + OFF_WH, smem + OFF_WL, row, 32 * half, v);
        }
        proxy_fence();
        tc_fence_before();
        __syncthreads();

        // ---- U^T += S_0 (-W)^T;  S_0 Q^T ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idw = idesc(64, false, true);
            const uint32_t idq = idesc(64, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bwh = sdesc(sbase + OFF_WH + kk * 2048, 16384, 1024);
                const uint64_t bwl = sdesc(sbase + OFF_WL + kk * 2048, 16384, 1024);
                const uint32_t ah = tbase + T_SH + 8 * kk, al = tbase + T_SL + 8 * kk;
                umma_ts(tbase + T_U, ah, bwh, idw, 1);
                umma_ts(tbase + T_U, ah, bwl, idw, 1);
                umma_ts(tbase + T_U, al, bwh, idw, 1);
                if (rd) {
                    const uint64_t bq = sdesc(inKQ + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    umma_ts(tbase + T_O, ah, bq, idq, kk > 0);
                    umma_ts(tbase + T_O, al, bq, idq, 1);
                }
            }
            umma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mma_wait()) { ok = false; break; }
        mma_pending = false;

        // ---- U'' = c_t U as bf16 hi/lo (K-major A operand [d_v][t]) ----
        {
            float v[32];
            tmem_ld32(trow + T_U + 32 * half, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= sc_c[32 * half + j];
            st_split32(smem + OFF_UH, smem + OFF_UL, row, 32 * half, v);
        }
        proxy_fence();
        tc_fence_before();
        __syncthreads();

        // ---- U''^T P''^T (into the G columns);  St += U''^T K ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idp = idesc(64, false, false);
            const uint32_t ids = idesc(128, false, true);
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const uint64_t auh = sdesc(sbase + OFF_UH + kt * 32, 16, 1024);
                const uint64_t aul = sdesc(sbase + OFF_UL + kt * 32, 16, 1024);
                if (rd) {
                    const uint64_t bph = sdesc(sbase + OFF_PH + kt * 32, 16, 1024);
                    const uint64_t bpl = sdesc(sbase + OFF_PL + kt * 32, 16, 1024);
                    umma_ss(tbase + T_G, auh, bph, idp, kt > 0);
                    umma_ss(tbase + T_G, auh, bpl, idp, 1);
                    umma_ss(tbase + T_G, aul, bph, idp, 1);
                }
                const uint64_t bk = sdesc(inKQ + kt * 2048, 16384, 1024);   // K: MN-major over d_k
                umma_ss(tbase + T_S, auh, bk, ids, 1);
                umma_ss(tbase + T_S, aul, bk, ids, 1);
            }
            umma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mma_wait()) { ok = false; break; }
        mma_pending = false;

        // ---- readout o_t = gamma_t (S_0 Q^T)[:, t] + (U''^T P''^T)[:, t] ----
        if (rd) {
            float a[32], b[32];
            tmem_ld32(trow + T_O + 32 * half, a);
            tmem_ld32(trow + T_G + 32 * half, b);
            OutT* ob = reinterpret_cast<OutT*>(p.o) + (size_t)h * D + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int t = 32 * half + j;
                if (t < clen) {
                    const float ov = fmaf(sc_g[t], a[j], b[j]);
                    OutT* op = ob + (size_t)(o_row0 + cur.begin + t) * (size_t)H * D;
                    if constexpr (OUT_BF16)
                        *op = __float2bfloat16_rn(ov);
                    else
                        *op = ov;
                }
            }
        }
        // ---- running scale; fold it into St at checkpoints, at the end and below the floor ----
        sigma = single ? 1.f : sigma0 * sc_g[clen - 1];
        const int chunk_end = cur.begin + clen;
        while (ck_dump < ck_end && p.ckpts[ck_dump].pos < chunk_end) ++ck_dump;
        const bool dump = ck_dump < ck_end && p.ckpts[ck_dump].pos == chunk_end;
        const bool last = chunk_end >= len;
        if (dump || last || sigma < kSigmaFloor) {
            float* d1 = dump ? p.ckpt_states + (size_t)p.ckpts[ck_dump].slot * (size_t)H * D * D + head_state : nullptr;
            float* d2 = (last && job.s_final) ? job.s_final + head_state : nullptr;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int c0 = 64 * half + 32 * cb;
                float v[32];
                tmem_ld32(trow + T_S + c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= sigma;
                tmem_st32(trow + T_S + c0, v);
                if (d1) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(d1 + (size_t)row * D + c0 + j) =
                            make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
                if (d2) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(d2 + (size_t)row * D + c0 + j) =
                            make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
            tmem_st_wait();
            sigma = 1.f;
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        cur = nxt;
        ++chunk_no;
    }

    if (ok && len == 0 && job.s_final) {
        // empty range: the final state is the initial one
        const float* s0 = job.s0;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            const int c0 = 64 * half + 32 * cb;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s0) x = __ldg(reinterpret_cast<const float4*>(s0 + head_state + (size_t)row * D + c0 + j));
                *reinterpret_cast<float4*>(job.s_final + head_state + (size_t)row * D + c0 + j) = x;
            }
        }
    }
    if (!ok && tid == 0) {
        // never leave with a copy or an MMA still writing into this CTA's shared memory or TMEM
        for (int cc = chunk_no; cc < kq_issued; ++cc) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&bar_in[cc & 1], (uint32_t)((cc >> 1) & 1)))
                if (global_ns() - t0 > drain_limit) break;
        }
        for (int cc = chunk_no; cc < v_issued; ++cc) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bar_v, (uint32_t)(cc & 1)))
                if (global_ns() - t0 > drain_limit) break;
        }
        if (mma_pending) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(bar_mma, (mma_phase - 1) & 1))
                if (global_ns() - t0 > drain_limit) break;
        }
        atomicOr(p.status, STATUS_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(512));
}

template <bool OUT_BF16, bool READOUT>
cudaError_t launch_chunk_tc(const Params& p, int grid, cudaStream_t stream) {
    auto kern = gdn_chunk_tc_kernel<OUT_BF16, READOUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, NTHREADS, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

// instantiated in inst_chunk_tc.cu
cudaError_t launch(const Params& p, int grid, bool readout, bool out_bf16, cudaStream_t stream);

}  // namespace tc
}  // namespace gdn
