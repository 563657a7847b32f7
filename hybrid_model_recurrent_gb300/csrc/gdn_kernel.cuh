// gdn_kernel.cuh - sm_103a state-scan kernel for the Gated DeltaNet recurrence.
//
// Operation (notes page "Tail-Replay: Escaping the Curse of Linear Attention in
// Prefix Caching for Hybrid LLMs", section 2.3, equation (1), right-multiplied
// for S in R^{d_v x d_k}):
//     u = S_{t-1} k_t,  w = beta_t (v_t - alpha_t u),  S_t = alpha_t S_{t-1} + w k_t^T,
//     o_t = S_t q_t.
// (alpha S (I - beta k k^T) + beta v k^T expands to exactly this.)
//
// Design (one CTA = one (job, head, block of state rows)):
//  * Row i of S evolves only from v_{t,i}: the key-space operator acts from the
//    right, so the rows of a head split across lanes, warps and CTAs with no
//    exchange.  Lanes form 4 row groups of 8 column lanes; a lane holds a register
//    tile of (d_k/8) columns and 4 rows at d_k = 128 (two groups of 2 run half a
//    token apart; a warp owns 16 state rows, "slots"), 2 rows (one group; 8 rows
//    a warp) below.  The dot products S k and S q of a group reduce over the 8
//    column lanes with a reduce-scatter that leaves lanes 4s..4s+3 of a row group
//    with slot s's sums.  Two consumer warps share each SM sub-partition (at
//    d_k = 128, and at 64 with d_v = 64), hiding each other's per-token chain.
//  * The state is kept in a running scale: S = s * St.  With s_t = alpha_t s_{t-1}
//    the update becomes St += c k^T with c = (beta/s_t) v - beta (St_{t-1} k), so
//    each state element costs exactly three FMAs per token (update, S k, S q),
//    issued as packed fp32x2 FMAs.  The input staging computes s_t and beta/s_t
//    per token (sequential left-to-right product) and schedules renormalisation
//    (St *= s, s = 1) whenever the scale would fall below 2^-32, at every
//    checkpoint and after the last token, so dumps and results are plain states
//    and the arithmetic after a checkpoint does not depend on the path before it.
//  * k, q, v tiles of 32 tokens arrive by TMA in a 3-deep shared-memory ring
//    guarded by mbarriers; bf16 k and q are widened to fp32 once per CTA (then
//    read with conflict-free broadcast loads) and the per-token scalars are
//    published beside them.  With d_k < 128 a producer warp does this; with
//    d_k = 128 the warps do it themselves, a share each (a producer as a ninth
//    warp would cap every thread at 168 registers).  Every wait is bounded by a
//    wall-clock limit; on expiry the kernel records the device status and
//    returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

namespace gdn {

constexpr int kChunk = 32;     // tokens per pipeline stage
constexpr int kStages = 3;     // depth of the shared-memory ring
constexpr int kMaxJobs = 256;  // jobs per launch (host splits larger batches)
constexpr int kMaxCkpts = 1536;
// A lane holds row_slots(d_k) state rows x (d_k / kColLanes) columns.  At d_k = 128 the 4 rows split into two
// groups that run half a token apart (see the consumer loop): shared memory serves a warp's broadcast 16-byte
// load in 2 cycles (64 floats a cycle to an SM, against 128 FMAs) and every float of k or q a lane loads feeds
// one FMA per row it holds, so 4 rows keep the loads under the FMA time (measured: 2 rows and 16 warps, +24 %).
// Below d_k = 128 the latency of each warp's dependent shuffles and arithmetic, not the loads, bounds the loop,
// and 2 rows a lane give twice the warps for a head (measured at d_k = 32: -8 %).
constexpr int kColLanes = 8;
__host__ __device__ constexpr int row_slots(int dk) { return dk == 128 ? 4 : 2; }
constexpr int kMaxConsumerWarps = 8;
// state rows (slots) held by one consumer warp
__host__ __device__ constexpr int slots_per_warp(int dk) { return (32 / kColLanes) * row_slots(dk); }
// With d_k = 128 the warps stage their own inputs (see the kernel): 8 warps of 64-register tiles then may use
// 255 registers, where a producer warp as a ninth would cap them at 168 (measured: -20 % time).  The smaller
// sizes keep a producer warp (at most 8 + 1 warps of under 100 registers, under no cap), which spares them the
// staging work.
__host__ __device__ constexpr bool staging_in_warps(int dk) { return dk == 128; }
constexpr float kRenormFloor = 0x1p-32f;
// Bound of the wait for this CTA's own copies in flight before it exits (independent of the
// user's wait limit, so that even a tiny limit never lets a CTA leave with a copy pending).
constexpr uint64_t kDrainLimitNs = 1000000000ull;

enum : uint32_t { FLAG_RENORM = 1u, FLAG_DUMP = 2u, FLAG_INDEX_SHIFT = 8u };
enum : unsigned { STATUS_TIMEOUT = 1u };

// One scan over a contiguous token range, the same for all heads.
struct Job {
    int64_t tok_begin;      // absolute stream row of the job's first token
    void* o;                // output row of the job's first token ([rows, H, dv]); nullptr: no readout
    const float* s0;        // [H, dv, dk] initial state, nullptr = zeros
    const float* s0_twin;   // [H, dv, dk] initial state of the twin (twin kernels)
    float* s_final;         // [H, dv, dk] state after the last token
    float* s_final_twin;    // [H, dv, dk] twin state after the last token
    int32_t len;            // tokens
    int32_t ck_begin;       // first entry of the launch's checkpoint table
    int32_t ck_count;       // entries for this job
    int32_t t_row0;         // two-pass chunked path: first row of this job's block of T rows (H x len rows)
};
static_assert(sizeof(Job) == 64, "Job layout");

struct Ckpt {
    int32_t pos;   // 1-based token position within the job
    int32_t slot;  // destination slot in ckpt_states ([slot, H, dv, dk])
};

struct Params {
    CUtensorMap tm_q;   // [T, H, dk] box (dk, 1, kChunk)
    CUtensorMap tm_k;   // [T, H, dk] box (dk, 1, kChunk)
    CUtensorMap tm_v;   // [T, H, dv] box (rows_per_cta, 1, kChunk)
    const float* alpha; // [T, H]
    const float* beta;  // [T, H]
    float* ckpt_states; // [slots, H, dv, dk]
    unsigned int* status;
    unsigned long long wait_limit_ns;
    int32_t H;
    int32_t dv;
    int32_t nw;             // consumer warps per CTA
    int32_t rows_per_cta;   // real state rows per CTA
    int32_t ctas_per_head;  // dv / rows_per_cta
    int32_t n_jobs;
    int32_t stall_after;    // testing hook: stop issuing input copies after this many chunks (-1: off)
    int32_t o_vec16;        // every job's o is 16-byte aligned: the chunked kernel may write it in 16-byte pieces
    // two-pass chunked path only: the chunk schedule and T = (I + L)^-1 of every chunk, computed by
    // parallel passes before the state scan (workspace buffers)
    CUtensorMap tm_t;       // t_ops as [4 * t_rows, 64] bf16, box (64, 64), 128-byte swizzle
    int32_t* chunk_beg;     // [rows]: chunk c of (job, head) starts at token chunk_beg[t_row0 + head * len + c]
    int32_t* chunk_cnt;     // [n_jobs, H]: chunks of (job, head)
    void* t_ops;            // bf16 [4][t_rows][64]: T diag(beta gamma) hi, lo, T diag(beta) hi, lo; row
                            // t_row0 + head * len + t holds row t - begin of its chunk
    int32_t t_rows;         // rows of each of the four planes
    int32_t pad2_;
    Job jobs[kMaxJobs];
    Ckpt ckpts[kMaxCkpts];
};
static_assert(sizeof(Params) <= 32764, "kernel parameter block");

// ------------------------------------------------------------------------------------
// PTX helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
        "p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// the same probe, letting the hardware suspend the thread for up to `hint_ns` while the phase is pending
// (it resumes as soon as the phase completes), so that a long wait issues a few instructions, not a spin
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, "
        "p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete, for at most limit_ns.  Called by
// all 32 lanes of a warp; the warp agrees on the outcome.
// orders this thread's (and, after a barrier, the CTA's) generic-proxy shared-memory accesses before later
// async-proxy ones (TMA copies into the same bytes)
__device__ __forceinline__ void proxy_fence_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        // suspend in slices of at most 1/8 of the limit (and 20 us), so that the limit is still honoured
        const uint64_t slice = limit_ns / 8;
        const uint32_t hint = slice < 20000u ? (uint32_t)slice : 20000u;
        const uint64_t t0 = global_ns();
        while (!(ok = mbar_try_wait_suspend(bar, parity, hint))) {
            if (global_ns() - t0 > limit_ns) break;
        }
    }
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Sum over the NCL column lanes of a row group of a group's two per-row partial sums v[0], v[1].  The lanes
// with bit NCL / 2 set end up with slot 1's sum, the others with slot 0's: the first round keeps one sum and
// sends the other to the lane NCL / 2 away, then the lanes that share a slot add up.  With SWAPPED the caller
// already holds its own slot's sum in v[0] and no select is needed; both forms add the same operands in the
// same order.
template <int NCL, bool SWAPPED>
__device__ __forceinline__ float reduce_pair(float (&v)[2], int lane) {
    float keep = v[0], send = v[1];
    if constexpr (!SWAPPED) {
        const bool up = (lane & (NCL / 2)) != 0;
        send = up ? v[0] : v[1];
        keep = up ? v[1] : v[0];
    }
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, NCL / 2);
#pragma unroll
    for (int step = NCL / 4; step >= 1; step /= 2) v[0] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], step);
    return v[0];
}

// Whether a lane holds the two rows of each group in the order "its own slot first" (see the consumer setup).
// This removes the selects from every reduction; measured on GB300 it pays at d_k = 64 and 32 (6-7 % per
// token) but costs 4 % at d_k = 128, where the loop sits at the register limit.
__host__ __device__ constexpr bool swapped_rows(int dk) { return dk != 128; }

// Shared-memory layout of one pipeline stage.
//   kf, qf : [kChunk][dk] fp32, read by the consumers
//   v      : [kChunk][rows] input dtype
//   sc     : [kChunk] float4 {s_t, beta_t / s_t, beta_t, flags}
//   kr, qr : [kChunk][dk] bf16 TMA landing buffers (bf16 inputs only)
struct StageLayout {
    uint32_t kf_off, qf_off, v_off, sc_off, kr_off, qr_off, bytes, tx_bytes;
};
__host__ __device__ constexpr uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }
__host__ __device__ inline StageLayout stage_layout(int dk, int in_bytes, int rows, bool readout) {
    StageLayout L{};
    const uint32_t kf = (uint32_t)(kChunk * dk * 4);
    const uint32_t kr = (uint32_t)(kChunk * dk * in_bytes);
    const uint32_t vb = (uint32_t)(kChunk * rows * in_bytes);
    const bool raw = in_bytes != 4;
    uint32_t off = 0;
    L.kf_off = off;
    off += align128(kf);
    L.qf_off = off;
    if (readout) off += align128(kf);
    L.v_off = off;
    off += align128(vb);
    L.sc_off = off;
    off += align128(kChunk * 16u);
    L.kr_off = off;
    if (raw) off += align128(kr);
    L.qr_off = off;
    if (raw && readout) off += align128(kr);
    L.bytes = align128(off);
    L.tx_bytes = kr * (readout ? 2u : 1u) + vb;
    return L;
}
// after the stages: barriers raw[kStages] and full[kStages], the scan carry (8 B), done counters
// [kStages] and the issued count (4 B each), then up to 127 B of alignment of the base
__host__ __device__ inline uint32_t smem_bytes(int dk, int in_bytes, int rows, bool readout) {
    return stage_layout(dk, in_bytes, rows, readout).bytes * kStages + 256u + 128u;
}

// ------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------
template <int DK, bool IN_BF16, bool OUT_BF16, bool READOUT, bool TWIN>
__global__ void __launch_bounds__(32 * (kMaxConsumerWarps + (staging_in_warps(DK) ? 0 : 1)), 1)
    gdn_scan_kernel(const __grid_constant__ Params p) {
    constexpr int ES = IN_BF16 ? 2 : 4;
    constexpr int NCL = kColLanes;           // column lanes per row group
    constexpr int RT = row_slots(DK);        // row slots per lane
    constexpr int RG = 2;                    // slots of a row group (reduced together)
    constexpr int NG = RT / RG;              // row groups per lane: A (slots 0, 1) and, with 4 slots, B (2, 3)
    constexpr int LPG = NCL / RG;            // lanes that end up holding one slot's sums in a group reduction
    constexpr int CT = DK / NCL;             // columns per lane (16, 8, 4)
    constexpr int CT2 = CT / 2;
    constexpr int CH4 = CT / 4;              // fp32 float4 chunks per lane and vector
    constexpr int NRG = 32 / NCL;            // row groups per warp
    constexpr int HALF = TWIN ? RT / 2 : RT; // real rows per lane per state
    constexpr int WR = NRG * HALF;           // real rows per warp (16, or 8 with the twin)
    static_assert(CH4 >= 1 && CT % 4 == 0, "lane tile");
    static_assert(NRG * RT == slots_per_warp(DK) && (NG == 1 || NG == 2), "slots per warp");
    using OutT = typename std::conditional<OUT_BF16, __nv_bfloat16, float>::type;
    constexpr bool FOLD = staging_in_warps(DK);   // the warps stage their inputs themselves (no producer warp)

    // the 128-byte aligned base is formed by pointer arithmetic on the shared array (not through an integer),
    // so that the compiler keeps its address space and reads the stages with shared-memory loads
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);

    const int nw = p.nw;
    const int RB = p.rows_per_cta;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const StageLayout L = stage_layout(DK, ES, RB, READOUT);
    uint64_t* rawb = reinterpret_cast<uint64_t*>(smem + L.bytes * kStages);   // [kStages] a chunk's copies landed
    uint64_t* full = rawb + kStages;   // [kStages] a chunk widened and its scalars written
    uint64_t* empty = full + kStages;  // [kStages] (with the producer warp) every warp done with a stage's chunk
    float* carry_s = reinterpret_cast<float*>(empty + kStages);   // running scale after the last scanned chunk
    int* carry_ck = reinterpret_cast<int*>(carry_s + 1);         // checkpoint cursor after it
    int* done_cnt = carry_ck + 1;                                // [kStages] warps done with a stage's chunk
    int* issued_sh = done_cnt + kStages;                         // chunks whose copies were issued

    const int per_job = p.H * p.ctas_per_head;
    const int job_idx = blockIdx.x / per_job;
    const int rem = blockIdx.x - job_idx * per_job;
    const int h = rem / p.ctas_per_head;
    const int rb = rem - h * p.ctas_per_head;
    const int64_t tok_begin = p.jobs[job_idx].tok_begin;
    const int len = p.jobs[job_idx].len;
    const int nchunks = (len + kChunk - 1) / kChunk;
    const uint64_t limit = p.wait_limit_ns;
    const int H = p.H;
    const int dv = p.dv;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&rawb[s], 1);
            mbar_init(&full[s], FOLD ? (uint32_t)nw : 1u);   // every warp, or the producer
            mbar_init(&empty[s], (uint32_t)nw);
            done_cnt[s] = 0;
        }
        *carry_s = 1.0f;
        *carry_ck = p.jobs[job_idx].ck_begin;
        *issued_sh = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if constexpr (!FOLD) {
        if (warp == nw) {
            // ============================== producer warp ==============================
            const size_t gate0 = (size_t)tok_begin * (size_t)H + (size_t)h;
            const int ck_end = p.jobs[job_idx].ck_begin + p.jobs[job_idx].ck_count;
            int ck_cur = p.jobs[job_idx].ck_begin;
            float s_carry = 1.0f;
            int issued = 0;
            bool ok = true;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages;
                if (p.stall_after >= 0 && c >= p.stall_after) break;   // testing hook (see Params)
                if (c >= kStages && !warp_wait(&empty[st], (uint32_t)(((c / kStages) + 1) & 1), limit)) {
                    ok = false;
                    break;
                }
                unsigned char* stage = smem + (size_t)st * L.bytes;
                uint64_t* landing = IN_BF16 ? &rawb[st] : &full[st];
                if (lane == 0) {
                    // bf16: the landing barrier completes on the copies alone (one arrival
                    // here); fp32: the copies land on `full`, which the producer arrives
                    // on after publishing the scalars
                    if constexpr (IN_BF16)
                        mbar_arrive_expect_tx(landing, L.tx_bytes);
                    else
                        mbar_expect_tx(landing, L.tx_bytes);
                    const int t0 = (int)(tok_begin + (int64_t)c * kChunk);
                    tma_load_3d(stage + (IN_BF16 ? L.kr_off : L.kf_off), &p.tm_k, 0, h, t0, landing);
                    if (READOUT) tma_load_3d(stage + (IN_BF16 ? L.qr_off : L.qf_off), &p.tm_q, 0, h, t0, landing);
                    tma_load_3d(stage + L.v_off, &p.tm_v, rb * RB, h, t0, landing);
                }
                issued = c + 1;
                const int base = c * kChunk;
                const int tau = base + lane;
                float a = 1.0f, b = 0.0f;
                if (tau < len) {
                    a = __ldg(p.alpha + gate0 + (size_t)tau * (size_t)H);
                    b = __ldg(p.beta + gate0 + (size_t)tau * (size_t)H);
                }
                float a_look = 1.0f;
                if (base + kChunk < len) a_look = __ldg(p.alpha + gate0 + (size_t)(base + kChunk) * (size_t)H);
                uint32_t fl = 0;
                while (ck_cur < ck_end && p.ckpts[ck_cur].pos <= base + kChunk) {
                    if (p.ckpts[ck_cur].pos - 1 == tau)
                        fl = FLAG_DUMP | FLAG_RENORM | ((uint32_t)ck_cur << FLAG_INDEX_SHIFT);
                    ++ck_cur;
                }
                if (tau == len - 1) fl |= FLAG_RENORM;
                // running scale, left to right (chunk-boundary independent)
                float s = s_carry, my_s = 1.0f;
                uint32_t my_fl = fl;
    #pragma unroll 4
                for (int j = 0; j < kChunk; ++j) {
                    const float aj = __shfl_sync(0xffffffffu, a, j);
                    const float an_sh = __shfl_sync(0xffffffffu, a, (j + 1) & 31);
                    const uint32_t fj = __shfl_sync(0xffffffffu, fl, j);
                    const float an = (j + 1 < kChunk) ? an_sh : a_look;
                    s = s * aj;
                    const bool valid = base + j < len;
                    const bool ren =
                        valid && ((fj & FLAG_RENORM) != 0u || (base + j + 1 < len && s * an < kRenormFloor));
                    if (lane == j) {
                        my_s = s;
                        my_fl = fj | (ren ? FLAG_RENORM : 0u);
                    }
                    if (ren) s = 1.0f;
                }
                s_carry = s;
                const float b1 = __fdiv_rn(b, my_s);
                reinterpret_cast<float4*>(stage + L.sc_off)[lane] = make_float4(my_s, b1, b, __uint_as_float(my_fl));
                if constexpr (IN_BF16) {
                    // widen k (and q) to fp32 once for all consumer warps
                    if (!warp_wait(&rawb[st], (uint32_t)((c / kStages) & 1), limit)) {
                        ok = false;
                        break;   // this chunk's copy stays accounted for by the drain below
                    }
                    constexpr int NV4 = kChunk * DK / 4;   // groups of 4 elements
    #pragma unroll 4
                    for (int g = lane; g < NV4; g += 32) {
                        const uint2 w = reinterpret_cast<const uint2*>(stage + L.kr_off)[g];
                        const float2 lo = bf16x2_to_float2(w.x), hi = bf16x2_to_float2(w.y);
                        reinterpret_cast<float4*>(stage + L.kf_off)[g] = make_float4(lo.x, lo.y, hi.x, hi.y);
                        if (READOUT) {
                            const uint2 u = reinterpret_cast<const uint2*>(stage + L.qr_off)[g];
                            const float2 ql = bf16x2_to_float2(u.x), qh = bf16x2_to_float2(u.y);
                            reinterpret_cast<float4*>(stage + L.qf_off)[g] = make_float4(ql.x, ql.y, qh.x, qh.y);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[st]);
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
                warp_wait(IN_BF16 ? &rawb[c % kStages] : &full[c % kStages], (uint32_t)((c / kStages) & 1),
                          limit > kDrainLimitNs ? limit : kDrainLimitNs);
            if (!ok && lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
            return;
        }
    }

    // ================================ consumer warps ===============================
    // With 4 slots the lane's rows form two row groups, A (slots 0, 1) and B (2, 3), run half a token apart:
    // group B's reduction, c and readout of one token are issued between group A's FMAs of the next, and
    // group A's between group B's, so that neither group waits for its own shuffles.  With the twin, A is
    // the scan and B the twin.  With 2 slots there is only group A (with the twin: slot 0 the scan's row,
    // slot 1 the twin's).
    const int cl = lane & (NCL - 1);
    const int rg = lane / NCL;
    const int row0 = warp * WR + rg * HALF;                              // CTA row of this group's slot 0
    const int gslot = cl / LPG;                                          // slot (within a group) of this lane's sums
    // With swapped_rows(DK) the lanes whose sums end up in slot 1 of a group hold the group's two rows in
    // swapped registers, so that every lane's first reduction round keeps register 0 and sends register 1:
    // register i of group g then holds slot g * RG + (i ^ gslot) (else slot i).
    static_assert(LPG == NCL / 2 && (!TWIN || NG == 1 || HALF == RG),
                  "two slots per group, reduced over the column lanes; the twin form's groups are its two states");
    constexpr bool SWAP = swapped_rows(DK);
    const int rswap = SWAP ? gslot : 0;
    auto slot_of = [&](int i) {
        if constexpr (SWAP) return (i / RG) * RG + ((i % RG) ^ rswap);
        else return i;
    };
    auto reduce_group = [&](float (&v)[RG]) { return reduce_pair<NCL, SWAP>(v, lane); };
    // CTA-relative real rows of those slots (one group with the twin: slot 0 the scan's row, slot 1 the twin's)
    const int rowA = row0 + ((TWIN && NG == 1) ? 0 : gslot);
    const int rowB = row0 + (TWIN ? gslot : RG + gslot);
    const int grow_base = rb * RB + row0;                                // head row of slot 0
    const size_t head_state = (size_t)h * (size_t)dv * DK;

    // state tile: S[i][2*j4 + e] holds columns 4*(cl + 8*j4) + 2*e .. +1 of slot slot_of(i)
    float2 S[RT][CT2];
#pragma unroll
    for (int i = 0; i < RT; ++i) {
        // with the twin, group g (two groups) or slot g (one group) is state g
        const int state = TWIN ? (NG == 2 ? i / RG : slot_of(i)) : 0;
        const int grow = grow_base + (TWIN ? slot_of(i) % HALF : slot_of(i));
        const float* src = state == 0 ? p.jobs[job_idx].s0 : p.jobs[job_idx].s0_twin;
#pragma unroll
        for (int j4 = 0; j4 < CH4; ++j4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (src) x = __ldg(reinterpret_cast<const float4*>(src + head_state + (size_t)grow * DK) + cl + NCL * j4);
            S[i][2 * j4 + 0] = make_float2(x.x, x.y);
            S[i][2 * j4 + 1] = make_float2(x.z, x.w);
        }
    }

    // this lane's 4-column piece j4 of a staged fp32 vector (k or q of one token)
    auto piece = [&](const unsigned char* tok, int j4, float2& lo, float2& hi) {
        const float4 w = reinterpret_cast<const float4*>(tok)[cl + NCL * j4];
        lo = make_float2(w.x, w.y);
        hi = make_float2(w.z, w.w);
    };
    auto load_v = [&](const unsigned char* stage, int tau, int row) -> float {
        const unsigned char* pv = stage + L.v_off + ((size_t)tau * RB + row) * ES;
        if constexpr (IN_BF16)
            return __uint_as_float(((uint32_t) * reinterpret_cast<const unsigned short*>(pv)) << 16);
        else
            return *reinterpret_cast<const float*>(pv);
    };
    // per-slot partial sums of St x over this lane's columns for the slots g*RG .. g*RG+RG-1
    auto dot_group = [&](int g, const unsigned char* x, float (&out)[RG]) {
        float2 acc[RG];
#pragma unroll
        for (int i = 0; i < RG; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j4 = 0; j4 < CH4; ++j4) {
            float2 x0, x1;
            piece(x, j4, x0, x1);
#pragma unroll
            for (int i = 0; i < RG; ++i) acc[i] = __ffma2_rn(S[g * RG + i][2 * j4], x0, acc[i]);
#pragma unroll
            for (int i = 0; i < RG; ++i) acc[i] = __ffma2_rn(S[g * RG + i][2 * j4 + 1], x1, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < RG; ++i) out[i] = acc[i].x + acc[i].y;
    };
    // c = (beta / s) v - beta (St k) from the token's scalars {s, beta / s, beta, flags}, rounded the same way
    // at every call site (an explicit FMA, never a contraction the compiler chooses per site), so that the
    // restart after a checkpoint and a resumed job's first token agree bit for bit
    auto c_of = [](const float4& sc, float v, float pk) { return __fmaf_rn(sc.y, v, -__fmul_rn(sc.z, pk)); };
    // c of the group's slot whose sums this lane holds, to every column lane of its row group (as (c, c))
    auto broadcast_c = [&](float c_mine, float2 (&cc)[RG]) {
        const int grp = lane & ~(NCL - 1);
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const float c = __shfl_sync(0xffffffffu, c_mine, grp | ((i ^ rswap) * LPG));
            cc[i] = make_float2(c, c);
        }
    };
    // one group's pass over token t: St += c k_t^T, then the partial sums of St k_{t+1} and St q_t
    auto group_pass = [&](int g, const float2 (&cc)[RG], const float2 (&kc)[CT2], const float2 (&kn)[CT2],
                          const unsigned char* qtok, float (&pk)[RG], float (&pq)[RG]) {
        float2 ak[RG], aq[RG];
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            ak[i] = make_float2(0.f, 0.f);
            aq[i] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int j4 = 0; j4 < CH4; ++j4) {
            float2 q0 = make_float2(0.f, 0.f), q1 = make_float2(0.f, 0.f);
            if constexpr (READOUT) piece(qtok, j4, q0, q1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int jj = 2 * j4 + e;
                const float2 qe = e ? q1 : q0;
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    float2& x = S[g * RG + i][jj];
                    x = __ffma2_rn(cc[i], kc[jj], x);
                    ak[i] = __ffma2_rn(x, kn[jj], ak[i]);
                    if constexpr (READOUT) aq[i] = __ffma2_rn(x, qe, aq[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            pk[i] = ak[i].x + ak[i].y;
            pq[i] = aq[i].x + aq[i].y;
        }
    };
    auto load_k = [&](const unsigned char* tok, float2 (&k)[CT2]) {
#pragma unroll
        for (int j4 = 0; j4 < CH4; ++j4) piece(tok, j4, k[2 * j4], k[2 * j4 + 1]);
    };
    // write the slots of one state (0: the scan, 1: the twin) to dst_head [dv, dk]
    auto store_state = [&](float* dst_head, int which) {
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            if ((TWIN ? (NG == 2 ? i / RG : slot_of(i)) : 0) != which) continue;
            const int grow = grow_base + (TWIN ? slot_of(i) % HALF : slot_of(i));
#pragma unroll
            for (int j4 = 0; j4 < CH4; ++j4) {
                const float2 a0 = S[i][2 * j4 + 0], a1 = S[i][2 * j4 + 1];
                reinterpret_cast<float4*>(dst_head + (size_t)grow * DK)[cl + NCL * j4] =
                    make_float4(a0.x, a0.y, a1.x, a1.y);
            }
        }
    };

    void* const o_job = p.jobs[job_idx].o;
    OutT* const o_head = reinterpret_cast<OutT*>(o_job) + (size_t)h * (size_t)dv + (size_t)(rb * RB);
    const bool o_lane = READOUT && o_job != nullptr && (cl % LPG) == 0 && (NG == 2 || !TWIN || gslot == 0);
    auto store_o = [&](OutT* o_tok, int row, float val) {
        OutT* op = o_tok + row;
        if constexpr (OUT_BF16)
            *op = __float2bfloat16_rn(val);
        else
            *op = val;
    };

    // Restart from the state in registers before token t of stage `stg` at row tau (the job start, and after
    // every renormalisation): group A's c_t from a direct St k_t, group B's partial sums of St k_t.
    float2 ccA[RG], ccB[RG];
    float pBk[RG], pBq[RG];
    auto restart = [&](const unsigned char* ktok, const float4& sc, const unsigned char* stg, int tau) {
        float pk[RG];
        dot_group(0, ktok, pk);
        const float pkr = reduce_group(pk);
        broadcast_c(c_of(sc, load_v(stg, tau, rowA), pkr), ccA);
        if constexpr (NG == 2) dot_group(1, ktok, pBk);
    };

    // ---- (d_k = 128) input staging by the warps themselves (no producer warp: a ninth warp would cap every
    //      thread at 168 registers, which costs the token loop ~20 %).  Chunk k's k, q, v tiles are copied by TMA
    //      into stage k % 3; the warp that finishes chunk k - 3 last issues them.  At the start of chunk k - 1 every warp
    //      prepares chunk k: it waits for the copies, widens its share of bf16 k and q to fp32, and warp k % nw
    //      also writes the chunk's per-token scalars (the running scale s_t, beta_t / s_t, beta_t and the
    //      renormalisation / checkpoint flags, left to right from the carry of chunk k - 1); each warp then
    //      arrives on the chunk's `full` barrier, which every warp waits for before the last token of chunk
    //      k - 1 reads chunk k's first token.  No barrier of the whole CTA: a warp that is slower at one chunk
    //      holds the others back only through the stage ring. ----
    const size_t gate0 = (size_t)tok_begin * (size_t)H + (size_t)h;
    const int ck_end = p.jobs[job_idx].ck_begin + p.jobs[job_idx].ck_count;
    auto issue = [&](int k) {   // one thread
        if (p.stall_after >= 0 && k >= p.stall_after) return;   // testing hook (see Params)
        const int s = k % kStages;
        unsigned char* stage = smem + (size_t)s * L.bytes;
        proxy_fence_shared();   // the warps' reads of this stage (chunk k - 3) come before the copies' writes
        mbar_arrive_expect_tx(&rawb[s], L.tx_bytes);
        const int t0 = (int)(tok_begin + (int64_t)k * kChunk);
        tma_load_3d(stage + (IN_BF16 ? L.kr_off : L.kf_off), &p.tm_k, 0, h, t0, &rawb[s]);
        if (READOUT) tma_load_3d(stage + (IN_BF16 ? L.qr_off : L.qf_off), &p.tm_q, 0, h, t0, &rawb[s]);
        tma_load_3d(stage + L.v_off, &p.tm_v, rb * RB, h, t0, &rawb[s]);
        atomicMax(issued_sh, k + 1);
    };
    // this warp's gates for the next chunk it scans (chunk k with k % nw == warp), loaded nw chunks ahead
    float ga = 1.f, gb = 0.f, gal = 1.f;
    auto load_gates = [&](int k) {
        const int base = k * kChunk, tau = base + lane;
        ga = 1.f;
        gb = 0.f;
        if (tau < len) {
            ga = __ldg(p.alpha + gate0 + (size_t)tau * (size_t)H);
            gb = __ldg(p.beta + gate0 + (size_t)tau * (size_t)H);
        }
        gal = 1.f;
        if (base + kChunk < len) gal = __ldg(p.alpha + gate0 + (size_t)(base + kChunk) * (size_t)H);
    };
    auto prepare = [&](int k) -> bool {
        const int s = k % kStages;
        unsigned char* stage = smem + (size_t)s * L.bytes;
        if (!warp_wait(&rawb[s], (uint32_t)((k / kStages) & 1), limit)) return false;
        if constexpr (IN_BF16) {
            constexpr int NV4 = kChunk * DK / 4;   // groups of 4 elements
#pragma unroll 2
            for (int g = warp * 32 + lane; g < NV4; g += 32 * nw) {
                const uint2 w = reinterpret_cast<const uint2*>(stage + L.kr_off)[g];
                const float2 lo = bf16x2_to_float2(w.x), hi = bf16x2_to_float2(w.y);
                reinterpret_cast<float4*>(stage + L.kf_off)[g] = make_float4(lo.x, lo.y, hi.x, hi.y);
                if (READOUT) {
                    const uint2 u = reinterpret_cast<const uint2*>(stage + L.qr_off)[g];
                    const float2 ql = bf16x2_to_float2(u.x), qh = bf16x2_to_float2(u.y);
                    reinterpret_cast<float4*>(stage + L.qf_off)[g] = make_float4(ql.x, ql.y, qh.x, qh.y);
                }
            }
        }
        if (k % nw == warp) {
            // the per-token scalars, left to right from the carry (chunk-boundary independent); the carry was
            // written by the scan of chunk k - 1, which this warp has seen complete through that chunk's `full`
            const int base = k * kChunk;
            const int tau = base + lane;
            int ck_cur = *carry_ck;
            uint32_t fl = 0;
            while (ck_cur < ck_end && p.ckpts[ck_cur].pos <= base + kChunk) {
                if (p.ckpts[ck_cur].pos - 1 == tau) fl = FLAG_DUMP | FLAG_RENORM | ((uint32_t)ck_cur << FLAG_INDEX_SHIFT);
                ++ck_cur;
            }
            if (tau == len - 1) fl |= FLAG_RENORM;
            float sc_run = *carry_s, my_s = 1.0f;
            uint32_t my_fl = fl;
#pragma unroll 4
            for (int j = 0; j < kChunk; ++j) {
                const float aj = __shfl_sync(0xffffffffu, ga, j);
                const float an_sh = __shfl_sync(0xffffffffu, ga, (j + 1) & 31);
                const uint32_t fj = __shfl_sync(0xffffffffu, fl, j);
                const float an = (j + 1 < kChunk) ? an_sh : gal;
                sc_run = sc_run * aj;
                const bool valid = base + j < len;
                const bool ren =
                    valid && ((fj & FLAG_RENORM) != 0u || (base + j + 1 < len && sc_run * an < kRenormFloor));
                if (lane == j) {
                    my_s = sc_run;
                    my_fl = fj | (ren ? FLAG_RENORM : 0u);
                }
                if (ren) sc_run = 1.0f;
            }
            const float b1 = __fdiv_rn(gb, my_s);
            reinterpret_cast<float4*>(stage + L.sc_off)[lane] = make_float4(my_s, b1, gb, __uint_as_float(my_fl));
            if (lane == 0) {
                *carry_s = sc_run;
                *carry_ck = ck_cur;
            }
            if (k + nw < nchunks) load_gates(k + nw);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        return true;
    };
    // this warp is done with chunk c: the last of the warps hands its stage to chunk c + 3
    auto release = [&](int c) {
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const int s = c % kStages;
            if (atomicAdd(&done_cnt[s], 1) == nw - 1) {
                atomicExch(&done_cnt[s], 0);
                __threadfence_block();
                if (c + kStages < nchunks) issue(c + kStages);
            }
        }
    };

    bool ok = true;
    float4 sct = make_float4(1.f, 0.f, 0.f, 0.f);   // scalars of the current token
    float4 scp = sct;                               // scalars of the token before
#pragma unroll
    for (int i = 0; i < RG; ++i) {
        ccA[i] = ccB[i] = make_float2(0.f, 0.f);
        pBk[i] = pBq[i] = 0.f;
    }
    if (len > 0) {
        if constexpr (FOLD) {
            if (threadIdx.x == 0)
                for (int k = 0; k < kStages && k < nchunks; ++k) issue(k);
            if (warp < nchunks) load_gates(warp);   // the first chunk each warp scans
            ok = prepare(0);
        }
        ok = ok && warp_wait(&full[0], 0u, limit);
        if (ok) {
            sct = reinterpret_cast<const float4*>(smem + L.sc_off)[0];
            restart(smem + L.kf_off, sct, smem, 0);
        }
    }

    // Chunks of the stage ring outside, tokens inside: per token only pointer steps, no index division.  A chunk
    // runs as two segments, tokens 0 .. n-2 (the next token is in this stage) and token n-1 (the next token, if
    // any, is the first of the next stage, waited for in between), and a renormalising token leaves the token loop:
    // the wait, the renormalisation, the restart and the checkpoint dump stay out of the loop body, whose code the
    // compiler then schedules on its own (measured: the same loop with that code inside it ran 1.4x longer).
    OutT* o_t = o_head;   // output row of the current token
    const size_t o_step = (size_t)H * (size_t)dv;
    int tg = 0;
    for (int c = 0; ok && c < nchunks; ++c) {
        const int st = c % kStages;
        const int stn = (c + 1) % kStages;
        const unsigned char* stage = smem + (size_t)st * L.bytes;
        const unsigned char* stage_n = smem + (size_t)stn * L.bytes;
        const int n = min(kChunk, len - c * kChunk);
        const bool more = c + 1 < nchunks;
        if constexpr (FOLD) {
            if (more && !prepare(c + 1)) {
                ok = false;
                break;
            }
        }
        int tau = 0;
        for (int seg = 0; seg < 2; ++seg) {
            const int tau_end = seg == 0 ? n - 1 : n;
            if (seg == 1 && more) {
                if (!warp_wait(&full[stn], (uint32_t)(((c + 1) / kStages) & 1), limit)) {
                    ok = false;
                    break;
                }
            }
            const unsigned char* nst = seg == 0 ? stage : stage_n;   // stage of the next token
            const bool has_next = seg == 0 || more;                 // the next token exists
            while (tau < tau_end) {
                int tau_r = -1;   // a token after which the state renormalises
                for (; tau < tau_end; ++tau, ++tg, o_t += o_step) {
                    const int taun = seg == 0 ? tau + 1 : 0;
                    // k of the next token (the last token dots with its own k; those sums are never used).  Past
                    // the last token the next-token reads below stay inside the stage ring and are not used either.
                    const unsigned char* k_cur = stage + L.kf_off + (size_t)tau * DK * 4;
                    const unsigned char* k_nxt = has_next ? nst + L.kf_off + (size_t)taun * DK * 4 : k_cur;
                    const unsigned char* q_cur = stage + L.qf_off + (size_t)tau * DK * 4;
                    const float4 scn = reinterpret_cast<const float4*>(nst + L.sc_off)[taun];
                    float2 kc[CT2], kn[CT2];
                    load_k(k_cur, kc);
                    load_k(k_nxt, kn);

                    // group B: c_t from St_{t-1} k_t, and its readout of token t-1
                    if constexpr (NG == 2) {
                        const float pkr = reduce_group(pBk);
                        broadcast_c(c_of(sct, load_v(stage, tau, rowB), pkr), ccB);
                        if constexpr (READOUT) {
                            const float pqr = reduce_group(pBq);
                            if (o_lane && !TWIN && tg > 0) store_o(o_t - o_step, rowB, scp.x * pqr);
                        }
                    }
                    // group A: token t
                    float pAk[RG], pAq[RG];
                    group_pass(0, ccA, kc, kn, q_cur, pAk, pAq);
                    // group A: c_{t+1} and its readout of token t (issued between group B's FMAs)
                    {
                        const float pkr = reduce_group(pAk);
                        broadcast_c(c_of(scn, load_v(nst, taun, rowA), pkr), ccA);
                        if constexpr (READOUT) {
                            const float pqr = reduce_group(pAq);
                            if (o_lane) store_o(o_t, rowA, sct.x * pqr);
                        }
                    }
                    // group B: token t
                    if constexpr (NG == 2) group_pass(1, ccB, kc, kn, q_cur, pBk, pBq);

                    const bool renorm = (__float_as_uint(sct.w) & FLAG_RENORM) != 0u;
                    scp = sct;
                    sct = scn;
                    if (renorm) {
                        tau_r = tau;
                        ++tau;
                        ++tg;
                        o_t += o_step;
                        break;
                    }
                }
                if (tau_r >= 0) {
                    // after token tau_r (its scalars now in scp, the next token's in sct): St <- s St, then the
                    // next token's c and partial sums from the renormalised state, and a checkpoint if one is due
                    const uint32_t fl = __float_as_uint(scp.w);
                    const float2 ss = make_float2(scp.x, scp.x);
#pragma unroll
                    for (int i = 0; i < RT; ++i)
#pragma unroll
                        for (int jj = 0; jj < CT2; ++jj) S[i][jj] = __fmul2_rn(S[i][jj], ss);
                    const int taun_r = seg == 0 ? tau_r + 1 : 0;
                    if (has_next) restart(nst + L.kf_off + (size_t)taun_r * DK * 4, sct, nst, taun_r);
                    if (fl & FLAG_DUMP) {
                        const int slot = p.ckpts[fl >> FLAG_INDEX_SHIFT].slot;
                        store_state(p.ckpt_states + (size_t)slot * (size_t)H * (size_t)dv * DK + head_state, 0);
                    }
                }
            }
        }
        if (!ok) break;
        if constexpr (FOLD) {
            release(c);
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
    }
    // group B's readout of the last token
    if constexpr (READOUT && NG == 2) {
        if (ok && len > 0) {
            const float pqr = reduce_group(pBq);
            if (o_lane && !TWIN) store_o(o_head + (size_t)(len - 1) * (size_t)H * (size_t)dv, rowB, scp.x * pqr);
        }
    }

    // never leave with copies in flight into this CTA's shared memory (after a wait ran out, copies of chunks
    // not prepared may still be landing): every warp is out of its loops, then warp 0 waits for the last ones
    if constexpr (FOLD) {
        __syncthreads();   // (with the producer warp, that warp drains its own copies)
        if (warp == 0) {
        const int iss = *issued_sh;
        for (int k = iss > kStages ? iss - kStages : 0; k < iss; ++k)
            warp_wait(&rawb[k % kStages], (uint32_t)((k / kStages) & 1), limit > kDrainLimitNs ? limit : kDrainLimitNs);
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
        return;
    }
    // final state(s): the last token always renormalises, so St is the state
    float* fin = p.jobs[job_idx].s_final;
    if (fin) store_state(fin + head_state, 0);
    if constexpr (TWIN) {
        float* fin2 = p.jobs[job_idx].s_final_twin;
        if (fin2) store_state(fin2 + head_state, 1);
    }
}

// The dynamic shared-memory opt-in of a kernel, made once per device (again only for a larger size): the
// attribute call costs host time, and a short kernel's successor must not wait for it on the device.
constexpr int kMaxOptinDevices = 64;
inline cudaError_t smem_optin(const void* kern, int bytes, std::atomic<int>* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool track = dev >= 0 && dev < kMaxOptinDevices;
    if (track && done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && track) {
        int cur = done[dev].load();
        while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes)) {
        }
    }
    return e;
}

// Launch one kernel instance; instantiated per d_k in inst_dk*.cu.
template <int DK, bool IN_BF16, bool OUT_BF16, bool READOUT, bool TWIN>
cudaError_t launch_scan(const Params& p, int grid, size_t smem, cudaStream_t stream) {
    auto kern = gdn_scan_kernel<DK, IN_BF16, OUT_BF16, READOUT, TWIN>;
    static std::atomic<int> optin[kMaxOptinDevices];
    cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), (int)smem, optin);
    if (e != cudaSuccess) return e;
    kern<<<grid, 32 * (p.nw + (staging_in_warps(DK) ? 0 : 1)), smem, stream>>>(p);
    return cudaGetLastError();
}

using LaunchFn = cudaError_t (*)(const Params&, int, size_t, cudaStream_t);

// index: ((in_bf16 * 2 + out_bf16) * 2 + readout) * 2 + twin
template <int DK>
LaunchFn launch_table(int idx);
template <>
LaunchFn launch_table<32>(int idx);
template <>
LaunchFn launch_table<64>(int idx);
template <>
LaunchFn launch_table<128>(int idx);

}  // namespace gdn
