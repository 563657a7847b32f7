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
// U''_s = c_s u_s, c_s = 1/(sigma_0 gamma_s):
//   U^T    = U~^T + St (-sigma_0 W)^T                (S_0 = sigma_0 St)
//   St_n   = St_0 + U''^T K                           (the accumulator is never rescaled per chunk)
//   o_t    = sigma_0 gamma_t (St Q^T + U''^T P^T)[:, t],  P[t][s] = q_t.k_s for s <= t
// What keeps every factor finite for any alpha in (0, 1]:
//   * a chunk ends before the token at which gamma would fall below 2^-32, so 1/gamma <= 2^32;
//   * a chunk of one token with alpha < 2^-32 scales St to alpha_1 S_0 / 1 (sigma -> 1) before its
//     update, takes c = 1, and reads out o_1 = sigma_0 alpha_1 St q_1 + (q_1.k_1) u_1 directly;
//   * sigma is folded into St (St <- sigma St, sigma <- 1) when it falls below 2^-40, at every
//     checkpoint and at the end, so checkpoints are plain states and a resume from one repeats
//     the full run's arithmetic bit for bit.
// Chunk ends depend only on the checkpoint list and on the gates after the previous chunk end,
// which the full run and a resume see alike.
//
// Operands that are not exact in bf16 (T diag(.), W, U'', P, St) are split x = hi + lo into two
// bf16 halves and multiplied as hi*hi + hi*lo + lo*hi (or hi*x + lo*x against the exact q, k, v),
// accumulated in fp32 in TMEM.
//
// Three warp roles run a software pipeline over the chunks of one (job, head):
//   chain (warps 0-3) - the state-dependent conversions of chunk j: St into the bf16 A operand,
//       U'' from U, readout, checkpoints;
//   prep (warps 4-11) - the state-independent work of chunk j+1: G, L, T, the
//       T diag(.) operands, -sigma_0 W, P, and (one warp) the gates and the chunk schedule one
//       chunk further ahead;
//   issue (warp 12, one lane; without a readout warps 12 and 13, one lane each) - every tcgen05.mma: the
//       chain's U^T += St (-sigma_0 W)^T, St Q^T, St += U''^T K, U''^T P^T and the prep's [K; Q] K^T (L and
//       P), W^T, U~^T, each as soon as the mbarriers of its operands have fired, so that no converting warp
//       waits on a full MMA queue.
// The prep warps stage the K/Q tiles of chunk j+1 as soon as they have read P_j out of the G
// columns, so [K; Q] K^T of the next chunk runs beside W^T, U~^T of this one and L is waiting in
// TMEM when the next iteration starts.
// They hand over through mbarriers; each group agrees on every wait by a barrier reduction, so a
// wait that runs out ends every loop without leaving a named barrier half-entered.
//
// TMEM (512 columns x 128 lanes of 32 bit):
//   [0,128) St   [128,192) U^T   [192,256) W^T   [256,320) O^T   [320,384) [K; Q] K^T
//   [384,448) St hi (bf16 pairs)   [448,512) St lo
// W^T directly follows U^T so that U^T += St (-sigma_0 W)^T takes [W_hi | W_lo] as one N = 128 operand:
// the W columns, zeroed once W is read out, then collect the S_hi W_lo^T half, added when U is read.
#pragma once

#include <climits>

#include "gdn_kernel.cuh"

namespace gdn {
namespace tc {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NCHAIN = 128;                  // warps 0-3
constexpr int NPREP = 256;                   // warps 4-11
// + warp 12 (MMA issue), and warp 13 (a second MMA-issuing thread) without a readout
__host__ __device__ constexpr int nthreads(bool readout) { return NCHAIN + NPREP + (readout ? 32 : 64); }
constexpr int BAR_CHAIN = 1, BAR_PREP = 2;   // named barriers
constexpr int kRing = 4;                     // chunk schedule entries in flight

struct Pos {   // chunk schedule cursor
    int begin, len;
};

// Per-chunk schedule and scalars, written by the gate warp, read by both groups.
struct Ring {
    int begin, n, single, fold, dump_slot, last, next_begin, next_len;
    float sigma0, sigma_after, prescale, qk0;
    int pad_[4];
    float rs[C];   // readout scale sigma_0 gamma_t (single: sigma_0 alpha_1)
    float c[C];    // U'' scale 1/(sigma_0 gamma_t) (single: 1); 0 past the chunk
};
static_assert(sizeof(Ring) == 576, "Ring layout");

// ---- shared memory (bytes); swizzled operand tiles are 1024-aligned ----
constexpr int OFF_KQ = 0;              // 2 x 32 KB: [K;Q] as two 64-column blocks of [128 rows][128 B]
constexpr int OFF_V = 65536;           // 16 KB: V as two 64-column blocks of [64 rows][128 B]
constexpr int OFF_T1H = 81920;         // [64 t][64 s] bf16 (T diag(beta gamma)) hi
constexpr int OFF_T1L = 90112;         //   lo
constexpr int OFF_T2H = 98304;         // (T diag(beta)) hi
constexpr int OFF_T2L = 106496;        //   lo
constexpr int OFF_PH = 114688;         // [64 t][64 s] P hi
constexpr int OFF_PL = 122880;         //   lo
constexpr int OFF_WH = 131072;         // [128 dk][64 t] -sigma_0 W^T hi (MN-major B operand)
constexpr int OFF_WL = 147456;         //   lo
constexpr int OFF_UH = 163840;         // [128 dv][64 t] U''^T hi (K-major A operand)
constexpr int OFF_UL = 180224;         //   lo
constexpr int OFF_LF = 196608;         // fp32 [64][68]: L, then T in place
constexpr int OFF_LD = 214016;         // fp32 4 x [16][17] diagonal blocks of L; later [32][kLdY] scratch
constexpr int OFF_PSC = 218624;        // fp32 prep scalars [2][4][64]: gamma, 1/gamma, beta gamma, beta
constexpr int OFF_RING = 220672;       // Ring[kRing]
constexpr int OFF_BAR = OFF_RING + kRing * 576;
constexpr int kBarBytes = 256;
constexpr int OFF_OST = OFF_BAR + kBarBytes;   // 8 KB: readout staging, a [tokens][32 rows] tile per reading warp
constexpr int OFF_U0 = OFF_LF + C * C * 4;     // two-pass: fp32 [2][128] u_1 of single-token chunks (after the T tile)
static_assert(OFF_U0 + 2 * 128 * 4 <= OFF_LD, "u_1 buffer inside the L area");
constexpr int kSmemBytes = OFF_OST + 4 * 2048 + 1024;
static_assert(kSmemBytes <= 232448, "227 KB of shared memory per block");
constexpr int kLdF = 68;
// Row strides of the merge scratch, chosen so that the mma.sync fragments (rows g8 and 2 t4, 2 t4 + 1) and the
// float pairs written back fall in distinct banks: level B [32][36] in the L area, level A [16][20] in a warp's
// two spent diagonal blocks of L.
constexpr int kLdY = 36, kLdS = 20;
static_assert(OFF_LD + 32 * kLdY * 4 <= OFF_PSC, "level-B scratch inside the L area");
static_assert(16 * kLdS <= 2 * 16 * 17, "level-A scratch inside two diagonal blocks");
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(OFF_PSC + 2 * 4 * C * 4 == OFF_RING, "scalar area");

constexpr uint32_t T_S = 0, T_U = 128, T_W = 192, T_O = 256, T_G = 320, T_SH = 384, T_SL = 448;
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
// two 32-column pieces for one wait: the second load's latency hides behind the first's (one asm, so no
// register is read before the wait)
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32], float (&vb)[32]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
          "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]),
          "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]),
          "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[32 + i]);
    }
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
// ldmatrix (four / two 8x8 b16 matrices) and mma.sync m16n8k16 (row.col, bf16 -> fp32)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x = hi + lo, both tf32 (10 explicit mantissa bits each)
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(x - __uint_as_float(hi)));
}
// d (16 x 8, m16n8 accumulator layout) += A (16 x 8, row-major at a, row stride lda) B (8 x 8, row-major
// at b, row stride ldb) as hi*hi, and c += hi*lo + lo*hi (mma.sync m16n8k8 tf32, fp32 accumulate); two
// accumulators keep the dependent MMA chains short; the caller adds c to d at the end
__device__ __forceinline__ void mma_tf32x3(float (&d)[4], float (&c)[4], const float* a, int lda, const float* b,
                                           int ldb, int g8, int t4) {
    uint32_t ah[4], al[4], bh[2], bl[2];
    tf32_split(a[g8 * lda + t4], ah[0], al[0]);
    tf32_split(a[(g8 + 8) * lda + t4], ah[1], al[1]);
    tf32_split(a[g8 * lda + t4 + 4], ah[2], al[2]);
    tf32_split(a[(g8 + 8) * lda + t4 + 4], ah[3], al[3]);
    tf32_split(b[t4 * ldb + g8], bh[0], bl[0]);
    tf32_split(b[(t4 + 4) * ldb + g8], bh[1], bl[1]);
#define GDN_MMA_TF32(D, A, B)                                                                                   \
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, " \
                 "{%0,%1,%2,%3};"                                                                               \
                 : "+f"(D[0]), "+f"(D[1]), "+f"(D[2]), "+f"(D[3])                                              \
                 : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(B[0]), "r"(B[1]))
    GDN_MMA_TF32(c, al, bh);
    GDN_MMA_TF32(d, ah, bh);
    GDN_MMA_TF32(c, ah, bl);
#undef GDN_MMA_TF32
}
// gamma over a window of up to 64 tokens held by one warp (token lane in a0, token 32 + lane in a1; 1 past
// the window): inclusive products g0, g1 in token order, the same rounding wherever a chunk's gates are formed
__device__ __forceinline__ void gate_prefix(float a0, float a1, float& g0, float& g1, int lane) {
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
}
// first token of the window whose gamma falls below 2^-32 (C if none); the chunk ends before it, or
// after it when it is the first token
__device__ __forceinline__ int gamma_first(float g0, float g1) {
    const unsigned m0 = __ballot_sync(0xffffffffu, g0 < kGammaFloor);
    const unsigned m1 = __ballot_sync(0xffffffffu, g1 < kGammaFloor);
    return m0 ? __ffs(m0) - 1 : (m1 ? 31 + __ffs(m1) : C);
}
// d (16 x 8) += A (16 x 16, fp32 row-major at a, row stride lda) B (16 x 8, fp32 row-major at b, row stride
// ldb) as hi*hi, and c += hi*lo + lo*hi, every operand split x = hi + lo into bf16 (mma.sync m16n8k16, fp32
// accumulate): half the instructions of the tf32 form for the same K; the caller adds c to d at the end
__device__ __forceinline__ void mma_bf16x3(float (&d)[4], float (&c)[4], const float* a, int lda, const float* b,
                                           int ldb, int g8, int t4) {
    // A pairs as 8-byte loads (a and lda even at every call): with lda = 68 the 32 lanes' pairs fill each bank
    // exactly twice, the minimum for 256 bytes
    uint32_t ah[4], al[4], bh[2], bl[2];
    const float2 a0 = *reinterpret_cast<const float2*>(a + g8 * lda + 2 * t4);
    const float2 a1 = *reinterpret_cast<const float2*>(a + (g8 + 8) * lda + 2 * t4);
    const float2 a2 = *reinterpret_cast<const float2*>(a + g8 * lda + 2 * t4 + 8);
    const float2 a3 = *reinterpret_cast<const float2*>(a + (g8 + 8) * lda + 2 * t4 + 8);
    split_pair(a0.x, a0.y, ah[0], al[0]);
    split_pair(a1.x, a1.y, ah[1], al[1]);
    split_pair(a2.x, a2.y, ah[2], al[2]);
    split_pair(a3.x, a3.y, ah[3], al[3]);
    split_pair(b[(2 * t4) * ldb + g8], b[(2 * t4 + 1) * ldb + g8], bh[0], bl[0]);
    split_pair(b[(2 * t4 + 8) * ldb + g8], b[(2 * t4 + 9) * ldb + g8], bh[1], bl[1]);
    mma_bf16_16816(c, al, bh[0], bh[1]);
    mma_bf16_16816(d, ah, bh[0], bh[1]);
    mma_bf16_16816(c, ah, bl[0], bl[1]);
}
__device__ __forceinline__ void group_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// barrier over a warp group that also returns whether every thread passed `v`
__device__ __forceinline__ bool group_all(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
// bounded wait for the phase of `parity`; gives up when another role has given up
__device__ __forceinline__ bool wait_phase(uint64_t* b, uint32_t parity, volatile int* abort_flag, uint64_t limit) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(b, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit) {
            *abort_flag = 1;
            return false;
        }
    }
}
// wait by one poller while the rest of the group sleeps in the barrier; afterwards every thread
// observes the completed phase itself (one probe that succeeds at once), for its own acquire
__device__ __forceinline__ bool group_wait(uint64_t* b, uint32_t parity, bool poller, int id, int n,
                                           volatile int* abort_flag, uint64_t limit) {
    bool ok = true;
    if (poller) ok = wait_phase(b, parity, abort_flag, limit);
    ok = group_all(id, n, ok);
    if (ok) (void)mbar_try_wait(b, parity);
    return ok;
}
// non-blocking probe (try_wait may suspend the thread for a while; a poller over several barriers
// must not wait on one of them)
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void drain_phase(uint64_t* b, uint32_t parity, uint64_t limit) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(b, parity))
        if (global_ns() - t0 > limit) break;
}

// ------------------------------------------------------------------------------------
// the kernel: one CTA = one (job, head)
// ------------------------------------------------------------------------------------
template <bool OUT_BF16, bool READOUT, bool PRE_T>
__global__ void __launch_bounds__(nthreads(READOUT), 1) gdn_chunk_tc_kernel(const __grid_constant__ Params p) {
    using OutT = typename std::conditional<OUT_BF16, __nv_bfloat16, float>::type;
    extern __shared__ unsigned char smem_raw[];
    // aligned by pointer arithmetic on the shared array (not through an integer), so that the compiler keeps
    // its address space and plain C++ accesses below compile to shared-memory loads and stores
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // TMA and MMA completions (one arrival each)
    uint64_t* bar_kq = bars + 0;       // [2] K/Q tiles landed
    uint64_t* bar_v = bars + 2;        // V tile landed
    uint64_t* bar_g = bars + 3;        // [K; Q] K^T done (its K rows give L, its Q rows P)
    uint64_t* bar_wu = bars + 4;       // W^T, U~^T done
    uint64_t* bar_uo = bars + 5;       // U^T done
    uint64_t* bar_st = bars + 6;       // state update and every MMA issued before it done
    uint64_t* bar_o = bars + 7;        // St Q^T + U''^T P^T done
    // operands ready for the issuing warp, or results read
    uint64_t* bar_gin = bars + 8;      // prep: K/Q tiles padded, G columns free             (1 arrival)
    uint64_t* bar_wuin = bars + 9;     // prep: T diag(.) operands in shared memory           (1)
    uint64_t* bar_wready = bars + 10;  // prep: -sigma_0 W in shared memory                   (NPREP)
    uint64_t* bar_pready = bars + 11;  // prep: P in shared memory                            (NPREP)
    uint64_t* bar_split = bars + 12;   // chain: St split into TMEM (and prescaled)           (NCHAIN)
    uint64_t* bar_ofree = bars + 13;   // chain: O^T read out                                 (NCHAIN)
    uint64_t* bar_ufree = bars + 14;   // chain: U'' in shared memory, U^T columns free       (NCHAIN)
    uint64_t* bar_ring = bars + 15;    // [kRing] schedule entry written by the gate warp     (32)
    uint64_t* bar_t = bars + 19;       // T tile of the chunk landed (T computed by the first passes)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 160);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 164);
    int* cnt = reinterpret_cast<int*>(smem + OFF_BAR + 168);   // K/Q, V chunks issued; commits g, wu, uo, st, o; T
    Ring* ring = reinterpret_cast<Ring*>(smem + OFF_RING);
    float* psc = reinterpret_cast<float*>(smem + OFF_PSC);
    float* Lf = reinterpret_cast<float*>(smem + OFF_LF);
    float* Ld = reinterpret_cast<float*>(smem + OFF_LD);
    float* Yb = Ld;   // the diagonal blocks are consumed before the merge scratch is written

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3;                 // TMEM lane quarter of this warp
    const int row = 32 * lq + lane;          // TMEM lane = accumulator row
    const int job_idx = blockIdx.x / p.H;
    const int h = blockIdx.x - job_idx * p.H;
    const int H = p.H;
    const Job& job = p.jobs[job_idx];
    const int64_t tok_begin = job.tok_begin;
    const int len = job.len;
    const int ck_end = job.ck_begin + job.ck_count;
    void* const o_job = job.o;
    const bool rd = READOUT && o_job != nullptr;
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = limit > kDrainLimitNs ? limit : kDrainLimitNs;
    const size_t head_state = (size_t)h * D * D;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int i = 0; i < 10; ++i) mbar_init(&bars[i], 1);
        mbar_init(bar_wready, NPREP);
        mbar_init(bar_pready, NPREP);
        mbar_init(bar_split, NCHAIN);
        mbar_init(bar_ofree, PRE_T ? NPREP : NCHAIN);   // the group that reads O out
        mbar_init(bar_ufree, NCHAIN);
        for (int i = 0; i < kRing; ++i) mbar_init(&bar_ring[i], 32);
        mbar_init(bar_t, 1);
        *abort_flag = 0;
        for (int i = 0; i < 8; ++i) cnt[i] = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t trow = tbase + ((uint32_t)(32 * lq) << 16);   // this warp's lane quarter
    // W follows U in TMEM, so U^T += St [W_hi | W_lo]^T runs as one N = 128 product per k step whose second
    // half (zeroed once W is read) is added when U is read
    constexpr uint32_t TW = T_W, TO = T_O, TG = T_G;

    auto allowed = [&](int c) { return p.stall_after < 0 || c < p.stall_after; };   // testing hook
    auto issue_kq = [&](int c, int pos) {
        const int buf = c & 1;
        proxy_fence();
        mbar_arrive_expect_tx(&bar_kq[buf], 4u * 8192u);
        unsigned char* dst = smem + OFF_KQ + buf * 32768;
        const int t0 = (int)(tok_begin + pos);
        tma_load_3d(dst + 0, &p.tm_k, 0, h, t0, &bar_kq[buf]);
        tma_load_3d(dst + 8192, &p.tm_q, 0, h, t0, &bar_kq[buf]);
        tma_load_3d(dst + 16384, &p.tm_k, 64, h, t0, &bar_kq[buf]);
        tma_load_3d(dst + 16384 + 8192, &p.tm_q, 64, h, t0, &bar_kq[buf]);
        atomicMax(&cnt[0], c + 1);
    };
    // T diag(beta gamma), T diag(beta) (bf16 hi, lo) of chunk c (starting at token pos) from the rows the
    // first passes wrote, straight into the operand tiles (the copy's 128-byte swizzle is the MMA layout)
    auto issue_t = [&](int c, int pos) {
        proxy_fence();
        mbar_arrive_expect_tx(bar_t, 4u * 8192u);
#pragma unroll
        for (int pl = 0; pl < 4; ++pl)
            tma_load_2d(smem + OFF_T1H + pl * 8192, &p.tm_t, 0, pl * p.t_rows + job.t_row0 + h * len + pos, bar_t);
        atomicMax(&cnt[7], c + 1);
    };
    auto issue_v = [&](int c, int pos) {
        proxy_fence();
        mbar_arrive_expect_tx(bar_v, 2u * 8192u);
        const int t0 = (int)(tok_begin + pos);
        tma_load_3d(smem + OFF_V, &p.tm_v, 0, h, t0, bar_v);
        tma_load_3d(smem + OFF_V + 8192, &p.tm_v, 64, h, t0, bar_v);
        atomicMax(&cnt[1], c + 1);
    };

    if (len == 0) {
        // empty range: the final state is the initial one
        if (warp < 4 && job.s_final) {
            for (int c0 = 0; c0 < D; c0 += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (job.s0) x = __ldg(reinterpret_cast<const float4*>(job.s0 + head_state + (size_t)row * D + c0));
                *reinterpret_cast<float4*>(job.s_final + head_state + (size_t)row * D + c0) = x;
            }
        }
    } else if (warp < 4) {
        // ============================ chain group ============================
        // state rows 32 lq .. 32 lq + 31, columns c0 .. c0 + 31 (one per lane's v) to dst [d_v][d_k]: through a
        // 32 x 8 tile per pass so that every store instruction writes whole 32-byte sectors
        float* dstg = reinterpret_cast<float*>(smem + (PRE_T ? OFF_LD : OFF_OST) + lq * (PRE_T ? 1024 : 2048));
        auto dump_cols = [&](float* dst, int c0, const float (&v)[32]) {
#pragma unroll
            for (int ps = 0; ps < 4; ++ps) {
                __syncwarp();
                *reinterpret_cast<float4*>(dstg + lane * 8) =
                    make_float4(v[8 * ps], v[8 * ps + 1], v[8 * ps + 2], v[8 * ps + 3]);
                *reinterpret_cast<float4*>(dstg + lane * 8 + 4) =
                    make_float4(v[8 * ps + 4], v[8 * ps + 5], v[8 * ps + 6], v[8 * ps + 7]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = 32 * k + lane, r = e >> 1, hq = e & 1;
                    *reinterpret_cast<float4*>(dst + (size_t)(32 * lq + r) * D + c0 + 8 * ps + 4 * hq) =
                        *reinterpret_cast<const float4*>(dstg + r * 8 + 4 * hq);
                }
            }
        };
        // St -> bf16 hi/lo pairs (the A operand of chunk Rn).  First, when the previous chunk Rp asks for it,
        // sigma is folded into St and the folded state dumped (checkpoint); a single small-alpha token then
        // scales St.  One pass over St: the fold costs no second read.
        auto split_state = [&](const Ring& Rn, const Ring* Rp) {
            const bool single = Rn.single != 0;
            const float f = Rn.prescale;
            const bool fold = Rp && Rp->fold != 0;
            const float ff = fold ? Rp->sigma_after : 1.f;
            float* d1 = (fold && Rp->dump_slot >= 0)
                            ? p.ckpt_states + (size_t)Rp->dump_slot * (size_t)H * D * D + head_state
                            : nullptr;
            auto split_block = [&](int cb, float(&v)[32]) {
                if (fold) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= ff;
                    if (!single) tmem_st32(trow + T_S + 32 * cb, v);
                    if (d1) dump_cols(d1, 32 * cb, v);
                }
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) split_pair(v[2 * e], v[2 * e + 1], hw[e], lw[e]);
                tmem_st16(trow + T_SH + 16 * cb, hw);
                tmem_st16(trow + T_SL + 16 * cb, lw);
                if (single) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= f;
                    tmem_st32(trow + T_S + 32 * cb, v);
                }
            };
            if constexpr (PRE_T) {   // two 32-column blocks per TMEM round trip (in the fused kernel the
                                     // extra registers cost more than the round trip saves)
#pragma unroll 1
                for (int cp = 0; cp < 2; ++cp) {
                    float v2[2][32];
                    tmem_ld32x2(trow + T_S + 64 * cp, trow + T_S + 64 * cp + 32, v2[0], v2[1]);
                    split_block(2 * cp, v2[0]);
                    split_block(2 * cp + 1, v2[1]);
                }
            } else {
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tmem_ld32(trow + T_S + 32 * cb, v);
                    split_block(cb, v);
                }
            }
            tmem_st_wait();
        };
        auto fold_state = [&](const Ring& R) {
            float* d1 = R.dump_slot >= 0 ? p.ckpt_states + (size_t)R.dump_slot * (size_t)H * D * D + head_state : nullptr;
            float* d2 = (R.last && job.s_final) ? job.s_final + head_state : nullptr;
            const float f = R.sigma_after;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
                tmem_ld32(trow + T_S + 32 * cb, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= f;
                tmem_st32(trow + T_S + 32 * cb, v);
                if (d1) dump_cols(d1, 32 * cb, v);
                if (d2) dump_cols(d2, 32 * cb, v);
            }
            tmem_st_wait();
        };
        auto readout = [&](const Ring& R, float u0) {
            // every schedule field into registers first: the output stores may alias shared memory
            const int n = R.n;
            const bool single = R.single != 0;
            const float qk0 = R.qk0;
            const size_t tstride = (size_t)H * D;
            const bool vec = p.o_vec16 != 0;
            OutT* ob = reinterpret_cast<OutT*>(o_job) + (size_t)R.begin * tstride + (size_t)h * D +
                       (vec ? 32 * lq : row);
            OutT* stg = reinterpret_cast<OutT*>(smem + OFF_OST + lq * 2048);
            constexpr int kTok = 2048 / (32 * (int)sizeof(OutT));   // tokens per staged tile: 32 bf16, 16 fp32
            constexpr int kSeg = 32 * (int)sizeof(OutT) / 16;        // 16-byte pieces per token and warp
            float vo[2][32];
            tmem_ld32x2(trow + TO, trow + TO + 32, vo[0], vo[1]);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                if (32 * cb >= n) break;
                float(&v)[32] = vo[cb];
                float rs[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(&R.rs[32 * cb + i]);
                    rs[i] = x.x;
                    rs[i + 1] = x.y;
                    rs[i + 2] = x.z;
                    rs[i + 3] = x.w;
                }
                if (cb == 0 && single) v[0] = fmaf(qk0, u0, rs[0] * v[0]);
                else if (cb == 0) v[0] *= rs[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) v[j] *= rs[j];
                if (cb == 1) v[0] *= rs[0];
                const int m = n - 32 * cb;
                if (vec) {
                    // through a [tokens][32 rows] tile: each token's 32 rows leave as whole 16-byte pieces
#pragma unroll
                    for (int ps = 0; ps < 32 / kTok; ++ps) {
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < kTok; ++i) {
                            if constexpr (OUT_BF16)
                                stg[i * 32 + lane] = __float2bfloat16_rn(v[ps * kTok + i]);
                            else
                                stg[i * 32 + lane] = v[ps * kTok + i];
                        }
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < kTok * kSeg / 32; ++k) {
                            const int e = 32 * k + lane, i = e / kSeg, u = e % kSeg;
                            const int t = ps * kTok + i;
                            if (t < m)
                                *reinterpret_cast<uint4*>(ob + (size_t)(32 * cb + t) * tstride + u * (16 / sizeof(OutT))) =
                                    *reinterpret_cast<const uint4*>(stg + i * 32 + u * (16 / sizeof(OutT)));
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < m) {
                            OutT* op = ob + (size_t)(32 * cb + j) * tstride;
                            if constexpr (OUT_BF16)
                                *op = __float2bfloat16_rn(v[j]);
                            else
                                *op = v[j];
                        }
                    }
                }
            }
        };

        // St = S_0 (sigma = 1)
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (job.s0) x = __ldg(reinterpret_cast<const float4*>(job.s0 + head_state + (size_t)row * D + 32 * cb + i));
                v[i] = x.x;
                v[i + 1] = x.y;
                v[i + 2] = x.z;
                v[i + 3] = x.w;
            }
            tmem_st32(trow + T_S + 32 * cb, v);
        }
        tmem_st_wait();
        bool ok = group_wait(&bar_ring[0], 0, tid == 0, BAR_CHAIN, NCHAIN, abort_flag, limit);
        if (ok) {
            split_state(ring[0], nullptr);
            tc_fence_before();
            mbar_arrive(bar_split);
            float u0_prev = 0.f;
            for (int j = 0;; ++j) {
                const Ring& R = ring[j % kRing];
                // ---- readout of the previous chunk while U^T of this one is computed ----
                if (rd && j > 0) {
                    if (!group_wait(bar_o, (uint32_t)((j - 1) & 1), tid == 0, BAR_CHAIN, NCHAIN, abort_flag, limit)) break;
                    tc_fence_after();
                    if (!PRE_T) {   // with T given the prep group reads O out; U''^T P^T is done with U'' all the same
                        readout(ring[(j - 1) % kRing], u0_prev);
                        tc_fence_before();
                        mbar_arrive(bar_ofree);
                    }
                }
                // ---- U'' = c_t U as bf16 hi/lo (K-major A operand [d_v][t]) ----
                if (!group_wait(bar_uo, (uint32_t)(j & 1), tid == 0, BAR_CHAIN, NCHAIN, abort_flag, limit)) break;
                tc_fence_after();
                float u0 = 0.f;
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    float v[32], c[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 x = *reinterpret_cast<const float4*>(&R.c[32 * cb + i]);
                        c[i] = x.x;
                        c[i + 1] = x.y;
                        c[i + 2] = x.z;
                        c[i + 3] = x.w;
                    }
                    {
                        float w[32];
                        tmem_ld32x2(trow + T_U + 32 * cb, trow + TW + 32 * cb, v, w);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] += w[i];
                    }
                    if (cb == 0) {
                        u0 = v[0];
                        if (PRE_T) reinterpret_cast<float*>(smem + OFF_U0)[(j & 1) * 128 + row] = u0;
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= c[i];
                    // U''^T as the products' A operand in TMEM, bf16 pairs: hi over the U columns, lo over the W
                    // columns, each into the 16 columns this thread has just read (block cb = 0) or read before
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) split_pair(v[2 * e], v[2 * e + 1], hw[e], lw[e]);
                    tmem_st16(trow + T_U + 16 * cb, hw);
                    tmem_st16(trow + TW + 16 * cb, lw);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar_ufree);
                // ---- after St += U''^T K: checkpoint / end / small scale -> fold sigma into St ----
                if (!group_wait(bar_st, (uint32_t)(j & 1), tid == 0, BAR_CHAIN, NCHAIN, abort_flag, limit)) break;
                tc_fence_after();
                const bool fold = R.fold != 0, last = R.last != 0;
                if (fold && last) fold_state(R);   // otherwise folded in the next split
                u0_prev = u0;
                if (last) {
                    if (rd && !PRE_T) {
                        if (!group_wait(bar_o, (uint32_t)(j & 1), tid == 0, BAR_CHAIN, NCHAIN, abort_flag, limit)) break;
                        tc_fence_after();
                        readout(R, u0_prev);
                    }
                    break;
                }
                // ---- next chunk: its K/Q two chunks ahead into the buffer just freed, then split St ----
                const int jn = j + 1;
                if (!group_wait(&bar_ring[jn % kRing], (uint32_t)((jn / kRing) & 1), tid == 0, BAR_CHAIN, NCHAIN,
                                abort_flag, limit))
                    break;
                const Ring& Rn = ring[jn % kRing];
                if (tid == 0 && Rn.next_len > 0 && allowed(j + 2)) issue_kq(j + 2, Rn.next_begin);
                split_state(Rn, &R);
                tc_fence_before();
                mbar_arrive(bar_split);
            }
        }
    } else if (warp < 12) {
        // ============================ prep group ============================
        const int ptid = tid - NCHAIN;           // 0..255
        const int pw = warp - 4;                 // 0..7
        const int half = pw >> 2;                // column half of G / W handled by this warp
        const bool leader = ptid == 0;
        // gate warp (pw == 3) state: schedule cursors, running scale, the next window's gates
        // the next checkpoint not yet reached, cached in registers (the table lives in the parameter block,
        // where an indexed read is slow): every checkpoint ends a window, so one cursor serves the
        // schedule and the dumps
        int g_ck = job.ck_begin;
        int g_ck_pos = g_ck < ck_end ? p.ckpts[g_ck].pos : INT_MAX;
        int g_ck_slot = g_ck < ck_end ? p.ckpts[g_ck].slot : -1;
        float g_sigma = 1.f;
        Pos g_win{0, 0};
        float ga0 = 1.f, ga1 = 1.f, gb0 = 0.f, gb1 = 0.f;
        auto next_window = [&](int pos) -> Pos {   // 64 tokens from pos, cut at the next checkpoint
            int end = pos + C < len ? pos + C : len;
            if (g_ck_pos < end) end = g_ck_pos;
            return Pos{pos, end - pos};
        };
        auto load_gates = [&](Pos c) {
            ga0 = ga1 = 1.f;
            gb0 = gb1 = 0.f;
            const size_t gbase = (size_t)(tok_begin + c.begin) * (size_t)H + (size_t)h;
            if (lane < c.len) {
                ga0 = __ldg(p.alpha + gbase + (size_t)lane * H);
                gb0 = __ldg(p.beta + gbase + (size_t)lane * H);
            }
            if (lane + 32 < c.len) {
                ga1 = __ldg(p.alpha + gbase + (size_t)(lane + 32) * H);
                gb1 = __ldg(p.beta + gbase + (size_t)(lane + 32) * H);
            }
        };
        // schedule and scalars of chunk jj (window g_win), published in ring[jj % kRing]
        auto compute_chunk = [&](int jj) {
            float a0 = ga0, a1 = ga1, b0 = gb0, b1 = gb1;
            float g0, g1;
            gate_prefix(a0, a1, g0, g1, lane);
            int n = g_win.len;
            const int first = gamma_first(g0, g1);
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
                gate_prefix(a0, a1, g0, g1, lane);
            }
            const float gfirst = __shfl_sync(0xffffffffu, g0, 0);
            const float glast = __shfl_sync(0xffffffffu, n > 32 ? g1 : g0, (n - 1) & 31);
            const bool single = n == 1 && gfirst < kGammaFloor;
            const int chunk_end = g_win.begin + n;
            const bool dump = g_ck_pos == chunk_end;
            const int dump_slot = g_ck_slot;
            if (dump) {
                ++g_ck;
                g_ck_pos = g_ck < ck_end ? p.ckpts[g_ck].pos : INT_MAX;
                g_ck_slot = g_ck < ck_end ? p.ckpts[g_ck].slot : -1;
            }
            const bool last = chunk_end >= len;
            const float sigma0 = g_sigma;
            const float s_after = single ? 1.f : sigma0 * glast;
            const bool fold = dump || last || s_after < kSigmaFloor;
            const Pos nx = last ? Pos{len, 0} : next_window(chunk_end);
            float* ps = psc + (jj & 1) * 4 * C;
            ps[lane] = g0;
            ps[lane + 32] = g1;
            ps[C + lane] = __frcp_rn(g0);
            ps[C + lane + 32] = __frcp_rn(g1);
            ps[2 * C + lane] = b0 * g0;
            ps[2 * C + lane + 32] = b1 * g1;
            ps[3 * C + lane] = b0;
            ps[3 * C + lane + 32] = b1;
            Ring& R = ring[jj % kRing];
            R.rs[lane] = single ? (lane == 0 ? sigma0 * g0 : 0.f) : sigma0 * g0;
            R.rs[lane + 32] = single ? 0.f : sigma0 * g1;
            R.c[lane] = lane < n ? (single ? 1.f : __frcp_rn(sigma0 * g0)) : 0.f;
            R.c[lane + 32] = lane + 32 < n ? __frcp_rn(sigma0 * g1) : 0.f;
            if (lane == 0) {
                R.begin = g_win.begin;
                R.n = n;
                R.single = single ? 1 : 0;
                R.fold = fold ? 1 : 0;
                R.dump_slot = dump ? dump_slot : -1;
                R.last = last ? 1 : 0;
                R.next_begin = nx.begin;
                R.next_len = nx.len;
                R.sigma0 = sigma0;
                R.sigma_after = s_after;
                R.prescale = single ? sigma0 * gfirst : 1.f;
                R.qk0 = 0.f;
            }
            g_sigma = fold ? 1.f : s_after;
            g_win = nx;
            if (nx.len > 0) load_gates(nx);
            mbar_arrive(&bar_ring[jj % kRing]);
        };

        if (pw == 3) {
            g_win = next_window(0);
            load_gates(g_win);
            if (lane == 0 && allowed(0)) {
                issue_kq(0, 0);
                issue_v(0, 0);
                if (PRE_T) issue_t(0, 0);
            }
            compute_chunk(0);
            if (lane == 0 && ring[0].next_len > 0 && allowed(1)) issue_kq(1, ring[0].next_begin);
        }
        // T is lower triangular: the rows 0-31, columns 32-63 of the T diag(.) operand tiles stay zero
        for (int i = ptid; i < 4 * 32 * 4; i += NPREP) {
            const int tile = i >> 7, r = (i >> 2) & 31, q = i & 3;
            *reinterpret_cast<uint4*>(smem + OFF_T1H + tile * 8192 + sw128(r, 32 + 8 * q)) = make_uint4(0u, 0u, 0u, 0u);
        }
        proxy_fence();
        group_sync(BAR_PREP, NPREP);

        // chunk jj's K/Q landed and its rows past the chunk zeroed; then [K; Q] K^T can be issued
        auto stage_kq = [&](int jj) -> bool {
            tc_fence_before();   // the G columns were last read by the previous chunk's P extraction
            if (!group_wait(&bar_kq[jj & 1], (uint32_t)((jj >> 1) & 1), leader, BAR_PREP, NPREP, abort_flag, limit))
                return false;
            const int nn = ring[jj % kRing].n;
            if (nn < C) {   // a full chunk needs no barrier beyond the wait's own
                const int nz = C - nn;
                for (int i = ptid; i < 4 * nz * 8; i += NPREP) {
                    const int seg = i & 7, rz = (i >> 3) % nz, part = (i >> 3) / nz;   // K / Q x two column blocks
                    unsigned char* base = smem + OFF_KQ + (jj & 1) * 32768 + (part >> 1) * 16384 + (part & 1) * 8192;
                    *reinterpret_cast<uint4*>(base + (nn + rz) * 128 + seg * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                proxy_fence();
                group_sync(BAR_PREP, NPREP);
            }
            if (leader) mbar_arrive(bar_gin);
            return true;
        };
        bool staged = stage_kq(0);

        if constexpr (PRE_T) {
            // T of every chunk was computed by the first passes: the group converts it, serves the chain as
            // before (P, -sigma_0 W, padded tiles) and reads O out.
            // o of chunk jj: rows 32 lq .. + 31 of this warp's lane quarter, tokens 32 half .. + 31, through a
            // [tokens][32 rows] tile of 1 KB so that whole 16-byte pieces leave (scalar stores if o is unaligned)
            auto read_o = [&](int jj) {
                const Ring& Ro = ring[jj % kRing];
                const int n = Ro.n, t0 = 32 * half;
                if (t0 >= n) return;
                float v[32], rs[32];
                tmem_ld32(trow + TO + t0, v);
                const bool single = Ro.single != 0;
                const float qk0 = Ro.qk0;
                const size_t tstride = (size_t)H * D;
                const bool vec = p.o_vec16 != 0;
                OutT* ob = reinterpret_cast<OutT*>(o_job) + (size_t)(Ro.begin + t0) * tstride + (size_t)h * D +
                           (vec ? 32 * lq : row);
                OutT* stg = reinterpret_cast<OutT*>(smem + OFF_OST + pw * 1024);
                constexpr int kTok = 1024 / (32 * (int)sizeof(OutT));   // tokens per tile: 16 bf16, 8 fp32
                constexpr int kSeg = 32 * (int)sizeof(OutT) / 16;        // 16-byte pieces per token
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(&Ro.rs[t0 + i]);
                    rs[i] = x.x;
                    rs[i + 1] = x.y;
                    rs[i + 2] = x.z;
                    rs[i + 3] = x.w;
                }
                if (t0 == 0 && single)
                    v[0] = fmaf(qk0, reinterpret_cast<const float*>(smem + OFF_U0)[(jj & 1) * 128 + row], rs[0] * v[0]);
                else
                    v[0] *= rs[0];
#pragma unroll
                for (int i = 1; i < 32; ++i) v[i] *= rs[i];
                const int m = n - t0;
                if (vec) {
#pragma unroll
                    for (int ps = 0; ps < 32 / kTok; ++ps) {
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < kTok; ++i) {
                            if constexpr (OUT_BF16)
                                stg[i * 32 + lane] = __float2bfloat16_rn(v[ps * kTok + i]);
                            else
                                stg[i * 32 + lane] = v[ps * kTok + i];
                        }
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < kTok * kSeg / 32; ++k) {
                            const int e = 32 * k + lane, i = e / kSeg, u = e % kSeg;
                            const int t = ps * kTok + i;
                            if (t < m)
                                *reinterpret_cast<uint4*>(ob + (size_t)t * tstride + u * (16 / sizeof(OutT))) =
                                    *reinterpret_cast<const uint4*>(stg + i * 32 + u * (16 / sizeof(OutT)));
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (i < m) {
                            if constexpr (OUT_BF16)
                                ob[(size_t)i * tstride] = __float2bfloat16_rn(v[i]);
                            else
                                ob[(size_t)i * tstride] = v[i];
                        }
                    }
                }
            };
            for (int j = 0; staged; ++j) {
                const Ring& R = ring[j % kRing];
                const int n = R.n;
                const bool single = R.single != 0;
                const bool last = R.last != 0;

                // ---- this chunk's V and T operand tiles; rows past the chunk (later tokens) zeroed ----
                if (!group_wait(bar_v, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
                if (!group_wait(bar_t, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
                if (n < C) {
                    const int nz = C - n;
                    for (int i = ptid; i < 6 * nz * 8; i += NPREP) {   // V: two column blocks; T: four planes
                        const int seg = i & 7, rz = (i >> 3) % nz, part = (i >> 3) / nz;
                        unsigned char* base = part < 2 ? smem + OFF_V + part * 8192 : smem + OFF_T1H + (part - 2) * 8192;
                        *reinterpret_cast<uint4*>(base + (n + rz) * 128 + seg * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    proxy_fence();
                    group_sync(BAR_PREP, NPREP);   // a full chunk's tiles are all the copies' own
                }
                if (leader) mbar_arrive(bar_wuin);
                if (pw == 3 && !last) compute_chunk(j + 1);   // the gate warp runs one chunk ahead, off the barriers

                // ---- W^T = K^T T1^T, U~^T = V^T T2^T; then -sigma_0 W^T as the MN-major B operand: first, as
                //      the chain's next U^T waits for it, while P waits for the previous readout ----
                if (!group_wait(bar_wu, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
                tc_fence_after();
                if (leader && !last && allowed(j + 1)) {   // the V and T tiles are free again
                    issue_v(j + 1, R.next_begin);
                    issue_t(j + 1, R.next_begin);
                }
                {
                    const float f = -R.sigma0;
                    float v[32];
                    tmem_ld32(trow + TW + 32 * half, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= f;
                    st_split32(smem + OFF_WH, smem + OFF_WL, row, 32 * half, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    tmem_st32(trow + TW + 32 * half, v);   // U^T's second half accumulates from zero
                    tmem_st_wait();
                }
                proxy_fence();
                tc_fence_before();
                mbar_arrive(bar_wready);

                // ---- once the chain's previous U''^T P^T is done: read O of the previous chunk out, then P =
                //      mask(q_t . k_s) from the Q rows of [K; Q] K^T; then the next chunk's K/Q tiles ----
                if (rd) {
                    if (j > 0) {
                        if (!group_wait(bar_o, (uint32_t)((j - 1) & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
                        tc_fence_after();
                        read_o(j - 1);
                        tc_fence_before();
                        mbar_arrive(bar_ofree);
                    }
                    if (!group_wait(bar_g, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
                    tc_fence_after();
                    if (lq >= 2) {
                        float v[32];
                        tmem_ld32(trow + TG + 32 * half, v);
                        const int t = row - 64, s0 = 32 * half;
                        if (single && t == 0 && half == 0) ring[j % kRing].qk0 = v[0];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = (!single && s0 + i <= t) ? v[i] : 0.f;
                        st_split32(smem + OFF_PH, smem + OFF_PL, t, s0, v);
                    }
                    tc_fence_before();
                    proxy_fence();
                    mbar_arrive(bar_pready);
                }
                if (!last && !(staged = stage_kq(j + 1))) break;

                if (last) {
                    // the last chunk's O
                    if (rd && group_wait(bar_o, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) {
                        tc_fence_after();
                        read_o(j);
                    }
                    break;
                }
            }
        } else {
        for (int j = 0; staged; ++j) {
            const Ring& R = ring[j % kRing];
            const int n = R.n;
            const bool single = R.single != 0;
            const bool last = R.last != 0;
            const float* ps = psc + (j & 1) * 4 * C;

            // ---- this chunk's [K; Q] K^T, issued a chunk ago ----
            if (!group_wait(bar_g, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
            tc_fence_after();
            // ---- L (fp32, zero on and above the diagonal) from the K rows of [K; Q] K^T; diagonal blocks to Ld ----
            if (lq < 2) {
                const int t = row, s0 = 32 * half;
                float gi[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(ps + C + s0 + i);
                    gi[i] = x.x;
                    gi[i + 1] = x.y;
                    gi[i + 2] = x.z;
                    gi[i + 3] = x.w;
                }
                const float f = ps[2 * C + t];
                float v[32];
                tmem_ld32(trow + TG + 32 * half, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = (s0 + i < t) ? f * gi[i] * v[i] : 0.f;
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    *reinterpret_cast<float4*>(Lf + t * kLdF + s0 + 4 * q4) =
                        make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                if ((t >> 5) == half) {   // the diagonal 16-block of row t lies in this half
                    float* dst = Ld + (t >> 4) * 16 * 17 + (t & 15) * 17;
#pragma unroll
                    for (int i = 0; i < 16; ++i) dst[i] = (lane & 16) ? v[16 + i] : v[i];
                }
            }
            group_sync(BAR_PREP, NPREP);
            const float* sg_bg = ps + 2 * C;
            const float* sg_b = ps + 3 * C;
            // T1 = T diag(beta gamma), T2 = T diag(beta) as bf16 hi/lo, K-major [t][s]: two adjacent columns
            auto put_t12 = [&](int t, int s, float x0, float x1) {
                uint32_t h1, l1, h2, l2;
                split_pair(x0 * sg_bg[s], x1 * sg_bg[s + 1], h1, l1);
                split_pair(x0 * sg_b[s], x1 * sg_b[s + 1], h2, l2);
                const uint32_t o = sw128(t, s);
                *reinterpret_cast<uint32_t*>(smem + OFF_T1H + o) = h1;
                *reinterpret_cast<uint32_t*>(smem + OFF_T1L + o) = l1;
                *reinterpret_cast<uint32_t*>(smem + OFF_T2H + o) = h2;
                *reinterpret_cast<uint32_t*>(smem + OFF_T2L + o) = l2;
            };
            // ---- T = (I + L)^-1 = [[T_AA, 0], [T_BA, T_BB]] in 32-blocks.  Warp 6 (rows 0-31 of G, columns
            //      0-31) and warp 9 (rows 32-63, columns 32-63) each take a whole diagonal 32-block of L and
            //      invert it alone: two 16x16 forward substitutions and one merge; the gate warp (7) runs a
            //      chunk ahead.  Warps 6 and 9 sit on SM sub-partitions 2 and 1 (warp % 4), away from the
            //      MMA-issue warp's poll loop on sub-partition 0, which slows a warp beside it by ~40 % here.  Then the whole group writes the T operands of both diagonal blocks and merges
            //      the lower-left block.  The merges run on mma.sync with every operand split into bf16
            //      hi + lo. ----
            if (pw == 2 || pw == 5) {
                const int qw = pw == 5 ? 1 : 0;            // diagonal quadrant: rows / columns 32 qw .. + 31
                {
                    // lanes 0-15: column jc of block 2 qw; lanes 16-31: of block 2 qw + 1 (forward substitution,
                    // each dot product in four partial sums)
                    {
                        const int bb = 2 * qw + (lane >> 4), jc = lane & 15;
                        const float* Lb = Ld + bb * 16 * 17;
                        float x[16];
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int s2 = 0; s2 < r; ++s2) acc[s2 & 3] = fmaf(Lb[r * 17 + s2], x[s2], acc[s2 & 3]);
                            x[r] = ((r == jc) ? 1.f : 0.f) - ((acc[0] + acc[1]) + (acc[2] + acc[3]));
                        }
#pragma unroll
                        for (int r = 0; r < 16; ++r) Lf[(16 * bb + r) * kLdF + 16 * bb + jc] = x[r];
                    }
                    __syncwarp();
                    // merge: T_ib,jb = -T_ib,ib (L_ib,jb T_jb,jb), (jb, ib) = (2 qw, 2 qw + 1), bf16 hi/lo x 3 on
                    // mma.sync (two 8-column tiles, one k step each)
                    {
                        const int jb = 2 * qw, ib = jb + 1, g8 = lane >> 2, t4 = lane & 3;
                        float* sc = Ld + jb * 16 * 17;   // this warp's diagonal blocks of L are no longer needed
                        float y[2][4], yc[2][4];
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) y[nt][e] = yc[nt][e] = 0.f;
                            mma_bf16x3(y[nt], yc[nt], Lf + (16 * ib) * kLdF + 16 * jb, kLdF,
                                       Lf + (16 * jb) * kLdF + 16 * jb + 8 * nt, kLdF, g8, t4);
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            sc[g8 * kLdS + 8 * nt + 2 * t4] = y[nt][0] + yc[nt][0];
                            sc[g8 * kLdS + 8 * nt + 2 * t4 + 1] = y[nt][1] + yc[nt][1];
                            sc[(g8 + 8) * kLdS + 8 * nt + 2 * t4] = y[nt][2] + yc[nt][2];
                            sc[(g8 + 8) * kLdS + 8 * nt + 2 * t4 + 1] = y[nt][3] + yc[nt][3];
                        }
                        __syncwarp();
                        float x[2][4], xc[2][4];
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) x[nt][e] = xc[nt][e] = 0.f;
                            mma_bf16x3(x[nt], xc[nt], Lf + (16 * ib) * kLdF + 16 * ib, kLdF, sc + 8 * nt, kLdS, g8, t4);
                        }
                        float* dst = Lf + (16 * ib) * kLdF + 16 * jb;
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            dst[g8 * kLdF + 8 * nt + 2 * t4] = -(x[nt][0] + xc[nt][0]);
                            dst[g8 * kLdF + 8 * nt + 2 * t4 + 1] = -(x[nt][1] + xc[nt][1]);
                            dst[(g8 + 8) * kLdF + 8 * nt + 2 * t4] = -(x[nt][2] + xc[nt][2]);
                            dst[(g8 + 8) * kLdF + 8 * nt + 2 * t4 + 1] = -(x[nt][3] + xc[nt][3]);
                        }
                    }
                }
            } else if (pw == 3 && !last) {
                compute_chunk(j + 1);   // the gate warp runs one chunk ahead
            }
            group_sync(BAR_PREP, NPREP);
            {   // the diagonal 32-blocks' T operands, spread over the whole group: one row piece of 8 columns
                // (one 16-byte store per plane) per thread
                const int t = 32 * (ptid >> 7) + ((ptid >> 2) & 31), s0 = 32 * (ptid >> 7) + 8 * (ptid & 3);
                const float4 x0 = *reinterpret_cast<const float4*>(Lf + t * kLdF + s0);
                const float4 x1 = *reinterpret_cast<const float4*>(Lf + t * kLdF + s0 + 4);
                const float4 a0 = *reinterpret_cast<const float4*>(sg_bg + s0);
                const float4 a1 = *reinterpret_cast<const float4*>(sg_bg + s0 + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(sg_b + s0);
                const float4 b1 = *reinterpret_cast<const float4*>(sg_b + s0 + 4);
                uint32_t h1[4], l1[4], h2[4], l2[4];
                split_pair(x0.x * a0.x, x0.y * a0.y, h1[0], l1[0]);
                split_pair(x0.z * a0.z, x0.w * a0.w, h1[1], l1[1]);
                split_pair(x1.x * a1.x, x1.y * a1.y, h1[2], l1[2]);
                split_pair(x1.z * a1.z, x1.w * a1.w, h1[3], l1[3]);
                split_pair(x0.x * b0.x, x0.y * b0.y, h2[0], l2[0]);
                split_pair(x0.z * b0.z, x0.w * b0.w, h2[1], l2[1]);
                split_pair(x1.x * b1.x, x1.y * b1.y, h2[2], l2[2]);
                split_pair(x1.z * b1.z, x1.w * b1.w, h2[3], l2[3]);
                const uint32_t o = sw128(t, s0);
                *reinterpret_cast<uint4*>(smem + OFF_T1H + o) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T1L + o) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T2H + o) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
                *reinterpret_cast<uint4*>(smem + OFF_T2L + o) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
            }
            {   // T_BA = -T_BB (L_BA T_AA) for the lower-left 32x32 block; warp = (row, column) tile
                const int g8 = lane >> 2, t4 = lane & 3;
                const int mt = pw >> 2, nt = pw & 3;
                float y[4] = {0.f, 0.f, 0.f, 0.f}, yc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16x3(y, yc, Lf + (32 + 16 * mt) * kLdF + 16 * ks, kLdF, Lf + (16 * ks) * kLdF + 8 * nt, kLdF,
                               g8, t4);
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] += yc[e];
                // L_BA T_AA as [32][kLdY] scratch
                Yb[(16 * mt + g8) * kLdY + 8 * nt + 2 * t4] = y[0];
                Yb[(16 * mt + g8) * kLdY + 8 * nt + 2 * t4 + 1] = y[1];
                Yb[(16 * mt + g8 + 8) * kLdY + 8 * nt + 2 * t4] = y[2];
                Yb[(16 * mt + g8 + 8) * kLdY + 8 * nt + 2 * t4 + 1] = y[3];
                group_sync(BAR_PREP, NPREP);
                float x[4] = {0.f, 0.f, 0.f, 0.f}, xc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16x3(x, xc, Lf + (32 + 16 * mt) * kLdF + 32 + 16 * ks, kLdF, Yb + (16 * ks) * kLdY + 8 * nt, kLdY,
                               g8, t4);
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] += xc[e];
                put_t12(32 + 16 * mt + g8, 8 * nt + 2 * t4, -x[0], -x[1]);
                put_t12(32 + 16 * mt + g8 + 8, 8 * nt + 2 * t4, -x[2], -x[3]);
            }
            // ---- this chunk's V (rows past the chunk zeroed): landed while T was formed.  The T operand
            //      stores are made visible to the MMA by the wait's own barrier (one more for padding) ----
            proxy_fence();
            if (!group_wait(bar_v, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
            if (n < C) {
                const int nz = C - n;
                for (int i = ptid; i < 2 * nz * 8; i += NPREP) {
                    const int seg = i & 7, rz = (i >> 3) % nz, part = (i >> 3) / nz;
                    *reinterpret_cast<uint4*>(smem + OFF_V + part * 8192 + (n + rz) * 128 + seg * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                proxy_fence();
                group_sync(BAR_PREP, NPREP);
            }
            if (leader) mbar_arrive(bar_wuin);

            // ---- while W^T and U~^T are computed: P = mask(q_t . k_s) from the Q rows of [K; Q] K^T, once the
            //      chain's previous U''^T P^T is done ----
            if (rd) {
                if (j > 0 && !group_wait(bar_o, (uint32_t)((j - 1) & 1), leader, BAR_PREP, NPREP, abort_flag, limit))
                    break;
                tc_fence_after();
                if (lq >= 2) {
                    float v[32];
                    tmem_ld32(trow + TG + 32 * half, v);
                    const int t = row - 64, s0 = 32 * half;
                    if (single && t == 0 && half == 0) ring[j % kRing].qk0 = v[0];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (!single && s0 + i <= t) ? v[i] : 0.f;
                    st_split32(smem + OFF_PH, smem + OFF_PL, t, s0, v);
                }
                proxy_fence();
                tc_fence_before();
                mbar_arrive(bar_pready);
            }
            // ---- the next chunk's [K; Q] K^T, now that the G columns are free: it runs beside this chunk's
            //      W and U~ and is ready when the next iteration starts ----
            if (!last && !(staged = stage_kq(j + 1))) break;
            // ---- W^T = K^T T1^T, U~^T = V^T T2^T; then -sigma_0 W^T as the MN-major B operand ----
            if (!group_wait(bar_wu, (uint32_t)(j & 1), leader, BAR_PREP, NPREP, abort_flag, limit)) break;
            tc_fence_after();
            if (leader && !last && allowed(j + 1)) issue_v(j + 1, R.next_begin);   // the V buffer is free again
            {
                const float f = -R.sigma0;
                float v[32];
                tmem_ld32(trow + TW + 32 * half, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= f;
                st_split32(smem + OFF_WH, smem + OFF_WL, row, 32 * half, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
                tmem_st32(trow + TW + 32 * half, v);   // U^T's second half accumulates from zero
                tmem_st_wait();
            }
            proxy_fence();
            tc_fence_before();
            mbar_arrive(bar_wready);

            if (last) break;
        }
        }
    } else if (lane == 0) {
        // ============================ MMA issue (warp 12, and warp 13 without a readout) ============================
        if constexpr (!READOUT) {
            // Without a readout: two issuing threads, one per stream, each in its stream's order: the prep stream
            // (warp 12) G_j, WU_j and the chain stream (warp 13) U_j, St_j.  An item is issued once the mbarriers of
            // its operands have fired; each thread blocks in the barrier wait (suspended in hardware, so it takes no
            // issue slot from the warps that share its SM sub-partition).  Each thread commits its own products; a
            // product that reads what the other stream wrote waits for that stream's completion barrier.
            const uint32_t id64 = idesc(64, false, false), id64b = idesc(64, false, true), id64a = idesc(64, true, false);
            const uint32_t id128b = idesc(128, false, true);
            auto wait = [&](uint64_t* b, uint32_t parity) { return wait_phase(b, parity, abort_flag, limit); };
            if (warp == 12) {
                for (int jp = 0;; ++jp) {
                    const uint32_t inKQ = sbase + OFF_KQ + (jp & 1) * 32768;
                    if (!wait(bar_gin, jp & 1)) break;
                    tc_fence_after();
                    // [K; Q] K^T: its K rows give L, its Q rows P (with T given only P, and only with a readout)
                    if (!PRE_T || rd) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                            umma_ss(tbase + TG, sdesc(inKQ + off, 16, 1024), sdesc(inKQ + off, 16, 1024), id64, kk > 0);
                        }
                        umma_commit(bar_g);
                        ++cnt[2];
                    }
                    // the U and W columns hold the previous chunk's U'' until its last product (U''^T P^T with a
                    // readout, else the state update) is done
                    if (!wait(bar_wuin, jp & 1)) break;
                    if (jp > 0 && !wait(rd ? bar_o : bar_st, (jp - 1) & 1)) break;
                    tc_fence_after();
                    // W^T = K^T T1^T, U~^T = V^T T2^T
                    const uint32_t inV = sbase + OFF_V;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ak = sdesc(inKQ + ks * 2048, 16384, 1024);   // K^T: MN-major, d_k blocks 16 KB apart
                        const uint64_t av = sdesc(inV + ks * 2048, 8192, 1024);     // V^T: MN-major, d_v blocks 8 KB apart
                        umma_ss(tbase + TW, ak, sdesc(sbase + OFF_T1H + ks * 32, 16, 1024), id64a, ks > 0);
                        umma_ss(tbase + TW, ak, sdesc(sbase + OFF_T1L + ks * 32, 16, 1024), id64a, 1);
                        umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2H + ks * 32, 16, 1024), id64a, ks > 0);
                        umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2L + ks * 32, 16, 1024), id64a, 1);
                    }
                    umma_commit(bar_wu);
                    ++cnt[3];
                    if (ring[jp % kRing].last) break;
                }
            } else if (warp == 13) {
                for (int jc = 0;; ++jc) {
                    const Ring& R = ring[jc % kRing];
                    const uint32_t inKQ = sbase + OFF_KQ + (jc & 1) * 32768;
                    if (!wait(bar_split, jc & 1) || !wait(bar_wready, jc & 1)) break;
                    tc_fence_after();
                    // U^T += St (-sigma_0 W)^T  (St from TMEM as bf16 hi/lo pairs)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bwh = sdesc(sbase + OFF_WH + kk * 2048, 16384, 1024);
                        const uint32_t ah = tbase + T_SH + 8 * kk, al = tbase + T_SL + 8 * kk;
                        // [U | W] += S_hi [W_hi | W_lo]^T (N = 128: W_lo follows W_hi at the block stride)
                        umma_ts(tbase + T_U, ah, bwh, id128b, 1);
                        umma_ts(tbase + T_U, al, bwh, id64b, 1);
                    }
                    umma_commit(bar_uo);
                    ++cnt[4];
                    if (rd) {
                        if (jc > 0 && !wait(bar_ofree, (jc - 1) & 1)) break;
                        tc_fence_after();
                        // O^T = St Q^T
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t bq = sdesc(inKQ + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                            umma_ts(tbase + TO, tbase + T_SH + 8 * kk, bq, id64, kk > 0);
                            umma_ts(tbase + TO, tbase + T_SL + 8 * kk, bq, id64, 1);
                        }
                    }
                    if (!wait(bar_ufree, jc & 1)) break;
                    tc_fence_after();
                    // St += U''^T K
#pragma unroll
                    for (int kt = 0; kt < 4; ++kt) {
                        const uint64_t bk = sdesc(inKQ + kt * 2048, 16384, 1024);   // K: MN-major over d_k
                        umma_ts(tbase + T_S, tbase + T_U + 8 * kt, bk, id128b, 1);   // U'' hi
                        umma_ts(tbase + T_S, tbase + TW + 8 * kt, bk, id128b, 1);    // U'' lo
                    }
                    umma_commit(bar_st);
                    ++cnt[5];
                    if (rd) {
                        if (!wait(bar_pready, jc & 1)) break;
                        tc_fence_after();
                        if (!R.single) {
                            // O^T += U''^T P^T
#pragma unroll
                            for (int kt = 0; kt < 4; ++kt) {
                                const uint64_t bph = sdesc(sbase + OFF_PH + kt * 32, 16, 1024);
                                const uint64_t bpl = sdesc(sbase + OFF_PL + kt * 32, 16, 1024);
                                umma_ts(tbase + TO, tbase + T_U + 8 * kt, bph, id64, 1);
                                umma_ts(tbase + TO, tbase + T_U + 8 * kt, bpl, id64, 1);
                                umma_ts(tbase + TO, tbase + TW + 8 * kt, bph, id64, 1);
                            }
                        }
                        umma_commit(bar_o);
                        ++cnt[6];
                    }
                    if (R.last) break;
                }
            }
        } else if (warp == 12) {
            // With a readout: one thread polls both streams and serves the prep's products first.  (Measured: two
            // sleeping threads shorten the replays, whose chain is short, and lengthen the prefill, where the
            // order in which the single thread interleaves the streams matters more.)
            // Two streams, each in its own order: prep G_j, WU_j and chain U_j, O1_j, St_j, O2_j; the prep stream
            // is served first when the prep group bounds the pipeline (T computed here), else the chain.
            // An item is issued once the mbarriers of its operands have fired; a stream ends after its last chunk.
            int jc = 0, sc = 0, jp = 0, sp = 0;
            bool chain_done = false, prep_done = false;
            uint64_t t_last = global_ns();
            const uint32_t id64 = idesc(64, false, false), id64b = idesc(64, false, true), id64a = idesc(64, true, false);
            const uint32_t id128b = idesc(128, false, true);
            while (!(chain_done && prep_done)) {
                bool progressed = false;
                auto serve_prep = [&]() {
                if (!prep_done) {
                    const uint32_t inKQ = sbase + OFF_KQ + (jp & 1) * 32768;
                    if (sp == 0 && mbar_test(bar_gin, jp & 1)) {
                        tc_fence_after();
                        // [K; Q] K^T: its K rows give L, its Q rows P (with T given only P, and only with a readout)
                        if (!PRE_T || rd) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                umma_ss(tbase + TG, sdesc(inKQ + off, 16, 1024), sdesc(inKQ + off, 16, 1024), id64,
                                        kk > 0);
                            }
                            umma_commit(bar_g);
                            ++cnt[2];
                        }
                        sp = 1;
                        progressed = true;
                    }
                    // the U and W columns hold the previous chunk's U'' until its last product (U''^T P^T with a
                    // readout, else the state update) is done
                    if (sp == 1 && mbar_test(bar_wuin, jp & 1) &&
                        (jp == 0 || mbar_test(rd ? bar_o : bar_st, (jp - 1) & 1))) {
                        tc_fence_after();
                        // W^T = K^T T1^T, U~^T = V^T T2^T
                        const uint32_t inV = sbase + OFF_V;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ak = sdesc(inKQ + ks * 2048, 16384, 1024);   // K^T: MN-major, d_k blocks 16 KB apart
                            const uint64_t av = sdesc(inV + ks * 2048, 8192, 1024);     // V^T: MN-major, d_v blocks 8 KB apart
                            umma_ss(tbase + TW, ak, sdesc(sbase + OFF_T1H + ks * 32, 16, 1024), id64a, ks > 0);
                            umma_ss(tbase + TW, ak, sdesc(sbase + OFF_T1L + ks * 32, 16, 1024), id64a, 1);
                            umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2H + ks * 32, 16, 1024), id64a, ks > 0);
                            umma_ss(tbase + T_U, av, sdesc(sbase + OFF_T2L + ks * 32, 16, 1024), id64a, 1);
                        }
                        umma_commit(bar_wu);
                        ++cnt[3];
                        progressed = true;
                        if (ring[jp % kRing].last) prep_done = true;
                        else {
                            ++jp;
                            sp = 0;
                        }
                    }
                }
                };
                auto serve_chain = [&]() {
                if (!chain_done) {
                    const Ring& R = ring[jc % kRing];
                    const uint32_t inKQ = sbase + OFF_KQ + (jc & 1) * 32768;
                    if (sc == 0) {
                        if (mbar_test(bar_split, jc & 1) && mbar_test(bar_wready, jc & 1)) {
                            tc_fence_after();
                            // U^T += St (-sigma_0 W)^T  (St from TMEM as bf16 hi/lo pairs)
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t bwh = sdesc(sbase + OFF_WH + kk * 2048, 16384, 1024);
                                const uint32_t ah = tbase + T_SH + 8 * kk, al = tbase + T_SL + 8 * kk;
                                // [U | W] += S_hi [W_hi | W_lo]^T (N = 128: W_lo follows W_hi at the block stride)
                                umma_ts(tbase + T_U, ah, bwh, id128b, 1);
                                umma_ts(tbase + T_U, al, bwh, id64b, 1);
                            }
                            umma_commit(bar_uo);
                            ++cnt[4];
                            sc = rd ? 1 : 2;
                            progressed = true;
                        }
                    }
                    if (sc == 1) {
                        if (jc == 0 || mbar_test(bar_ofree, (jc - 1) & 1)) {
                            tc_fence_after();
                            // O^T = St Q^T
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t bq = sdesc(inKQ + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                                umma_ts(tbase + TO, tbase + T_SH + 8 * kk, bq, id64, kk > 0);
                                umma_ts(tbase + TO, tbase + T_SL + 8 * kk, bq, id64, 1);
                            }
                            sc = 2;
                            progressed = true;
                        }
                    }
                    if (sc == 2) {
                        if (mbar_test(bar_ufree, jc & 1)) {
                            tc_fence_after();
                            // St += U''^T K
#pragma unroll
                            for (int kt = 0; kt < 4; ++kt) {
                                const uint64_t bk = sdesc(inKQ + kt * 2048, 16384, 1024);   // K: MN-major over d_k
                                umma_ts(tbase + T_S, tbase + T_U + 8 * kt, bk, id128b, 1);   // U'' hi
                                umma_ts(tbase + T_S, tbase + TW + 8 * kt, bk, id128b, 1);    // U'' lo
                            }
                            umma_commit(bar_st);
                            ++cnt[5];
                            sc = rd ? 3 : 4;
                            progressed = true;
                        }
                    }
                    if (sc == 3) {
                        if (mbar_test(bar_pready, jc & 1)) {
                            tc_fence_after();
                            if (!R.single) {
                                // O^T += U''^T P^T
#pragma unroll
                                for (int kt = 0; kt < 4; ++kt) {
                                    const uint64_t bph = sdesc(sbase + OFF_PH + kt * 32, 16, 1024);
                                    const uint64_t bpl = sdesc(sbase + OFF_PL + kt * 32, 16, 1024);
                                    umma_ts(tbase + TO, tbase + T_U + 8 * kt, bph, id64, 1);
                                    umma_ts(tbase + TO, tbase + T_U + 8 * kt, bpl, id64, 1);
                                    umma_ts(tbase + TO, tbase + TW + 8 * kt, bph, id64, 1);
                                }
                            }
                            umma_commit(bar_o);
                            ++cnt[6];
                            sc = 4;
                            progressed = true;
                        }
                    }
                    if (sc == 4) {
                        if (R.last) chain_done = true;
                        else {
                            ++jc;
                            sc = 0;
                        }
                    }
                }
                };
                // with T computed beforehand the state chain is the critical path: its products go first
                if (PRE_T) {
                    serve_chain();
                    serve_prep();
                } else {
                    serve_prep();
                    serve_chain();
                }
                if (progressed) {
                    t_last = global_ns();
                } else {
                    __nanosleep(20);
                    if (*abort_flag) break;
                    if (global_ns() - t_last > limit) {
                        *abort_flag = 1;
                        break;
                    }
                }
            }
        }
    }

    // ---- leave only with no copy and no MMA still writing into this CTA's shared memory or TMEM ----
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        const int kq = cnt[0];
        for (int b = 0; b < 2; ++b) {
            const int c = ((kq - 1) & 1) == b ? kq - 1 : kq - 2;
            if (c >= 0) drain_phase(&bar_kq[b], (uint32_t)((c >> 1) & 1), drain_limit);
        }
        if (cnt[1] > 0) drain_phase(bar_v, (uint32_t)((cnt[1] - 1) & 1), drain_limit);
        if (cnt[7] > 0) drain_phase(bar_t, (uint32_t)((cnt[7] - 1) & 1), drain_limit);
        for (int i = 0; i < 5; ++i)
            if (cnt[2 + i] > 0) drain_phase(&bars[3 + i], (uint32_t)((cnt[2 + i] - 1) & 1), drain_limit);
        atomicOr(p.status, STATUS_TIMEOUT);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(512));
}

template <bool OUT_BF16, bool READOUT, bool PRE_T>
cudaError_t launch_chunk_tc(const Params& p, int grid, cudaStream_t stream) {
    auto kern = gdn_chunk_tc_kernel<OUT_BF16, READOUT, PRE_T>;
    static std::atomic<int> optin[kMaxOptinDevices];
    cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), kSmemBytes, optin);
    if (e != cudaSuccess) return e;
    kern<<<grid, nthreads(READOUT), kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

// instantiated in inst_chunk_tc.cu; pre_t: T of every chunk is in p.t_rows (two-pass path)
cudaError_t launch(const Params& p, int grid, bool readout, bool out_bf16, bool pre_t, cudaStream_t stream);
// the first passes of the two-pass path (gdn_tprep.cu): the chunk schedule of every (job, head) into
// p.chunk_beg / p.chunk_cnt, then T of every chunk into p.t_rows; n_streams = jobs x heads
cudaError_t launch_schedule(const Params& p, int n_streams, cudaStream_t stream);
cudaError_t launch_tprep(const Params& p, int n_streams, cudaStream_t stream);

}  // namespace tc
}  // namespace gdn
