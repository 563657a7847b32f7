// gdn_tprep.cu - the two parallel passes of the two-pass chunked scan (d_k = d_v = 128, bf16 k).
//
// The chunkwise form of the Gated DeltaNet recurrence ("Tail-Replay" notes page, section 2.3,
// equation (1), regrouped over chunks of up to 64 tokens; derivation in gdn_chunk_tc.cuh) needs per
// chunk T = (I + L)^-1 with L[t][s] = beta_t (gamma_t / gamma_s) k_t.k_s for s < t.  T depends only on
// the chunk's own k, alpha and beta, not on the state, so every chunk of every (job, head) can be
// inverted at once, on every SM, before the state scan runs:
//   schedule_kernel - the chunk starts of each (job, head): windows of 64 tokens from the previous
//       chunk end, cut at the next checkpoint and before the token where gamma falls below 2^-32
//       (the rule the scan kernel's gate warp applies, with the same rounding);
//   tprep_kernel    - T of every chunk in fp32 (bf16 hi/lo x 3 merges and K K^T on mma.sync), stored
//       as the scan's MMA operands T diag(beta gamma) and T diag(beta), each split into bf16 hi + lo, in rows
//       indexed by token, so the storage is bounded by the tokens scanned.
#include <cuda_runtime.h>

#include <climits>

#include "gdn_chunk_tc.cuh"

namespace gdn {
namespace tc {

namespace {

constexpr int kSchedThreads = 256;
constexpr int kSchedTile = 8192;   // gates of one (job, head) staged per pass
constexpr int kSchedWins = 256;    // windows judged at once

// ---- chunk schedule: one block per (job, head).  The windows a walk without gamma cuts would take (64
//      tokens from the previous end, cut at the next checkpoint) are listed first, all of them judged at once
//      by the 8 warps with the same rule and rounding as the scan's gate warp; the walk then takes the windows
//      in order up to the first that is cut early, and lists the windows again from its end. ----
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const __grid_constant__ Params p) {
    __shared__ float sa[kSchedTile + C];
    __shared__ int ws[kSchedWins], wl[kSchedWins], wn[kSchedWins], wck[kSchedWins];
    __shared__ int s_pos, s_cnt, s_ck, s_nw;
    const int s = blockIdx.x, H = p.H;
    const int jb = s / H, h = s - jb * H;
    const Job& job = p.jobs[jb];
    const int len = job.len;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t* beg = p.chunk_beg + (size_t)job.t_row0 + (size_t)h * (size_t)len;
    const int ck_end = job.ck_begin + job.ck_count;
    if (threadIdx.x == 0) {
        s_pos = 0;
        s_cnt = 0;
        s_ck = job.ck_begin;
    }
    __syncthreads();
    while (s_pos < len) {
        const int tile0 = s_pos;
        const int tile_n = min(len - tile0, kSchedTile + C);
        for (int i = threadIdx.x; i < tile_n; i += kSchedThreads)
            sa[i] = __ldg(p.alpha + (size_t)(job.tok_begin + tile0 + i) * (size_t)H + (size_t)h);
        __syncthreads();
        // every window that lies inside the staged tile
        while (s_pos < len && s_pos - tile0 + min(C, len - s_pos) <= tile_n) {
            if (threadIdx.x == 0) {   // the windows of a walk without cuts, from here
                int pos = s_pos, ck = s_ck, nw = 0;
                while (nw < kSchedWins && pos < len && pos - tile0 + min(C, len - pos) <= tile_n) {
                    const int ck_pos = ck < ck_end ? p.ckpts[ck].pos : INT_MAX;
                    int end = pos + C < len ? pos + C : len;
                    if (ck_pos < end) end = ck_pos;
                    if (ck_pos == end) ++ck;
                    ws[nw] = pos;
                    wl[nw] = end - pos;
                    wck[nw] = ck;   // the checkpoint cursor after the window
                    ++nw;
                    pos = end;
                }
                s_nw = nw;
            }
            __syncthreads();
            const int nw = s_nw;
            for (int i = warp; i < nw; i += kSchedThreads / 32) {
                const int w0 = ws[i] - tile0, win = wl[i];
                const float a0 = lane < win ? sa[w0 + lane] : 1.f;
                const float a1 = lane + 32 < win ? sa[w0 + lane + 32] : 1.f;
                float g0, g1;
                gate_prefix(a0, a1, g0, g1, lane);
                const int first = gamma_first(g0, g1);
                if (lane == 0) wn[i] = first < win ? (first > 0 ? first : 1) : win;
            }
            __syncthreads();
            if (threadIdx.x == 0) {   // take the windows in order up to the first cut early
                int pos = s_pos, cnt = s_cnt, ck = s_ck;
                for (int i = 0; i < nw; ++i) {
                    beg[cnt++] = ws[i];
                    if (wn[i] < wl[i]) {   // ends before its window: the cursor stays, the windows shift
                        pos = ws[i] + wn[i];
                        break;
                    }
                    pos = ws[i] + wl[i];
                    ck = wck[i];
                }
                s_pos = pos;
                s_cnt = cnt;
                s_ck = ck;
            }
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) p.chunk_cnt[s] = s_cnt;
}

// ---- T of every chunk: 4 warps per chunk; the next chunk's K is copied in once K K^T is done, and its
//      gates are loaded a chunk ahead ----
constexpr int kTpThreads = 128;
constexpr int kTpBlocksPerSm = 5;
constexpr int kTpLd = 68;                    // fp32 elements per row of L / T in shared memory
constexpr int TP_K = 0;                      // 16 KB: K as two 64-column blocks of [64 rows][128 B], swizzled
constexpr int TP_L = 16384;                  // fp32 [64][68]: L, then T in place
constexpr int TP_Y = TP_L + C * kTpLd * 4;   // fp32 [32][33] scratch of the merges
constexpr int TP_G = TP_Y + 32 * 33 * 4;     // fp32 [3][64]: beta gamma, 1/gamma, beta
constexpr int TP_BAR = TP_G + 3 * C * 4;     // 1 mbarrier
constexpr int kTpSmemBytes = TP_BAR + 64 + 1024;

// shared-memory address of K element (row, col), col % 8 == 0, in a swizzled buffer at kbase
__device__ __forceinline__ uint32_t k_addr(uint32_t kbase, int row, int col) {
    return kbase + (uint32_t)((col >> 6) * 8192) + sw128(row, col & 63);
}

__global__ void __launch_bounds__(kTpThreads, kTpBlocksPerSm) tprep_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char tp_raw[];
    // aligned by pointer arithmetic on the shared array (not through an integer), so that the compiler keeps
    // its address space and plain C++ accesses below compile to shared-memory loads and stores
    unsigned char* smem = tp_raw + ((1024u - (smem_addr(tp_raw) & 1023u)) & 1023u);
    float* sl = reinterpret_cast<float*>(smem + TP_L);
    float* sy = reinterpret_cast<float*>(smem + TP_Y);
    float* sbg = reinterpret_cast<float*>(smem + TP_G);
    float* sgi = sbg + C;
    float* sbe = sbg + 2 * C;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + TP_BAR);
    const uint32_t kbase0 = smem_addr(smem + TP_K);

    const int s = blockIdx.y, H = p.H;
    const int jb = s / H, h = s - jb * H;
    const Job& job = p.jobs[jb];
    const int len = job.len;
    const int nch = p.chunk_cnt[s];
    const int32_t* beg = p.chunk_beg + (size_t)job.t_row0 + (size_t)h * (size_t)len;
    const size_t trow0 = (size_t)job.t_row0 + (size_t)h * (size_t)len;
    const size_t plane = (size_t)p.t_rows * C;
    __nv_bfloat16* tout = reinterpret_cast<__nv_bfloat16*>(p.t_ops) + trow0 * C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = limit > kDrainLimitNs ? limit : kDrainLimitNs;
    if (blockIdx.x >= nch) return;

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        fence_barrier_init();
    }
    // the blocks above the diagonal of L and T are never written: zero them once
    for (int i = tid; i < C * C; i += kTpThreads) {
        const int r = i >> 6, c = i & 63;
        if ((c >> 4) > (r >> 4)) sl[r * kTpLd + c] = 0.f;
    }
    __syncthreads();

    int issued = 0;   // thread 0: copies issued
    auto issue_k = [&](int c) {
        const int t0 = (int)(job.tok_begin + beg[c]);
        unsigned char* dst = smem + TP_K;
        proxy_fence();
        mbar_arrive_expect_tx(&bar[0], 16384u);
        tma_load_3d(dst, &p.tm_k, 0, h, t0, &bar[0]);
        tma_load_3d(dst + 8192, &p.tm_k, 64, h, t0, &bar[0]);
        ++issued;
    };
    // warp 0: alpha, beta of a chunk (1 and 0 past its end), held in registers a chunk ahead
    float ga0 = 1.f, ga1 = 1.f, gb0 = 0.f, gb1 = 0.f;
    auto load_gates = [&](int c) {
        const int bc = beg[c];
        const int nc = (c + 1 < nch ? beg[c + 1] : len) - bc;
        const size_t g = (size_t)(job.tok_begin + bc) * (size_t)H + (size_t)h;
        ga0 = lane < nc ? __ldg(p.alpha + g + (size_t)lane * H) : 1.f;
        ga1 = lane + 32 < nc ? __ldg(p.alpha + g + (size_t)(lane + 32) * H) : 1.f;
        gb0 = lane < nc ? __ldg(p.beta + g + (size_t)lane * H) : 0.f;
        gb1 = lane + 32 < nc ? __ldg(p.beta + g + (size_t)(lane + 32) * H) : 0.f;
    };
    if (tid == 0) issue_k(blockIdx.x);
    if (warp == 0) load_gates(blockIdx.x);

    bool ok = true;
    for (int i = 0;; ++i) {
        const int c = blockIdx.x + i * gridDim.x;
        if (c >= nch) break;
        const int b = beg[c];
        const int n = (c + 1 < nch ? beg[c + 1] : len) - b;
        const bool more = c + (int)gridDim.x < nch;
        // gates of the chunk: gamma (the scan's rounding), beta gamma and 1/gamma; then the next chunk's
        if (warp == 0) {
            const float a0 = ga0, a1 = ga1, b0 = gb0, b1 = gb1;
            if (more) load_gates(c + gridDim.x);
            float g0, g1;
            gate_prefix(a0, a1, g0, g1, lane);
            sbg[lane] = b0 * g0;
            sbg[lane + 32] = b1 * g1;
            sgi[lane] = __frcp_rn(g0);
            sgi[lane + 32] = __frcp_rn(g1);
            sbe[lane] = b0;
            sbe[lane + 32] = b1;
        }
        // this chunk's K (bounded wait by one poller; then every thread observes the phase itself)
        {
            bool got = true;
            if (tid == 0) {
                const uint32_t par = (uint32_t)(i & 1);
                if (!mbar_try_wait(&bar[0], par)) {
                    const uint64_t t0 = global_ns();
                    while (!(got = mbar_try_wait(&bar[0], par)))
                        if (global_ns() - t0 > limit) break;
                }
            }
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            mbar_try_wait(&bar[0], (uint32_t)(i & 1));
        }
        const uint32_t kb = kbase0;
        unsigned char* kp = smem + TP_K;
        if (n < C) {   // rows past the chunk belong to later tokens: zero them
            const int nz = C - n;
            for (int e = tid; e < 2 * nz * 8; e += kTpThreads) {
                const int seg = e & 7, rz = (e >> 3) % nz, part = (e >> 3) / nz;
                *reinterpret_cast<uint4*>(kp + part * 8192 + (n + rz) * 128 + seg * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();

        // ---- G = K K^T on or below the diagonal 16-blocks, turned into L (zero on and above the diagonal):
        //      warps 0, 1 take row blocks 0 and 3, warps 2, 3 row blocks 1 and 2; warp parity = n8 half ----
        {
            const int nh = warp & 1;
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                const int rb = warp < 2 ? (pass == 0 ? 3 : 0) : (pass == 0 ? 2 : 1);
                float acc[4][4];
#pragma unroll
                for (int cb = 0; cb < 4; ++cb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[cb][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a[4];
                    ldsm_x4(k_addr(kb, 16 * rb + (lane & 7) + ((lane >> 3) & 1) * 8, 16 * ks + (lane >> 4) * 8), a);
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        if (cb > rb) continue;
                        uint32_t b0, b1;
                        ldsm_x2(k_addr(kb, 16 * cb + 8 * nh + (lane & 7), 16 * ks + ((lane >> 3) & 1) * 8), b0, b1);
                        mma_bf16_16816(acc[cb], a, b0, b1);
                    }
                }
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    if (cb > rb) continue;
                    const int s0 = 16 * cb + 8 * nh + 2 * t4;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int t = 16 * rb + g8 + 8 * hh;
                        const float f = sbg[t];
                        sl[t * kTpLd + s0] = s0 < t ? f * sgi[s0] * acc[cb][2 * hh] : 0.f;
                        sl[t * kTpLd + s0 + 1] = s0 + 1 < t ? f * sgi[s0 + 1] * acc[cb][2 * hh + 1] : 0.f;
                    }
                }
            }
        }
        __syncthreads();
        if (tid == 0 && more) issue_k(c + gridDim.x);   // K K^T is done: the buffer takes the next chunk's K
        // ---- the four 16x16 diagonal blocks of T by forward substitution: warp w, block w, lane = column ----
        {
            const int jc = lane & 15;
            const float* Lb = sl + (16 * warp) * kTpLd + 16 * warp;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s2 = 0; s2 < r; ++s2) acc[s2 & 3] = fmaf(Lb[r * kTpLd + s2], x[s2], acc[s2 & 3]);
                x[r] = ((r == jc) ? 1.f : 0.f) - ((acc[0] + acc[1]) + (acc[2] + acc[3]));
            }
            __syncwarp();
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) sl[(16 * warp + r) * kTpLd + 16 * warp + jc] = x[r];
            }
        }
        __syncthreads();
        // ---- level A: T_ib,jb = -T_ib,ib (L_ib,jb T_jb,jb) for (jb, ib) = (0, 1) (warps 0, 1) and (2, 3)
        //      (warps 2, 3); warp parity = 8-column half ----
        {
            const int pr = warp >> 1, hf = warp & 1, jb = 2 * pr, ib = jb + 1;
            float* yp = sy + pr * 256;   // [16][16]
            float y[4] = {0.f, 0.f, 0.f, 0.f}, yc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16x3(y, yc, sl + (16 * ib) * kTpLd + 16 * jb, kTpLd, sl + (16 * jb) * kTpLd + 16 * jb + 8 * hf, kTpLd,
                       g8, t4);
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] += yc[e];
            yp[g8 * 16 + 8 * hf + 2 * t4] = y[0];
            yp[g8 * 16 + 8 * hf + 2 * t4 + 1] = y[1];
            yp[(g8 + 8) * 16 + 8 * hf + 2 * t4] = y[2];
            yp[(g8 + 8) * 16 + 8 * hf + 2 * t4 + 1] = y[3];
            __syncthreads();   // every read of L_ib,jb is done before T_ib,jb overwrites it
            float xx[4] = {0.f, 0.f, 0.f, 0.f}, xc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16x3(xx, xc, sl + (16 * ib) * kTpLd + 16 * ib, kTpLd, yp + 8 * hf, 16, g8, t4);
            float* dst = sl + (16 * ib) * kTpLd + 16 * jb + 8 * hf;
            dst[g8 * kTpLd + 2 * t4] = -(xx[0] + xc[0]);
            dst[g8 * kTpLd + 2 * t4 + 1] = -(xx[1] + xc[1]);
            dst[(g8 + 8) * kTpLd + 2 * t4] = -(xx[2] + xc[2]);
            dst[(g8 + 8) * kTpLd + 2 * t4 + 1] = -(xx[3] + xc[3]);
        }
        __syncthreads();
        // ---- level B: T_BA = -T_BB (L_BA T_AA) for the lower-left 32-block; warp w = columns 8w .. 8w + 7 ----
        {
            float y[2][4], yc[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) y[mt][e] = yc[mt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                if (16 * ks + 15 < 8 * warp) continue;   // rows of T_AA above column 8w are zero
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
                    mma_bf16x3(y[mt], yc[mt], sl + (32 + 16 * mt) * kTpLd + 16 * ks, kTpLd,
                               sl + (16 * ks) * kTpLd + 8 * warp, kTpLd, g8, t4);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float* yr = sy + (16 * mt) * 33 + 8 * warp + 2 * t4;
                yr[g8 * 33] = y[mt][0] + yc[mt][0];
                yr[g8 * 33 + 1] = y[mt][1] + yc[mt][1];
                yr[(g8 + 8) * 33] = y[mt][2] + yc[mt][2];
                yr[(g8 + 8) * 33 + 1] = y[mt][3] + yc[mt][3];
            }
            __syncthreads();   // every read of L_BA is done before T_BA overwrites it
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float xx[4] = {0.f, 0.f, 0.f, 0.f}, xc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    if (ks > mt) continue;   // T_BB is zero above its diagonal
                    mma_bf16x3(xx, xc, sl + (32 + 16 * mt) * kTpLd + 32 + 16 * ks, kTpLd, sy + (16 * ks) * 33 + 8 * warp,
                               33, g8, t4);
                }
                float* dst = sl + (32 + 16 * mt) * kTpLd + 8 * warp + 2 * t4;
                dst[g8 * kTpLd] = -(xx[0] + xc[0]);
                dst[g8 * kTpLd + 1] = -(xx[1] + xc[1]);
                dst[(g8 + 8) * kTpLd] = -(xx[2] + xc[2]);
                dst[(g8 + 8) * kTpLd + 1] = -(xx[3] + xc[3]);
            }
        }
        __syncthreads();
        // ---- rows 0 .. n-1 of T diag(beta gamma) and T diag(beta), split x = hi + lo into bf16, to their
        //      tokens' rows of the four planes; 8 columns per item ----
        for (int e = tid; e < n * 8; e += kTpThreads) {
            const int r = e >> 3, c0 = 8 * (e & 7);
            const float4 x0 = *reinterpret_cast<const float4*>(sl + r * kTpLd + c0);
            const float4 x1 = *reinterpret_cast<const float4*>(sl + r * kTpLd + c0 + 4);
            const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int s0 = c0 + 2 * q;
                split_pair(x[2 * q] * sbg[s0], x[2 * q + 1] * sbg[s0 + 1], h1[q], l1[q]);
                split_pair(x[2 * q] * sbe[s0], x[2 * q + 1] * sbe[s0 + 1], h2[q], l2[q]);
            }
            __nv_bfloat16* dst = tout + (size_t)(b + r) * C + c0;
            *reinterpret_cast<uint4*>(dst) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
            *reinterpret_cast<uint4*>(dst + plane) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
            *reinterpret_cast<uint4*>(dst + 2 * plane) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            *reinterpret_cast<uint4*>(dst + 3 * plane) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
        }
        __syncthreads();   // T and the K buffer are free for the next chunk
    }
    if (!ok && tid == 0) {
        // a copy may still be in flight into the buffer: wait for it (bounded) before leaving
        if (issued > 0) drain_phase(&bar[0], (uint32_t)((issued - 1) & 1), drain_limit);
        atomicOr(p.status, STATUS_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_schedule(const Params& p, int n_streams, cudaStream_t stream) {
    if (n_streams <= 0) return cudaSuccess;
    schedule_kernel<<<n_streams, kSchedThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tprep(const Params& p, int n_streams, cudaStream_t stream) {
    if (n_streams <= 0) return cudaSuccess;
    static std::atomic<int> optin[kMaxOptinDevices];
    static std::atomic<int> slots_of[kMaxOptinDevices];   // resident blocks on the whole device, once known
    cudaError_t e = smem_optin(reinterpret_cast<const void*>(tprep_kernel), kTpSmemBytes, optin);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int slots = (dev >= 0 && dev < kMaxOptinDevices) ? slots_of[dev].load() : 0;
    if (slots <= 0) {
        int sms = 0, per_sm = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tprep_kernel, kTpThreads, kTpSmemBytes)) !=
            cudaSuccess)
            return e;
        slots = sms * (per_sm > 0 ? per_sm : 1);
        if (dev >= 0 && dev < kMaxOptinDevices) slots_of[dev].store(slots);
    }
    // one wave: the chunks of a (job, head) are dealt round robin to its blocks
    const int per_stream = slots / n_streams > 1 ? slots / n_streams : 1;
    const dim3 grid((unsigned)per_stream, (unsigned)n_streams);
    tprep_kernel<<<grid, kTpThreads, kTpSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
