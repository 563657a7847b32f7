// gdn_api.cu - host side of the C ABI: argument validation, the exact index
// plan (replay start, checkpoint selection), the ragged job table (longest job
// first), TMA descriptors and kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/gdn_scan.h"
#include "gdn_chunk.cuh"
#include "gdn_chunk_tc.cuh"
#include "gdn_group.cuh"
#include "gdn_kernel.cuh"

#define GDN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int32_t> g_stall_after{-1};
constexpr size_t kWorkspaceBytes = 256;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_d(int d) { return d == 32 || d == 64 || d == 128; }

// [T, H, d] stream, box (box_x, 1, box_t)
bool make_stream_map(CUtensorMap* m, const void* base, bool bf16, int64_t T, int H, int d, int box_x,
                     int box_t = gdn::kChunk, bool swizzle128 = false) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const size_t es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)std::max<int64_t>(T, 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(d * es), (cuuint64_t)((size_t)H * d * es)};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1u, (cuuint32_t)box_t};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool chunked_ok(const gdn_problem* p) {
    return p->d_k == gdn::chunk::D && p->d_v == gdn::chunk::D && p->qkv_dtype == GDN_BF16;
}

bool use_chunked(const gdn_problem* p) { return p->algo != GDN_ALGO_PER_TOKEN && chunked_ok(p); }

// Common validation of the problem description; fills seq lengths.
gdn_status check_problem(const gdn_problem* p, std::vector<int64_t>& lens) {
    if (!p || !p->cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (p->num_seqs < 1 || p->num_heads < 1 || p->d_k < 1 || p->d_v < 1) return GDN_ERR_INVALID_ARG;
    if ((p->qkv_dtype != GDN_F32 && p->qkv_dtype != GDN_BF16) || (p->out_dtype != GDN_F32 && p->out_dtype != GDN_BF16))
        return GDN_ERR_INVALID_ARG;
    if (p->algo != GDN_ALGO_AUTO && p->algo != GDN_ALGO_PER_TOKEN && p->algo != GDN_ALGO_CHUNKED &&
        p->algo != GDN_ALGO_CHUNKED_MMA && p->algo != GDN_ALGO_CHUNKED_TWO_PASS)
        return GDN_ERR_INVALID_ARG;
    if (!supported_d(p->d_k) || !supported_d(p->d_v)) return GDN_ERR_UNSUPPORTED;
    if ((p->algo == GDN_ALGO_CHUNKED || p->algo == GDN_ALGO_CHUNKED_MMA || p->algo == GDN_ALGO_CHUNKED_TWO_PASS) &&
        !chunked_ok(p))
        return GDN_ERR_UNSUPPORTED;
    if (p->cu_seqlens[0] != 0) return GDN_ERR_INVALID_ARG;
    lens.resize(p->num_seqs);
    for (int b = 0; b < p->num_seqs; ++b) {
        const int64_t n = p->cu_seqlens[b + 1] - p->cu_seqlens[b];
        if (n < 0) return GDN_ERR_INVALID_ARG;
        lens[b] = n;
    }
    const int64_t T = p->cu_seqlens[p->num_seqs];
    if (T >= ((int64_t)1 << 31) - gdn::kChunk) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)p->num_heads * p->d_v * p->d_k > ((int64_t)1 << 40)) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)p->num_heads > (1 << 20)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

gdn_status check_streams(const gdn_problem* p, const void* q, const void* k, const void* v, const float* alpha,
                         const float* beta, bool need_q, bool need_any) {
    if (!need_any) return GDN_OK;
    if (!k || !v || !alpha || !beta || (need_q && !q)) return GDN_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || (need_q && !aligned(q, 16))) return GDN_ERR_INVALID_ARG;
    if (!aligned(alpha, 4) || !aligned(beta, 4)) return GDN_ERR_INVALID_ARG;
    (void)p;
    return GDN_OK;
}

gdn_status check_workspace(void* ws, size_t bytes) {
    if (!ws || bytes < kWorkspaceBytes || !aligned(ws, 16)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

// Workspace of the two-pass chunked path: after the status word, the chunk counts [streams], the chunk
// starts [rows] and the T operands [4][rows][64] bf16, where rows = sum over the call's ranges of len x H.
struct TwoPassLayout {
    size_t cnt_off, beg_off, t_off, total;
};
constexpr int64_t kMaxTwoPassRows = ((int64_t)1 << 29) - gdn::tc::C;   // 4 planes of rows keep copy coordinates in int32
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
TwoPassLayout two_pass_layout(int64_t rows, int64_t streams) {
    TwoPassLayout l;
    l.cnt_off = kWorkspaceBytes;
    l.beg_off = round_up(l.cnt_off + 4 * (size_t)streams, 256);
    l.t_off = round_up(l.beg_off + 4 * (size_t)rows, 256);
    l.total = l.t_off + (size_t)rows * 4 * gdn::tc::C * 2;
    return l;
}

// Validate one sequence's checkpoint list: strictly increasing in [1, n].
bool ckpts_valid(const int64_t* c, int64_t M, int64_t n) {
    for (int64_t i = 0; i < M; ++i) {
        if (c[i] < 1 || c[i] > n) return false;
        if (i > 0 && c[i] <= c[i - 1]) return false;
    }
    return true;
}

struct HostJob {
    gdn::Job job;
    std::vector<gdn::Ckpt> ckpts;
};

struct LaunchSpec {
    const gdn_problem* p;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    void* o;
    float* ckpt_states;
    unsigned int* status;
    bool readout;
    bool twin;
    size_t ws_bytes;   // bytes at status (the caller's workspace)
};

// rows and streams of the two-pass path for a job list (the exact twins counted when `twin`)
void two_pass_extent(const LaunchSpec& L, const std::vector<HostJob>& jobs, int64_t& rows, int64_t& streams) {
    const int64_t H = L.p->num_heads, f = L.twin ? 2 : 1;
    rows = 0;
    for (const HostJob& j : jobs) rows += (int64_t)j.job.len * H * f;
    streams = (int64_t)jobs.size() * H * f;
}
// the T kernel's grid has a block row per (job, head) of a launch: at most 65535
bool two_pass_supported(const LaunchSpec& L) { return (int64_t)L.p->num_heads * gdn::kMaxJobs <= 65535; }
bool two_pass_fits(const LaunchSpec& L, const std::vector<HostJob>& jobs) {
    int64_t rows, streams;
    two_pass_extent(L, jobs, rows, streams);
    if (!two_pass_supported(L) || rows > kMaxTwoPassRows) return false;
    return L.ws_bytes >= two_pass_layout(rows, streams).total;
}
// GDN_ALGO_CHUNKED_TWO_PASS with too small a workspace is an invalid argument, found before anything is enqueued
gdn_status check_two_pass(const LaunchSpec& L, const std::vector<HostJob>& jobs) {
    if (L.p->algo != GDN_ALGO_CHUNKED_TWO_PASS) return GDN_OK;
    if (!two_pass_supported(L)) return GDN_ERR_UNSUPPORTED;
    return two_pass_fits(L, jobs) ? GDN_OK : GDN_ERR_INVALID_ARG;
}

// Batch jobs into parameter blocks and launch each with `launch(params, n_jobs)`.
template <class F>
gdn_status launch_batches(gdn::Params& prm, std::vector<HostJob>& jobs, F&& launch) {
    size_t i = 0;
    while (i < jobs.size()) {
        int nj = 0, nc = 0;
        while (i + nj < jobs.size() && nj < gdn::kMaxJobs &&
               nc + (int)jobs[i + nj].ckpts.size() <= gdn::kMaxCkpts) {
            gdn::Job j = jobs[i + nj].job;
            j.ck_begin = nc;
            j.ck_count = (int32_t)jobs[i + nj].ckpts.size();
            for (const gdn::Ckpt& c : jobs[i + nj].ckpts) prm.ckpts[nc++] = c;
            prm.jobs[nj++] = j;
        }
        if (nj == 0) return GDN_ERR_UNSUPPORTED;  // one job with more checkpoints than a launch holds
        prm.n_jobs = nj;
        if (launch(prm, nj) != cudaSuccess) return GDN_ERR_CUDA;
        i += nj;
    }
    return GDN_OK;
}

// Chunked tensor-core paths (d_k = d_v = 128, bf16): one CTA per (job, head); tcgen05 by default,
// warp-level mma.sync for GDN_ALGO_CHUNKED_MMA.
gdn_status run_jobs_chunked(const LaunchSpec& L, std::vector<HostJob>& jobs, cudaStream_t stream) {
    const gdn_problem* p = L.p;
    const int H = p->num_heads;
    if ((int64_t)H * gdn::kMaxJobs > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    // the exact twin runs as a second job over the same tokens from S_a
    if (L.twin) {
        const size_t n = jobs.size();
        for (size_t i = 0; i < n; ++i) {
            HostJob t = jobs[i];
            t.job.s0 = jobs[i].job.s0_twin;
            t.job.s_final = jobs[i].job.s_final_twin;
            t.job.o = nullptr;
            t.job.s0_twin = nullptr;
            t.job.s_final_twin = nullptr;
            jobs.push_back(t);
        }
    }
    std::stable_sort(jobs.begin(), jobs.end(),
                     [](const HostJob& a, const HostJob& b) { return a.job.len > b.job.len; });
    const int64_t T = p->cu_seqlens[p->num_seqs];
    auto prm = std::make_unique<gdn::Params>();
    std::memset(prm.get(), 0, sizeof(gdn::Params));
    const int D = gdn::chunk::D, C = gdn::chunk::C;
    // two passes when asked for, or by default when the workspace holds T of every chunk
    const bool warp_mma = p->algo == GDN_ALGO_CHUNKED_MMA;
    bool two_pass = false;
    if (p->algo == GDN_ALGO_CHUNKED_TWO_PASS || p->algo == GDN_ALGO_AUTO) {
        LaunchSpec whole = L;
        whole.twin = false;   // the twins are in `jobs` now
        two_pass = two_pass_fits(whole, jobs);
        if (p->algo == GDN_ALGO_CHUNKED_TWO_PASS && !two_pass) return GDN_ERR_INVALID_ARG;
    }
    if (two_pass) {
        int64_t rows = 0;
        for (HostJob& j : jobs) {
            j.job.t_row0 = (int32_t)rows;
            rows += (int64_t)j.job.len * H;
        }
        const TwoPassLayout lay = two_pass_layout(rows, (int64_t)jobs.size() * H);
        unsigned char* ws = reinterpret_cast<unsigned char*>(L.status);
        prm->chunk_cnt = reinterpret_cast<int32_t*>(ws + lay.cnt_off);
        prm->chunk_beg = reinterpret_cast<int32_t*>(ws + lay.beg_off);
        prm->t_ops = ws + lay.t_off;
        prm->t_rows = (int32_t)std::max<int64_t>(rows, 1);
        EncodeTiledFn enc = encode_fn();
        if (!enc) return GDN_ERR_CUDA;
        cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(4 * (int64_t)prm->t_rows)};
        cuuint64_t strides[1] = {(cuuint64_t)(C * 2)};
        cuuint32_t box[2] = {(cuuint32_t)C, (cuuint32_t)C};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(&prm->tm_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, prm->t_ops, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GDN_ERR_CUDA;
    }
    bool maps = true;
    if (L.k) maps = maps && make_stream_map(&prm->tm_k, L.k, true, T, H, D, 64, C, true);
    if (L.q) maps = maps && make_stream_map(&prm->tm_q, L.q, true, T, H, D, 64, C, true);
    if (L.v) maps = maps && make_stream_map(&prm->tm_v, L.v, true, T, H, D, 64, C, true);
    if (!maps) return GDN_ERR_CUDA;
    // without a readout the q tiles are still staged: point them at k
    if (!L.q && L.k) prm->tm_q = prm->tm_k;
    prm->alpha = L.alpha;
    prm->beta = L.beta;
    prm->o_vec16 = 1;
    for (const HostJob& j : jobs)
        if (j.job.o && !aligned(j.job.o, 16)) prm->o_vec16 = 0;
    prm->ckpt_states = L.ckpt_states;
    prm->status = L.status;
    prm->wait_limit_ns = g_wait_ns.load();
    prm->stall_after = g_stall_after.load();
    prm->H = H;
    prm->dv = D;
    const bool out_bf16 = p->out_dtype == GDN_BF16;
    return launch_batches(*prm, jobs, [&](const gdn::Params& pr, int nj) -> cudaError_t {
        const int grid = nj * H;
        if (two_pass) {
            cudaError_t e = gdn::tc::launch_schedule(pr, grid, stream);
            if (e == cudaSuccess) e = gdn::tc::launch_tprep(pr, grid, stream);
            if (e == cudaSuccess) e = gdn::tc::launch(pr, grid, L.readout, out_bf16, true, stream);
            return e;
        }
        if (!warp_mma) return gdn::tc::launch(pr, grid, L.readout, out_bf16, false, stream);
        if (L.readout)
            return out_bf16 ? gdn::chunk::launch_chunk<true, true>(pr, grid, stream)
                            : gdn::chunk::launch_chunk<false, true>(pr, grid, stream);
        return gdn::chunk::launch_chunk<false, false>(pr, grid, stream);
    });
}

// Sort jobs longest first and launch them in batches that fit one parameter block.
gdn_status run_jobs(const LaunchSpec& L, std::vector<HostJob>& jobs, cudaStream_t stream) {
    const gdn_problem* p = L.p;
    if (use_chunked(p)) return run_jobs_chunked(L, jobs, stream);
    const int H = p->num_heads, dv = p->d_v, dk = p->d_k;
    const bool in_bf16 = p->qkv_dtype == GDN_BF16;
    const bool out_bf16 = p->out_dtype == GDN_BF16;
    const int wr = gdn::slots_per_warp(dk) / (L.twin ? 2 : 1);   // real rows per consumer warp
    const int nw = std::min(gdn::kMaxConsumerWarps, dv / wr);
    const int rows = nw * wr;
    const int ctas_per_head = dv / rows;
    if (nw < 1 || rows * ctas_per_head != dv) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)H * ctas_per_head * gdn::kMaxJobs > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;

    std::stable_sort(jobs.begin(), jobs.end(),
                     [](const HostJob& a, const HostJob& b) { return a.job.len > b.job.len; });

    const int64_t T = p->cu_seqlens[p->num_seqs];
    auto prm = std::make_unique<gdn::Params>();
    std::memset(prm.get(), 0, sizeof(gdn::Params));
    // A map is encoded only for a stream that is given; the kernel issues no
    // copy for a job without tokens, and streams are validated non-NULL whenever
    // any job has tokens.
    bool maps = true;
    if (L.k) maps = maps && make_stream_map(&prm->tm_k, L.k, in_bf16, T, H, dk, dk);
    if (L.readout && L.q) maps = maps && make_stream_map(&prm->tm_q, L.q, in_bf16, T, H, dk, dk);
    if (L.v) maps = maps && make_stream_map(&prm->tm_v, L.v, in_bf16, T, H, dv, rows);
    if (!maps) return GDN_ERR_CUDA;
    prm->alpha = L.alpha;
    prm->beta = L.beta;
    prm->ckpt_states = L.ckpt_states;
    prm->status = L.status;
    prm->wait_limit_ns = g_wait_ns.load();
    prm->stall_after = g_stall_after.load();
    prm->H = H;
    prm->dv = dv;
    prm->nw = nw;
    prm->rows_per_cta = rows;
    prm->ctas_per_head = ctas_per_head;

    const int idx = (((in_bf16 ? 1 : 0) * 2 + (out_bf16 ? 1 : 0)) * 2 + (L.readout ? 1 : 0)) * 2 + (L.twin ? 1 : 0);
    gdn::LaunchFn fn = nullptr;
    switch (dk) {
        case 32: fn = gdn::launch_table<32>(idx); break;
        case 64: fn = gdn::launch_table<64>(idx); break;
        case 128: fn = gdn::launch_table<128>(idx); break;
        default: return GDN_ERR_UNSUPPORTED;
    }
    if (!fn) return GDN_ERR_UNSUPPORTED;
    const size_t smem = gdn::smem_bytes(dk, in_bf16 ? 2 : 4, rows, L.readout);

    return launch_batches(*prm, jobs, [&](const gdn::Params& pr, int nj) -> cudaError_t {
        return fn(pr, nj * H * ctas_per_head, smem, stream);
    });
}

}  // namespace

// ---------------------------------------------------------------------------------------
// host-only helpers
// ---------------------------------------------------------------------------------------
GDN_EXPORT gdn_status gdn_replay_plan(int64_t m, int32_t r_num, int32_t r_den, int64_t* a, int64_t* k) {
    if (!a || !k || m < 0 || m > ((int64_t)1 << 40) || r_den <= 0 || r_num < 0 || r_num > r_den)
        return GDN_ERR_INVALID_ARG;
    // k = ceil(r_num * m / r_den) in exact integers (no floating point)
    const int64_t prod = (int64_t)r_num * m;
    const int64_t q = prod / r_den;
    const int64_t kk = q + ((q * r_den != prod) ? 1 : 0);
    *k = kk;
    *a = m - kk;
    return GDN_OK;
}

GDN_EXPORT gdn_status gdn_select_ckpt(const int64_t* c, int32_t M, int64_t d, int32_t* j) {
    if (!j || M < 0 || (M > 0 && !c)) return GDN_ERR_INVALID_ARG;
    for (int32_t i = 1; i < M; ++i)
        if (c[i] <= c[i - 1]) return GDN_ERR_INVALID_ARG;
    // binary search for the last c_i <= d
    int32_t lo = 0, hi = M;  // answer in [lo-1, hi-1]
    while (lo < hi) {
        const int32_t mid = lo + (hi - lo) / 2;
        if (c[mid] <= d)
            lo = mid + 1;
        else
            hi = mid;
    }
    *j = lo - 1;
    return GDN_OK;
}

GDN_EXPORT size_t gdn_workspace_size(void) { return kWorkspaceBytes; }

GDN_EXPORT size_t gdn_workspace_size_two_pass(int64_t tokens, int32_t num_heads, int32_t num_ranges) {
    if (tokens < 0 || num_heads < 1 || num_ranges < 0) return 0;
    if (tokens > kMaxTwoPassRows / num_heads) return 0;
    return two_pass_layout(tokens * num_heads, (int64_t)num_ranges * num_heads).total;
}

GDN_EXPORT void gdn_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

GDN_EXPORT void gdn_debug_stall_after(int32_t chunks) { g_stall_after.store(chunks < 0 ? -1 : chunks); }

GDN_EXPORT const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
    }
    return "GDN_ERR_UNKNOWN";
}

GDN_EXPORT gdn_status gdn_clear_status(void* workspace, size_t ws_bytes, gdn_stream_t stream) {
    gdn_status st = check_workspace(workspace, ws_bytes);
    if (st != GDN_OK) return st;
    return cudaMemsetAsync(workspace, 0, sizeof(unsigned int), (cudaStream_t)stream) == cudaSuccess ? GDN_OK
                                                                                                     : GDN_ERR_CUDA;
}

GDN_EXPORT gdn_status gdn_read_status(const void* workspace, size_t ws_bytes, gdn_stream_t stream) {
    gdn_status st = check_workspace(const_cast<void*>(workspace), ws_bytes);
    if (st != GDN_OK) return st;
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    return (word & gdn::STATUS_TIMEOUT) ? GDN_ERR_DEVICE_TIMEOUT : GDN_OK;
}

// ---------------------------------------------------------------------------------------
// prefill with sparse checkpoints
// ---------------------------------------------------------------------------------------
// Address of output row `row` of a [rows, H, d_v] buffer (nullptr when there is no buffer).
static void* out_row(void* o, const gdn_problem* p, int64_t row) {
    if (!o) return nullptr;
    const size_t es = p->out_dtype == GDN_BF16 ? 2 : 4;
    return static_cast<unsigned char*>(o) + (size_t)row * (size_t)p->num_heads * (size_t)p->d_v * es;
}

// Every check of a prefill and its job table, nothing enqueued.
static gdn_status prefill_prepare(const gdn_problem* p, const void* q, const void* k, const void* v,
                                  const float* alpha, const float* beta, const float* S0, void* o, float* S_final,
                                  const int64_t* ckpt_pos, const int64_t* cu_ckpt, float* ckpt_states,
                                  void* workspace, size_t ws_bytes, std::vector<HostJob>& jobs, LaunchSpec& L) {
    std::vector<int64_t> lens;
    gdn_status st = check_problem(p, lens);
    if (st != GDN_OK) return st;
    const int64_t T = p->cu_seqlens[p->num_seqs];
    if ((st = check_streams(p, q, k, v, alpha, beta, o != nullptr, T > 0)) != GDN_OK) return st;
    if ((st = check_workspace(workspace, ws_bytes)) != GDN_OK) return st;
    if (!S_final || !aligned(S_final, 16) || (S0 && !aligned(S0, 16))) return GDN_ERR_INVALID_ARG;
    if (o && !aligned(o, p->out_dtype == GDN_BF16 ? 2 : 4)) return GDN_ERR_INVALID_ARG;
    const int B = p->num_seqs;
    int64_t n_ck = 0;
    if (cu_ckpt) {
        if (cu_ckpt[0] != 0) return GDN_ERR_INVALID_ARG;
        for (int b = 0; b < B; ++b)
            if (cu_ckpt[b + 1] < cu_ckpt[b]) return GDN_ERR_INVALID_ARG;
        n_ck = cu_ckpt[B];
        if (n_ck > 0 && (!ckpt_pos || !ckpt_states || !aligned(ckpt_states, 16))) return GDN_ERR_INVALID_ARG;
        for (int b = 0; b < B; ++b)
            if (!ckpts_valid(ckpt_pos + cu_ckpt[b], cu_ckpt[b + 1] - cu_ckpt[b], lens[b])) return GDN_ERR_INVALID_ARG;
        if (n_ck >= ((int64_t)1 << 23)) return GDN_ERR_UNSUPPORTED;
    }
    const size_t D = (size_t)p->num_heads * p->d_v * p->d_k;
    jobs.assign(B, HostJob{});
    for (int b = 0; b < B; ++b) {
        gdn::Job& j = jobs[b].job;
        std::memset(&j, 0, sizeof(j));
        j.tok_begin = p->cu_seqlens[b];
        j.len = (int32_t)lens[b];
        j.o = out_row(o, p, p->cu_seqlens[b]);
        j.s0 = S0 ? S0 + (size_t)b * D : nullptr;
        j.s_final = S_final + (size_t)b * D;
        if (cu_ckpt)
            for (int64_t i = cu_ckpt[b]; i < cu_ckpt[b + 1]; ++i)
                jobs[b].ckpts.push_back(gdn::Ckpt{(int32_t)ckpt_pos[i], (int32_t)i});
    }
    L = LaunchSpec{p, q, k, v, alpha, beta, o, ckpt_states, static_cast<unsigned int*>(workspace), o != nullptr,
                   false, ws_bytes};
    return check_two_pass(L, jobs);
}

GDN_EXPORT gdn_status gdn_prefill_ckpt(const gdn_problem* p, const void* q, const void* k, const void* v,
                                       const float* alpha, const float* beta, const float* S0, void* o,
                                       float* S_final, const int64_t* ckpt_pos, const int64_t* cu_ckpt,
                                       float* ckpt_states, void* workspace, size_t ws_bytes, gdn_stream_t stream) {
    std::vector<HostJob> jobs;
    LaunchSpec L{};
    gdn_status st = prefill_prepare(p, q, k, v, alpha, beta, S0, o, S_final, ckpt_pos, cu_ckpt, ckpt_states,
                                    workspace, ws_bytes, jobs, L);
    if (st != GDN_OK) return st;
    return run_jobs(L, jobs, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------------------
// resume from the deepest checkpoint at or below d
// ---------------------------------------------------------------------------------------
// Every check of a resume, its index plan (chosen checkpoint and packed output offset per probe) and
// its job table, nothing enqueued.
static gdn_status resume_prepare(const gdn_problem* p, const void* q, const void* k, const void* v,
                                 const float* alpha, const float* beta, const float* S0, const float* ckpt_states,
                                 const int64_t* ckpt_pos, const int64_t* cu_ckpt, int32_t num_probes,
                                 const int32_t* probe_seq, const int64_t* probe_depth, float* S_out, void* o_out,
                                 void* workspace, size_t ws_bytes, std::vector<HostJob>& jobs, LaunchSpec& L,
                                 std::vector<int64_t>& chosen, std::vector<int64_t>& offs) {
    std::vector<int64_t> lens;
    gdn_status st = check_problem(p, lens);
    if (st != GDN_OK) return st;
    if (num_probes < 0) return GDN_ERR_INVALID_ARG;
    if (num_probes > 0 && (!probe_seq || !probe_depth || !S_out || !aligned(S_out, 16))) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(workspace, ws_bytes)) != GDN_OK) return st;
    if (S0 && !aligned(S0, 16)) return GDN_ERR_INVALID_ARG;
    if (o_out && !aligned(o_out, p->out_dtype == GDN_BF16 ? 2 : 4)) return GDN_ERR_INVALID_ARG;
    const int B = p->num_seqs;
    if (cu_ckpt) {
        if (cu_ckpt[0] != 0) return GDN_ERR_INVALID_ARG;
        for (int b = 0; b < B; ++b)
            if (cu_ckpt[b + 1] < cu_ckpt[b]) return GDN_ERR_INVALID_ARG;
        if (cu_ckpt[B] > 0 && (!ckpt_pos || !ckpt_states || !aligned(ckpt_states, 16))) return GDN_ERR_INVALID_ARG;
        for (int b = 0; b < B; ++b)
            if (!ckpts_valid(ckpt_pos + cu_ckpt[b], cu_ckpt[b + 1] - cu_ckpt[b], lens[b])) return GDN_ERR_INVALID_ARG;
    }
    const size_t D = (size_t)p->num_heads * p->d_v * p->d_k;
    jobs.assign(num_probes, HostJob{});
    chosen.assign(num_probes, 0);
    offs.assign(num_probes + 1, 0);
    int64_t total = 0;
    for (int32_t i = 0; i < num_probes; ++i) {
        const int s = probe_seq[i];
        const int64_t d = probe_depth[i];
        if (s < 0 || s >= B || d < 0 || d > lens[s]) return GDN_ERR_INVALID_ARG;
        int32_t j = -1;
        if (cu_ckpt && cu_ckpt[s + 1] > cu_ckpt[s]) {
            if (gdn_select_ckpt(ckpt_pos + cu_ckpt[s], (int32_t)(cu_ckpt[s + 1] - cu_ckpt[s]), d, &j) != GDN_OK)
                return GDN_ERR_INVALID_ARG;
        }
        const int64_t c = j < 0 ? 0 : ckpt_pos[cu_ckpt[s] + j];
        chosen[i] = c;
        offs[i] = total;
        total += d - c;
        gdn::Job& jb = jobs[i].job;
        std::memset(&jb, 0, sizeof(jb));
        jb.tok_begin = p->cu_seqlens[s] + c;
        jb.len = (int32_t)(d - c);
        jb.o = out_row(o_out, p, offs[i]);
        jb.s0 = j < 0 ? (S0 ? S0 + (size_t)s * D : nullptr) : ckpt_states + (size_t)(cu_ckpt[s] + j) * D;
        jb.s_final = S_out + (size_t)i * D;
    }
    offs[num_probes] = total;
    if ((st = check_streams(p, q, k, v, alpha, beta, o_out != nullptr, total > 0)) != GDN_OK) return st;
    L = LaunchSpec{p, q, k, v, alpha, beta, o_out, nullptr, static_cast<unsigned int*>(workspace), o_out != nullptr,
                   false, ws_bytes};
    return check_two_pass(L, jobs);
}

GDN_EXPORT gdn_status gdn_resume_from_ckpt(const gdn_problem* p, const void* q, const void* k, const void* v,
                                           const float* alpha, const float* beta, const float* S0,
                                           const float* ckpt_states, const int64_t* ckpt_pos,
                                           const int64_t* cu_ckpt, int32_t num_probes, const int32_t* probe_seq,
                                           const int64_t* probe_depth, float* S_out, void* o_out,
                                           int64_t* chosen_pos, int64_t* o_offsets, void* workspace,
                                           size_t ws_bytes, gdn_stream_t stream) {
    std::vector<HostJob> jobs;
    LaunchSpec L{};
    std::vector<int64_t> chosen, offs;
    gdn_status st = resume_prepare(p, q, k, v, alpha, beta, S0, ckpt_states, ckpt_pos, cu_ckpt, num_probes, probe_seq,
                                   probe_depth, S_out, o_out, workspace, ws_bytes, jobs, L, chosen, offs);
    if (st != GDN_OK) return st;
    if (chosen_pos) std::copy(chosen.begin(), chosen.end(), chosen_pos);
    if (o_offsets) std::copy(offs.begin(), offs.end(), o_offsets);
    if (num_probes == 0) return GDN_OK;
    return run_jobs(L, jobs, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------------------
// Tail-Replay
// ---------------------------------------------------------------------------------------
// Tail replay with a given tail length k_b per sequence (rows [m_b - k_b, m_b)): every check and the job
// table, nothing enqueued.
static gdn_status replay_prepare(const gdn_problem* p, const void* q, const void* k, const void* v,
                                 const float* alpha, const float* beta, const int64_t* m, const int64_t* kv,
                                 const float* S_a, float* S_hat, float* S_exact, void* o, void* workspace,
                                 size_t ws_bytes, std::vector<HostJob>& jobs, LaunchSpec& L) {
    std::vector<int64_t> lens;
    gdn_status st = check_problem(p, lens);
    if (st != GDN_OK) return st;
    if (!m || !kv || !S_hat || !aligned(S_hat, 16)) return GDN_ERR_INVALID_ARG;
    if ((S_a == nullptr) != (S_exact == nullptr)) return GDN_ERR_INVALID_ARG;
    if (S_a && (!aligned(S_a, 16) || !aligned(S_exact, 16))) return GDN_ERR_INVALID_ARG;
    if (o && !aligned(o, p->out_dtype == GDN_BF16 ? 2 : 4)) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(workspace, ws_bytes)) != GDN_OK) return st;
    const int B = p->num_seqs;
    const size_t D = (size_t)p->num_heads * p->d_v * p->d_k;
    jobs.assign(B, HostJob{});
    int64_t total = 0;
    for (int b = 0; b < B; ++b) {
        if (m[b] < 0 || m[b] > lens[b] || kv[b] < 0 || kv[b] > m[b]) return GDN_ERR_INVALID_ARG;
        const int64_t a = m[b] - kv[b];
        total += kv[b];
        gdn::Job& j = jobs[b].job;
        std::memset(&j, 0, sizeof(j));
        j.tok_begin = p->cu_seqlens[b] + a;
        j.len = (int32_t)kv[b];
        j.o = out_row(o, p, p->cu_seqlens[b] + a);
        j.s0 = nullptr;
        j.s0_twin = S_a ? S_a + (size_t)b * D : nullptr;
        j.s_final = S_hat + (size_t)b * D;
        j.s_final_twin = S_exact ? S_exact + (size_t)b * D : nullptr;
    }
    if ((st = check_streams(p, q, k, v, alpha, beta, o != nullptr, total > 0)) != GDN_OK) return st;
    L = LaunchSpec{p, q, k, v, alpha, beta, o, nullptr, static_cast<unsigned int*>(workspace), o != nullptr,
                   S_a != nullptr, ws_bytes};
    return check_two_pass(L, jobs);
}

static gdn_status replay_k(const gdn_problem* p, const void* q, const void* k, const void* v, const float* alpha,
                           const float* beta, const int64_t* m, const int64_t* kv, const float* S_a, float* S_hat,
                           float* S_exact, void* o, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    std::vector<HostJob> jobs;
    LaunchSpec L{};
    gdn_status st = replay_prepare(p, q, k, v, alpha, beta, m, kv, S_a, S_hat, S_exact, o, workspace, ws_bytes,
                                   jobs, L);
    if (st != GDN_OK) return st;
    return run_jobs(L, jobs, stream);
}

static gdn_status plan_all(int B, const int64_t* m, int32_t r_num, int32_t r_den, std::vector<int64_t>& av,
                           std::vector<int64_t>& kv) {
    if (B < 1 || !m) return GDN_ERR_INVALID_ARG;
    av.resize(B);
    kv.resize(B);
    for (int b = 0; b < B; ++b)
        if (gdn_replay_plan(m[b], r_num, r_den, &av[b], &kv[b]) != GDN_OK) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

GDN_EXPORT gdn_status gdn_tail_replay(const gdn_problem* p, const void* q, const void* k, const void* v,
                                      const float* alpha, const float* beta, const int64_t* m, int32_t r_num,
                                      int32_t r_den, const float* S_a, float* S_hat, float* S_exact, void* o,
                                      int64_t* a_out, int64_t* k_out, void* workspace, size_t ws_bytes,
                                      gdn_stream_t stream) {
    if (!p) return GDN_ERR_INVALID_ARG;
    std::vector<int64_t> av, kv;
    gdn_status st = plan_all(p->num_seqs, m, r_num, r_den, av, kv);
    if (st != GDN_OK) return st;
    st = replay_k(p, q, k, v, alpha, beta, m, kv.data(), S_a, S_hat, S_exact, o, workspace, ws_bytes,
                  (cudaStream_t)stream);
    if (st == GDN_OK || st == GDN_ERR_CUDA) {
        if (a_out) std::copy(av.begin(), av.end(), a_out);
        if (k_out) std::copy(kv.begin(), kv.end(), k_out);
    }
    return st;
}

GDN_EXPORT gdn_status gdn_tail_replay_k(const gdn_problem* p, const void* q, const void* k, const void* v,
                                        const float* alpha, const float* beta, const int64_t* m,
                                        const int64_t* k_replay, const float* S_a, float* S_hat, float* S_exact,
                                        void* o, void* workspace, size_t ws_bytes, gdn_stream_t stream) {
    return replay_k(p, q, k, v, alpha, beta, m, k_replay, S_a, S_hat, S_exact, o, workspace, ws_bytes,
                    (cudaStream_t)stream);
}

GDN_EXPORT gdn_status gdn_tail_replay_overlap(const gdn_problem* p, const void* q, const void* k, const void* v,
                                              const float* alpha, const float* beta, const int64_t* m,
                                              int32_t r_num, int32_t r_den, const float* S_a, float* S_hat,
                                              float* S_exact, void* o, int64_t* a_out, int64_t* k_out,
                                              const void* kv_host, void* kv_dev, size_t kv_bytes, void* workspace,
                                              size_t ws_bytes, gdn_stream_t stream, gdn_stream_t copy_stream) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (kv_bytes > 0 && (!kv_host || !kv_dev)) return GDN_ERR_INVALID_ARG;
    std::vector<int64_t> av, kv;
    gdn_status st = plan_all(p->num_seqs, m, r_num, r_den, av, kv);
    if (st != GDN_OK) return st;
    // every check of the replay before anything is enqueued
    std::vector<HostJob> jobs;
    LaunchSpec L{};
    if ((st = replay_prepare(p, q, k, v, alpha, beta, m, kv.data(), S_a, S_hat, S_exact, o, workspace, ws_bytes, jobs,
                             L)) != GDN_OK)
        return st;
    const cudaStream_t cs = (cudaStream_t)stream, xs = (cudaStream_t)copy_stream;
    cudaEvent_t before = nullptr, copied = nullptr;
    if (kv_bytes > 0) {
        if (cudaEventCreateWithFlags(&before, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&copied, cudaEventDisableTiming) != cudaSuccess) {
            if (before) cudaEventDestroy(before);
            return GDN_ERR_CUDA;
        }
        // the copy waits for the caller's earlier work on `stream` (which may still use kv_dev), then runs
        // beside the replay
        bool ok = cudaEventRecord(before, cs) == cudaSuccess && cudaStreamWaitEvent(xs, before, 0) == cudaSuccess &&
                  cudaMemcpyAsync(kv_dev, kv_host, kv_bytes, cudaMemcpyHostToDevice, xs) == cudaSuccess &&
                  cudaEventRecord(copied, xs) == cudaSuccess;
        if (!ok) {
            cudaEventDestroy(before);
            cudaEventDestroy(copied);
            return GDN_ERR_CUDA;
        }
    }
    st = run_jobs(L, jobs, cs);
    if (kv_bytes > 0) {
        // later work on `stream` (the new suffix) sees the copied KV
        if (cudaStreamWaitEvent(cs, copied, 0) != cudaSuccess && st == GDN_OK) st = GDN_ERR_CUDA;
        cudaEventDestroy(before);
        cudaEventDestroy(copied);
    }
    if (st == GDN_OK || st == GDN_ERR_CUDA) {
        if (a_out) std::copy(av.begin(), av.end(), a_out);
        if (k_out) std::copy(kv.begin(), kv.end(), k_out);
    }
    return st;
}

// ---------------------------------------------------------------------------------------
// one serving step: prefills, resumes and tail replays in a single launch
// ---------------------------------------------------------------------------------------
// Two launch lanes per device for gdn_step: streams of the library's own, the long jobs' of the highest and the
// short jobs' of the lowest priority (so that the long jobs' CTAs are placed first whatever the order in which
// the two launches become ready), and the events that fork them from the caller's stream and join them back to
// it; made on the first call that needs them.
struct SideLane {
    cudaStream_t hi = nullptr, lo = nullptr;
    cudaEvent_t fork = nullptr, join_hi = nullptr, join_lo = nullptr;
    int sms = 0;
    bool ready = false;
};
static std::mutex g_side_mutex;
static SideLane g_side[gdn::kMaxOptinDevices];

static SideLane* side_lane() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gdn::kMaxOptinDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideLane& L = g_side[dev];
    if (!L.ready) {
        if (!L.sms && cudaDeviceGetAttribute(&L.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
        if (!L.hi && cudaStreamCreateWithPriority(&L.hi, cudaStreamNonBlocking, greatest) != cudaSuccess)
            return nullptr;
        if (!L.lo && cudaStreamCreateWithPriority(&L.lo, cudaStreamNonBlocking, least) != cudaSuccess) return nullptr;
        for (cudaEvent_t* e : {&L.fork, &L.join_hi, &L.join_lo})
            if (!*e && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        L.ready = true;
    }
    return &L;
}

// Jobs sorted longest first split into a head of long jobs whose CTAs (one per job and head) all fit on the
// SMs together and a tail of jobs at most a quarter of the previous one's length; 0 when there is no such split.
static size_t split_point(const std::vector<HostJob>& jobs, int64_t heads, int sms) {
    for (size_t b = 1; b < jobs.size(); ++b) {
        if ((int64_t)b * heads > sms) return 0;
        if ((int64_t)jobs[b].job.len * 4 <= (int64_t)jobs[b - 1].job.len) return b;
    }
    return 0;
}

static bool ranges_overlap(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
    if (!a || !b || a_bytes == 0 || b_bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

GDN_EXPORT gdn_status gdn_step(const gdn_problem* p, const void* q, const void* k, const void* v,
                               const float* alpha, const float* beta, const gdn_prefill_args* prefill,
                               const gdn_resume_args* resume, const gdn_replay_args* replay, void* workspace,
                               size_t ws_bytes, gdn_stream_t stream) {
    if (!p) return GDN_ERR_INVALID_ARG;
    std::vector<HostJob> all, part;
    LaunchSpec L{};
    gdn_status st = GDN_OK;
    bool readout = false;
    float* ckpt_out = nullptr;
    if (prefill) {
        if ((st = prefill_prepare(p, q, k, v, alpha, beta, prefill->S0, prefill->o, prefill->S_final,
                                  prefill->ckpt_pos, prefill->cu_ckpt, prefill->ckpt_states, workspace, ws_bytes,
                                  part, L)) != GDN_OK)
            return st;
        readout = readout || L.readout;
        ckpt_out = prefill->ckpt_states;
        all.insert(all.end(), part.begin(), part.end());
    }
    std::vector<int64_t> chosen, offs;
    if (resume) {
        if ((st = resume_prepare(p, q, k, v, alpha, beta, resume->S0, resume->ckpt_states, resume->ckpt_pos,
                                 resume->cu_ckpt, resume->num_probes, resume->probe_seq, resume->probe_depth,
                                 resume->S_out, resume->o_out, workspace, ws_bytes, part, L, chosen, offs)) != GDN_OK)
            return st;
        // the resumes read checkpoints that this launch must not be writing
        if (prefill && prefill->cu_ckpt && resume->cu_ckpt) {
            const size_t state_bytes = (size_t)p->num_heads * p->d_v * p->d_k * sizeof(float);
            const int B = p->num_seqs;
            if (ranges_overlap(prefill->ckpt_states, (size_t)prefill->cu_ckpt[B] * state_bytes,
                               resume->ckpt_states, (size_t)resume->cu_ckpt[B] * state_bytes))
                return GDN_ERR_INVALID_ARG;
        }
        readout = readout || L.readout;
        all.insert(all.end(), part.begin(), part.end());
    }
    std::vector<int64_t> av, kv;
    if (replay) {
        if ((st = plan_all(p->num_seqs, replay->m, replay->r_num, replay->r_den, av, kv)) != GDN_OK) return st;
        if ((st = replay_prepare(p, q, k, v, alpha, beta, replay->m, kv.data(), replay->S_a, replay->S_hat,
                                 replay->S_exact, replay->o, workspace, ws_bytes, part, L)) != GDN_OK)
            return st;
        readout = readout || L.readout;
        // the exact twins as jobs of their own: the same tokens from S_a, no readout
        const size_t n = part.size();
        for (size_t i = 0; i < n; ++i) {
            if (!part[i].job.s0_twin) continue;
            HostJob t = part[i];
            t.job.s0 = part[i].job.s0_twin;
            t.job.s_final = part[i].job.s_final_twin;
            t.job.o = nullptr;
            t.job.s0_twin = nullptr;
            t.job.s_final_twin = nullptr;
            part[i].job.s0_twin = nullptr;
            part[i].job.s_final_twin = nullptr;
            part.push_back(t);
        }
        all.insert(all.end(), part.begin(), part.end());
    }
    if (readout && !q) return GDN_ERR_INVALID_ARG;
    LaunchSpec M{p, q, k, v, alpha, beta, nullptr, ckpt_out, static_cast<unsigned int*>(workspace), readout, false,
                 ws_bytes};
    if ((st = check_two_pass(M, all)) != GDN_OK) return st;
    if (resume) {
        if (resume->chosen_pos) std::copy(chosen.begin(), chosen.end(), resume->chosen_pos);
        if (resume->o_offsets) std::copy(offs.begin(), offs.end(), resume->o_offsets);
    }
    if (replay) {
        if (replay->a_out) std::copy(av.begin(), av.end(), replay->a_out);
        if (replay->k_out) std::copy(kv.begin(), kv.end(), replay->k_out);
    }
    if (all.empty()) return GDN_OK;
    // On the fused tensor-core path a few long scans (prefills) beside many short ones (resumes, replays) run
    // best as two launches side by side: the long jobs' CTAs placed first, the short ones on the remaining SMs.
    // (One launch of all of them places the long CTAs less well; so does letting the short launch reach the
    // GPU first.)
    const cudaStream_t cs = (cudaStream_t)stream;
    const bool fused = use_chunked(p) &&
                       (p->algo == GDN_ALGO_CHUNKED || (p->algo == GDN_ALGO_AUTO && !two_pass_fits(M, all)));
    if (fused) {
        std::stable_sort(all.begin(), all.end(),
                         [](const HostJob& a, const HostJob& b) { return a.job.len > b.job.len; });
        SideLane* lane = side_lane();
        const size_t b = lane ? split_point(all, p->num_heads, lane->sms) : 0;
        if (b > 0) {
            std::vector<HostJob> head(all.begin(), all.begin() + b), tail(all.begin() + b, all.end());
            std::lock_guard<std::mutex> lock(g_side_mutex);   // the lanes' events are shared by every caller
            if (cudaEventRecord(lane->fork, cs) != cudaSuccess ||
                cudaStreamWaitEvent(lane->hi, lane->fork, 0) != cudaSuccess ||
                cudaStreamWaitEvent(lane->lo, lane->fork, 0) != cudaSuccess)
                return GDN_ERR_CUDA;
            // Both lanes take the fused kernel: each lane alone might fit the caller's workspace for the two-pass
            // path, but the two lanes run at the same time and would share its schedule and T areas.
            LaunchSpec F = M;
            F.ws_bytes = kWorkspaceBytes;
            const gdn_status s1 = run_jobs(F, head, lane->hi);
            const gdn_status s2 = run_jobs(F, tail, lane->lo);
            if (cudaEventRecord(lane->join_hi, lane->hi) != cudaSuccess ||
                cudaEventRecord(lane->join_lo, lane->lo) != cudaSuccess ||
                cudaStreamWaitEvent(cs, lane->join_hi, 0) != cudaSuccess ||
                cudaStreamWaitEvent(cs, lane->join_lo, 0) != cudaSuccess)
                return GDN_ERR_CUDA;
            return s1 != GDN_OK ? s1 : s2;
        }
    }
    return run_jobs(M, all, cs);
}

GDN_EXPORT gdn_status gdn_adaptive_replay_plan(const gdn_problem* p, const float* alpha, const int64_t* m,
                                               float eps, int32_t rmax_num, int32_t rmax_den, int64_t* k_out,
                                               int32_t* exact_out, gdn_stream_t stream) {
    std::vector<int64_t> lens;
    gdn_status st = check_problem(p, lens);
    if (st != GDN_OK) return st;
    if (!alpha || !m || !k_out || !exact_out || !(eps >= 0.f) || !(eps < 1.f)) return GDN_ERR_INVALID_ARG;
    const int B = p->num_seqs, H = p->num_heads;
    std::vector<int64_t> av, kmax;
    if ((st = plan_all(B, m, rmax_num, rmax_den, av, kmax)) != GDN_OK) return st;
    for (int b = 0; b < B; ++b)
        if (m[b] > lens[b]) return GDN_ERR_INVALID_ARG;
    std::vector<float> tail;
    for (int b = 0; b < B; ++b) {
        const int64_t K = kmax[b];
        int64_t need = 0;
        bool reached = true;
        if (K > 0) {
            tail.resize((size_t)K * H);
            // gates of rows [m_b - K, m_b): the budget's tail of every head
            // on the caller's stream, after the work that writes the gates
            const cudaStream_t cs = (cudaStream_t)stream;
            if (cudaMemcpyAsync(tail.data(), alpha + (size_t)(p->cu_seqlens[b] + m[b] - K) * H,
                                sizeof(float) * tail.size(), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
                cudaStreamSynchronize(cs) != cudaSuccess)
                return GDN_ERR_CUDA;
            for (int h = 0; h < H; ++h) {
                // smallest k with alpha_m * alpha_{m-1} * ... * alpha_{m-k+1} <= eps (fp32, newest gate first)
                float prod = 1.f;
                int64_t kh = -1;
                for (int64_t i = 1; i <= K; ++i) {
                    prod *= tail[(size_t)(K - i) * H + h];
                    if (prod <= eps) {
                        kh = i;
                        break;
                    }
                }
                if (kh < 0) {
                    reached = false;
                    kh = K;
                }
                need = std::max(need, kh);
            }
        } else {
            reached = m[b] == 0;   // an empty budget recovers only an empty prefix
        }
        k_out[b] = need;
        exact_out[b] = reached ? 0 : 1;
    }
    return GDN_OK;
}

// ------------------------------------------------------------------------------------
// In-group chained replay ("Tail-Replay" notes page, section 2.2 step 3, section 2.4)
// ------------------------------------------------------------------------------------
namespace {

size_t group_row_floats(const gdn_group* g) {
    return 2 * (size_t)g->d_model + 4 * (size_t)g->heads * g->d_head + 2 * (size_t)g->heads;
}
size_t group_layer_floats(const gdn_group* g) {
    return (4 * (size_t)g->heads * g->d_head + 2 * (size_t)g->heads) * (size_t)g->d_model;
}
bool group_ok(const gdn_group* g) {
    return g && g->layers >= 1 && g->layers <= 64 && g->heads >= 1 && g->heads <= 1024 && g->d_model >= 1 &&
           g->d_model <= 8192 && (g->d_head == 32 || g->d_head == 64 || g->d_head == 128) &&
           (int64_t)g->heads * g->d_head <= 8192;
}

// One chain through the group over `rows` input rows: per layer project, scan from a zero state (readout
// except after the last layer), mix into the next layer's input.
gdn_status group_chain(const gdn_group* g, const float* h_in, int64_t rows, const float* weights, float* S_out,
                       float* scratch, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    const int Dm = g->d_model, H = g->heads, d = g->d_head, Hd = H * d;
    float* hA = scratch;
    float* hB = hA + (size_t)rows * Dm;
    float* q = hB + (size_t)rows * Dm;
    float* k = q + (size_t)rows * Hd;
    float* v = k + (size_t)rows * Hd;
    float* o = v + (size_t)rows * Hd;
    float* al = o + (size_t)rows * Hd;
    float* be = al + (size_t)rows * H;
    const float* cur = h_in;
    const int64_t cu[2] = {0, rows};
    gdn_problem p{};
    p.num_seqs = 1;
    p.num_heads = H;
    p.d_k = p.d_v = d;
    p.cu_seqlens = cu;
    p.qkv_dtype = GDN_F32;
    p.out_dtype = GDN_F32;
    p.algo = GDN_ALGO_AUTO;
    const size_t LW = group_layer_floats(g);
    for (int l = 0; l < g->layers; ++l) {
        const float* W = weights + (size_t)l * LW;
        const float* Wq = W;
        const float* Wk = Wq + (size_t)Hd * Dm;
        const float* Wv = Wk + (size_t)Hd * Dm;
        const float* wa = Wv + (size_t)Hd * Dm;
        const float* wb = wa + (size_t)H * Dm;
        const float* Wo = wb + (size_t)H * Dm;
        const bool last = l + 1 == g->layers;
        if (gdn::group::project(cur, rows, Dm, H, d, Wq, Wk, Wv, wa, wb, q, k, v, al, be, stream) != cudaSuccess)
            return GDN_ERR_CUDA;
        // the end of the group needs only the state: the next group reads its own cached input
        const gdn_status st = gdn_prefill_ckpt(&p, last ? nullptr : q, k, v, al, be, nullptr, last ? nullptr : o,
                                               S_out + (size_t)l * H * d * d, nullptr, nullptr, nullptr, workspace,
                                               ws_bytes, stream);
        if (st != GDN_OK) return st;
        if (!last) {
            float* nxt = cur == hA ? hB : hA;
            if (gdn::group::mix(cur, o, rows, Dm, Hd, Wo, nxt, stream) != cudaSuccess) return GDN_ERR_CUDA;
            cur = nxt;
        }
    }
    return GDN_OK;
}

}  // namespace

GDN_EXPORT size_t gdn_group_scratch_bytes(const gdn_group* g, int64_t rows) {
    if (!group_ok(g) || rows < 0) return 0;
    return (size_t)rows * group_row_floats(g) * sizeof(float);
}

GDN_EXPORT gdn_status gdn_group_replay(const gdn_group* g, const float* h, int64_t m, int32_t r_num, int32_t r_den,
                                       const float* weights, float* S_hat, float* S_exact, int64_t* a_out,
                                       int64_t* k_out, void* scratch, size_t scratch_bytes, void* workspace,
                                       size_t ws_bytes, gdn_stream_t stream) {
    if (!group_ok(g)) return GDN_ERR_INVALID_ARG;
    if (m < 0 || m >= ((int64_t)1 << 31) - 64 || !h || !weights || !S_hat || !aligned(S_hat, 16) || !aligned(h, 16) ||
        !aligned(weights, 16))
        return GDN_ERR_INVALID_ARG;
    if (S_exact && !aligned(S_exact, 16)) return GDN_ERR_INVALID_ARG;
    int64_t a = 0, kk = 0;
    if (gdn_replay_plan(m, r_num, r_den, &a, &kk) != GDN_OK) return GDN_ERR_INVALID_ARG;
    const int64_t rows = S_exact ? m : kk;
    if (!scratch || !aligned(scratch, 16) || scratch_bytes < gdn_group_scratch_bytes(g, rows))
        return GDN_ERR_INVALID_ARG;
    gdn_status st;
    if ((st = check_workspace(workspace, ws_bytes)) != GDN_OK) return st;
    if (a_out) *a_out = a;
    if (k_out) *k_out = kk;
    const cudaStream_t s = (cudaStream_t)stream;
    if (S_exact && (st = group_chain(g, h, m, weights, S_exact, static_cast<float*>(scratch), workspace, ws_bytes, s)) !=
                       GDN_OK)
        return st;
    return group_chain(g, h + (size_t)a * g->d_model, kk, weights, S_hat, static_cast<float*>(scratch), workspace,
                       ws_bytes, s);
}
