// gdn_noalloc.cu - prefill with sparse checkpoints for callers that cannot
// allocate device memory.
//
// The regular entry points take a small caller-provided workspace. Some callers
// cannot provide one: they are handed their input and output buffers but have no
// device allocator of their own. Examples are a plugin inside a serving engine
// whose memory pool owns all of HBM, or a latency-critical loop that cannot
// afford the implicit device synchronisation of cudaMalloc. For them this file
// keeps the scan's scratch (the device status word) in a fixed-size static
// device array. It is allocated when the library is loaded onto a GPU and
// stays there until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdn_scan.h"

#define GDN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Largest scratch this entry point can hold. The scan needs gdn_workspace_size() bytes.
constexpr size_t kNoallocScratchBytes = 256;
constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

// One copy per GPU that loads the library, shared by every call on that GPU.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

GDN_EXPORT gdn_status gdn_prefill_ckpt_noalloc(const gdn_problem* p, const void* q, const void* k, const void* v,
                                               const float* alpha, const float* beta, const float* S0, void* o,
                                               float* S_final, const int64_t* ckpt_pos, const int64_t* cu_ckpt,
                                               float* ckpt_states, gdn_stream_t stream) {
    if (gdn_workspace_size() > kNoallocScratchBytes) return GDN_ERR_UNSUPPORTED;  // scratch too small

    // Per-device set-up: host code may not pass the array's name to a kernel (on the
    // host it is only a stand-in). Ask the runtime for its device address once per
    // device, with that device current, and reuse it for the rest of the process
    // (a cudaDeviceReset would invalidate it; the header rules that case out).
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return GDN_ERR_CUDA;
    if (dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_addr[dev]) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return GDN_ERR_CUDA;
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }

    // The array keeps the previous call's contents: the status word must start at zero.
    if (cudaMemsetAsync(scratch, 0, kNoallocScratchBytes, (cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status st = gdn_prefill_ckpt(p, q, k, v, alpha, beta, S0, o, S_final, ckpt_pos, cu_ckpt, ckpt_states,
                                     scratch, kNoallocScratchBytes, stream);
    if (st != GDN_OK) return st;
    // Report device-side wait expiries now; the caller has no workspace to read later.
    return gdn_read_status(scratch, kNoallocScratchBytes, stream);
}
