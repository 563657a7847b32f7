// gdn_group.cu - the layer-to-layer steps of in-group chained replay ("Tail-Replay" notes page,
// section 2.2 step 3 and section 2.4): a group of linear-attention layers is replayed one layer after
// the other, each layer reading the previous layer's outputs.  The pages fix no model, so the group
// here is synthetic (its weights are inputs), per layer l and head h:
//   q_t = normalise(W_q h_t), k_t = normalise(W_k h_t), v_t = W_v h_t          (d_head each, per head)
//   alpha_t = 1 - 0.1 sigmoid(w_a . h_t),  beta_t = sigmoid(w_b . h_t)           (per head)
//   h'_t = h_t + W_o [o_t,1; ...; o_t,H]                                        (residual, d_model)
// The GDN scans between these steps are the library's own kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_group.cuh"

namespace gdn {
namespace group {

// One block per (row t, head), d_head threads (a multiple of 32): q, k, v of that head, and the two
// gates from the first two warps' reductions.
__global__ void project_kernel(const float* __restrict__ h, int64_t rows, int Dm, int H, int d,
                               const float* __restrict__ Wq, const float* __restrict__ Wk, const float* __restrict__ Wv,
                               const float* __restrict__ wa, const float* __restrict__ wb, float* __restrict__ q,
                               float* __restrict__ k, float* __restrict__ v, float* __restrict__ alpha,
                               float* __restrict__ beta) {
    extern __shared__ float sh[];   // h_t [Dm], then 2 x 32 partial sums
    float* red = sh + Dm;
    const int64_t t = blockIdx.x;
    const int hh = blockIdx.y, e = threadIdx.x;
    if (t >= rows) return;
    for (int i = e; i < Dm; i += blockDim.x) sh[i] = h[t * Dm + i];
    __syncthreads();
    const size_t r = (size_t)hh * d + e;
    float aq = 0.f, ak = 0.f, av = 0.f;
    for (int i = 0; i < Dm; ++i) {
        const float x = sh[i];
        aq = fmaf(Wq[r * Dm + i], x, aq);
        ak = fmaf(Wk[r * Dm + i], x, ak);
        av = fmaf(Wv[r * Dm + i], x, av);
    }
    // L2 norms of q and k over the head's d_head entries
    float sq = aq * aq, sk = ak * ak;
    for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    const int w = e >> 5, nw = blockDim.x >> 5;
    if ((e & 31) == 0) {
        red[w] = sq;
        red[32 + w] = sk;
    }
    __syncthreads();
    float nq = 0.f, nk = 0.f;
    for (int i = 0; i < nw; ++i) {
        nq += red[i];
        nk += red[32 + i];
    }
    const size_t o = ((size_t)t * H + hh) * d + e;
    q[o] = aq * rsqrtf(nq);
    k[o] = ak * rsqrtf(nk);
    v[o] = av;
    // gates: warp 0 reduces w_a . h_t, warp 1 w_b . h_t (warp 0 both when d_head = 32)
    auto gate_dot = [&](const float* wrow) {
        float acc = 0.f;
        for (int i = e & 31; i < Dm; i += 32) acc = fmaf(wrow[i], sh[i], acc);
        for (int s2 = 16; s2 > 0; s2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s2);
        return acc;
    };
    if (w == 0) {
        const float z = gate_dot(wa + (size_t)hh * Dm);
        if (e == 0) alpha[(size_t)t * H + hh] = 1.f - 0.1f / (1.f + expf(-z));
    }
    if (w == 1 || (nw == 1 && w == 0)) {
        const float z = gate_dot(wb + (size_t)hh * Dm);
        if ((e & 31) == 0) beta[(size_t)t * H + hh] = 1.f / (1.f + expf(-z));
    }
}

// One block per row t: h_out = h_in + W_o o_t (Dm outputs, each a dot product over H d_head).
__global__ void mix_kernel(const float* __restrict__ h_in, const float* __restrict__ o, int64_t rows, int Dm, int Hd,
                           const float* __restrict__ Wo, float* __restrict__ h_out) {
    extern __shared__ float so[];   // o_t [Hd]
    const int64_t t = blockIdx.x;
    if (t >= rows) return;
    for (int i = threadIdx.x; i < Hd; i += blockDim.x) so[i] = o[t * Hd + i];
    __syncthreads();
    for (int j = threadIdx.x; j < Dm; j += blockDim.x) {
        float acc = 0.f;
        for (int i = 0; i < Hd; ++i) acc = fmaf(Wo[(size_t)j * Hd + i], so[i], acc);
        h_out[t * Dm + j] = h_in[t * Dm + j] + acc;
    }
}

cudaError_t project(const float* h, int64_t rows, int Dm, int H, int d, const float* Wq, const float* Wk,
                    const float* Wv, const float* wa, const float* wb, float* q, float* k, float* v, float* alpha,
                    float* beta, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)rows, (unsigned)H);
    project_kernel<<<grid, d, (Dm + 64) * sizeof(float), stream>>>(h, rows, Dm, H, d, Wq, Wk, Wv, wa, wb, q, k, v,
                                                                   alpha, beta);
    return cudaGetLastError();
}

cudaError_t mix(const float* h_in, const float* o, int64_t rows, int Dm, int Hd, const float* Wo, float* h_out,
                cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    mix_kernel<<<(unsigned)rows, 256, Hd * sizeof(float), stream>>>(h_in, o, rows, Dm, Hd, Wo, h_out);
    return cudaGetLastError();
}

}  // namespace group
}  // namespace gdn
