// gdn_group.cuh - launchers of the layer-to-layer kernels of in-group chained replay (gdn_group.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace group {

// q, k (unit norm per head), v [rows, H, d]; alpha, beta [rows, H] from h [rows, Dm] (all fp32, row-major)
cudaError_t project(const float* h, int64_t rows, int Dm, int H, int d, const float* Wq, const float* Wk,
                    const float* Wv, const float* wa, const float* wb, float* q, float* k, float* v, float* alpha,
                    float* beta, cudaStream_t stream);

// h_out = h_in + W_o o (o [rows, Hd], W_o [Dm, Hd], h [rows, Dm])
cudaError_t mix(const float* h_in, const float* o, int64_t rows, int Dm, int Hd, const float* Wo, float* h_out,
                cudaStream_t stream);

}  // namespace group
}  // namespace gdn
