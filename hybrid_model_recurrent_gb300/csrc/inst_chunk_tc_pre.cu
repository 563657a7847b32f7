// inst_chunk_tc_pre.cu - instantiations of the tcgen05 chunkwise kernel that reads T from the first
// passes of the two-pass path (own translation unit, compiled in parallel).
#include "gdn_chunk_tc.cuh"

namespace gdn {
namespace tc {

cudaError_t launch_given_t(const Params& p, int grid, bool readout, bool out_bf16, cudaStream_t stream) {
    if (readout)
        return out_bf16 ? launch_chunk_tc<true, true, true>(p, grid, stream)
                        : launch_chunk_tc<false, true, true>(p, grid, stream);
    return launch_chunk_tc<false, false, true>(p, grid, stream);
}

}  // namespace tc
}  // namespace gdn
