// inst_chunk_tc.cu - instantiations of the tcgen05 chunkwise kernel that computes T itself (own
// translation unit so that it compiles in parallel with the rest of the library).
#include "gdn_chunk_tc.cuh"

namespace gdn {
namespace tc {

cudaError_t launch_given_t(const Params& p, int grid, bool readout, bool out_bf16, cudaStream_t stream);

cudaError_t launch(const Params& p, int grid, bool readout, bool out_bf16, bool pre_t, cudaStream_t stream) {
    if (pre_t) return launch_given_t(p, grid, readout, out_bf16, stream);
    if (readout)
        return out_bf16 ? launch_chunk_tc<true, true, false>(p, grid, stream)
                        : launch_chunk_tc<false, true, false>(p, grid, stream);
    return launch_chunk_tc<false, false, false>(p, grid, stream);
}

}  // namespace tc
}  // namespace gdn
