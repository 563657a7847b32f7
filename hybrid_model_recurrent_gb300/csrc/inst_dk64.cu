// Kernel instances for d_k = 64: every (input dtype, output dtype, readout,
// twin) combination the host dispatcher can ask for.
#include "gdn_kernel.cuh"

namespace gdn {

template <>
LaunchFn launch_table<64>(int idx) {
    // index: ((in_bf16 * 2 + out_bf16) * 2 + readout) * 2 + twin; without a
    // readout the output dtype is irrelevant and maps to the fp32 instance.
    static const LaunchFn table[16] = {
        launch_scan<64, false, false, false, false>, launch_scan<64, false, false, false, true>,
        launch_scan<64, false, false, true, false>,  launch_scan<64, false, false, true, true>,
        launch_scan<64, false, false, false, false>, launch_scan<64, false, false, false, true>,
        launch_scan<64, false, true, true, false>,   launch_scan<64, false, true, true, true>,
        launch_scan<64, true, false, false, false>,  launch_scan<64, true, false, false, true>,
        launch_scan<64, true, false, true, false>,   launch_scan<64, true, false, true, true>,
        launch_scan<64, true, false, false, false>,  launch_scan<64, true, false, false, true>,
        launch_scan<64, true, true, true, false>,    launch_scan<64, true, true, true, true>,
    };
    return (idx >= 0 && idx < 16) ? table[idx] : nullptr;
}

}  // namespace gdn
