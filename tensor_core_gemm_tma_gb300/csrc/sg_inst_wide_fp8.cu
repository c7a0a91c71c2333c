// sg_inst_wide_fp8.cu -- kernel instantiations: mode 6 (wide paired tiles, two 256-column accumulators), FP8 E4M3 operands.
#include "sg_launch.cuh"

namespace sg {

LaunchFn launcher_wide_e4m3(int out, bool residual) {
    switch (out * 2 + (residual ? 1 : 0)) {
        case SG_F32 * 2 + 0: return &launch_kernel<256, SG_F32, 6, false, 1>;
        case SG_F32 * 2 + 1: return &launch_kernel<256, SG_F32, 6, true, 1>;
        case SG_F16 * 2 + 0: return &launch_kernel<256, SG_F16, 6, false, 1>;
        case SG_F16 * 2 + 1: return &launch_kernel<256, SG_F16, 6, true, 1>;
        case SG_BF16 * 2 + 0: return &launch_kernel<256, SG_BF16, 6, false, 1>;
        case SG_BF16 * 2 + 1: return &launch_kernel<256, SG_BF16, 6, true, 1>;
        default: return nullptr;
    }
}

}  // namespace sg
