// sg_inst_panel.cu -- kernel instantiations: mode 4 (B resident in shared memory) and mode 5 (an
// int8-coded B decoded into that resident panel), tile width 128.
#include "sg_launch.cuh"

namespace sg {

LaunchFn launcher_panel(int out, bool residual, int esz) {
    switch ((out * 2 + (residual ? 1 : 0)) * 4 + esz) {
        case (SG_F32 * 2 + 0) * 4 + 1: return &launch_kernel<128, SG_F32, 4, false, 1>;
        case (SG_F32 * 2 + 0) * 4 + 2: return &launch_kernel<128, SG_F32, 4, false, 2>;
        case (SG_F32 * 2 + 1) * 4 + 1: return &launch_kernel<128, SG_F32, 4, true, 1>;
        case (SG_F32 * 2 + 1) * 4 + 2: return &launch_kernel<128, SG_F32, 4, true, 2>;
        case (SG_F16 * 2 + 0) * 4 + 1: return &launch_kernel<128, SG_F16, 4, false, 1>;
        case (SG_F16 * 2 + 0) * 4 + 2: return &launch_kernel<128, SG_F16, 4, false, 2>;
        case (SG_F16 * 2 + 1) * 4 + 1: return &launch_kernel<128, SG_F16, 4, true, 1>;
        case (SG_F16 * 2 + 1) * 4 + 2: return &launch_kernel<128, SG_F16, 4, true, 2>;
        case (SG_BF16 * 2 + 0) * 4 + 1: return &launch_kernel<128, SG_BF16, 4, false, 1>;
        case (SG_BF16 * 2 + 0) * 4 + 2: return &launch_kernel<128, SG_BF16, 4, false, 2>;
        case (SG_BF16 * 2 + 1) * 4 + 1: return &launch_kernel<128, SG_BF16, 4, true, 1>;
        case (SG_BF16 * 2 + 1) * 4 + 2: return &launch_kernel<128, SG_BF16, 4, true, 2>;
        default: return nullptr;
    }
}

LaunchFn launcher_decoded(int out) {
    switch (out) {
        case SG_F32: return &launch_kernel<128, SG_F32, 5, false, 2>;
        case SG_F16: return &launch_kernel<128, SG_F16, 5, false, 2>;
        case SG_BF16: return &launch_kernel<128, SG_BF16, 5, false, 2>;
        default: return nullptr;
    }
}

}  // namespace sg
