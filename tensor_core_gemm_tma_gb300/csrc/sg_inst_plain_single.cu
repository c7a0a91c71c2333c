// sg_inst_plain_single.cu -- kernel instantiations: no residual, single-CTA mode.
#include "sg_launch.cuh"

namespace sg {

LaunchFn launcher_plain_single(int bn, int out) {
    switch (bn * 4 + out) {
        case 128 * 4 + SG_F32: return &launch_kernel<128, SG_F32, 1, false, 2>;
        case 128 * 4 + SG_F16: return &launch_kernel<128, SG_F16, 1, false, 2>;
        case 128 * 4 + SG_BF16: return &launch_kernel<128, SG_BF16, 1, false, 2>;
        case 192 * 4 + SG_F32: return &launch_kernel<192, SG_F32, 1, false, 2>;
        case 192 * 4 + SG_F16: return &launch_kernel<192, SG_F16, 1, false, 2>;
        case 192 * 4 + SG_BF16: return &launch_kernel<192, SG_BF16, 1, false, 2>;
        case 256 * 4 + SG_F32: return &launch_kernel<256, SG_F32, 1, false, 2>;
        case 256 * 4 + SG_F16: return &launch_kernel<256, SG_F16, 1, false, 2>;
        case 256 * 4 + SG_BF16: return &launch_kernel<256, SG_BF16, 1, false, 2>;
        default: return nullptr;
    }
}

}  // namespace sg
