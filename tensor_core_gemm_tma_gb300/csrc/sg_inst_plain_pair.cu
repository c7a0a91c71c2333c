// sg_inst_plain_pair.cu -- kernel instantiations: no residual, CTA-pair mode (paired MMA).
#include "sg_launch.cuh"

namespace sg {

LaunchFn launcher_plain_pair(int bn, int out, int mode) {
    switch ((bn * 4 + out) * 4 + mode) {
        case (128 * 4 + SG_F32) * 4 + 3: return &launch_kernel<128, SG_F32, 3, false, 2>;
        case (128 * 4 + SG_F16) * 4 + 3: return &launch_kernel<128, SG_F16, 3, false, 2>;
        case (128 * 4 + SG_BF16) * 4 + 3: return &launch_kernel<128, SG_BF16, 3, false, 2>;
        case (256 * 4 + SG_F32) * 4 + 3: return &launch_kernel<256, SG_F32, 3, false, 2>;
        case (256 * 4 + SG_F16) * 4 + 3: return &launch_kernel<256, SG_F16, 3, false, 2>;
        case (256 * 4 + SG_BF16) * 4 + 3: return &launch_kernel<256, SG_BF16, 3, false, 2>;
        default: return nullptr;
    }
}

}  // namespace sg
