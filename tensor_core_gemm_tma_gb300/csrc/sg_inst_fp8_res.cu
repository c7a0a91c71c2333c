// sg_inst_fp8_res.cu -- kernel instantiations: FP8 E4M3 operands, with a residual.
#include "sg_launch.cuh"

namespace sg {

LaunchFn launcher_fp8_res(int bn, int out, int mode) {
    switch ((bn * 4 + out) * 4 + mode) {
        case (128 * 4 + SG_F32) * 4 + 1: return &launch_kernel<128, SG_F32, 1, true, 1>;
        case (256 * 4 + SG_F32) * 4 + 1: return &launch_kernel<256, SG_F32, 1, true, 1>;
        case (256 * 4 + SG_F32) * 4 + 3: return &launch_kernel<256, SG_F32, 3, true, 1>;
        case (128 * 4 + SG_F16) * 4 + 1: return &launch_kernel<128, SG_F16, 1, true, 1>;
        case (256 * 4 + SG_F16) * 4 + 1: return &launch_kernel<256, SG_F16, 1, true, 1>;
        case (256 * 4 + SG_F16) * 4 + 3: return &launch_kernel<256, SG_F16, 3, true, 1>;
        case (128 * 4 + SG_BF16) * 4 + 1: return &launch_kernel<128, SG_BF16, 1, true, 1>;
        case (256 * 4 + SG_BF16) * 4 + 1: return &launch_kernel<256, SG_BF16, 1, true, 1>;
        case (256 * 4 + SG_BF16) * 4 + 3: return &launch_kernel<256, SG_BF16, 3, true, 1>;
        default: return nullptr;
    }
}

}  // namespace sg
