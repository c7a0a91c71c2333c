// sg_inst_wide.cu -- kernel instantiations: mode 6 (wide paired tiles, two 256-column accumulators), 16-bit operands.
#include "sg_launch.cuh"

namespace sg {

static LaunchFn launcher_wide_16(int out, bool residual) {
    switch (out * 2 + (residual ? 1 : 0)) {
        case SG_F32 * 2 + 0: return &launch_kernel<256, SG_F32, 6, false, 2>;
        case SG_F32 * 2 + 1: return &launch_kernel<256, SG_F32, 6, true, 2>;
        case SG_F16 * 2 + 0: return &launch_kernel<256, SG_F16, 6, false, 2>;
        case SG_F16 * 2 + 1: return &launch_kernel<256, SG_F16, 6, true, 2>;
        case SG_BF16 * 2 + 0: return &launch_kernel<256, SG_BF16, 6, false, 2>;
        case SG_BF16 * 2 + 1: return &launch_kernel<256, SG_BF16, 6, true, 2>;
        default: return nullptr;
    }
}

LaunchFn launcher_wide_e4m3(int out, bool residual);  // sg_inst_wide_fp8.cu

LaunchFn launcher_wide(int out, bool residual, int esz) {
    return esz == 1 ? launcher_wide_e4m3(out, residual) : launcher_wide_16(out, residual);
}

}  // namespace sg
