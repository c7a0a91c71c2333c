// sg_launch.cuh -- launching one instantiation of the GEMM kernel.
//
// The instantiations are spread over several translation units
// (sg_inst_*.cu), compiled in parallel; each exports a lookup from
// (tile width, output type, mode) to its launcher.  The host API file only
// sees these declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "sg_kernel.cuh"

namespace sg {

struct LaunchArgs {
    const CUtensorMap* ta;
    const CUtensorMap* tb;
    const CUtensorMap* tc;
    const CUtensorMap* tr;
    const Params* prm;
    int grid;             // CTAs requested (a multiple of the cluster size)
    int smem;             // dynamic shared memory per CTA
    int smem_optin;       // the device's opt-in maximum, set once as the kernel's attribute
    cudaStream_t stream;
    std::mutex* mu;       // guards the two per-device caches below
    bool* attr_done;      // this instantiation's attribute is set on this device
    int* max_clusters;    // co-resident clusters of this instantiation (0: not queried, -1: unknown)
};

// Returns 0, or -1 when a CUDA call fails.
using LaunchFn = int (*)(LaunchArgs&);

template <int BN, int OUT, int MODE, bool RES, int ESZ>
int launch_kernel(LaunchArgs& a) {
    constexpr int CM = (MODE == 3 || MODE == 6) ? 2 : 1;  // CTAs per cluster
    auto kern = sg_gemm_kernel<BN, OUT, MODE, RES, ESZ>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(a.smem);
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int grid = a.grid;
    {
        std::lock_guard<std::mutex> lk(*a.mu);
        if (!*a.attr_done) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem_optin) != cudaSuccess)
                return -1;
            *a.attr_done = true;
        }
        if (CM > 1) {
            int& mc = *a.max_clusters;
            if (mc == 0) {
                cfg.gridDim = dim3(static_cast<unsigned>(a.grid), 1, 1);
                int n = 0;
                mc = (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) ? n : -1;
                cudaGetLastError();  // a failed query is not a launch error
            }
            // a persistent grid larger than what can be co-resident only adds a tail
            if (mc > 0 && grid > mc * CM) grid = mc * CM;
        }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, *a.ta, *a.tb, *a.tc, *a.tr, *a.prm) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// The launcher of one instantiation, or nullptr if it does not exist.
// Defined by the instantiation units.  16-bit operands:
LaunchFn launcher_plain_single(int bn, int out);  // mode 1, no residual
LaunchFn launcher_plain_pair(int bn, int out, int mode);  // mode 3 (paired MMA), no residual
LaunchFn launcher_res_single(int bn, int out);
LaunchFn launcher_res_pair(int bn, int out, int mode);
// FP8 E4M3 operands (tile widths 128 and 256; the paired MMA only at 256):
LaunchFn launcher_fp8_plain(int bn, int out, int mode);
LaunchFn launcher_fp8_res(int bn, int out, int mode);
// Mode 4 (resident B), tile width 128, either element size (esz 1 or 2):
LaunchFn launcher_panel(int out, bool residual, int esz);
LaunchFn launcher_decoded(int out);  // mode 5: 16-bit A, int8-coded B decoded into the resident panel
// Mode 6 (wide paired tiles: two 256-column accumulators), either element size:
LaunchFn launcher_wide(int out, bool residual, int esz);

}  // namespace sg
