// The small-M stream-K kernels (narrow MMA side of 16, 32 or 64 rows), which
// sum split tiles through a global-memory workspace.
#include "kernel_streamk.cuh"
#include "launch.h"

namespace gemm_gb300 {
namespace {

template <class Cfg, class T, bool F8>
struct StreamKLauncher {
    static cudaError_t prepare() {
        return cudaFuncSetAttribute(gemm_streamk_kernel<Cfg, T, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg::SMEM_BYTES);
    }
    static cudaError_t launch(const CUtensorMap& w, const CUtensorMap& x, const StreamKParams& p,
                              int grid_ctas, cudaStream_t stream) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
        cfg.attrs = attr;
        return cudaLaunchKernelEx(&cfg, gemm_streamk_kernel<Cfg, T, F8>, w, x, p);
    }
    static const StreamKOps& ops() {
        static const StreamKOps o = {Cfg::MN, Cfg::STAGES, Cfg::SMEM_BYTES, Cfg::TMEM_COLS, &prepare, &launch};
        return o;
    }
};

template <class Cfg>
const StreamKOps& streamk_ops_for(int dtype) {
    if (dtype >= 2) return StreamKLauncher<Cfg, __nv_bfloat16, true>::ops();
    if (dtype == 1) return StreamKLauncher<Cfg, __nv_bfloat16, false>::ops();
    return StreamKLauncher<Cfg, __half, false>::ops();
}

}  // namespace

const StreamKOps& streamk_ops(int mn, int dtype) {
    if (mn <= 16) return streamk_ops_for<CfgStreamK16>(dtype);
    if (mn <= 32) return streamk_ops_for<CfgStreamK32>(dtype);
    return streamk_ops_for<CfgStreamK64>(dtype);
}

}  // namespace gemm_gb300
