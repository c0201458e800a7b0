// The small-M column-range kernels (narrow MMA side of 16, 32 or 64 rows),
// launched in clusters of P CTAs (the K pieces of one column range).
#include "kernel_skinny.cuh"
#include "launch.h"

namespace gemm_gb300 {
namespace {

template <class Cfg, class T, bool F8>
struct SkinnyLauncher {
    static cudaError_t prepare() {
        return cudaFuncSetAttribute(gemm_skinny_kernel<Cfg, T, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg::SMEM_BYTES);
    }
    static cudaError_t max_active(int pieces, int* out) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(pieces), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(pieces);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaOccupancyMaxActiveClusters(out, gemm_skinny_kernel<Cfg, T, F8>, &cfg);
    }
    static cudaError_t launch(const CUtensorMap& w, const CUtensorMap& x, const SkinnyParams& p,
                              int grid_ctas, cudaStream_t stream) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        // programmatic stream serialisation (see the tiled launcher); a cluster
        // of P CTAs when the K loop is split
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
        if (p.pieces > 1) {
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = static_cast<unsigned>(p.pieces);
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        cfg.attrs = attr;
        return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<Cfg, T, F8>, w, x, p);
    }
    static const SkinnyOps& ops() {
        static const SkinnyOps o = {Cfg::MN,         Cfg::RING_BYTES, Cfg::X_BYTES, Cfg::MAX_ATOMS,
                                    Cfg::SMEM_BYTES, Cfg::TMEM_COLS,  &prepare,     &max_active,
                                    &launch};
        return o;
    }
};

template <class Cfg>
const SkinnyOps& skinny_ops_for(int dtype) {
    if (dtype >= 2) return SkinnyLauncher<Cfg, __nv_bfloat16, true>::ops();
    if (dtype == 1) return SkinnyLauncher<Cfg, __nv_bfloat16, false>::ops();
    return SkinnyLauncher<Cfg, __half, false>::ops();
}

}  // namespace

const SkinnyOps& skinny_ops(int mn, int dtype) {
    if (mn <= 16) return skinny_ops_for<CfgSkinny16>(dtype);
    if (mn <= 32) return skinny_ops_for<CfgSkinny32>(dtype);
    return skinny_ops_for<CfgSkinny64>(dtype);
}

}  // namespace gemm_gb300
