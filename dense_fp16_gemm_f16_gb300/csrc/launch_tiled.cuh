// launch_tiled.cuh -- builds the TiledOps table of one tiled configuration.
#pragma once

#include "kernel_tiled.cuh"
#include "launch.h"

namespace gemm_gb300 {

template <class Cfg, class T, bool F8>
struct TiledLauncher {
    // 1-CTA configurations also come with two K blocks per ring stage (for
    // launches made only of narrow column pieces)
    static constexpr int kMaxAtoms = Cfg::CG == 1 ? 2 : 1;

    static cudaError_t prepare() {
        cudaError_t e = cudaFuncSetAttribute(gemm_tiled_kernel<Cfg, T, F8, 1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if constexpr (kMaxAtoms > 1) {
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemm_tiled_kernel<Cfg, T, F8, 2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        }
        return e;
    }

    static cudaError_t max_active(int* out) {
        if constexpr (Cfg::CG > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(Cfg::CG, 1, 1);
            cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
            cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = Cfg::CG;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaOccupancyMaxActiveClusters(out, gemm_tiled_kernel<Cfg, T, F8>, &cfg);
        } else {
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gemm_tiled_kernel<Cfg, T, F8>, Cfg::THREADS,
                                                                 Cfg::SMEM_BYTES);
        }
    }

    static cudaError_t max_active_split(int pieces, int* out) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(Cfg::CG * pieces), 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(Cfg::CG * pieces);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaOccupancyMaxActiveClusters(out, gemm_tiled_kernel<Cfg, T, F8>, &cfg);
    }

    static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b_piece,
                              const CUtensorMap& d, const TiledParams& p, int grid_ctas, cudaStream_t stream) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        // programmatic stream serialisation: this grid may be scheduled while the
        // previous kernel in the stream finishes; it waits (griddepcontrol.wait)
        // before its first global access
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
        // clusters: a CTA pair, or with split K ksplit MMA groups on one tile
        const int cluster = Cfg::CG * (p.ksplit > 1 ? p.ksplit : 1);
        if (cluster > 1) {
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        cfg.attrs = attr;
        if constexpr (kMaxAtoms > 1) {
            if (p.stage_atoms == 2)
                return cudaLaunchKernelEx(&cfg, gemm_tiled_kernel<Cfg, T, F8, 2>, a, b, b_piece, d, p);
        }
        if (p.stage_atoms != 1) return cudaErrorInvalidValue;
        return cudaLaunchKernelEx(&cfg, gemm_tiled_kernel<Cfg, T, F8, 1>, a, b, b_piece, d, p);
    }

    static const TiledOps& ops() {
        static const TiledOps o = {Cfg::CG, Cfg::BM, Cfg::BN, Cfg::STAGES, Cfg::SMEM_BYTES,
                                   Cfg::TMEM_COLS, Cfg::CG, Cfg::B_ROWS, kMaxAtoms,
                                   &prepare, &max_active, &max_active_split, &launch};
        return o;
    }
};

// The table for a gemm_dtype_t: fp16 operands and D (0), bf16 (1), or 8-bit
// operands (2 = E4M3, 3 = E5M2; one kernel, the format is a launch
// parameter) with a bf16 D.
template <class Cfg>
const TiledOps& tiled_ops_for(int dtype) {
    if (dtype >= 2) return TiledLauncher<Cfg, __nv_bfloat16, true>::ops();
    if (dtype == 1) return TiledLauncher<Cfg, __nv_bfloat16, false>::ops();
    return TiledLauncher<Cfg, __half, false>::ops();
}

}  // namespace gemm_gb300
