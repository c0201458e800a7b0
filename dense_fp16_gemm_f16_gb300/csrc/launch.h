// launch.h -- host-side entry points into each compiled kernel variant.  Each
// variant lives in its own translation unit; the C-ABI layer (api.cu) only
// sees these function tables.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "config.h"

namespace gemm_gb300 {

struct TiledOps {
    // tile_m: rows of one tile (per CTA pair when cta_group == 2); cluster: CTAs
    // per cluster; b_box_rows: rows of B per TMA box (each CTA's B rows);
    // max_stage_atoms: the most K blocks per ring stage a launch may ask for
    int cta_group, tile_m, tile_n, stages, smem_bytes, tmem_cols, cluster, b_box_rows, max_stage_atoms;
    // set the kernel's shared-memory limit on the current device
    cudaError_t (*prepare)();
    // co-resident clusters (cta_group 2) or CTAs per SM (cta_group 1) on the current device
    cudaError_t (*max_active)(int* out);
    // co-resident split-K clusters of `pieces` MMA groups on the current device
    cudaError_t (*max_active_split)(int pieces, int* out);
    // b_piece: B with a box of (B rows per CTA) / split rows, for the column
    // pieces of the last round's tiles
    cudaError_t (*launch)(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b_piece,
                          const CUtensorMap& d, const TiledParams& p, int grid_ctas, cudaStream_t stream);
};

struct SkinnyOps {
    // the ring holds min(max_atoms, ring_bytes / (B slot + x_bytes)) K blocks
    int mn, ring_bytes, x_bytes, max_atoms, smem_bytes, tmem_cols;
    cudaError_t (*prepare)();
    // co-resident clusters of `pieces` CTAs on the current device
    cudaError_t (*max_active)(int pieces, int* out);
    cudaError_t (*launch)(const CUtensorMap& w, const CUtensorMap& x, const SkinnyParams& p,
                          int grid_ctas, cudaStream_t stream);
};

struct StreamKOps {
    int mn, stages, smem_bytes, tmem_cols;
    cudaError_t (*prepare)();
    cudaError_t (*launch)(const CUtensorMap& w, const CUtensorMap& x, const StreamKParams& p,
                          int grid_ctas, cudaStream_t stream);
};

// dtype: 0 = fp16 operands and output, 1 = bf16, 2 / 3 = E4M3 / E5M2 operands
// with a bf16 output
const TiledOps& tiled_ops_2cta256(int dtype);
const TiledOps& tiled_ops_2cta512(int dtype);   // two consumers per CTA
const TiledOps& tiled_ops_1cta128(int dtype);
const TiledOps& tiled_ops_1cta256(int dtype);
const SkinnyOps& skinny_ops(int mn, int dtype);    // mn = 16, 32 or 64
const StreamKOps& streamk_ops(int mn, int dtype);  // mn = 16, 32 or 64

}  // namespace gemm_gb300
