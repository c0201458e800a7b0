// The 1-CTA (cta_group::1) persistent kernels: 128 x 128 and 128 x 256 tiles.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_1cta128(int dtype) {
    return dtype == 1 ? TiledLauncher<Cfg1cta128, __nv_bfloat16>::ops() : TiledLauncher<Cfg1cta128, __half>::ops();
}
const TiledOps& tiled_ops_1cta256(int dtype) {
    return dtype == 1 ? TiledLauncher<Cfg1cta256, __nv_bfloat16>::ops() : TiledLauncher<Cfg1cta256, __half>::ops();
}
}  // namespace gemm_gb300
