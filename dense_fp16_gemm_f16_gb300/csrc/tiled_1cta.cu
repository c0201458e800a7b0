// The 1-CTA (cta_group::1) persistent kernels: 128 x 128 and 128 x 256 tiles.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_1cta128(int dtype) {
    return tiled_ops_for<Cfg1cta128>(dtype);
}
const TiledOps& tiled_ops_1cta256(int dtype) {
    return tiled_ops_for<Cfg1cta256>(dtype);
}
}  // namespace gemm_gb300
