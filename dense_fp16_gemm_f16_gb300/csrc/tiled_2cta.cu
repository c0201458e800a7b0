// The 2-CTA (cta_group::2) persistent kernel: 256 x 256 tile per CTA pair.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_2cta256(int dtype) {
    return tiled_ops_for<Cfg2cta256>(dtype);
}
}  // namespace gemm_gb300
