// The 2-CTA (cta_group::2) persistent kernel with two MMA consumers per CTA
// sharing each staged B tile: a 512 x 256 tile per CTA pair.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_2cta512(int dtype) {
    return tiled_ops_for<Cfg2cta512>(dtype);
}
}  // namespace gemm_gb300
