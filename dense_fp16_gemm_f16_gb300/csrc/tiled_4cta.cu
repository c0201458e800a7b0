// Two CTA pairs per 4-CTA cluster, sharing each B block by multicast: a
// 512 x 256 tile per cluster.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_4cta512(int dtype) {
    return tiled_ops_for<Cfg4cta512>(dtype);
}
}  // namespace gemm_gb300
