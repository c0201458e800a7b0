// Two CTA pairs per 4-CTA cluster, sharing each B block by multicast: a
// 512 x 256 tile per cluster.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_4cta512(int dtype) {
    return dtype == 1 ? TiledLauncher<Cfg4cta512, __nv_bfloat16>::ops() : TiledLauncher<Cfg4cta512, __half>::ops();
}
}  // namespace gemm_gb300
