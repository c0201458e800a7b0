// The 1-CTA (cta_group::1) persistent kernels: 128 x 128 and 128 x 256 tiles.
#include "launch_tiled.cuh"

namespace gemm_gb300 {
const TiledOps& tiled_ops_1cta128() { return TiledLauncher<Cfg1cta128>::ops(); }
const TiledOps& tiled_ops_1cta256() { return TiledLauncher<Cfg1cta256>::ops(); }
}  // namespace gemm_gb300
