// MXFP4 caches (OCP MX: E2M1 elements, E8M0 scales per 32 head dims), head_dim
// 128: tile-kernel instantiations (two tiles per warp step, FP16 P and V).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_fp4_d128(int wide) {
  if (!wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true, 2, 5, false, true>);
  return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true, 2, 9, false, true>);
}
}  // namespace pa
