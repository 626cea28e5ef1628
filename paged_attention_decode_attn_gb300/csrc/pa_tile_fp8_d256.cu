// FP8 e4m3 caches, head_dim 256 (at most 32 query rows): tile-kernel instantiations.
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_fp8_d256(int vtok) {
  if (!vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 256, 1, false, 1, 5>);
  return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 256, 1, true, 1, 5>);
}
}  // namespace pa
