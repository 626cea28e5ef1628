// FP8 e4m3 caches, head_dim 128: tile-kernel instantiations (two tiles per warp step).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_fp8_d128(int vtok, int wide) {
  if (!vtok && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, false, 2, 5>);
  if (vtok && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true, 2, 5>);
  if (!vtok && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, false, 2, 9>);
  return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true, 2, 9>);
}
}  // namespace pa
