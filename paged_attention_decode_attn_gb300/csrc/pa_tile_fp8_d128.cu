// FP8 e4m3 caches, head_dim 128: tile-kernel instantiations.
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_fp8_d128(int nt, int vtok) {
  if (nt == 1 && !vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, false>);
  if (nt == 1 && vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true>);
  if (nt == 2 && !vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 2, false>);
  if (nt == 2 && vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 2, true>);
  return nullptr;
}
}  // namespace pa
