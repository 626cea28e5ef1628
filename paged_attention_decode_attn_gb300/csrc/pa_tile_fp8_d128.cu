// FP8 e4m3 caches, head_dim 128: tile-kernel instantiations (two tiles per warp step).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_fp8_d128(int nt, int vtok, int tw) {
  if (tw != 2) return nullptr;
  if (nt == 1 && !vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, false, 2>);
  if (nt == 1 && vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 1, true, 2>);
  if (nt == 2 && !vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 2, false, 2>);
  if (nt == 2 && vtok) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<true, 128, 2, true, 2>);
  return nullptr;
}
}  // namespace pa
