// BF16 caches: tile-kernel instantiations.
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16(int d, int nt, int tw) {
  if (tw != 1) return nullptr;
  if (d == 128 && nt == 1) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1>);
  if (d == 128 && nt == 2) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 2, false, 1>);
  if (d == 256 && nt == 1) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1>);
  return nullptr;
}
}  // namespace pa
