// BF16 caches: tile-kernel instantiations.
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16(int d, int wide) {
  if (d == 128 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 5>);
  if (d == 128 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 9>);
  if (d == 256 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1, 5>);
  return nullptr;
}
}  // namespace pa
