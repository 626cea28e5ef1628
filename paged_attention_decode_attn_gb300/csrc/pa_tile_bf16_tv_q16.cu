// BF16 caches with transposed V and FP16 queries (split into BF16 hi + lo):
// tile-kernel instantiations.
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16_tv_q16(int d, int wide) {
  if (d == 128 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 5, true, false, true>);
  if (d == 128 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 9, true, false, true>);
  if (d == 256 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1, 5, true, false, true>);
  if (d == 64 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 5, true, false, true>);
  if (d == 64 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 9, true, false, true>);
  return nullptr;
}
}  // namespace pa
