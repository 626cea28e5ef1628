// BF16 caches with FP16 queries: tile-kernel instantiations (each query is
// split exactly into BF16 hi + lo, two MMAs per K step of S).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16_q16(int d, int wide) {
  if (d == 128 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 5, true>);
  if (d == 128 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 9, true>);
  if (d == 256 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1, 5, true>);
  if (d == 64 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 5, true>);
  if (d == 64 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 9, true>);
  return nullptr;
}
}  // namespace pa
