// BF16 caches with V in the transposed layout (chunks of 8 tokens per head
// dim): tile-kernel instantiations with BF16 queries (FP16 queries:
// pa_tile_bf16_tv_q16.cu).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16_tv(int d, int wide, int q_f16) {
  if (q_f16) return tile_kernel_bf16_tv_q16(d, wide);
  if (d == 128 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 5, false, false, true>);
  if (d == 128 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 9, false, false, true>);
  if (d == 256 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1, 5, false, false, true>);
  if (d == 64 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 5, false, false, true>);
  if (d == 64 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 9, false, false, true>);
  return nullptr;
}
}  // namespace pa
