// BF16 caches: tile-kernel instantiations (BF16 queries; FP16 queries are
// built in pa_tile_bf16_q16.cu).
#include "pa_tile.cuh"

namespace pa {
const void* tile_kernel_bf16(int d, int wide, int q_f16) {
  if (q_f16) return tile_kernel_bf16_q16(d, wide);
  if (d == 128 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 5>);
  if (d == 128 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 128, 1, false, 1, 9>);
  if (d == 256 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 256, 1, false, 1, 5>);
  // head_dim 64: one 128-byte block per token row, like FP8 head_dim 128
  if (d == 64 && !wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 5>);
  if (d == 64 && wide) return reinterpret_cast<const void*>(&dev::pa_tile_kernel<false, 64, 1, false, 1, 9>);
  return nullptr;
}
}  // namespace pa
