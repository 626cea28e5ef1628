// BF16 caches: tensor-memory consumer instantiations (head_dim 128, 16 or 32
// rows per softmax warpgroup).
#include "pa_mtp.cuh"

namespace pa {
const void* mtp_kernel_bf16(int d, int rh) {
  if (d == 128 && rh == 16) return reinterpret_cast<const void*>(&dev::pa_mtp_kernel<false, 128, false, 16>);
  if (d == 128 && rh == 32) return reinterpret_cast<const void*>(&dev::pa_mtp_kernel<false, 128, false, 32>);
  return nullptr;
}
}  // namespace pa
