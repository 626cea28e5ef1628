// BF16 caches: tensor-memory consumer instantiations (head_dim 128: two
// warpgroups of 16 rows, two of 32 or four of 16).
#include "pa_mtp.cuh"

namespace pa {
const void* mtp_kernel_bf16(int d, int rh, int nwg) {
  if (d != 128) return nullptr;
  if (rh == 16 && nwg == 2) return reinterpret_cast<const void*>(&dev::pa_mtp_kernel<false, 128, false, 16, 2>);
  if (rh == 32 && nwg == 2) return reinterpret_cast<const void*>(&dev::pa_mtp_kernel<false, 128, false, 32, 2>);
  if (rh == 16 && nwg == 4) return reinterpret_cast<const void*>(&dev::pa_mtp_kernel<false, 128, false, 16, 4>);
  return nullptr;
}
}  // namespace pa
