// FP8 e4m3 caches: tensor-memory consumer instantiations (head_dim 128 with
// 16 or 32 rows per softmax warpgroup, head_dim 256 with 16), and the
// dispatch over all tensor-memory instantiations.
#include "pa_mtp.cuh"

namespace pa {
const void* mtp_kernel_bf16(int d, int rh);

const void* mtp_kernel(int fp8, int d, int vtok, int rh) {
  if (!fp8) return mtp_kernel_bf16(d, rh);
  if (d == 128 && rh == 16)
    return vtok ? reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 128, true, 16>)
                : reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 128, false, 16>);
  if (d == 128 && rh == 32)
    return vtok ? reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 128, true, 32>)
                : reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 128, false, 32>);
  if (d == 256 && rh == 16)
    return vtok ? reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 256, true, 16>)
                : reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, 256, false, 16>);
  return nullptr;
}
}  // namespace pa
