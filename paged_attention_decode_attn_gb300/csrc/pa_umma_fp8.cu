// FP8 e4m3 caches: tcgen05-consumer instantiations (head_dim 128 and 256).
#include "pa_umma.cuh"

namespace pa {
const void* umma_kernel_fp8(int d, int vtok) {
  if (d == 128) return vtok ? reinterpret_cast<const void*>(&dev::pa_umma_kernel<true, 128, true>)
                            : reinterpret_cast<const void*>(&dev::pa_umma_kernel<true, 128, false>);
  if (d == 256) return vtok ? reinterpret_cast<const void*>(&dev::pa_umma_kernel<true, 256, true>)
                            : reinterpret_cast<const void*>(&dev::pa_umma_kernel<true, 256, false>);
  return nullptr;
}
}  // namespace pa
