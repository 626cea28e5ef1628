// BF16 caches: tcgen05-consumer instantiation (head_dim 128), and the
// dispatch over all tcgen05 instantiations.
#include "pa_umma.cuh"

namespace pa {
const void* umma_kernel_fp8(int d, int vtok);

const void* umma_kernel(int fp8, int d, int vtok) {
  if (fp8) return umma_kernel_fp8(d, vtok);
  if (d == 128) return reinterpret_cast<const void*>(&dev::pa_umma_kernel<false, 128, false>);
  return nullptr;
}
}  // namespace pa
