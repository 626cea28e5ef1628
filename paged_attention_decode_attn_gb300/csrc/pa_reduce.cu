// Standalone partition reducer (the fallback merge: one CTA per unit).
#include "pa_tile.cuh"

namespace pa {
namespace dev {
__global__ void __launch_bounds__(128) pa_reduce_kernel_d64(const __grid_constant__ PaParams p) { reduce_unit<64>(p); }
__global__ void __launch_bounds__(128) pa_reduce_kernel_d128(const __grid_constant__ PaParams p) { reduce_unit<128>(p); }
__global__ void __launch_bounds__(128) pa_reduce_kernel_d256(const __grid_constant__ PaParams p) { reduce_unit<256>(p); }
}  // namespace dev

const void* reduce_kernel(int d) {
  if (d == 64) return reinterpret_cast<const void*>(&dev::pa_reduce_kernel_d64);
  if (d == 128) return reinterpret_cast<const void*>(&dev::pa_reduce_kernel_d128);
  if (d == 256) return reinterpret_cast<const void*>(&dev::pa_reduce_kernel_d256);
  return nullptr;
}
}  // namespace pa
