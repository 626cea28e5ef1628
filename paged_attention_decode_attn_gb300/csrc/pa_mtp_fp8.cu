// FP8 e4m3 caches: tensor-memory consumer instantiations (head_dim 128 with
// two warpgroups of 16 rows, two of 32 or four of 16; head_dim 256 with two of
// 16), and the dispatch over all tensor-memory instantiations.
#include "pa_mtp.cuh"

namespace pa {
const void* mtp_kernel_bf16(int d, int rh, int nwg);

namespace {
template <int D, int RH, int NWG>
const void* fp8_kernel(int vtok) {
  return vtok ? reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, D, true, RH, NWG>)
              : reinterpret_cast<const void*>(&dev::pa_mtp_kernel<true, D, false, RH, NWG>);
}
}  // namespace

const void* mtp_kernel(int fp8, int d, int vtok, int rh, int nwg) {
  if (!fp8) return mtp_kernel_bf16(d, rh, nwg);
  if (d == 128 && rh == 16 && nwg == 2) return fp8_kernel<128, 16, 2>(vtok);
  if (d == 128 && rh == 32 && nwg == 2) return fp8_kernel<128, 32, 2>(vtok);
  if (d == 128 && rh == 16 && nwg == 4) return fp8_kernel<128, 16, 4>(vtok);
  if (d == 256 && rh == 16 && nwg == 2) return fp8_kernel<256, 16, 2>(vtok);
  return nullptr;
}
}  // namespace pa
