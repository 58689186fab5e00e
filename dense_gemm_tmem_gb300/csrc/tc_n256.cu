// Instantiations with a 256-column MMA tile (large shapes).
#include "tc_launch.cuh"

namespace dg {
cudaError_t launch_tc_n256(const TcLaunch& L) {
  if (L.trans) return cudaErrorInvalidValue;
  return L.out_f16 ? launch_tc_inst<256, true, false>(L) : launch_tc_inst<256, false, false>(L);
}
}  // namespace dg
