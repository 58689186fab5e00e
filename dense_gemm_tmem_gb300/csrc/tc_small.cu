// Instantiations with 16/32/64-column MMA tiles: swapped operands for skinny M.
#include "tc_launch.cuh"

namespace dg {
cudaError_t launch_tc_small(const TcLaunch& L) {
  if (!L.trans) return cudaErrorInvalidValue;
  switch (L.bn) {
    case 16:
      return L.out_f16 ? launch_tc_inst<16, true, true>(L) : launch_tc_inst<16, false, true>(L);
    case 32:
      return L.out_f16 ? launch_tc_inst<32, true, true>(L) : launch_tc_inst<32, false, true>(L);
    case 64:
      return L.out_f16 ? launch_tc_inst<64, true, true>(L) : launch_tc_inst<64, false, true>(L);
    default:
      return cudaErrorInvalidValue;
  }
}
}  // namespace dg
