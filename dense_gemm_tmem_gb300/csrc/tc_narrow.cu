// Instantiations with 32/64-column MMA tiles, operands not swapped: small
// shapes split into more, narrower output tiles instead of a k-split.
#include "tc_launch.cuh"

namespace dg {
cudaError_t launch_tc_narrow(const TcLaunch& L) {
  if (L.trans) return cudaErrorInvalidValue;
  switch (L.bn) {
    case 32:
      return L.out_f16 ? launch_tc_inst<32, true, false>(L) : launch_tc_inst<32, false, false>(L);
    case 64:
      return L.out_f16 ? launch_tc_inst<64, true, false>(L) : launch_tc_inst<64, false, false>(L);
    default:
      return cudaErrorInvalidValue;
  }
}

int lean_stages_narrow(int bn) {
  auto both = [](int a, int b) { return a < b ? a : b; };
  switch (bn) {
    case 32:
      return both(stages_for_two_per_sm<32, false, false>(kLeanMinStages),
                  stages_for_two_per_sm<32, true, false>(kLeanMinStages));
    case 64:
      return both(stages_for_two_per_sm<64, false, false>(kLeanMinStages),
                  stages_for_two_per_sm<64, true, false>(kLeanMinStages));
    default:
      return 0;
  }
}
}  // namespace dg
