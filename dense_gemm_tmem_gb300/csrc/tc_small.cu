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

int lean_stages_small(int bn) {
  auto both = [](int a, int b) { return a < b ? a : b; };
  switch (bn) {
    case 16:
      return both(stages_for_two_per_sm<16, false, true>(kLeanMinStages),
                  stages_for_two_per_sm<16, true, true>(kLeanMinStages));
    case 32:
      return both(stages_for_two_per_sm<32, false, true>(kLeanMinStages),
                  stages_for_two_per_sm<32, true, true>(kLeanMinStages));
    case 64:
      return both(stages_for_two_per_sm<64, false, true>(kLeanMinStages),
                  stages_for_two_per_sm<64, true, true>(kLeanMinStages));
    default:
      return 0;
  }
}
}  // namespace dg
