// Instantiations with a 128-column MMA tile (mid shapes; swapped skinny M up to 128 when forced).
#include "tc_launch.cuh"

namespace dg {
cudaError_t launch_tc_n128(const TcLaunch& L) {
  if (L.trans)
    return L.out_f16 ? launch_tc_inst<128, true, true>(L) : launch_tc_inst<128, false, true>(L);
  return L.out_f16 ? launch_tc_inst<128, true, false>(L) : launch_tc_inst<128, false, false>(L);
}

// Cluster-split capacity: every instantiation uses one CTA per SM and about
// the same shared memory, so one of them stands for all.
int tc_max_active_clusters(int s) { return max_active_clusters_inst<128, false, false>(s); }

int lean_stages_n128(bool trans) {
  auto both = [](int a, int b) { return a < b ? a : b; };
  if (trans)
    return both(stages_for_two_per_sm<128, false, true>(kLeanMinStages),
                stages_for_two_per_sm<128, true, true>(kLeanMinStages));
  return both(stages_for_two_per_sm<128, false, false>(kLeanMinStages),
              stages_for_two_per_sm<128, true, false>(kLeanMinStages));
}
}  // namespace dg
