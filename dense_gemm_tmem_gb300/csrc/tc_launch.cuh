// tc_launch.cuh: launcher template for one tc_gemm_kernel instantiation.
#pragma once

#include "internal.h"

namespace dg {

template <int BN, bool OUT_F16, bool TRANS>
cudaError_t launch_tc_inst(const TcLaunch& L) {
  using Cfg = TcConfig<BN>;
  auto kern = tc_gemm_kernel<BN, OUT_F16, TRANS>;
  // The attribute is per device context; setting it each launch is cheap and
  // keeps multi-device use correct.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kTcThreads, Cfg::kSmemBytes, L.stream>>>(L.tmA, L.tmB, L.args);
  return cudaGetLastError();
}

}  // namespace dg
