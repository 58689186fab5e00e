// Instantiations of the two-SM (cta_group::2) kernel: fp16 or fp32 output.
#include "internal.h"
#include "tc2_kernel.cuh"

namespace dg {

namespace {
template <bool OUT_F16, int G>
cudaError_t launch_tc2_inst(const TcLaunch& L) {
  auto kern = tc2_gemm_kernel<OUT_F16, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Tc2Config::kSmemBytes);
  if (e != cudaSuccess) return e;
  // the cluster shape (2, 1, 1) is compiled into the kernel; grid is even
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(unsigned(L.grid), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = Tc2Config::kSmemBytes;
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1u : 0u;
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmC, L.args);
}
}  // namespace

cudaError_t launch_tc2(const TcLaunch& L) {
  if (L.trans || L.grid <= 0 || (L.grid & 1)) return cudaErrorInvalidValue;
  switch (L.args.kgroup) {  // k-blocks per stage: the operands' maps are encoded for it
    case 1: return L.out_f16 ? launch_tc2_inst<true, 1>(L) : launch_tc2_inst<false, 1>(L);
    case 2: return L.out_f16 ? launch_tc2_inst<true, 2>(L) : launch_tc2_inst<false, 2>(L);
    case 3: return L.out_f16 ? launch_tc2_inst<true, 3>(L) : launch_tc2_inst<false, 3>(L);
    default: return cudaErrorInvalidValue;
  }
}

int tc2_max_active_clusters(bool out_f16) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = Tc2Config::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e;
  if (out_f16) {
    e = cudaFuncSetAttribute(tc2_gemm_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tc2Config::kSmemBytes);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, tc2_gemm_kernel<true, 1>, &cfg);
  } else {
    e = cudaFuncSetAttribute(tc2_gemm_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tc2Config::kSmemBytes);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, tc2_gemm_kernel<false, 1>, &cfg);
  }
  return e == cudaSuccess ? n : -1;
}

}  // namespace dg
