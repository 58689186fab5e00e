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
  const int s = L.args.work.csplit;
  if (s > 8 || (s > 1 && L.grid % s != 0)) return cudaErrorInvalidValue;
  // Programmatic launch (the prologue may overlap the previous kernel; the
  // kernel waits for it before touching global memory) and, for the cluster
  // split, clusters of s CTAs along x, one tile per cluster.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (L.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (s > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = unsigned(s);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  const int stages = L.args.stages > 0 ? L.args.stages : Cfg::kStages;
  if (stages > Cfg::kStages) return cudaErrorInvalidValue;
  // whole groups of k-blocks; an MN-major box is at most 256 k deep
  const int J = L.args.kgroup;
  if (J < 1 || J > 4 || stages % J != 0) return cudaErrorInvalidValue;
  // a cluster split of a tile wider than 64 parks its partial in the ring
  if (s > 1 && BN > 64 &&
      int64_t(stages) * Cfg::kStageBytes < int64_t(kBM) * (BN + 4) * 4)
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3(unsigned(L.grid), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::smem_bytes(stages);
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(n);
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmC, L.args);
}

// The most ring stages (>= min_stages) with which two CTAs of this
// instantiation fit on one SM, or 0 if none do.
// The count comes from the kernel's registers and the SM's register file and
// shared memory (each CTA also holds the shared memory the system reserves).
template <int BN, bool OUT_F16, bool TRANS>
int stages_for_two_per_sm(int min_stages) {
  using Cfg = TcConfig<BN>;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, tc_gemm_kernel<BN, OUT_F16, TRANS>) != cudaSuccess) return 0;
  int dev = 0, regs_sm = 0, smem_sm = 0, reserved = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess)
    return 0;
  // registers are given out per warp, in units of 256
  const int warp_regs = ((fa.numRegs * 32 + 255) / 256) * 256;
  if (2 * (kTcThreads / 32) * warp_regs > regs_sm) return 0;
  for (int st = Cfg::kStages; st >= min_stages; --st)
    if (2 * (Cfg::smem_bytes(st) + fa.sharedSizeBytes + reserved) <= smem_sm) return st;
  return 0;
}

// Clusters of `s` CTAs of this instantiation that fit on the device at once.
template <int BN, bool OUT_F16, bool TRANS>
int max_active_clusters_inst(int s) {
  using Cfg = TcConfig<BN>;
  auto kern = tc_gemm_kernel<BN, OUT_F16, TRANS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::kSmemBytes) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(s);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(s), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess ? n : -1;
}

}  // namespace dg
