// Instantiations of the 64-row one-SM kernel (tc64_kernel.cuh): 32/64/128-wide
// tiles, fp16 or fp32 output.
#include "internal.h"
#include "tc64_kernel.cuh"

namespace dg {

namespace {
template <int BN, bool OUT_F16>
cudaError_t launch_tc64_inst(const TcLaunch& L) {
  using Cfg = Tc64Config<BN>;
  auto kern = tc64_gemm_kernel<BN, OUT_F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int stages = L.args.stages > 0 ? L.args.stages : Cfg::kStages;
  const int J = L.args.kgroup;
  if (stages > Cfg::kStages || L.args.work.csplit > 1 || L.args.work.sk_tiles > 0)
    return cudaErrorInvalidValue;  // whole tiles only
  // whole groups of J k-blocks; an MN-major box is at most 256 k deep
  if (J < 1 || J > 4 || stages % J != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(unsigned(L.grid), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::smem_bytes(stages);
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = L.pdl ? 1u : 0u;
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.args);
}
}  // namespace

cudaError_t launch_tc64(const TcLaunch& L) {
  if (L.trans) return cudaErrorInvalidValue;
  switch (L.bn) {
    case 32: return L.out_f16 ? launch_tc64_inst<32, true>(L) : launch_tc64_inst<32, false>(L);
    case 64: return L.out_f16 ? launch_tc64_inst<64, true>(L) : launch_tc64_inst<64, false>(L);
    case 128:
      return L.out_f16 ? launch_tc64_inst<128, true>(L) : launch_tc64_inst<128, false>(L);
    default: return cudaErrorInvalidValue;
  }
}

int tc64_stages_for(int bn) {
  switch (bn) {
    case 32: return Tc64Config<32>::kStages;
    case 64: return Tc64Config<64>::kStages;
    default: return Tc64Config<128>::kStages;
  }
}

}  // namespace dg
