// simt_f16.cu: the fp16-input instantiations of the CUDA-core GEMM
// (simt_kernel.cuh): fp16 A and B widened to fp32, fp32 accumulation, fp16 or
// fp32 output.  Used for fp16 operands whose base address or leading
// dimension breaks the TMA rules of the tensor-core path.
#include "simt_kernel.cuh"

namespace dg {

cudaError_t launch_simt_f16(const SimtLaunch& L) {
  if (!L.in_f16) return cudaErrorInvalidValue;
  if (L.out_f16) return simt_detail::launch_simt_typed<__half, __half>(L);
  return simt_detail::launch_simt_typed<__half, float>(L);
}

}  // namespace dg
