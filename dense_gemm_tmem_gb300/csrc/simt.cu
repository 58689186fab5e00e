// simt.cu: the fp32-input instantiations of the CUDA-core GEMM
// (simt_kernel.cuh), its host-side queries, and the K == 0 fill kernel.
#include "simt_kernel.cuh"

namespace dg {

int simt_a_stride() { return simt_detail::aligned_stride(kSimtBM, 32, 4); }
int simt_b_stride() { return simt_detail::aligned_stride(kSimtBN, 32, 4); }

int simt_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, simt_detail::simt_sgemm_kernel<float, float, kSimtBM, kSimtBN, false, false, true>,
          kSimtThreads, 0) != cudaSuccess)
    return -1;
  return n;
}

cudaError_t launch_simt(const SimtLaunch& L) {
  if (L.in_f16) return launch_simt_f16(L);
  if (L.out_f16) return cudaErrorInvalidValue;  // fp32 inputs give fp32 outputs
  return simt_detail::launch_simt_typed<float, float>(L);
}

// ---------------------------------------------------------------- K == 0 --
namespace {
template <bool OUT_F16>
__global__ void fill_bias_kernel(int64_t M, int64_t N, const float* bias, void* C) {
  const int64_t total = M * N;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float v = bias ? bias[i % N] : 0.f;
    if (OUT_F16)
      reinterpret_cast<__half*>(C)[i] = __float2half_rn(v);
    else
      reinterpret_cast<float*>(C)[i] = v;
  }
}
}  // namespace

cudaError_t launch_fill(int64_t M, int64_t N, const float* bias, void* C, bool out_f16,
                        cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (out_f16)
    fill_bias_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(M, N, bias, C);
  else
    fill_bias_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(M, N, bias, C);
  return cudaGetLastError();
}

}  // namespace dg
