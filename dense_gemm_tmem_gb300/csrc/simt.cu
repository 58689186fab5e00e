// simt.cu: fp32 CUDA-core GEMM, C = A·B (+bias), true FFMA (no TF32).
//
// Each technique of the "TVM Matrix Multiplication Optimization" ladder
// (kimm240.github.io/tvm, Steps 1-6) has its place here:
//   Step 1 data-parallel 2-D thread map    -> 2-D grid of 128x128 output tiles
//   Step 2 tiling + loop reordering        -> each thread owns an 8x8 register tile
//                                             and runs the k loop outermost
//   Step 3 shared memory, cooperative fetch-> all 256 threads stage a 128x8 A block
//                                             and an 8x128 B block per k-step
//   Step 4 vectorisation + register caching-> float4 global and shared loads;
//                                             accumulators live in registers
//   Step 5 software pipelining             -> two shared-memory buffers; the next
//                                             block is fetched into registers
//                                             while the current one is consumed
//   Step 6 unrolling                       -> the k-step and the 8x8 FMA nest are
//                                             fully unrolled
// The staging rows are padded as storage_align(factor 32, offset 4) pads them
// (leiblog.wang, the storage_align answer: the stride is raised to the next
// value congruent to offset mod factor), 128 -> 132 floats, which makes the
// transposed A stores free of bank conflicts.
#include "internal.h"

namespace dg {

namespace {

// storage_align(factor, offset) applied to a row of `extent` elements.
constexpr int aligned_stride(int extent, int factor, int offset) {
  return extent + (factor + offset - extent % factor) % factor;
}
constexpr int kAS = aligned_stride(kSimtBM, 32, 4);
constexpr int kBS = aligned_stride(kSimtBN, 32, 4);
static_assert(kAS == 132 && kBS == 132, "padded staging strides");

struct SimtArgs {
  int64_t M, N, K;
  const float* A;
  const float* B;
  const float* bias;
  float* C;
  bool vec_a, vec_b, vec_c;  // float4 access allowed (16-byte aligned rows)
};

template <bool A_COL, bool B_COL>
__global__ void __launch_bounds__(kSimtThreads, 2) simt_sgemm_kernel(const SimtArgs a) {
  constexpr int BM = kSimtBM, BN = kSimtBN, BK = kSimtBK;
  __shared__ __align__(16) float As[2][BK][kAS];
  __shared__ __align__(16) float Bs[2][BK][kBS];

  const int t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;
  const int64_t m0 = int64_t(blockIdx.y) * BM;
  const int64_t n0 = int64_t(blockIdx.x) * BN;
  const int64_t M = a.M, N = a.N, K = a.K;

  float ra[4], rb[4];
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // Global -> registers for k-block k0 (zero outside the matrix).
  auto fetch = [&](int64_t k0) {
    if (!A_COL) {  // A row-major: row m, 4 consecutive k
      const int64_t m = m0 + (t >> 1), k = k0 + (t & 1) * 4;
      const float* p = a.A + m * K + k;
      if (a.vec_a && m < M && k + 3 < K) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        ra[0] = v.x; ra[1] = v.y; ra[2] = v.z; ra[3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) ra[i] = (m < M && k + i < K) ? __ldg(p + i) : 0.f;
      }
    } else {       // A column-major (K x M storage): row k, 4 consecutive m
      const int64_t k = k0 + (t >> 5), m = m0 + (t & 31) * 4;
      const float* p = a.A + k * M + m;
      if (a.vec_a && k < K && m + 3 < M) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        ra[0] = v.x; ra[1] = v.y; ra[2] = v.z; ra[3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) ra[i] = (k < K && m + i < M) ? __ldg(p + i) : 0.f;
      }
    }
    if (!B_COL) {  // B row-major: row k, 4 consecutive n
      const int64_t k = k0 + (t >> 5), n = n0 + (t & 31) * 4;
      const float* p = a.B + k * N + n;
      if (a.vec_b && k < K && n + 3 < N) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        rb[0] = v.x; rb[1] = v.y; rb[2] = v.z; rb[3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) rb[i] = (k < K && n + i < N) ? __ldg(p + i) : 0.f;
      }
    } else {       // B column-major (N x K storage): column n, 4 consecutive k
      const int64_t n = n0 + (t >> 1), k = k0 + (t & 1) * 4;
      const float* p = a.B + n * K + k;
      if (a.vec_b && n < N && k + 3 < K) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        rb[0] = v.x; rb[1] = v.y; rb[2] = v.z; rb[3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) rb[i] = (n < N && k + i < K) ? __ldg(p + i) : 0.f;
      }
    }
  };

  // Registers -> shared buffer `buf`, as As[k][m] and Bs[k][n].
  auto stage = [&](int buf) {
    if (!A_COL) {
      const int m = t >> 1, k = (t & 1) * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) As[buf][k + i][m] = ra[i];
    } else {
      const int k = t >> 5, m = (t & 31) * 4;
      *reinterpret_cast<float4*>(&As[buf][k][m]) = make_float4(ra[0], ra[1], ra[2], ra[3]);
    }
    if (!B_COL) {
      const int k = t >> 5, n = (t & 31) * 4;
      *reinterpret_cast<float4*>(&Bs[buf][k][n]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
    } else {
      const int n = t >> 1, k = (t & 1) * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) Bs[buf][k + i][n] = rb[i];
    }
  };

  const int64_t nk = (K + BK - 1) / BK;
  fetch(0);
  stage(0);
  __syncthreads();
  for (int64_t kt = 0; kt < nk; ++kt) {
    const int buf = int(kt & 1);
    if (kt + 1 < nk) fetch((kt + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (kt + 1 < nk) stage(buf ^ 1);
    __syncthreads();
  }

  // Epilogue: + bias[n], rows ty*4+i (+64), columns tx*4+j (+64).
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t n = n0 + h * 64 + tx * 4;
      if (n >= N) continue;
      float o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = acc[i][h * 4 + j] + ((a.bias && n + j < N) ? __ldg(a.bias + n + j) : 0.f);
      float* dst = a.C + m * N + n;
      if (a.vec_c && n + 3 < N) {
        *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n + j < N) dst[j] = o[j];
      }
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int simt_a_stride() { return kAS; }
int simt_b_stride() { return kBS; }

cudaError_t launch_simt(const SimtLaunch& L) {
  SimtArgs a;
  a.M = L.M; a.N = L.N; a.K = L.K;
  a.A = L.A; a.B = L.B; a.bias = L.bias; a.C = L.C;
  a.vec_a = aligned16(L.A) && ((L.a_major == 0 ? L.K : L.M) % 4 == 0);
  a.vec_b = aligned16(L.B) && ((L.b_major == 0 ? L.N : L.K) % 4 == 0);
  a.vec_c = aligned16(L.C) && (L.N % 4 == 0);
  const int64_t gx = (L.N + kSimtBN - 1) / kSimtBN;
  const int64_t gy = (L.M + kSimtBM - 1) / kSimtBM;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid{unsigned(gx), unsigned(gy), 1u};
  if (L.a_major == 0 && L.b_major == 0)
    simt_sgemm_kernel<false, false><<<grid, kSimtThreads, 0, L.stream>>>(a);
  else if (L.a_major == 0)
    simt_sgemm_kernel<false, true><<<grid, kSimtThreads, 0, L.stream>>>(a);
  else if (L.b_major == 0)
    simt_sgemm_kernel<true, false><<<grid, kSimtThreads, 0, L.stream>>>(a);
  else
    simt_sgemm_kernel<true, true><<<grid, kSimtThreads, 0, L.stream>>>(a);
  return cudaGetLastError();
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
