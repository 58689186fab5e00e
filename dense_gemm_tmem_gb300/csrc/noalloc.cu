// noalloc.cu: gemm_run_noalloc, the tensor-core GEMM for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs inside a host application which owns the
// device's memory, for example a plugin in a framework whose caching allocator
// has reserved the memory up front (a cudaMalloc of its own may fail, or would
// bypass the framework's accounting), and latency-critical paths where a
// cudaMalloc or cudaFree would synchronise the device.  gemm_create allocates
// the split workspace with cudaMalloc; this entry point needs no handle and
// allocates nothing: its scratch lives in a fixed array compiled into the
// library, which every GPU that loads the library holds until the process exits.
//
// It launches the same tc_gemm_kernel that gemm_run launches, with the same
// picker, and points the kernel's split workspace, tile counters and status word
// into that array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc2_kernel.cuh"

namespace dg {
namespace {

// Scratch layout (bytes): fp32 partial tiles, then the split-tile counters,
// then one device status word.
constexpr size_t kNaPartialBytes = size_t(16) << 20;   // 16 MiB of partial tiles
constexpr int kNaCounters = 4096;                      // split tiles per call
constexpr size_t kNaCounterOff = kNaPartialBytes;
constexpr size_t kNaStatusOff = kNaCounterOff + sizeof(int) * kNaCounters;
constexpr size_t kNaScratchBytes = kNaStatusOff + 256;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

constexpr int kNaMaxDevices = 64;

struct DeviceScratch {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch
  int num_sms = 0;
  int pairs = 0;                  // CTA pairs of the two-SM kernel resident at once
  int csplit_clusters[9] = {};    // clusters of s one-SM CTAs resident at once
};

std::mutex g_na_mu;
DeviceScratch g_na_dev[kNaMaxDevices];

// Once per device, with that device current: the array's device address and
// the SM count.  Returns GEMM_OK or an error code.
int scratch_for_device(int device, DeviceScratch* out) {
  if (device < 0 || device >= kNaMaxDevices) return GEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(g_na_mu);
  DeviceScratch& d = g_na_dev[device];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return GEMM_ERR_CUDA;
    d.base = static_cast<unsigned char*>(ptr);
    d.num_sms = sms;
    const int pairs = tc2_max_active_clusters(true);
    d.pairs = pairs > 0 ? (pairs < sms / 2 ? pairs : sms / 2) : sms / 2;
    for (int s : {2, 4, 8}) {
      const int n = tc_max_active_clusters(s);
      d.csplit_clusters[s] = n > 0 ? (n < sms / s ? n : sms / s) : n == 0 ? -1 : sms / s;
    }
    d.ready = true;
  }
  *out = d;
  return GEMM_OK;
}

// One fp16 operand's tensor map, encoded per call (no cache: nothing to own).
// Same geometry as gemm_run's: K-major {K, rows} with a {64, box_rows} box,
// MN-major {rows, K} with a {64, 64} box, 128-byte swizzle, zero fill.
int encode_operand_na(CUtensorMap* out, const void* ptr, int64_t rows, int64_t K, int mn_major,
                      int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GEMM_ERR_CUDA;
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], estr[2] = {1, 1};
  if (!mn_major) {
    dims[0] = cuuint64_t(K);
    dims[1] = cuuint64_t(rows);
    strides[0] = cuuint64_t(K) * 2;
    box[0] = kBK;
    box[1] = cuuint32_t(box_rows);
  } else {
    dims[0] = cuuint64_t(rows);
    dims[1] = cuuint64_t(K);
    strides[0] = cuuint64_t(rows) * 2;
    box[0] = 64;
    box[1] = kBK;
  }
  const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace
}  // namespace dg

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                                const float* bias, void* C, gemm_layout_t layout,
                                void* stream_ptr, int* dev_status) {
  using namespace dg;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return GEMM_ERR_CUDA;
  DeviceScratch sc;
  int rc = scratch_for_device(device, &sc);
  if (rc != GEMM_OK) return rc;

  Options opt;
  opt.pair_clusters = sc.pairs;
  opt.pair_split = 0;  // two-SM plans stay whole tiles: their split needs more than the array
  for (int s = 0; s < 9; ++s) opt.csplit_clusters[s] = sc.csplit_clusters[s];
  gemm_plan_t plan;
  rc = plan_for(M, N, K, layout, sc.num_sms, opt, &plan);
  if (rc != GEMM_OK) return rc;
  if (plan.kernel == GEMM_KERNEL_NONE) return GEMM_OK;
  if (plan.kernel == GEMM_KERNEL_SIMT) return GEMM_ERR_UNSUPPORTED;  // fp16 inputs only
  if (!C) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  if (plan.kernel == GEMM_KERNEL_FILL)
    return launch_fill(M, N, bias, C, layout.out_dtype == GEMM_F16, stream) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
  if (!A || !B) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))
    return GEMM_ERR_UNSUPPORTED;

  // Fit the split into the fixed scratch: fewer CTAs if its partial tiles
  // would not fit, and a clear refusal if its tiles outnumber the counters.
  if (plan.workspace_bytes > int64_t(kNaPartialBytes)) {
    const int64_t per_cta = int64_t(2) * kBM * plan.tile_n * int64_t(sizeof(float));
    opt.force_grid = int(kNaPartialBytes / per_cta);
    rc = plan_for(M, N, K, layout, sc.num_sms, opt, &plan);
    if (rc != GEMM_OK) return rc;
  }
  // Only the Stream-K split counts arrivals per tile; the cluster split adds
  // its partials on chip and the whole-tile plans need no counters.
  if (plan.workspace_bytes > int64_t(kNaPartialBytes) ||
      (plan.kernel == GEMM_KERNEL_STREAMK && plan.sk_tiles > kNaCounters))
    return GEMM_ERR_UNSUPPORTED;

  float* partials = reinterpret_cast<float*>(sc.base);
  int* counters = reinterpret_cast<int*>(sc.base + kNaCounterOff);
  int* own_status = reinterpret_cast<int*>(sc.base + kNaStatusOff);
  int* status = dev_status ? dev_status : own_status;

  // The counters must start at zero, and so must the array's own status word
  // when it stands in for the caller's: the array keeps whatever the last
  // call (possibly an aborted one) left there.
  if (plan.kernel == GEMM_KERNEL_STREAMK &&
      cudaMemsetAsync(counters, 0, sizeof(int) * size_t(plan.sk_tiles), stream) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (!dev_status && cudaMemsetAsync(own_status, 0, sizeof(int), stream) != cudaSuccess)
    return GEMM_ERR_CUDA;

  const bool swap = plan.swap_ab != 0;
  const int64_t Mm = swap ? N : M;
  const int64_t Nm = swap ? M : N;
  const bool pair = plan.kernel == GEMM_KERNEL_TC2;  // whole tiles: no scratch but status
  TcLaunch L;
  L.bm = pair ? kPairBM : plan.tile_m;
  L.bn = plan.tile_n;
  L.out_f16 = layout.out_dtype == GEMM_F16;
  L.trans = swap;
  L.pair = pair;
  L.grid = plan.grid;
  L.stream = stream;
  rc = encode_operand_na(&L.tmA, swap ? B : A, Mm, K, plan.a_mn_major, pair ? kBM : plan.tile_m);
  if (rc != GEMM_OK) return rc;
  rc = encode_operand_na(&L.tmB, swap ? A : B, Nm, K, plan.b_mn_major,
                         pair ? kHalfBN : plan.tile_n);
  if (rc != GEMM_OK) return rc;
  TcArgs& a = L.args;
  a.work = spec_of(plan);
  a.Mm = int32_t(Mm);
  a.Nm = int32_t(Nm);
  a.C = C;
  a.ldc = N;
  a.bias = bias;
  a.workspace = partials;
  a.tickets = counters;
  a.status = status;
  a.wait_limit_ns = opt.wait_limit_ns;
  a.a_mn = plan.a_mn_major;
  a.b_mn = plan.b_mn_major;
  a.idesc = make_idesc_f16(pair ? kPairBM : plan.tile_m, plan.tile_n, plan.a_mn_major,
                           plan.b_mn_major);
  a.trace = nullptr;
  std::memset(&L.tmC, 0, sizeof(L.tmC));
  a.c_tma = 0;  // plain stores: no output tensor map to encode and keep
  const int64_t c_pitch = N * (layout.out_dtype == GEMM_F16 ? 2 : 4);
  a.c_vec = (!swap && (reinterpret_cast<uintptr_t>(C) & 15) == 0 && c_pitch % 16 == 0) ? 1 : 0;
  a.bias_init = 0;
  return launch_tc(L) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
