// internal.h: host-side declarations shared by the API and the kernel launch
// files (not part of the public C-ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gemm.h"
#include "tc_kernel.cuh"

namespace dg {

// Picker options (gemm_set_option; defaults below).
struct Options {
  int force_kernel = -1;
  int force_tile_n = -1;
  int force_grid = -1;
  int min_split_iters = 0;  // 0: per tile width, so k-work outweighs the partial
  int force_swap = -1;
  int group_m = 0;         // tile rows per raster group; 0: 2048 rows of A per group
  int pair = -1;           // two-SM kernel: 0 never, 1 whenever possible, -1 picker's rule
  int pair_clusters = 0;   // CTA pairs resident at once (0: SMs / 2); set per device
  int csplit = -1;         // cluster split: -1 picker's rule, 0 never, 2/4/8 forced
  int pdl = 1;             // programmatic dependent launch of the tensor-core kernels
  int pair_split = -1;     // two-SM kernel k-split: -1/0 none, 1 all tiles, 2 the tail
  int tma_store = -1;      // epilogue output by TMA store where C allows it: -1 for fp16
                           // output or more output tiles than CTAs, 1 always, 0 never
  int bias_init = 0;       // seed the accumulators with the bias
  int dyn_sched = 0;       // two-SM kernel, whole tiles: 1 tiles handed out at run time
  int stages = -1;         // one-SM kernel ring stages: -1 picker, n >= 1 forced
  int tile_m = -1;         // one-SM kernel tile rows: -1 picker, 64 or 128 forced
  int k_group = -1;        // k-blocks per TMA copy (64-row kernel): -1 picker, 1/2/4 forced
  // per tile width (16, 32, 64, 128, 256 -> 0..4) and operand order: the most
  // stages that let two CTAs share an SM (0: none); set per device
  int lean_stages[5][2] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}, {0, 0}};
  int csplit_clusters[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};  // clusters of s resident (0: SMs/s)
  int simt_per_sm = 0;     // 128 x 128 CUDA-core CTAs resident per SM (0: 2); set per device
  uint64_t wait_limit_ns = 2000000000ull;
};

// The tile picker (api.cu).
int plan_for(int64_t M, int64_t N, int64_t K, gemm_layout_t L, int num_sms,
             const Options& o, gemm_plan_t* p);
WorkSpec spec_of(const gemm_plan_t& p);

// cuTensorMapEncodeTiled, reached through the runtime's entry-point query
// (NULL if the driver does not provide it).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// One tensor-core launch, fully described.
struct TcLaunch {
  int bm = 128;       // MMA M tile of the one-SM kernels: 128, or 64 (tc64.cu)
  int bn;             // MMA N tile: 16, 32, 64, 128 or 256
  bool out_f16;
  bool trans;         // swapped operands, transposed store
  bool pair = false;  // two-SM kernel (cluster pairs, 256 x 256 tiles)
  bool pdl = true;    // programmatic launch: prologue may overlap the previous kernel
  int grid;
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmC;  // row-major C, 32 x 32 boxes; used only when args.c_tma
  TcArgs args;
  cudaStream_t stream;
};

// Launches the matching tc_gemm_kernel instantiation (sets its shared-memory
// attribute on first use).  Returns cudaErrorInvalidValue for a combination
// that has no instantiation.
cudaError_t launch_tc(const TcLaunch& L);
cudaError_t launch_tc_n256(const TcLaunch& L);
cudaError_t launch_tc_n128(const TcLaunch& L);
cudaError_t launch_tc_small(const TcLaunch& L);
cudaError_t launch_tc_narrow(const TcLaunch& L);
// Two-SM kernel (tc2.cu): even grid, not swapped, whole 256 x 256 tiles.
cudaError_t launch_tc2(const TcLaunch& L);
// One-SM kernel with 64-row tiles (tc64.cu): not swapped, whole tiles.
cudaError_t launch_tc64(const TcLaunch& L);
int tc64_stages_for(int bn);
// Clusters of two that fit on the device at once (-1 if the query fails).
int tc2_max_active_clusters(bool out_f16);
// Clusters of s one-SM CTAs (cluster split) that fit at once (-1 on failure).
int tc_max_active_clusters(int s);
int tc_stages_for(int bn);
int tc_smem_bytes_for(int bn);
// Fewest ring stages a launch of tile width bn with a cluster split of
// csplit may use (a tile wider than 64 parks its fp32 partial in the ring).
int tc_min_stages(int bn, int csplit);
// Fewest stages, and fewest bytes of loads in flight, a launch that shares
// its SMs with the next launch's CTAs may keep.
constexpr int kLeanMinStages = 3;
constexpr int64_t kLeanMinInflight = 88 * 1024;
// The most ring stages with which two CTAs of the one-SM kernel of tile width
// bn (either output type) fit on one SM, or 0: the per-file queries and the
// dispatcher over them.
int lean_stages_small(int bn);
int lean_stages_narrow(int bn);
int lean_stages_n128(bool trans);
int tc_lean_stages(int bn, bool trans);

// CUDA-core GEMM with fp32 accumulation (simt_kernel.cuh): fp32 inputs
// (simt.cu), or fp16 inputs the tensor-core path cannot read (simt_f16.cu).
struct SimtLaunch {
  int64_t M, N, K;
  const void* A;         // fp32, or fp16 when in_f16
  const void* B;
  const float* bias;
  void* C;               // fp32, or fp16 when out_f16 (fp16 inputs only)
  bool in_f16 = false;
  bool out_f16 = false;
  int a_major, b_major;  // 0 row, 1 column
  int tile = 128;        // square tile edge: kSimtBM (128) or kSimtSmallTile (64)
  WorkSpec work;         // grid, tiles, raster order and k-split (work.cuh)
  float* workspace = nullptr;  // split partials (2 tile slots per CTA) when work.sk_tiles > 0
  int* tickets = nullptr;      // split-tile arrival counters, all 0 between launches
  cudaStream_t stream;
};
cudaError_t launch_simt(const SimtLaunch& L);
cudaError_t launch_simt_f16(const SimtLaunch& L);
constexpr int kSimtBM = 128, kSimtBN = 128, kSimtBK = 16;
constexpr int kSimtThreads = 128;  // 128 x 128 tile: 16 x 8 outputs per thread
constexpr int kSimtSmallTile = 64;  // 64 x 64 tiles, 64 threads
constexpr int kSimtMinSplitIters = 8;  // fewest k-blocks a split CTA gets
// CTAs of the 128 x 128 kernel resident on one SM (-1 if the query fails).
int simt_ctas_per_sm();
int simt_a_stride();
int simt_b_stride();

// K == 0: C = bias (or 0) (fill.cu).
cudaError_t launch_fill(int64_t M, int64_t N, const float* bias, void* C, bool out_f16,
                        cudaStream_t stream);

// One CTA whose bounded wait never completes (selftest.cu).
cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, cudaStream_t stream);

}  // namespace dg
