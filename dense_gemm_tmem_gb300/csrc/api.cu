// api.cu: the C-ABI (include/gemm.h): handle, argument checks, tile picker,
// TMA descriptor encoding with a small cache, and kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/gemm.h"
#include "internal.h"
#include "tc2_kernel.cuh"

namespace dg {

constexpr int kMaxTileN = 256;
constexpr int kNarrowIters = 12;  // deepest K (in k-blocks) for which narrow whole tiles win
constexpr int kTicketCap = 16384;     // split tiles one launch may have
// after the tickets: the two-SM kernel's tile counter and finished-pair count
constexpr int kCounterInts = kTicketCap + 2;
constexpr int kTmapCacheSize = 32;
constexpr int64_t kMaxCoord = (int64_t(1) << 31) - 1024;  // TMA coordinates are int32

struct TmapKey {
  const void* ptr;
  int64_t rows, k;
  int mn_major, box_rows;
  int kind;  // 0 fp16 operand, 1 fp32 output, 2 fp16 output
  int kgroup;  // k-blocks per box (operands)
  bool operator==(const TmapKey& o) const {
    return ptr == o.ptr && rows == o.rows && k == o.k && mn_major == o.mn_major &&
           box_rows == o.box_rows && kind == o.kind && kgroup == o.kgroup;
  }
};

struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool valid = false;
};

namespace {

bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GEMM_LOG");
    return v && v[0] && v[0] != '0';
  }();
  return on;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile width 16, 32, 64, 128, 256 -> 0 ... 4 (Options::lean_stages).
int width_index(int bn) { return bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : 4; }

// Allocation-failure injection (gemm_inject_alloc_failure): when armed with n,
// the n-th device allocation from now fails as if the device were full.
std::atomic<int64_t> g_fail_alloc_in{0};

cudaError_t dev_malloc(void** p, size_t bytes) {
  int64_t n = g_fail_alloc_in.load();
  while (n > 0 && !g_fail_alloc_in.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 1) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

}  // namespace

// ------------------------------------------------------------ tile picker --
// The CUDA-core kernel's plan (fp32 inputs, and fp16 inputs the tensor-core
// path cannot read).
int plan_simt(int64_t M, int64_t N, int64_t K, int num_sms, const Options& o, gemm_plan_t* p) {
  // 128x128 tiles (256 threads, 2 CTAs per SM), their k-blocks split over the
  // resident CTAs when the tiles are too few.  Only when even that split
  // would run fewer than 8 CTAs do 64x64 tiles (64 threads) spread the work
  // wider.  Measured (graph replay, cold inputs, TFLOP/s, 128-tile split vs
  // 64-tiles): 1024^3 35.1 vs 22.7, 512^3 10.9 vs 5.5, 1536^3 47.0 vs 41.1,
  // 4096x256x4096 47.4 vs 23.8; 128^3 (one 128-tile) 0.25 vs 0.37.
  const int min_iters = o.min_split_iters > 0 ? o.min_split_iters : kSimtMinSplitIters;
  int tile;
  if (o.force_tile_n > 0) {
    if (o.force_tile_n != kSimtBM && o.force_tile_n != kSimtSmallTile)
      return GEMM_ERR_UNSUPPORTED;
    tile = o.force_tile_n;
  } else {
    const int64_t big = ceil_div(M, kSimtBM) * ceil_div(N, kSimtBN);
    const int64_t big_split = std::max(big, big * ceil_div(K, kSimtBK) / min_iters);
    tile = big_split >= 8 ? kSimtBM : kSimtSmallTile;
  }
  const int64_t tiles_m = ceil_div(M, tile), tiles_n = ceil_div(N, tile);
  const int64_t T = tiles_m * tiles_n;
  const int64_t I = ceil_div(K, kSimtBK);
  if (T > INT32_MAX / 2 || I > INT32_MAX / 2 || T * I > (int64_t(1) << 40))
    return GEMM_ERR_UNSUPPORTED;
  // Resident CTAs (the split's grid), capped so two partial slots per CTA
  // fit the handle's workspace.
  const int64_t per_sm = o.simt_per_sm > 0 ? std::min(o.simt_per_sm, 2) : 2;
  const int64_t S = per_sm * num_sms;
  int64_t dp = T, sk = 0, grid = T;
  if (o.force_grid > 0) {
    // forced grid: every tile's k-blocks split over that many CTAs
    dp = 0;
    sk = T;
    grid = std::min<int64_t>({o.force_grid, S, T * I});
    if (grid == T) {
      dp = T;
      sk = 0;
    }
  } else if (tile == kSimtBM && T >= S) {
    // the tensor-core rule over resident CTAs: whole waves stay whole; a
    // part-empty last wave is merged with the wave before it and split
    const int64_t full = T / S, rem = T % S;
    if (rem != 0 && full < 4) {
      dp = (full - 1) * S;
      sk = T - dp;
      grid = S;
    }
  } else if (tile == kSimtBM) {
    // fewer tiles than resident CTAs: split all k-blocks over up to S CTAs
    grid = std::min(S, std::max<int64_t>(T, T * I / min_iters));
    if (grid > T) {
      dp = 0;
      sk = T;
    } else {
      grid = T;
    }
  }
  if (sk > kTicketCap) return GEMM_ERR_UNSUPPORTED;
  p->kernel = GEMM_KERNEL_SIMT;
  p->tile_m = tile;
  p->tile_n = tile;
  p->tile_k = kSimtBK;
  p->stages = 2;
  p->tiles_m = int32_t(tiles_m);
  p->tiles_n = int32_t(tiles_n);
  p->grid = int32_t(grid);
  p->k_iters = int32_t(I);
  p->dp_tiles = int32_t(dp);
  p->sk_tiles = int32_t(sk);
  p->group_m = o.group_m > 0 ? o.group_m : 2048 / tile;
  p->workspace_bytes = sk > 0 ? int64_t(2) * grid * tile * tile * 4 : 0;
  return GEMM_OK;
}

// Chooses kernel, tile, split and grid for a shape.  Rules:
//  * fp32 inputs -> CUDA-core kernel, 128x128 tiles (64x64 only when a split
//    of the 128-tiles would still run fewer than 8 CTAs).  With 128-tiles
//    the tiles-vs-waves rule below is applied over the resident CTAs (2 per
//    SM), and a split hands out the k-blocks in runs of at least 8.
//  * fp16 inputs whose leading dimensions (or, in gemm_run, base addresses)
//    break the TMA rules -> the same CUDA-core kernel, fp16 widened to fp32.
//  * fp16 inputs -> tcgen05 kernels.  Shapes with at least half as many
//    256x256 tiles as CTA pairs -> the two-SM kernel.  Skinny M (M <= 64,
//    N >= 2M, A row-major) swaps the operands so N fills the 128-row MMA side
//    and M becomes the MMA N side (16/32/64 columns).  Measured (N = K =
//    4096, graph replay, cold inputs, us per launch, swapped vs not): M = 32
//    10.3 vs 12.8, 64 10.9 vs 12.9, but 80 13.0 vs 12.9, 128 13.6 vs 13.1 --
//    beyond 64 the swapped tile is 128 wide either way and its partials no
//    longer fit the push path.  Otherwise the tile
//    is 128x256 (128x128 when N <= 128 or when 256-wide tiles would fill fewer
//    than half the SMs).
//  * Decomposition of the one-SM kernel (the k-split the leiblog.wang
//    Stream-K post uses to keep SMs busy, where it pays here):
//      tiles fill under half the SMs: a cluster split of each tile's k-blocks
//        (partials added on chip), or, for shallow K, narrow whole tiles;
//        failing both, all k-blocks split evenly over up to one CTA per SM
//        (Stream-K), at least enough k-blocks per CTA that it reads 4x its
//        fp32 partial tile in operands (else whole tiles, one per CTA);
//      otherwise whole tiles, persistent over the SMs.
// k-blocks per TMA copy on a 128-row one-SM plan with `stages` ring slots:
// 2 by default where the ring then still has 3 stages (6 slots or more), else
// 1; GEMM_OPT_K_GROUP forces it.  Measured (graph replay, cold inputs, us per
// launch, 1 vs 2): 2048x1024x2048 16.5 vs 13.9, 1024x1024x768 8.1 vs 7.1,
// skinny M = 64 / 128 11.7 / 14.3 vs 10.9 / 13.7; the 5-slot short rings of
// skinny M <= 32 were slower as 2 stages of 2 (10.0 vs 10.8).  A K-major
// operand needs K a multiple of 64 (its 3-D view holds whole k-blocks); the
// ring keeps whole groups and at least `min_stages` slots.  Returns the group
// and trims *stages.
int one_sm_k_group(const Options& o, int64_t K, bool a_mn, bool b_mn, int* stages,
                   int min_stages) {
  if (K % kBK != 0 && !(a_mn && b_mn)) return 1;
  const int kg = o.k_group > 0 ? std::min(o.k_group, 4) : (*stages >= 6 ? 2 : 1);
  if (kg <= 1) return 1;
  const int st = *stages - *stages % kg;
  if (st < kg || st < min_stages) return 1;
  *stages = st;
  return kg;
}

// Whether row-major output tiles leave by TMA store (C's base and row pitch
// permitting, checked at launch): the tensor-core kernels that store 32-column
// chunks of row-major tiles, by default only on launches of many waves, 4 or
// more output tiles per CTA (per pair on the two-SM kernel) for fp32 output,
// 10 or more for fp16.  There TMA stores measured even or ahead (graph replay,
// cold inputs, us per launch, TMA vs plain: fp32 8192 x 8192 x 4096 312.2 vs
// 317.0, 6144^3 266.1 vs 267.0; fp16 8192^3 600.7 vs 601.4, 8192 x 8192 x
// 2048 156.9 vs 157.3); on fewer waves the staged plain stores measured
// faster (fp32 4096 x 4096 x 1024 37.1 vs 34.6, 3072^3 41.4 vs 40.3, 512^3
// 6.64 vs 6.92, one 128 x 128 tile 4.04 vs 4.41; fp16 2048^3 18.9 vs 17.9,
// 2048 x 2048 x 1024 13.0 vs 12.1, 4096^3 88.3 vs 87.4, 6144^3 258.4 vs 257.8).
int32_t plan_tma_store(const gemm_plan_t& p, const Options& o, bool out_f16) {
  const bool pair = p.kernel == GEMM_KERNEL_TC2;
  if (p.kernel != GEMM_KERNEL_TC && p.kernel != GEMM_KERNEL_STREAMK && !pair) return 0;
  if (p.swap_ab || p.tile_n < 32 || (!pair && p.tile_m != kBM)) return 0;
  if (o.tma_store >= 0) return o.tma_store > 0 ? 1 : 0;
  const int64_t tiles = int64_t(p.tiles_m) * p.tiles_n;
  const int64_t units = pair ? p.grid / 2 : p.grid;  // CTAs, or pairs
  return tiles >= (out_f16 ? 10 : 4) * units ? 1 : 0;
}

int plan_for_shape(int64_t M, int64_t N, int64_t K, gemm_layout_t L, int num_sms,
                   const Options& o, gemm_plan_t* p);

int plan_for(int64_t M, int64_t N, int64_t K, gemm_layout_t L, int num_sms,
             const Options& o, gemm_plan_t* p) {
  const int rc = plan_for_shape(M, N, K, L, num_sms, o, p);
  if (rc == GEMM_OK) p->tma_store = plan_tma_store(*p, o, L.out_dtype == GEMM_F16);
  return rc;
}

int plan_for_shape(int64_t M, int64_t N, int64_t K, gemm_layout_t L, int num_sms,
                   const Options& o, gemm_plan_t* p) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->k_group = 1;
  if (M < 0 || N < 0 || K < 0 || num_sms <= 0) return GEMM_ERR_INVALID_ARG;
  if (L.a_major > 1 || L.b_major > 1 || L.in_dtype > 1 || L.out_dtype > 1)
    return GEMM_ERR_INVALID_ARG;
  if (L.in_dtype == GEMM_F32 && L.out_dtype == GEMM_F16) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) {
    p->kernel = GEMM_KERNEL_NONE;
    return GEMM_OK;
  }
  if (K == 0) {
    p->kernel = GEMM_KERNEL_FILL;
    p->grid = 1;
    return GEMM_OK;
  }
  if (L.in_dtype == GEMM_F32) {
    if (o.force_kernel >= 0 && o.force_kernel != GEMM_KERNEL_SIMT) return GEMM_ERR_UNSUPPORTED;
    return plan_simt(M, N, K, num_sms, o, p);
  }
  // fp16: tensor-core path, unless asked for the CUDA-core kernel or the TMA
  // rules rule it out (int32 coordinates; leading dimensions a multiple of 8
  // elements, i.e. 16-byte row strides).
  const int64_t lda = L.a_major == GEMM_ROW_MAJOR ? K : M;
  const int64_t ldb = L.b_major == GEMM_ROW_MAJOR ? N : K;
  if (o.force_kernel == GEMM_KERNEL_SIMT || M > kMaxCoord || N > kMaxCoord || K > kMaxCoord ||
      lda % 8 != 0 || ldb % 8 != 0) {
    if (o.force_kernel >= 0 && o.force_kernel != GEMM_KERNEL_SIMT) return GEMM_ERR_UNSUPPORTED;
    return plan_simt(M, N, K, num_sms, o, p);
  }

  const bool forced_pair = o.force_kernel == GEMM_KERNEL_TC2;
  const bool swap = o.force_swap >= 0 ? (o.force_swap != 0)
                    : forced_pair     ? false
                                      : (L.a_major == GEMM_ROW_MAJOR && M <= 64 && N >= 2 * M);
  const int64_t Mm = swap ? N : M;
  const int64_t Nm = swap ? M : N;
  const int a_mn = swap ? (L.b_major == GEMM_ROW_MAJOR) : (L.a_major == GEMM_COL_MAJOR);
  const int b_mn = swap ? (L.a_major == GEMM_COL_MAJOR) : (L.b_major == GEMM_ROW_MAJOR);

  // Two-SM kernel (CTA pairs, 256 x 256 tiles, whole tiles): when asked for,
  // or when there are at least half as many pair tiles as resident pairs.  A
  // part-empty last wave of pair tiles costs less than splitting k: measured
  // (graph replay, cold inputs, TFLOP/s, two-SM kernel vs the one-SM
  // Stream-K/hybrid split) 2048^3 891 vs 458, 3072^3 1200 vs 828, 4096^3 1568
  // vs 1308, 4096x4096x1024 1043 vs 711, 1024x4096x4096 1014 vs 608.
  const int64_t pairs = o.pair_clusters > 0 ? o.pair_clusters : num_sms / 2;
  if (forced_pair && (swap || pairs < 1 || o.force_tile_n > 0)) return GEMM_ERR_UNSUPPORTED;
  if (!swap && pairs >= 1 && o.force_tile_n <= 0 &&
      (forced_pair || (o.force_kernel < 0 && o.pair != 0))) {
    const int64_t t2m = ceil_div(Mm, kPairBM), t2n = ceil_div(Nm, kPairBN);
    const int64_t T2 = t2m * t2n;
    const int64_t I2 = ceil_div(K, kBK);
    bool use = forced_pair || o.pair == 1;
    // Shallow products with at most one wave of pair tiles run faster as
    // one-SM 128 x 256 whole tiles: a pair tile's prologue and exposed
    // epilogue weigh more when each tile is short and nothing overlaps them.
    // Measured (graph replay, cold inputs, us per launch, one-SM whole vs
    // two-SM): 2048x2048x1024 13.19 vs 14.31, 1024x4864x512 11.03 vs 12.28;
    // with more waves the pairs win (4096x4096x1024, 3.4 waves: 1095 vs 1146
    // TFLOP/s; 1280x5120x1024, 1.3 waves: 696 vs 708), and from K = 1536 the
    // pairs are as fast or faster (2048^3 19.32 vs 19.40 us, 4096x2048x1536
    // 24.77 vs 24.33).
    const bool shallow_few = K <= 1024 && T2 <= pairs;
    if (!use && o.force_grid <= 0) use = 2 * T2 >= pairs && !shallow_few;
    if (use) {
      if (T2 > INT32_MAX / 2 || I2 > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
      int64_t np = std::min(pairs, T2);
      if (o.force_grid > 0) np = std::max<int64_t>(1, std::min<int64_t>(np, o.force_grid / 2));
      // Whole tiles by default.  Asked for, a Stream-K tail: the part-empty
      // last wave and the full wave before it split evenly over all pairs
      // (each pair's share ~1.5 tiles of k-blocks instead of 2 tiles for some
      // pairs and 1 for the rest).  Measured on 8192^3 (13.47 waves, 3.8 %
      // idle pair time in the last wave) the split ran 2.8 % slower than
      // whole tiles: publishing and re-reading the 128 KiB fp32 halves holds
      // the accumulators longer than the idle pairs cost.
      int64_t dp2 = T2, sk2 = 0;
      if (o.pair_split == 1) {
        // every tile split: up to all pairs, even more pairs than tiles
        np = o.force_grid > 0 ? std::max<int64_t>(1, std::min<int64_t>(pairs, o.force_grid / 2))
                              : pairs;
        np = std::min(np, T2 * I2);
        dp2 = 0;
        sk2 = T2;
      } else if (o.pair_split == 2) {
        const int64_t full = T2 / np, rem = T2 % np;
        if (rem != 0 && full >= 1) {
          dp2 = (full - 1) * np;
          sk2 = T2 - dp2;
        }
      }
      if (2 * sk2 > kTicketCap) return GEMM_ERR_UNSUPPORTED;  // a counter per CTA half
      // two k-blocks per stage and TMA copy (32 KiB boxes): each SM's TMA
      // unit then issues one copy per k-block instead of two, where a copy
      // of up to 32 KiB takes it about as long as a 16 KiB one.  A K-major
      // operand is read through a 3-D view of whole k-blocks (K a multiple
      // of 64).
      const bool kg_ok = I2 >= 2 && (K % kBK == 0 || (a_mn && b_mn));
      p->k_group = !kg_ok ? 1 : o.k_group > 0 ? int(std::min<int64_t>({o.k_group, 3, I2})) : 2;
      p->kernel = GEMM_KERNEL_TC2;
      p->swap_ab = 0;
      p->tile_m = kPairBM;
      p->tile_n = kPairBN;
      p->tile_k = kBK;
      p->stages = Tc2Config::kStages;
      p->grid = int32_t(2 * np);
      p->tiles_m = int32_t(t2m);
      p->tiles_n = int32_t(t2n);
      p->k_iters = int32_t(I2);
      p->dp_tiles = int32_t(dp2);
      p->sk_tiles = int32_t(sk2);
      p->a_mn_major = a_mn;
      p->b_mn_major = b_mn;
      // raster groups of 4096 rows of A (16 pair-tile rows), walked in the
      // static order: measured with two-k-block copies (same box, us per
      // launch, 20 / 400 launches of 8192^3): static 16 rows 606-608 / 660.9,
      // static 8 rows 615 / 667.7, run-time order 8 rows 621 / 677.4, run-time
      // 16 rows 616 / 674.9; 16384^3 static 16 rows 4658 / 5205 against
      // run-time 8 rows 4688 / 5259.
      p->group_m = o.group_m > 0 ? o.group_m : 4096 / kPairBM;
      // two partial slots per pair, each a 128 x 256 fp32 half per CTA
      p->workspace_bytes = sk2 > 0 ? int64_t(2) * np * 2 * kBM * kPairBN * 4 : 0;
      return GEMM_OK;
    }
  }

  int bn;
  bool narrow = false;  // whole 64-wide tiles for a small, shallow product
  if (o.force_tile_n > 0) {
    bn = o.force_tile_n;
  } else if (swap) {
    bn = Nm <= 16 ? 16 : Nm <= 32 ? 32 : Nm <= 64 ? 64 : 128;
    if (b_mn && bn < 64) bn = 64;
  } else {
    bn = Nm <= 128 ? 128 : 256;
    // too few 256-wide tiles to fill half the SMs: 128-wide tiles double the
    // count and halve each split partial
    if (bn == 256 && ceil_div(Mm, kBM) * ceil_div(Nm, 256) < num_sms / 2) bn = 128;
    // Few, shallow tiles (fewer 128-wide tiles than SMs, at most kNarrowIters
    // k-blocks): whole tiles 64 columns wide instead of a k-split, so no CTA
    // waits on a reduction and each has half the epilogue.  Measured (graph
    // replay, cold inputs, us per launch): 512^3 6.8 vs 8.2 for a cluster
    // split of 4; 1024x1024x512 7.1 vs 9.2; 256^3 5.8 vs 8.2.  Deeper K
    // favours the split (512x512x2048: 13.5 vs 10.0).
    if (o.force_kernel < 0 && o.force_grid <= 0 && o.csplit < 0 &&
        ceil_div(K, kBK) <= kNarrowIters && ceil_div(Mm, kBM) * ceil_div(Nm, bn) < num_sms &&
        ceil_div(Mm, kBM) * ceil_div(Nm, 64) <= num_sms) {
      bn = 64;
      narrow = true;
    }
  }
  const bool bn_ok = swap ? (bn == 16 || bn == 32 || bn == 64 || bn == 128)
                          : (bn == 32 || bn == 64 || bn == 128 || bn == 256);
  if (!bn_ok || (b_mn && bn % 64 != 0)) return GEMM_ERR_UNSUPPORTED;


  const int64_t tiles_m = ceil_div(Mm, kBM);
  int64_t tiles_n = ceil_div(Nm, bn);
  int64_t T = tiles_m * tiles_n;
  const int64_t I = ceil_div(K, kBK);
  if (T > INT32_MAX / 2 || I > INT32_MAX / 2 || T * I > (int64_t(1) << 40))
    return GEMM_ERR_UNSUPPORTED;
  const int64_t G = num_sms;
  int64_t dp = 0, sk = 0, grid = 0;
  const int64_t max_grid = o.force_grid > 0 ? std::min<int64_t>(o.force_grid, G) : G;

  // 64-row tiles for a small, shallow product taken as whole tiles: twice the
  // CTAs of 128-row tiles, each bringing in half the A rows and writing half
  // the output (a small single-wave launch is bound by what each SM moves).
  {
    const bool shape_ok = !swap && (bn == 32 || bn == 64 || bn == 128);
    const int64_t t64 = ceil_div(Mm, 64) * ceil_div(Nm, bn);
    const bool use64 = shape_ok && (o.tile_m == 64 || (o.tile_m < 0 && narrow && t64 <= G));
    if (o.tile_m == 64 &&
        (!use64 || (o.force_kernel >= 0 && o.force_kernel != GEMM_KERNEL_TC)))
      return GEMM_ERR_UNSUPPORTED;
    if (use64) {
      // Narrower still while the tiles fill under half the SMs (K-major B:
      // an MN-major B box is 64 wide).  Measured, graph replay, cold inputs:
      // one 128 x 128 output with K = 64, 8 tiles 32 wide 2.20 us against 4
      // tiles 64 wide 2.39; 512^3, 128 tiles 32 wide 5.03 against 64 tiles
      // 64 wide 4.96.
      if (o.force_tile_n <= 0 && o.tile_m < 0 && bn == 64 && !b_mn &&
          ceil_div(Mm, 64) * ceil_div(Nm, 32) < G / 2)
        bn = 32;
      const int64_t t64b = ceil_div(Mm, 64) * ceil_div(Nm, bn);
      const int64_t I64 = ceil_div(K, kBK);
      if (t64b > INT32_MAX / 2 || I64 > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
      const int full = tc64_stages_for(bn);
      // k-blocks per TMA copy: the unit takes about the same time per copy up
      // to 32 KiB, so a shallow product loads in a few deep boxes (up to 4
      // k-blocks: an MN-major box is at most 256 deep).  A K-major operand is
      // read through a 3-D view of whole k-blocks, so K must be a multiple of 64.
      int kg = I64 >= 4 ? 4 : I64 >= 2 ? 2 : 1;
      if (o.k_group > 0) kg = std::min<int64_t>(o.k_group, kg > 1 ? kg : 1);
      if (K % kBK != 0 && !(a_mn && b_mn)) kg = 1;
      p->k_group = kg;
      p->kernel = GEMM_KERNEL_TC;
      p->swap_ab = 0;
      p->tile_m = 64;
      p->tile_n = bn;
      p->tile_k = kBK;
      p->stages = o.stages > 0 ? std::min(o.stages, full) : full;
      p->stages = std::max(kg, p->stages - p->stages % kg);  // whole groups
      p->grid = int32_t(std::min(max_grid, t64b));
      p->tiles_m = int32_t(ceil_div(Mm, 64));
      p->tiles_n = int32_t(ceil_div(Nm, bn));
      p->k_iters = int32_t(I64);
      p->dp_tiles = int32_t(t64b);
      p->sk_tiles = 0;
      p->a_mn_major = a_mn;
      p->b_mn_major = b_mn;
      p->group_m = o.group_m > 0 ? o.group_m : 2048 / 64;
      p->workspace_bytes = 0;
      return GEMM_OK;
    }
  }

  // Cluster split: when the tiles fill few SMs, each tile's k-blocks are split
  // over a cluster of s CTAs (8, 4 or 2, whose clusters all fit at once and
  // leave every CTA >= 2 k-blocks).  The CTAs of a cluster add their fp32
  // partials through distributed shared memory: no global workspace, and the
  // hardware co-schedules the cluster, so its barrier always completes.
  {
    const bool forced = o.force_kernel == GEMM_KERNEL_SPLITC;
    int64_t cs = 0;
    auto fits = [&](int64_t tiles, int s) {
      // capacity: measured clusters resident at once; 0 = unknown (SMs / s); < 0 = none
      const int64_t cap = o.csplit_clusters[s] != 0 ? o.csplit_clusters[s] : G / s;
      return cap > 0 && tiles <= cap && tiles * s <= G;
    };
    if (forced) {
      cs = o.csplit >= 2 ? o.csplit : 4;
      if (I < cs) return GEMM_ERR_UNSUPPORTED;
    } else if (o.force_kernel < 0 && o.csplit != 0 && o.force_grid <= 0 && T < G && !narrow) {
      if (o.csplit >= 2) {
        if (fits(T, o.csplit) && I >= 2 * o.csplit) cs = o.csplit;
      } else {
        // Tile width and cluster size by the per-CTA cost: the operand bytes
        // it loads, (128 + w) x 128 B per k-block over ceil(I / s) k-blocks,
        // plus the fp32 partial bytes it exchanges, 128 x w x 4 B x (s-1)/s,
        // weighted 5x (distributed shared memory moves them that much slower
        // per SM than TMA brings operands in copies of two k-blocks).
        // Widths: the picker's, and 64 for unswapped tiles wider than that.
        // Measured (graph replay, cold inputs, us per launch, every width and
        // cluster size forced): the rule picks the fastest on 512x512x1024
        // (6.9), 512x512x2048 (7.9), 384x384x2048 (7.1), 512x512x8192 (13.4),
        // 512x1024x2048 (9.7: 64 wide in pairs), 768x768x1536 (9.0: 64 wide in
        // pairs), 256x512x4096 (8.9), 1024x1024x2048 (12.6), 1024x1024x8192
        // (24.6); 256x256x1024 5.9 against 5.8 for clusters of 8.
        int best_w = 0;
        double best_cost = 0;
        for (int w : {bn, (!swap && o.force_tile_n <= 0 && bn > 64) ? 64 : 0}) {
          if (w == 0) continue;
          const int64_t tw = tiles_m * ceil_div(Nm, w);
          if (tw >= G) continue;
          for (int sz : {8, 4, 2}) {
            if (!fits(tw, sz) || I < 2 * sz) continue;
            const double cost = double(kBM + w) * kBK * 2 * double(ceil_div(I, sz)) +
                                5.0 * kBM * w * 4 * double(sz - 1) / sz;
            if (cs == 0 || cost < best_cost) {
              best_w = w;
              cs = sz;
              best_cost = cost;
            }
          }
        }
        if (cs > 1 && best_w != bn) {
          bn = best_w;
          tiles_n = ceil_div(Nm, bn);
          T = tiles_m * tiles_n;
        }
      }
    }
    if (cs > 1) {
      p->kernel = GEMM_KERNEL_SPLITC;
      p->swap_ab = swap ? 1 : 0;
      p->tile_m = kBM;
      p->tile_n = bn;
      p->tile_k = kBK;
      p->stages = tc_stages_for(bn);
      // A split over more than half the SMs leaves too few idle for the next
      // launch's CTAs to start early: with a ring short enough that two CTAs
      // share an SM, they start beside this launch's and have their setup and
      // first loads done when it ends.  The split's own k-range needs few
      // stages.  (Parked partials need the ring to hold the partial tile.)
      // The short ring must still keep enough loads in flight for the
      // split's own streaming: measured, 5 stages of 18 KiB (16-wide tiles,
      // skinny M = 16: 9.86 -> 9.35 us) help, 3 of 24 KiB (64-wide, M = 64:
      // 10.84 -> 12.79 us) do not.  Tiles wider than 64 park their partial
      // in the ring: it must hold it.
      const int lean = o.lean_stages[width_index(bn)][swap ? 1 : 0];
      const int64_t lean_inflight = int64_t(lean) * (kBM + bn) * kBK * 2;
      if (lean >= tc_min_stages(bn, int(cs)) && lean_inflight >= kLeanMinInflight &&
          T * cs > G / 2)
        p->stages = std::min(p->stages, lean);
      if (o.stages > 0) p->stages = std::min(o.stages, tc_stages_for(bn));
      p->stages = std::max(p->stages, tc_min_stages(bn, int(cs)));
      p->k_group = one_sm_k_group(o, K, a_mn, b_mn, &p->stages, tc_min_stages(bn, int(cs)));
      p->grid = int32_t(T * cs);
      p->tiles_m = int32_t(tiles_m);
      p->tiles_n = int32_t(tiles_n);
      p->k_iters = int32_t(I);
      p->dp_tiles = 0;
      p->sk_tiles = int32_t(T);
      p->a_mn_major = a_mn;
      p->b_mn_major = b_mn;
      p->group_m = o.group_m > 0 ? o.group_m : 2048 / kBM;
      p->cluster_split = int32_t(cs);
      p->workspace_bytes = 0;
      return GEMM_OK;
    }
  }

  if (o.force_kernel == GEMM_KERNEL_TC || narrow) {
    dp = T;
    grid = std::min(max_grid, T);
  } else if (o.force_kernel == GEMM_KERNEL_STREAMK) {
    sk = T;
    grid = std::min(max_grid, T * I);
  } else if (max_grid < G && T > max_grid) {
    // a forced smaller grid: split everything over it
    sk = T;
    grid = max_grid;
  } else if (2 * T >= G) {
    // At least half as many tiles as SMs: whole tiles, a part-empty last wave
    // and all.  The Stream-K or hybrid split the leiblog.wang post suggests for
    // that tail measured slower here (graph replay, cold inputs, TFLOP/s):
    // 4096^3 1383 whole vs 1308 hybrid, 1024x2048x4096 707 vs 516 split,
    // 1536x1536x4096 796 vs 596, 2048x1024x2048 565 vs 337, 512x4096x8192 810
    // vs 665 -- its fixup reads every other contributor's partial serially.
    dp = T;
    grid = std::min(T, G);
  } else {
    const int64_t total = T * I;
    // A split CTA writes (and the tile's last CTA reads back) a 128 x bn fp32
    // partial; give each CTA at least 4x that many bytes of operand k-blocks.
    int min_iters = o.min_split_iters;
    if (min_iters <= 0) {
      const int64_t partial = int64_t(kBM) * bn * 4;
      const int64_t kblock = int64_t(kBM + bn) * kBK * 2;
      min_iters = int(ceil_div(4 * partial, kblock));
    }
    const int64_t want = std::max<int64_t>(T, total / min_iters);
    grid = std::min(max_grid, want);
    if (grid == T) {
      dp = T;  // one whole tile per CTA
    } else {
      sk = T;
    }
  }
  if (sk > kTicketCap) return GEMM_ERR_UNSUPPORTED;

  p->kernel = sk > 0 ? GEMM_KERNEL_STREAMK : GEMM_KERNEL_TC;
  p->swap_ab = swap ? 1 : 0;
  p->tile_m = kBM;
  p->tile_n = bn;
  p->tile_k = kBK;
  p->stages = o.stages > 0 ? std::min(o.stages, tc_stages_for(bn)) : tc_stages_for(bn);
  p->k_group = one_sm_k_group(o, K, a_mn, b_mn, &p->stages, 1);
  p->grid = int32_t(grid);
  p->tiles_m = int32_t(tiles_m);
  p->tiles_n = int32_t(tiles_n);
  p->k_iters = int32_t(I);
  p->dp_tiles = int32_t(dp);
  p->sk_tiles = int32_t(sk);
  p->a_mn_major = a_mn;
  p->b_mn_major = b_mn;
  p->group_m = o.group_m > 0 ? o.group_m : 2048 / kBM;
  p->workspace_bytes = sk > 0 ? int64_t(2) * grid * kBM * bn * 4 : 0;
  return GEMM_OK;
}

WorkSpec spec_of(const gemm_plan_t& p) {
  WorkSpec w;
  w.tiles_m = p.tiles_m;
  w.tiles_n = p.tiles_n;
  w.k_iters = p.k_iters;
  w.dp_tiles = p.dp_tiles;
  w.sk_tiles = p.sk_tiles;
  w.grid = p.kernel == GEMM_KERNEL_TC2 ? p.grid / 2 : p.grid;  // pairs work as one unit
  w.group_m = p.group_m;
  w.csplit = p.kernel == GEMM_KERNEL_SPLITC ? p.cluster_split : 0;
  return w;
}

// ------------------------------------------------------------- TMA maps --
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace dg

struct gemm_ctx {
  int device = 0;
  int num_sms = 0;
  float* workspace = nullptr;
  size_t workspace_bytes = 0;
  int* tickets = nullptr;
  int* status = nullptr;
  int last_detail = 0;
  uint64_t* trace = nullptr;  // caller's device buffer for phase stamps, or NULL
  int64_t trace_ctas = 0;     // CTA rows it holds (kTraceSlots stamps each)
  dg::Options opt;
  void* host_stage = nullptr;   // gemm_run_host: device copies of A, B, bias and C
  size_t host_stage_bytes = 0;  // grow-only
  std::mutex host_mu;           // serialises gemm_run_host's enqueueing
  cudaEvent_t host_done = nullptr;  // recorded after each gemm_run_host call's work
  bool host_done_recorded = false;
  std::mutex mu;  // guards the tensor-map cache
  dg::TmapEntry cache[dg::kTmapCacheSize];
  int cache_next = 0;
};

namespace dg {
namespace {

// An fp16 operand with `rows` rows (MMA view) and depth K, in boxes of
// `kgroup` k-blocks:
//   K-major  (K contiguous):    dims {K, rows}, box {64, box_rows}; for kgroup > 1
//                               (K a multiple of 64) the 3-D view {64, rows, K / 64}
//                               (strides K * 2 and 128 bytes), box {64, box_rows, kgroup}
//   MN-major (rows contiguous): dims {rows, K}, box {64, 64 * kgroup}
// 128-byte swizzle; out-of-range elements read as zero.
int encode_operand(gemm_ctx* h, CUtensorMap* out, const void* ptr, int64_t rows, int64_t K,
                   int mn_major, int box_rows, int kgroup = 1) {
  if (kgroup > 1 && ((!mn_major && K % kBK != 0) || kgroup * kBK > 256))
    return GEMM_ERR_UNSUPPORTED;
  const TmapKey key{ptr, rows, K, mn_major, box_rows, 0, kgroup};
  {
    std::lock_guard<std::mutex> g(h->mu);
    for (auto& e : h->cache)
      if (e.valid && e.key == key) {
        *out = e.map;
        return GEMM_OK;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GEMM_ERR_CUDA;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  cuuint32_t rank = 2;
  if (!mn_major && kgroup > 1) {
    rank = 3;
    dims[0] = kBK;
    dims[1] = cuuint64_t(rows);
    dims[2] = cuuint64_t(K / kBK);
    strides[0] = cuuint64_t(K) * 2;
    strides[1] = kBK * 2;
    box[0] = kBK;
    box[1] = cuuint32_t(box_rows);
    box[2] = cuuint32_t(kgroup);
  } else if (!mn_major) {
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
    box[1] = cuuint32_t(kBK * kgroup);
  }
  CUtensorMap map;
  const CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
  std::lock_guard<std::mutex> g(h->mu);
  TmapEntry& e = h->cache[h->cache_next];
  h->cache_next = (h->cache_next + 1) % kTmapCacheSize;
  e.key = key;
  e.map = map;
  e.valid = true;
  *out = map;
  return GEMM_OK;
}

// Row-major C (M x N, ldc = N) for the epilogue's TMA stores: 32 x 32 boxes,
// 128-byte swizzle for fp32 (128-byte box rows), 64-byte for fp16.  Returns
// false when C cannot take them (base not 16-byte aligned, row pitch not a
// multiple of 16 bytes, or the encode fails); the epilogue then stores with
// plain instructions.
bool encode_output(gemm_ctx* h, CUtensorMap* out, void* C, int64_t M, int64_t N, bool f16) {
  const int64_t pitch = N * (f16 ? 2 : 4);
  if ((reinterpret_cast<uintptr_t>(C) & 15) || pitch % 16 != 0 || M > kMaxCoord ||
      N > kMaxCoord)
    return false;
  const TmapKey key{C, M, N, 0, 32, f16 ? 2 : 1, 1};
  {
    std::lock_guard<std::mutex> g(h->mu);
    for (auto& e : h->cache)
      if (e.valid && e.key == key) {
        *out = e.map;
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(M)};
  const cuuint64_t strides[1] = {cuuint64_t(pitch)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap map;
  const CUresult r =
      fn(&map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C,
         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         f16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> g(h->mu);
  TmapEntry& e = h->cache[h->cache_next];
  h->cache_next = (h->cache_next + 1) % kTmapCacheSize;
  e.key = key;
  e.map = map;
  e.valid = true;
  *out = map;
  return true;
}

// Runs `f` with the handle's device current, restoring the caller's.
template <class F>
int on_device(int device, F&& f) {
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;
  const int rc = f();
  if (prev != device) cudaSetDevice(prev);
  return rc;
}

void log_plan(const gemm_plan_t& p, int64_t M, int64_t N, int64_t K) {
  std::fprintf(stderr,
               "[gemm] M=%lld N=%lld K=%lld kernel=%d swap=%d tile=%dx%dx%d stages=%d "
               "grid=%d tiles=%dx%d k_iters=%d dp=%d sk=%d a_mn=%d b_mn=%d k_group=%d "
               "csplit=%d tma_store=%d\n",
               (long long)M, (long long)N, (long long)K, p.kernel, p.swap_ab, p.tile_m,
               p.tile_n, p.tile_k, p.stages, p.grid, p.tiles_m, p.tiles_n, p.k_iters,
               p.dp_tiles, p.sk_tiles, p.a_mn_major, p.b_mn_major, p.k_group, p.cluster_split,
               p.tma_store);
}

}  // namespace

cudaError_t launch_tc(const TcLaunch& L) {
  if (L.pair) return launch_tc2(L);
  if (L.bm == 64) return launch_tc64(L);
  if (L.bn == 256) return launch_tc_n256(L);
  if (L.bn == 128) return launch_tc_n128(L);
  if (!L.trans) return launch_tc_narrow(L);
  return launch_tc_small(L);
}

int tc_lean_stages(int bn, bool trans) {
  switch (bn) {
    case 16: return trans ? lean_stages_small(16) : 0;
    case 32: return trans ? lean_stages_small(32) : lean_stages_narrow(32);
    case 64: return trans ? lean_stages_small(64) : lean_stages_narrow(64);
    case 128: return lean_stages_n128(trans);
    default: return 0;
  }
}

int tc_min_stages(int bn, int csplit) {
  if (csplit <= 1 || bn <= 64) return 1;  // no parked partial
  const int64_t park = int64_t(kBM) * (bn + 4) * 4;  // rows (or columns) padded by 4 floats
  const int64_t stage = int64_t(kBM + bn) * kBK * 2;
  return int((park + stage - 1) / stage);
}

int tc_stages_for(int bn) {
  switch (bn) {
    case 256: return TcConfig<256>::kStages;
    case 128: return TcConfig<128>::kStages;
    case 64: return TcConfig<64>::kStages;
    case 32: return TcConfig<32>::kStages;
    default: return TcConfig<16>::kStages;
  }
}

int tc_smem_bytes_for(int bn) {
  switch (bn) {
    case 256: return TcConfig<256>::kSmemBytes;
    case 128: return TcConfig<128>::kSmemBytes;
    case 64: return TcConfig<64>::kSmemBytes;
    case 32: return TcConfig<32>::kSmemBytes;
    default: return TcConfig<16>::kSmemBytes;
  }
}

}  // namespace dg

// ================================================================== C-ABI ==
extern "C" {

const char* gemm_strerror(int code) {
  switch (code) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: shape/layout/alignment not supported";
    case GEMM_ERR_ALLOC: return "GEMM_ERR_ALLOC: allocation failed";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA call failed";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a device-side wait expired";
    default: return "unknown gemm status";
  }
}

int gemm_plan_for(int64_t M, int64_t N, int64_t K, gemm_layout_t layout, int num_sms,
                  gemm_plan_t* out) {
  return dg::plan_for(M, N, K, layout, num_sms, dg::Options(), out);
}

int gemm_work_units(const gemm_plan_t* plan, int cta, int32_t* out, int max_units) {
  if (!plan || max_units < 0 || (max_units > 0 && !out)) return GEMM_ERR_INVALID_ARG;
  if (plan->kernel != GEMM_KERNEL_TC && plan->kernel != GEMM_KERNEL_STREAMK &&
      plan->kernel != GEMM_KERNEL_TC2 && plan->kernel != GEMM_KERNEL_SPLITC &&
      plan->kernel != GEMM_KERNEL_SIMT)
    return GEMM_ERR_INVALID_ARG;
  // for the two-SM kernel `cta` numbers CTA pairs
  const int units = plan->kernel == GEMM_KERNEL_TC2 ? plan->grid / 2 : plan->grid;
  if (cta < 0 || cta >= units) return GEMM_ERR_INVALID_ARG;
  const dg::WorkSpec w = dg::spec_of(*plan);
  dg::WorkIter it;
  // what the kernel runs: the tensor-core kernels use init_tc
  if (plan->kernel == GEMM_KERNEL_SIMT)
    it.init(w, cta);
  else
    it.init_tc(w, cta);
  dg::Unit u;
  int n = 0;
  while (it.next(w, u)) {
    if (n < max_units) {
      out[3 * n] = u.tile;
      out[3 * n + 1] = u.kb0;
      out[3 * n + 2] = u.kb1;
    }
    ++n;
  }
  return n;
}

int gemm_split_contributors(const gemm_plan_t* plan, int sk_tile, int32_t* first,
                            int32_t* last) {
  if (!plan || !first || !last ||
      (plan->kernel != GEMM_KERNEL_STREAMK && plan->kernel != GEMM_KERNEL_SIMT &&
       plan->kernel != GEMM_KERNEL_TC2) ||
      sk_tile < 0 || sk_tile >= plan->sk_tiles)
    return GEMM_ERR_INVALID_ARG;
  const dg::WorkSpec w = dg::spec_of(*plan);
  dg::split_contributors(w, sk_tile, *first, *last);
  return GEMM_OK;
}

int64_t gemm_drain_limit_ns(int64_t wait_limit_ns) {
  const uint64_t w = wait_limit_ns > 0 ? uint64_t(wait_limit_ns) : dg::Options().wait_limit_ns;
  return int64_t(dg::drain_limit_ns(w));
}

int gemm_simt_smem_strides(int32_t* a_stride, int32_t* b_stride) {
  if (!a_stride || !b_stride) return GEMM_ERR_INVALID_ARG;
  *a_stride = dg::simt_a_stride();
  *b_stride = dg::simt_b_stride();
  return GEMM_OK;
}

int gemm_create(gemm_handle_t* out, int device) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (device < 0 || device >= ndev) return GEMM_ERR_INVALID_ARG;
  gemm_ctx* h = new (std::nothrow) gemm_ctx();
  if (!h) return GEMM_ERR_ALLOC;
  h->device = device;
  const int rc = dg::on_device(device, [&]() -> int {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;
    h->num_sms = prop.multiProcessorCount;
    const int pairs = dg::tc2_max_active_clusters(true);
    h->opt.pair_clusters = pairs > 0 ? std::min(pairs, h->num_sms / 2) : h->num_sms / 2;
    for (int s : {2, 4, 8}) {
      const int n = dg::tc_max_active_clusters(s);
      // n == 0: clusters of s cannot be scheduled at all (-1 keeps the picker off them);
      // a failed query leaves the SMs / s estimate
      h->opt.csplit_clusters[s] = n > 0 ? std::min(n, h->num_sms / s) : n == 0 ? -1 : h->num_sms / s;
      if (dg::log_enabled())
        std::fprintf(stderr, "[gemm] device %d: clusters of %d resident at once: %d\n", device, s,
                     n);
    }
    if (dg::log_enabled())
      std::fprintf(stderr, "[gemm] device %d: CTA pairs resident at once: %d\n", device, pairs);
    for (int bn : {16, 32, 64, 128})
      for (int t = 0; t < 2; ++t) {
        h->opt.lean_stages[dg::width_index(bn)][t] = dg::tc_lean_stages(bn, t != 0);
        if (dg::log_enabled())
          std::fprintf(stderr, "[gemm] device %d: tile width %d%s: two CTAs per SM with %d stages\n",
                       device, bn, t ? " (swapped)" : "",
                       h->opt.lean_stages[dg::width_index(bn)][t]);
      }
    const int simt = dg::simt_ctas_per_sm();
    h->opt.simt_per_sm = simt > 0 ? simt : 2;
    h->workspace_bytes = size_t(2) * h->num_sms * dg::kBM * dg::kMaxTileN * sizeof(float);
    if (dg::dev_malloc(reinterpret_cast<void**>(&h->workspace), h->workspace_bytes) !=
        cudaSuccess)
      return GEMM_ERR_ALLOC;
    if (dg::dev_malloc(reinterpret_cast<void**>(&h->tickets), sizeof(int) * dg::kCounterInts) !=
        cudaSuccess)
      return GEMM_ERR_ALLOC;
    if (dg::dev_malloc(reinterpret_cast<void**>(&h->status), sizeof(int)) != cudaSuccess)
      return GEMM_ERR_ALLOC;
    if (cudaMemset(h->tickets, 0, sizeof(int) * dg::kCounterInts) != cudaSuccess ||
        cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return GEMM_ERR_CUDA;
    return GEMM_OK;
  });
  if (rc != GEMM_OK) {
    gemm_destroy(h);
    return rc;
  }
  *out = h;
  return GEMM_OK;
}

int gemm_destroy(gemm_handle_t h) {
  if (!h) return GEMM_OK;
  dg::on_device(h->device, [&]() -> int {
    if (h->workspace) cudaFree(h->workspace);
    if (h->tickets) cudaFree(h->tickets);
    if (h->status) cudaFree(h->status);
    if (h->host_stage) cudaFree(h->host_stage);
    if (h->host_done) cudaEventDestroy(h->host_done);
    return GEMM_OK;
  });
  delete h;
  return GEMM_OK;
}

int gemm_set_option(gemm_handle_t h, int option, int64_t value) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  dg::Options& o = h->opt;
  const dg::Options d;
  switch (option) {
    case GEMM_OPT_FORCE_KERNEL:
      if (value >= 0 && value != GEMM_KERNEL_TC && value != GEMM_KERNEL_STREAMK &&
          value != GEMM_KERNEL_SIMT && value != GEMM_KERNEL_TC2 && value != GEMM_KERNEL_SPLITC)
        return GEMM_ERR_INVALID_ARG;
      o.force_kernel = value < 0 ? d.force_kernel : int(value);
      return GEMM_OK;
    case GEMM_OPT_FORCE_TILE_N:
      if (value >= 0 && value != 16 && value != 32 && value != 64 && value != 128 &&
          value != 256)
        return GEMM_ERR_INVALID_ARG;
      o.force_tile_n = value < 0 ? d.force_tile_n : int(value);
      return GEMM_OK;
    case GEMM_OPT_FORCE_GRID:
      o.force_grid = value <= 0 ? d.force_grid : int(std::min<int64_t>(value, INT32_MAX));
      return GEMM_OK;
    case GEMM_OPT_WAIT_LIMIT_NS:
      o.wait_limit_ns = value <= 0 ? d.wait_limit_ns : uint64_t(value);
      return GEMM_OK;
    case GEMM_OPT_MIN_SPLIT_ITERS:
      o.min_split_iters = value <= 0 ? d.min_split_iters : int(std::min<int64_t>(value, 1 << 20));
      return GEMM_OK;
    case GEMM_OPT_FORCE_SWAP_AB:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.force_swap = value < 0 ? d.force_swap : int(value);
      return GEMM_OK;
    case GEMM_OPT_GROUP_M:
      o.group_m = value <= 0 ? d.group_m : int(std::min<int64_t>(value, 1 << 16));
      return GEMM_OK;
    case GEMM_OPT_PAIR:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.pair = value < 0 ? d.pair : int(value);
      return GEMM_OK;
    case GEMM_OPT_CLUSTER_SPLIT:
      if (value > 0 && value != 2 && value != 4 && value != 8) return GEMM_ERR_INVALID_ARG;
      o.csplit = value < 0 ? d.csplit : int(value);
      return GEMM_OK;
    case GEMM_OPT_PDL:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.pdl = value < 0 ? d.pdl : int(value);
      return GEMM_OK;
    case GEMM_OPT_PAIR_SPLIT:
      if (value > 2) return GEMM_ERR_INVALID_ARG;
      o.pair_split = value < 0 ? d.pair_split : int(value);
      return GEMM_OK;
    case GEMM_OPT_TMA_STORE:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.tma_store = value < 0 ? d.tma_store : int(value);
      return GEMM_OK;
    case GEMM_OPT_BIAS_INIT:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.bias_init = value < 0 ? d.bias_init : int(value);
      return GEMM_OK;
    case GEMM_OPT_DYNAMIC_TILES:
      if (value > 1) return GEMM_ERR_INVALID_ARG;
      o.dyn_sched = value < 0 ? d.dyn_sched : int(value);
      return GEMM_OK;
    case GEMM_OPT_STAGES:
      o.stages = value <= 0 ? d.stages : int(std::min<int64_t>(value, 64));
      return GEMM_OK;
    case GEMM_OPT_TILE_M:
      if (value >= 0 && value != 64 && value != 128) return GEMM_ERR_INVALID_ARG;
      o.tile_m = value < 0 ? d.tile_m : int(value);
      return GEMM_OK;
    case GEMM_OPT_K_GROUP:
      if (value >= 0 && (value < 1 || value > 4)) return GEMM_ERR_INVALID_ARG;
      o.k_group = value < 0 ? d.k_group : int(value);
      return GEMM_OK;
    default:
      return GEMM_ERR_INVALID_ARG;
  }
}

int gemm_query_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K, gemm_layout_t layout,
                    gemm_plan_t* out) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  return dg::plan_for(M, N, K, layout, h->num_sms, h->opt, out);
}

int gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
             const float* bias, void* C, gemm_layout_t layout, void* stream_ptr) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  gemm_plan_t plan;
  int rc = dg::plan_for(M, N, K, layout, h->num_sms, h->opt, &plan);
  if (rc != GEMM_OK) return rc;
  if (dg::log_enabled()) dg::log_plan(plan, M, N, K);
  if (plan.kernel == GEMM_KERNEL_NONE) return GEMM_OK;
  if (!C) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  if (plan.kernel == GEMM_KERNEL_FILL) {
    return dg::on_device(h->device, [&]() -> int {
      return dg::launch_fill(M, N, bias, C, layout.out_dtype == GEMM_F16, stream) == cudaSuccess
                 ? GEMM_OK
                 : GEMM_ERR_CUDA;
    });
  }
  if (!A || !B) return GEMM_ERR_INVALID_ARG;

  // fp16 operands the TMA cannot read (base not 16-byte aligned): the
  // CUDA-core kernel instead
  if (plan.kernel != GEMM_KERNEL_SIMT &&
      ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))) {
    dg::Options o = h->opt;
    o.force_kernel = GEMM_KERNEL_SIMT;
    o.force_tile_n = -1;
    rc = dg::plan_for(M, N, K, layout, h->num_sms, o, &plan);
    if (rc != GEMM_OK) return rc;
  }
  if (plan.kernel == GEMM_KERNEL_SIMT) {
    dg::SimtLaunch L;
    L.M = M; L.N = N; L.K = K;
    L.A = A;
    L.B = B;
    L.bias = bias;
    L.C = C;
    L.in_f16 = layout.in_dtype == GEMM_F16;
    L.out_f16 = layout.out_dtype == GEMM_F16;
    L.a_major = layout.a_major;
    L.b_major = layout.b_major;
    L.tile = plan.tile_m;
    L.work = dg::spec_of(plan);
    L.workspace = h->workspace;
    L.tickets = h->tickets;
    L.stream = stream;
    return dg::on_device(h->device, [&]() -> int {
      return dg::launch_simt(L) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    });
  }

  const bool swap = plan.swap_ab != 0;
  const void* opA = swap ? B : A;  // MMA-view A operand (rows Mm)
  const void* opB = swap ? A : B;  // MMA-view B operand (rows Nm)
  const int64_t Mm = swap ? N : M;
  const int64_t Nm = swap ? M : N;

  const bool pair = plan.kernel == GEMM_KERNEL_TC2;
  dg::TcLaunch L;
  L.bm = pair ? dg::kPairBM : plan.tile_m;
  L.bn = plan.tile_n;
  L.out_f16 = layout.out_dtype == GEMM_F16;
  L.trans = swap;
  L.pair = pair;
  L.pdl = h->opt.pdl != 0;
  L.grid = plan.grid;
  L.stream = stream;
  // each CTA loads 128 (or 64) rows of A; a pair CTA loads half of the
  // 256-column B tile
  const int kgroup = plan.k_group > 1 ? plan.k_group : 1;
  rc = dg::encode_operand(h, &L.tmA, opA, Mm, K, plan.a_mn_major, pair ? dg::kBM : plan.tile_m,
                          kgroup);
  if (rc != GEMM_OK) return rc;
  rc = dg::encode_operand(h, &L.tmB, opB, Nm, K, plan.b_mn_major,
                          pair ? dg::kHalfBN : plan.tile_n, kgroup);
  if (rc != GEMM_OK) return rc;
  dg::TcArgs& a = L.args;
  a.work = dg::spec_of(plan);
  a.Mm = int32_t(Mm);
  a.Nm = int32_t(Nm);
  a.C = C;
  a.ldc = N;
  a.bias = bias;
  a.workspace = h->workspace;
  a.tickets = h->tickets;
  a.status = h->status;
  a.wait_limit_ns = h->opt.wait_limit_ns;
  a.a_mn = plan.a_mn_major;
  a.b_mn = plan.b_mn_major;
  // Row-major output chunks of 32 columns leave by TMA store where the plan
  // takes it (plan_tma_store) and C allows it.
  std::memset(&L.tmC, 0, sizeof(L.tmC));
  a.c_tma = (plan.tma_store &&
             dg::encode_output(h, &L.tmC, C, M, N, layout.out_dtype == GEMM_F16))
                ? 1
                : 0;
  // whole, aligned 4-column groups for the plain stores of row-major output
  const int64_t c_pitch = N * (layout.out_dtype == GEMM_F16 ? 2 : 4);
  a.c_vec = (!swap && (reinterpret_cast<uintptr_t>(C) & 15) == 0 && c_pitch % 16 == 0) ? 1 : 0;
  a.bias_init = (h->opt.bias_init && bias) ? 1 : 0;
  // Asked for (GEMM_OPT_DYNAMIC_TILES), whole pair tiles are handed out at
  // run time in tile order (a counter the pairs draw from), so the tiles in
  // flight stay one compact block of the raster however the pairs drift
  // apart; the split tail and the bias seeding keep the static schedule.
  if (pair && plan.sk_tiles == 0 && !a.bias_init && h->opt.dyn_sched > 0)
    a.sched = h->tickets + dg::kTicketCap;
  a.stages = pair ? 0 : plan.stages;
  a.kgroup = kgroup;
  // phase stamps only if the caller's buffer holds one row per CTA
  a.trace = (h->trace && h->trace_ctas >= plan.grid) ? h->trace : nullptr;
  a.idesc = dg::make_idesc_f16(pair ? dg::kPairBM : plan.tile_m, plan.tile_n, plan.a_mn_major,
                               plan.b_mn_major);
  return dg::on_device(h->device, [&]() -> int {
    return dg::launch_tc(L) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  });
}

int gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                  const void* B, const float* bias, void* C, gemm_layout_t layout,
                  void* stream_ptr) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || layout.in_dtype > 1 || layout.out_dtype > 1)
    return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  const size_t in_sz = layout.in_dtype == GEMM_F16 ? 2 : 4;
  const size_t out_sz = layout.out_dtype == GEMM_F16 ? 2 : 4;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };  // 256-byte aligned parts
  const size_t a_bytes = size_t(M) * size_t(K) * in_sz, b_bytes = size_t(K) * size_t(N) * in_sz;
  const size_t bias_bytes = bias ? size_t(N) * 4 : 0, c_bytes = size_t(M) * size_t(N) * out_sz;
  const size_t need = up(a_bytes) + up(b_bytes) + up(bias_bytes) + up(c_bytes);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  std::lock_guard<std::mutex> lock(h->host_mu);
  return dg::on_device(h->device, [&]() -> int {
    if (!h->host_done && cudaEventCreateWithFlags(&h->host_done, cudaEventDisableTiming) != cudaSuccess) {
      h->host_done = nullptr;
      return GEMM_ERR_CUDA;
    }
    if (need > h->host_stage_bytes) {
      // the previous call (on any stream) may still use the old buffers
      if (h->host_done_recorded && cudaEventSynchronize(h->host_done) != cudaSuccess)
        return GEMM_ERR_CUDA;
      if (h->host_stage) cudaFree(h->host_stage);
      h->host_stage = nullptr;
      h->host_stage_bytes = 0;
      if (dg::dev_malloc(&h->host_stage, need) != cudaSuccess) {
        h->host_stage = nullptr;
        return GEMM_ERR_ALLOC;
      }
      h->host_stage_bytes = need;
    } else if (h->host_done_recorded && cudaStreamWaitEvent(stream, h->host_done, 0) != cudaSuccess) {
      // same buffers: this call's copies start after the previous call's work
      return GEMM_ERR_CUDA;
    }
    uint8_t* base = static_cast<uint8_t*>(h->host_stage);
    void* dA = base;
    void* dB = base + up(a_bytes);
    float* dbias = bias ? reinterpret_cast<float*>(base + up(a_bytes) + up(b_bytes)) : nullptr;
    void* dC = base + up(a_bytes) + up(b_bytes) + up(bias_bytes);
    int rc = GEMM_OK;
    if ((a_bytes && cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (b_bytes && cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (bias_bytes &&
         cudaMemcpyAsync(dbias, bias, bias_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)) {
      rc = GEMM_ERR_CUDA;
    } else {
      rc = gemm_run(h, M, N, K, dA, dB, dbias, dC, layout, stream_ptr);
      if (rc == GEMM_OK && cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        rc = GEMM_ERR_CUDA;
    }
    // whatever was enqueued, the next call waits for it
    if (cudaEventRecord(h->host_done, stream) == cudaSuccess)
      h->host_done_recorded = true;
    else if (rc == GEMM_OK)
      rc = GEMM_ERR_CUDA;
    return rc;
  });
}

int gemm_status(gemm_handle_t h, void* stream_ptr) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  return dg::on_device(h->device, [&]() -> int {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
      return GEMM_ERR_CUDA;
    h->last_detail = word;
    if (word == 0) return GEMM_OK;
    // a kernel stopped early: clear the word and the split counters it may
    // have left behind, so the handle is usable again
    if (cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(h->tickets, 0, sizeof(int) * dg::kCounterInts) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return GEMM_ERR_CUDA;
    return GEMM_ERR_DEVICE_TIMEOUT;
  });
}

int gemm_status_detail(gemm_handle_t h) { return h ? h->last_detail : 0; }

int gemm_inject_alloc_failure(int64_t n) {
  if (n < 0) return GEMM_ERR_INVALID_ARG;
  dg::g_fail_alloc_in.store(n);
  return GEMM_OK;
}

int gemm_set_trace(gemm_handle_t h, uint64_t* dev_buf, int64_t ctas) {
  if (!h || ctas < 0 || (ctas > 0 && !dev_buf)) return GEMM_ERR_INVALID_ARG;
  h->trace = ctas > 0 ? dev_buf : nullptr;
  h->trace_ctas = ctas;
  return GEMM_OK;
}

int gemm_selftest_wait_timeout(gemm_handle_t h, int64_t limit_ns, void* stream_ptr) {
  if (!h || limit_ns <= 0) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  return dg::on_device(h->device, [&]() -> int {
    return dg::launch_wait_selftest(uint64_t(limit_ns), h->status, stream) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
  });
}

}  // extern "C"
