// simt_kernel.cuh: the CUDA-core GEMM kernel, C = A·B (+bias) with fp32
// accumulation (true FFMA, no TF32), for fp32 inputs (simt.cu) and for fp16
// inputs that the tensor-core path cannot take (simt_f16.cu).
//
// Each technique of the "TVM Matrix Multiplication Optimization" ladder
// (kimm240.github.io/tvm, Steps 1-6) has its place here:
//   Step 1 data-parallel 2-D thread map    -> one CTA per BM x BN output tile
//   Step 2 tiling + loop reordering        -> each thread owns an 8x8 register tile
//                                             and runs the k loop outermost
//   Step 3 shared memory, cooperative fetch-> all threads stage a BM x 16 A block
//                                             and a 16 x BN B block per k-step
//   Step 4 vectorisation + register caching-> float4 global and shared loads;
//                                             accumulators live in registers, and
//                                             the FMAs are packed two lanes wide
//                                             (fma.rn.f32x2: a pair of A rows times
//                                             one B column per instruction)
//   Step 5 software pipelining             -> two shared-memory buffers; the next
//                                             block is fetched (into registers, or
//                                             by direct global-to-shared copies
//                                             for aligned fp32 operands stored
//                                             m/n-contiguous) while the current
//                                             one is consumed
//   Step 6 unrolling                       -> the k-step and the 8x8 FMA nest are
//                                             fully unrolled
// The staging rows are padded as storage_align(factor 32, offset 4) pads them
// (leiblog.wang, the storage_align answer: the stride is raised to the next
// value congruent to offset mod factor), 128 -> 132 and 64 -> 68 floats, which
// makes the transposed A stores free of bank conflicts.
//
// Two tile shapes: 128 x 128 with 256 threads, and 64 x 64 with 64 threads for
// products too small to give even a k-split of 128-tiles 8 CTAs (the 8x8
// thread tile, and so the ratio of shared loads to FMAs, is the same in
// both).
//
// Work is handed out as the tensor-core kernels hand it out (work.cuh): whole
// tiles first, then, when the tile count would leave the last wave of resident
// CTAs part-empty, the k-blocks of the remaining tiles split evenly over the
// CTAs (the Stream-K decomposition of the leiblog.wang Stream-K post).  A CTA
// whose unit covers part of a tile publishes its fp32 partial to the
// workspace; the last contributor to arrive adds all partials in ascending k
// order and stores the tile.  No CTA ever waits for another.
//
// fp16 inputs are widened to fp32 as they are staged (8-byte loads of four
// halves where aligned), so products and sums are the fp32 FMAs of the fp32
// path; an fp16 output is rounded once, after the bias add.  Each packed FMA
// lane is an IEEE fused multiply-add rounded to nearest, exactly fmaf, so the
// packing changes no result.
#pragma once

#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "work.cuh"

namespace dg {
namespace simt_detail {

// storage_align(factor, offset) applied to a row of `extent` elements.
__host__ __device__ constexpr int aligned_stride(int extent, int factor, int offset) {
  return extent + (factor + offset - extent % factor) % factor;
}
static_assert(aligned_stride(128, 32, 4) == 132 && aligned_stride(64, 32, 4) == 68,
              "padded staging strides");

struct SimtArgs {
  int64_t M, N, K;
  const void* A;             // TIn elements
  const void* B;             // TIn elements
  const float* bias;
  void* C;                   // TOut elements
  bool vec_a, vec_b, vec_c;  // 4-element vector access allowed (aligned rows)
  WorkSpec work;             // tiles, raster order and split of this launch
  float* workspace;          // split partials: 2 slots of BM x BN floats per CTA
  int* tickets;              // one arrival counter per split tile (left at 0)
};

// One 4-element piece of a k-block as fp32: consecutive elements along the
// storage row, starting at p; zero outside [0, limit) or when `inside` is false.
// fp16 elements are widened exactly (every fp16 value is an fp32 value).
__device__ __forceinline__ void load4(float (&r)[4], const float* p, bool vec, bool inside,
                                      int64_t first, int64_t limit) {
  if (vec && inside && first + 3 < limit) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = (inside && first + i < limit) ? __ldg(p + i) : 0.f;
  }
}
__device__ __forceinline__ void load4(float (&r)[4], const __half* p, bool vec, bool inside,
                                      int64_t first, int64_t limit) {
  if (vec && inside && first + 3 < limit) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));  // 4 halves, 8-byte aligned
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      r[i] = (inside && first + i < limit) ? __half2float(__ldg(p + i)) : 0.f;
  }
}

// d = a * b + d on two packed fp32 lanes ({low, high} halves of each 64-bit
// operand), each lane one IEEE fused multiply-add rounded to nearest: the
// results of two fmaf calls in one instruction, which halves the issue slots
// the FMAs take (the FMA pipe itself does the same 128 lanes per SM per clock).
__device__ __forceinline__ void fma2(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
// {x, x} as one packed operand.
__device__ __forceinline__ uint64_t dup2(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}

// 16 bytes global -> shared without passing through registers, cached in L2
// only; with inside == false nothing is read (src may be any valid address)
// and the 16 bytes are zero-filled.  Both addresses 16-byte aligned.  Awaited
// by cp_async_wait_all before the barrier that publishes the buffer.
__device__ __forceinline__ void cp_async16(float* smem_dst, const float* gsrc, bool inside) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
               ::"r"(d), "l"(gsrc), "r"(inside ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async16(float*, const __half*, bool) {}  // fp16: not used
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Four consecutive outputs of one row (n + j < N checked per element when the
// vector store is not allowed); one rounding to TOut.
__device__ __forceinline__ void store4(float* dst, const float (&o)[4], bool vec, int64_t n,
                                       int64_t N) {
  if (vec && n + 3 < N) {
    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n + j < N) dst[j] = o[j];
  }
}
__device__ __forceinline__ void store4(__half* dst, const float (&o)[4], bool vec, int64_t n,
                                       int64_t N) {
  if (vec && n + 3 < N) {
    const __half2 lo = __floats2half2_rn(o[0], o[1]);
    const __half2 hi = __floats2half2_rn(o[2], o[3]);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n + j < N) dst[j] = __float2half_rn(o[j]);
  }
}

// Rows of the register tile each thread of a BM-row tile owns: 16 for the
// 128-row tiles (128 threads), 8 for the 64-row tiles (64 threads).
template <int BM>
constexpr int kSimtTM = BM == 128 ? 16 : 8;

// BM x BN tile, NT = (BM/TM) x (BN/8) threads, each a TM x 8 register tile
// made of TM/4 groups of 4 rows, BM/(TM/4) apart, and two 4-column groups
// BN/2 apart.  A 1-D grid of a.work.grid CTAs walks the units that WorkIter
// hands it.  Residency asked of the compiler: 2 CTAs per SM for 128-tiles; 4
// for 64-tiles, which the picker uses only for products too small to give
// 128-tiles 8 CTAs.  ASYNC (fp32 only): the operands stored m/n-contiguous
// have 16-byte aligned rows and are copied global -> shared directly, holding
// no staging registers.
template <typename TIn, typename TOut, int BM, int BN, bool A_COL, bool B_COL, bool ASYNC>
__global__ void __launch_bounds__((BM / kSimtTM<BM>) * (BN / 8), BM == 128 ? 2 : 4)
    simt_sgemm_kernel(const SimtArgs a) {
  constexpr int BK = kSimtBK;
  constexpr int TM = kSimtTM<BM>;   // rows per thread
  constexpr int RG = TM / 4;        // groups of 4 rows per thread
  constexpr int RS = BM / RG;       // row distance between a thread's groups
  constexpr int NT = (BM / TM) * (BN / 8);
  constexpr int AS = aligned_stride(BM, 32, 4);
  constexpr int BS = aligned_stride(BN, 32, 4);
  constexpr int AV = BM * BK / 4 / NT;  // float4 pieces of A per thread per k-block
  constexpr int BV = BN * BK / 4 / NT;
  static_assert(AV >= 1 && BV >= 1 && AV * NT * 4 == BM * BK && BV * NT * 4 == BN * BK, "");
  static_assert(!ASYNC || std::is_same<TIn, float>::value, "direct copies are fp32 only");
  constexpr bool kAsyncA = ASYNC && A_COL;   // column-major A: m-contiguous
  constexpr bool kAsyncB = ASYNC && !B_COL;  // row-major B: n-contiguous
  __shared__ __align__(16) float As[2][BK][AS];
  __shared__ __align__(16) float Bs[2][BK][BS];
  __shared__ int last_flag;

  const int t = threadIdx.x;
  const int tx = t % (BN / 8), ty = t / (BN / 8);
  const int64_t M = a.M, N = a.N, K = a.K;
  const WorkSpec& W = a.work;
  const TIn* const Ap = static_cast<const TIn*>(a.A);
  const TIn* const Bp = static_cast<const TIn*>(a.B);

  float ra[AV][4], rb[BV][4];
  float acc[TM][8];
  // The main loop accumulates row pairs, P[i][j] = {acc[2i][j], acc[2i+1][j]},
  // with packed two-wide FMAs: a pair of A rows times one B column, {b, b}.
  uint64_t P[TM / 2][8];

  // Piece v of this thread for an operand stored k-contiguous (row-major A,
  // column-major B): pairs of threads cover 8 consecutive k of one row (a
  // 32-byte sector), RP = NT/2 rows per pass, the next 8 k in a later pass.
  // That keeps the transposed shared stores free of bank conflicts with the
  // padded stride (a warp's 32 stores hit 16 rows x 2 k-quarters 16 banks
  // apart).  An operand stored m/n-contiguous is read as piece f = t + v*NT:
  // k-row f/(BM/4), run of 4 f%(BM/4).
  constexpr int RP = NT / 2;
  static_assert(BK % 8 == 0 && BM % RP == 0 && BN % RP == 0, "piece map");
  auto kc_row = [&](int v, int rows) { return (t >> 1) + (v % (rows / RP)) * RP; };
  auto kc_kq = [&](int v, int rows) { return 2 * (v / (rows / RP)) + (t & 1); };

  // Global -> registers (or, for ASYNC operands, straight into shared buffer
  // `buf`) for the k-block starting at k0 of the tile at (m0, n0).
  auto fetch = [&](int64_t m0, int64_t n0, int64_t k0, int buf) {
#pragma unroll
    for (int v = 0; v < AV; ++v) {
      const int f = t + v * NT;
      if (!A_COL) {
        const int64_t m = m0 + kc_row(v, BM), k = k0 + kc_kq(v, BM) * 4;
        load4(ra[v], Ap + m * K + k, a.vec_a, m < M, k, K);
      } else {
        const int kr = f / (BM / 4), mr = (f % (BM / 4)) * 4;
        const int64_t k = k0 + kr, m = m0 + mr;
        if constexpr (kAsyncA) {
          // rows are whole vectors: a run is inside or outside as a whole
          const bool in = k < K && m < M;
          cp_async16(&As[buf][kr][mr], in ? Ap + k * M + m : Ap, in);
        } else {
          load4(ra[v], Ap + k * M + m, a.vec_a, k < K, m, M);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < BV; ++v) {
      const int f = t + v * NT;
      if (!B_COL) {
        const int kr = f / (BN / 4), nr = (f % (BN / 4)) * 4;
        const int64_t k = k0 + kr, n = n0 + nr;
        if constexpr (kAsyncB) {
          const bool in = k < K && n < N;
          cp_async16(&Bs[buf][kr][nr], in ? Bp + k * N + n : Bp, in);
        } else {
          load4(rb[v], Bp + k * N + n, a.vec_b, k < K, n, N);
        }
      } else {
        const int64_t n = n0 + kc_row(v, BN), k = k0 + kc_kq(v, BN) * 4;
        load4(rb[v], Bp + n * K + k, a.vec_b, n < N, k, K);
      }
    }
  };

  // Registers -> shared buffer `buf`, as As[k][m] and Bs[k][n] (operands that
  // were copied directly are already there).
  auto stage = [&](int buf) {
#pragma unroll
    for (int v = 0; v < AV && !kAsyncA; ++v) {
      const int f = t + v * NT;
      if (!A_COL) {
        const int m = kc_row(v, BM), k = kc_kq(v, BM) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) As[buf][k + i][m] = ra[v][i];
      } else {
        const int k = f / (BM / 4), m = (f % (BM / 4)) * 4;
        *reinterpret_cast<float4*>(&As[buf][k][m]) =
            make_float4(ra[v][0], ra[v][1], ra[v][2], ra[v][3]);
      }
    }
#pragma unroll
    for (int v = 0; v < BV && !kAsyncB; ++v) {
      const int f = t + v * NT;
      if (!B_COL) {
        const int k = f / (BN / 4), n = (f % (BN / 4)) * 4;
        *reinterpret_cast<float4*>(&Bs[buf][k][n]) =
            make_float4(rb[v][0], rb[v][1], rb[v][2], rb[v][3]);
      } else {
        const int n = kc_row(v, BN), k = kc_kq(v, BN) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) Bs[buf][k + i][n] = rb[v][i];
      }
    }
    if constexpr (kAsyncA || kAsyncB) cp_async_wait_all();
  };

  // Epilogue: + bias[n]; rows (i/4)*RS + ty*4 + i%4, columns tx*4+j (+BN/2).
  auto store_tile = [&](int64_t m0, int64_t n0) {
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int64_t m = m0 + (i / 4) * RS + ty * 4 + (i % 4);
      if (m >= M) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t n = n0 + h * (BN / 2) + tx * 4;
        if (n >= N) continue;
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = acc[i][h * 4 + j] + ((a.bias && n + j < N) ? __ldg(a.bias + n + j) : 0.f);
        store4(static_cast<TOut*>(a.C) + m * N + n, o, a.vec_c, n, N);
      }
    }
  };

  // The work iterator lives in shared memory, advanced by thread 0, so none of
  // its state occupies registers across the k loop.
  __shared__ WorkIter s_it;
  __shared__ Unit s_unit;
  __shared__ int s_more;
  if (t == 0) s_it.init(W, int32_t(blockIdx.x));
  for (;;) {
    if (t == 0) s_more = s_it.next(W, s_unit) ? 1 : 0;
    __syncthreads();
    if (!s_more) break;
    const Unit u = s_unit;
    int32_t tm, tn;
    tile_coords(W, u.tile, tm, tn);
    const int64_t m0 = int64_t(tm) * BM, n0 = int64_t(tn) * BN;
#pragma unroll
    for (int i = 0; i < TM / 2; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) P[i][j] = 0;  // two +0.0f

    // The previous unit ended with a barrier after its last shared reads, so
    // buffer 0 is free.
    fetch(m0, n0, int64_t(u.kb0) * BK, 0);
    stage(0);
    __syncthreads();
    for (int32_t kt = u.kb0; kt < u.kb1; ++kt) {
      const int buf = (kt - u.kb0) & 1;
      // buffer buf^1 was last read before the barrier that ended the step before
      if (kt + 1 < u.kb1) fetch(m0, n0, int64_t(kt + 1) * BK, buf ^ 1);
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        // row pairs (ty*4 + {0,1}) and (ty*4 + {2,3}) of each row group
        uint64_t av[TM / 2];
#pragma unroll
        for (int g = 0; g < RG; ++g) {
          const ulonglong2 ag =
              *reinterpret_cast<const ulonglong2*>(&As[buf][kk][g * RS + ty * 4]);
          av[2 * g] = ag.x;
          av[2 * g + 1] = ag.y;
        }
        // columns tx*4 + {0..3} and BN/2 + tx*4 + {0..3}, each as {b, b}
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][BN / 2 + tx * 4]);
        const uint64_t bv[8] = {dup2(b0.x), dup2(b0.y), dup2(b0.z), dup2(b0.w),
                                dup2(b1.x), dup2(b1.y), dup2(b1.z), dup2(b1.w)};
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) fma2(P[i][j], av[i], bv[j]);
      }
      if (kt + 1 < u.kb1) stage(buf ^ 1);
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM / 2; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[2 * i][j] = __uint_as_float(uint32_t(P[i][j]));
        acc[2 * i + 1][j] = __uint_as_float(uint32_t(P[i][j] >> 32));
      }

    if (!unit_is_partial(W, u)) {
      store_tile(m0, n0);
      continue;
    }
    // Split unit.  Publish the fp32 partial: float4 j of thread t (row j/2 of
    // its register tile, column half j%2) at float4 index j*NT + t of the slot,
    // so each warp's stores are contiguous.
    constexpr int kQuads = TM * 2;  // float4 per thread
    const int32_t st = u.tile - W.dp_tiles;
    const int32_t me = int32_t(blockIdx.x);
    const size_t slot_elems = size_t(BM) * BN;
    float4* mine = reinterpret_cast<float4*>(a.workspace +
                                             size_t(split_slot(W, me, st)) * slot_elems);
#pragma unroll
    for (int j = 0; j < kQuads; ++j)
      __stcg(mine + j * NT + t, make_float4(acc[j >> 1][(j & 1) * 4], acc[j >> 1][(j & 1) * 4 + 1],
                                            acc[j >> 1][(j & 1) * 4 + 2],
                                            acc[j >> 1][(j & 1) * 4 + 3]));
    __threadfence();
    __syncthreads();
    int32_t first, last;
    split_contributors(W, st, first, last);
    if (t == 0) {
      const int old = atomicAdd(&a.tickets[st], 1);
      last_flag = (old == last - first) ? 1 : 0;
    }
    __syncthreads();
    if (!last_flag) continue;
    // Last to arrive: every contributor's partial, this CTA's own included,
    // is in the workspace.  Add them in ascending k order, whichever CTA
    // arrived last, so the sum is the same on every run.
    // Every contributor after the first starts its range inside this tile, so
    // its partial is in its first slot (split_slot gives 2r for it).
    __threadfence();
    const int32_t first_slot = split_slot(W, first, st);
    // four float4 (one register-tile row pair) of every contributor at a time
#pragma unroll
    for (int jc = 0; jc < kQuads / 4; ++jc) {
      for (int32_t r = first; r <= last; ++r) {
        const float4* src = reinterpret_cast<const float4*>(
            a.workspace + size_t(r == first ? first_slot : 2 * r) * slot_elems);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = jc * 4 + jj;
          const float4 v = __ldcg(src + j * NT + t);
          float* d = &acc[j >> 1][(j & 1) * 4];
          if (r == first) {
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
          } else {
            d[0] += v.x; d[1] += v.y; d[2] += v.z; d[3] += v.w;
          }
        }
      }
    }
    if (t == 0) atomicExch(&a.tickets[st], 0);  // ready for the next launch
    store_tile(m0, n0);
  }
}

template <typename TIn, typename TOut, int BM, int BN, bool A_COL, bool B_COL>
cudaError_t launch_simt_layout(const SimtArgs& a, cudaStream_t s) {
  constexpr int NT = (BM / kSimtTM<BM>) * (BN / 8);
  const dim3 grid{unsigned(a.work.grid), 1u, 1u};
  // direct copies for the 128-tile fp32 kernel when its m/n-contiguous
  // operands have aligned rows (the 64-tile kernel has registers to spare)
  constexpr bool kCanAsync = BM == 128 && std::is_same<TIn, float>::value && (A_COL || !B_COL);
  if constexpr (kCanAsync) {
    if ((!A_COL || a.vec_a) && (B_COL || a.vec_b)) {
      simt_sgemm_kernel<TIn, TOut, BM, BN, A_COL, B_COL, true><<<grid, NT, 0, s>>>(a);
      return cudaGetLastError();
    }
  }
  simt_sgemm_kernel<TIn, TOut, BM, BN, A_COL, B_COL, false><<<grid, NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int BM, int BN>
cudaError_t launch_simt_tile(const SimtArgs& a, int a_major, int b_major, cudaStream_t s) {
  if (a.work.grid <= 0) return cudaErrorInvalidConfiguration;
  if (a_major == 0 && b_major == 0) return launch_simt_layout<TIn, TOut, BM, BN, false, false>(a, s);
  if (a_major == 0) return launch_simt_layout<TIn, TOut, BM, BN, false, true>(a, s);
  if (b_major == 0) return launch_simt_layout<TIn, TOut, BM, BN, true, false>(a, s);
  return launch_simt_layout<TIn, TOut, BM, BN, true, true>(a, s);
}

inline bool aligned_to(const void* p, uintptr_t n) {
  return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0;
}

// Argument block for launch L with TIn / TOut elements.
template <typename TIn, typename TOut>
SimtArgs simt_args(const SimtLaunch& L) {
  constexpr uintptr_t vin = 4 * sizeof(TIn), vout = 4 * sizeof(TOut);
  SimtArgs a;
  a.M = L.M; a.N = L.N; a.K = L.K;
  a.A = L.A; a.B = L.B; a.bias = L.bias; a.C = L.C;
  a.vec_a = aligned_to(L.A, vin) && ((L.a_major == 0 ? L.K : L.M) % 4 == 0);
  a.vec_b = aligned_to(L.B, vin) && ((L.b_major == 0 ? L.N : L.K) % 4 == 0);
  a.vec_c = aligned_to(L.C, vout) && (L.N % 4 == 0);
  a.work = L.work;
  a.workspace = L.workspace;
  a.tickets = L.tickets;
  return a;
}

template <typename TIn, typename TOut>
cudaError_t launch_simt_typed(const SimtLaunch& L) {
  const SimtArgs a = simt_args<TIn, TOut>(L);
  if (a.work.sk_tiles > 0 && (!a.workspace || !a.tickets)) return cudaErrorInvalidValue;
  if (L.tile == kSimtSmallTile)
    return launch_simt_tile<TIn, TOut, kSimtSmallTile, kSimtSmallTile>(a, L.a_major, L.b_major,
                                                                       L.stream);
  return launch_simt_tile<TIn, TOut, kSimtBM, kSimtBN>(a, L.a_major, L.b_major, L.stream);
}

}  // namespace simt_detail
}  // namespace dg
