// tc64_kernel.cuh: the one-SM tcgen05 GEMM with 64-row tiles, for small
// products that a 128-row tiling would spread over too few SMs.
//
//   D[64 x BN] = Aop[64 x K] · Bop[BN x K]ᵀ   (fp16 in, fp32 accumulate in TMEM)
//
// then C = D (+bias) rounded once to the output type.  Same roles as the
// 128-row kernel (tc_kernel.cuh): warp 0 one lane TMA producer, warp 1 one lane
// MMA issuer (and TMEM owner), warps 2-5 epilogue; every wait bounded.  Only
// whole tiles (no k-split), operands in place (not swapped), plain stores.
//
// Why it exists: a small single-wave launch is bound per SM, by the operand
// bytes each CTA must bring in and the output bytes it must write.  With 64
// rows a tile needs half the A rows of a 128-row one, so twice as many CTAs
// share the same product, each with fewer bytes to move.
//
// TMEM layout of an M = 64 accumulator: row r of D sits in lane
// 32 * (r / 16) + r % 16, column j in column j.  So each epilogue warp reads
// its 32-lane quarter as usual and only lanes 0-15 hold rows (16 per warp).
#pragma once

#include "tc_kernel.cuh"

namespace dg {

constexpr int kBM64 = 64;  // MMA M of this kernel

template <int BN>
struct Tc64Config {
  // the whole k range of a shallow product (up to 12 k-blocks; 8 for 128-wide tiles)
  static constexpr int kStages = BN == 128 ? 8 : 12;
  static constexpr int kABytes = kBM64 * kBK * 2;    // 8 KiB
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kBarBytes = 256;
  // epilogue staging: per warp 32 rows of 32 + 4 floats
  static constexpr int kEpiStageBytes = 4 * 32 * (32 + 4) * 4;
  static constexpr int smem_bytes(int stages) {
    return 1024 + stages * kStageBytes + kBarBytes + kEpiStageBytes;
  }
  static constexpr int kSmemBytes = smem_bytes(kStages);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(BN == 32 || BN == 64 || BN == 128, "tile width");
  static_assert((2 * kStages + 5) * 8 + 16 <= kBarBytes, "barrier area");
};

// The ring holds `stages` k-blocks, taken J = args.kgroup at a time: one TMA
// copy per operand brings J consecutive k-blocks (a 3-D box for a K-major
// operand, a box J k-blocks deep for an MN-major one), so a small launch
// issues a few large copies instead of two per k-block (the TMA unit of an SM
// takes about the same time per copy up to 32 KiB).  Group g of a tile
// covers k-blocks kb0 + g*J ...; the last group may be short: its box reads
// zeros (or unused k-blocks) past the tile's range, and its MMAs stop there.
template <int BN, bool OUT_F16>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc64_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const TcArgs args) {
  using Cfg = Tc64Config<BN>;
  const int J = args.kgroup > 1 ? args.kgroup : 1;
  const int S = (args.stages > 0 ? args.stages : Cfg::kStages) / J;  // ring stages of J blocks
  constexpr int CW = 32;  // TMEM columns per epilogue load

  const uint64_t t_entry = args.trace ? globaltimer_ns() : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                          // S x J x 8 KiB
  uint8_t* sB = smem + S * J * Cfg::kABytes;   // S x J x BN*128 B
  uint8_t* stage = sB + S * J * Cfg::kBBytes;  // epilogue staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + Cfg::kEpiStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* acc_full = bars + 2 * S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), kEpiThreads);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // As in the 128-row kernel: only this CTA's own resources so far; every
  // role prepares its first step and waits for the kernels ahead of this one
  // just before its first global access.
  pdl_launch_dependents();
  const WaitCtl wc{args.wait_limit_ns, args.status, abort_flag};
  const WorkSpec& W = args.work;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      WorkIter it;
      it.init_tc(W, blockIdx.x);
      Unit u;
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true, first = true, waited = false;
      while (ok && it.next(W, u)) {
        int32_t tm, tn;
        tile_coords(W, u.tile, tm, tn);
        for (int32_t kb = u.kb0; kb < u.kb1; kb += J) {
          if (!wait_bounded(smem_u32(&empty[s]), ph ^ 1, wc, kSiteProducer)) {
            ok = false;
            break;
          }
          if (!waited) {
            pdl_wait_prerequisites();
            waited = true;
            if (args.trace) {
              args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceEntry] = t_entry;
              trace_mark(args, blockIdx.x, kTraceStart);
            }
          }
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, J * Cfg::kStageBytes);  // whole boxes, zero-filled past K
          const uint32_t a_dst = smem_u32(sA + s * J * Cfg::kABytes);
          const uint32_t b_dst = smem_u32(sB + s * J * Cfg::kBBytes);
          const int32_t k0 = kb * kBK;
          // A: 64 rows x 64 J k, one box either way round
          if (args.a_mn)
            tma_load_2d(a_dst, &tmA, fb, tm * kBM64, k0);
          else if (J > 1)
            tma_load_3d(a_dst, &tmA, fb, 0, tm * kBM64, kb);
          else
            tma_load_2d(a_dst, &tmA, fb, k0, tm * kBM64);
          if (!args.b_mn) {
            if (J > 1)
              tma_load_3d(b_dst, &tmB, fb, 0, tn * BN, kb);
            else
              tma_load_2d(b_dst, &tmB, fb, k0, tn * BN);
          } else {
            if constexpr (BN >= 64) {
              // 64-column halves, each J k-blocks deep
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(b_dst + j * J * 8192, &tmB, fb, tn * BN + 64 * j, k0);
            }
          }
          if (first) {
            trace_mark(args, blockIdx.x, kTraceFirstLoad);
            first = false;
          }
          issued |= 1u << s;
          issued_par = (issued_par & ~(1u << s)) | (ph << s);
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!waited) pdl_wait_prerequisites();
      if (!ok) {  // copies still in flight land before the CTA exits
        for (int t = 0; t < S; ++t)
          if ((issued >> t) & 1) wait_drain(smem_u32(&full[t]), (issued_par >> t) & 1, wc);
      }
    } else {
      pdl_wait_prerequisites();
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    pdl_wait_prerequisites();
    if (lane == 0) {
      WorkIter it;
      it.init_tc(W, blockIdx.x);
      Unit u;
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true, any = false;
      // an MN-major B's 64-column halves sit J k-blocks apart
      const uint32_t a_lbo = args.a_mn ? 8192u : 16u;
      const uint32_t b_lbo = args.b_mn ? uint32_t(J) * 8192u : 16u;
      const uint32_t a_step = args.a_mn ? (2048u >> 4) : (32u >> 4);
      const uint32_t b_step = args.b_mn ? (2048u >> 4) : (32u >> 4);
      // k-block j of a group: A blocks are 8 KiB either way round; a K-major B
      // block holds BN rows, an MN-major one 64 k rows of each half
      const uint32_t b_blk = args.b_mn ? 8192u : uint32_t(Cfg::kBBytes);
      while (ok && it.next(W, u)) {
        if (!wait_bounded(smem_u32(&acc_empty[b]), aph, wc, kSiteMmaAccum)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(b * BN);
        for (int32_t kb = u.kb0; kb < u.kb1; kb += J) {
          if (!wait_bounded(smem_u32(&full[s]), ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!any) trace_mark(args, blockIdx.x, kTraceFirstData);
          const uint32_t a0 = smem_u32(sA + s * J * Cfg::kABytes);
          const uint32_t b0 = smem_u32(sB + s * J * Cfg::kBBytes);
          const int nj = u.kb1 - kb < J ? u.kb1 - kb : J;
#pragma unroll 1
          for (int j = 0; j < nj; ++j) {
            const uint64_t adesc = make_sdesc_sw128(a0 + uint32_t(j) * 8192u, a_lbo, 1024);
            const uint64_t bdesc = make_sdesc_sw128(b0 + uint32_t(j) * b_blk, b_lbo, 1024);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_f16(d_tmem, adesc + uint64_t(kk * a_step), bdesc + uint64_t(kk * b_step),
                         args.idesc, (kb > u.kb0 || j > 0 || kk > 0) ? 1u : 0u);
          }
          any = true;
          tc_commit(smem_u32(&empty[s]));
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        trace_mark(args, blockIdx.x, kTraceMmaDone);
        tc_commit(smem_u32(&acc_full[b]));
        if (++b == 2) {
          b = 0;
          aph ^= 1;
        }
      }
      if (!ok && any) {  // every MMA issued so far finishes before TMEM is freed
        tc_commit(smem_u32(drain));
        wait_drain(smem_u32(drain), 0, wc);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;   // TMEM lane quarter: rows 16q .. 16q + 15 in lanes 0-15
    const int et = threadIdx.x - 64;
    WorkIter it;
    it.init_tc(W, blockIdx.x);
    pdl_wait_prerequisites();  // C (and the bias) are global
    for (int b0 = 0; b0 < 2; ++b0) {
      tc_fence_before();
      mbar_arrive(smem_u32(&acc_empty[b0]));
    }
    Unit u;
    int b = 0;
    uint32_t aph = 0;
    int units = 0;
    float* sw = reinterpret_cast<float*>(stage) + q * 32 * (CW + 4);
    while (it.next(W, u)) {
      int32_t tm, tn;
      tile_coords(W, u.tile, tm, tn);  // while the MMAs still run
      const bool got = wait_bounded(smem_u32(&acc_full[b]), aph, wc, kSiteEpilogue);
      if (!epi_all(got)) break;
      tc_fence_after();
      if (et == 0) trace_mark(args, blockIdx.x, kTraceLastAccum);
      ++units;
      const int32_t mrow0 = tm * kBM64 + q * 16;  // first row of this warp's 16
      const int32_t nbase = tn * BN;
      const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(b * BN);
#pragma unroll 1
      for (int c = 0; c < BN / CW; ++c) {
        float v[CW];
        __syncwarp();
        tmem_load_chunk<CW>(taddr + c * CW, v);
        if (args.c_vec)
          store_rows_vec<CW, OUT_F16, 16>(args, sw, mrow0, lane, nbase + c * CW, v);
        else
          store_rows_staged<CW, OUT_F16, 16>(args, sw, mrow0, lane, nbase + c * CW, v);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acc_empty[b]));
      if (++b == 2) {
        b = 0;
        aph ^= 1;
      }
    }
    __syncwarp();
    if (et == 0) {
      trace_mark(args, blockIdx.x, kTraceEnd);
      if (args.trace) args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceUnits] = uint64_t(units);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
  if (args.trace) {
    __syncthreads();
    if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceExit);
  }
}

}  // namespace dg
