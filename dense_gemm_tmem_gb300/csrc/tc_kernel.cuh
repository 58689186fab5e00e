// tc_kernel.cuh: the tcgen05/TMEM tensor-core GEMM for sm_103a.
//
//   D[Mm x Nm] = Aop[Mm x K] · Bop[Nm x K]ᵀ   (fp16 in, fp32 accumulate in TMEM)
//
// then C = D (+bias) rounded once to fp16 or kept in fp32.  With TRANS the
// kernel has been handed swapped operands (Aop = Bᵀ, Bop = A) and writes Dᵀ,
// so a skinny M lands on the MMA's N side.
//
// Design, per CTA (192 threads, one CTA per SM, persistent over work units):
//   warp 0, one lane   TMA producer: 128x64 A block and BNx64 B block per
//                      k-block into an S-stage ring of 128B-swizzled shared
//                      memory (the swizzle takes the place of the padding the
//                      leiblog.wang bank-conflict post adds to a 128x256x32 tile).
//   warp 1, one lane   MMA issuer: 4 x tcgen05.mma (K = 16 each) per k-block into
//                      one of two TMEM accumulators (BN fp32 columns each);
//                      tcgen05.commit frees the stage and, after the unit's last
//                      k-block, hands the accumulator to the epilogue.  Warp 1
//                      also allocates and frees TMEM.
//   warps 2-5          epilogue: tcgen05.ld 32 lanes x 32 columns, + bias[n] in
//                      fp32, one rounding to the output type, then, on launches
//                      of many waves, a TMA store of the warp's 32 x 32 block
//                      from a swizzled shared box (otherwise, and where C cannot
//                      take TMA, plain stores staged through padded shared rows;
//                      lane-per-column stores for swapped operands).  For a Stream-K partial
//                      unit: publish the fp32 partial, take a ticket, and the
//                      last contributor sums all partials in ascending k order
//                      before the same epilogue.  Each drained accumulator is
//                      released to the MMA issuer, after seeding it with the
//                      next unit's bias when the reduction starts from the bias.
// The pipeline overlap of the A500 ladder's software-pipelining step
// (kimm240.github.io/tvm, Step 5) is the S-stage ring plus the two accumulators:
// the MMA of tile i+1 runs while the epilogue drains tile i.
//
// Every wait is bounded (wait_bounded): on expiry the CTA raises an abort flag,
// records the site in the device status word, waits (bounded) for its own copies
// and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"
#include "work.cuh"

namespace dg {

constexpr int kBM = 128;          // MMA M (TMEM lanes)
constexpr int kBK = 64;           // fp16 k-elements per stage = one 128-byte swizzle row
constexpr int kTcThreads = 192;   // 6 warps
constexpr int kEpiThreads = 128;  // warps 2-5

template <int BN>
struct TcConfig {
  static constexpr int kStages = BN == 256 ? 4 : BN == 128 ? 6 : BN == 64 ? 8 : 10;
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // power of two >= 32
  static constexpr int kChunk = BN < 32 ? BN : 32;             // TMEM columns per load
  static constexpr int kBarBytes = 256;
  // epilogue staging (after the stages, so 1024-byte aligned): per epilogue
  // warp 32 rows of kChunk + 4 floats, or a 4 KiB swizzled TMA store box
  // (64-column tiles: 32 KiB, which also holds the pushed partials of a
  // swapped cluster split, 128 rows x 64 columns of fp32)
  static constexpr int kEpiStageBytes = BN == 64 ? 32768 : 4 * 32 * (kChunk + 4) * 4;
  static_assert(kEpiStageBytes % 1024 == 0 && (kChunk != 32 || kEpiStageBytes >= 4 * 4096),
                "staging area");
  // dynamic shared memory of a launch with `stages` ring stages (at most kStages)
  static constexpr int smem_bytes(int stages) {
    return 1024 + stages * kStageBytes + kBarBytes + kEpiStageBytes;
  }
  static constexpr int kSmemBytes = smem_bytes(kStages);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert((2 * kStages + 5) * 8 + 16 <= kBarBytes, "barrier area");
};

struct TcArgs {
  WorkSpec work;
  int32_t Mm, Nm;         // MMA-view extents
  void* C;                // output, row-major, ldc elements per row
  int64_t ldc;
  const float* bias;      // NULL or one fp32 per output column of C
  float* workspace;       // split partials: 2 slots per CTA of kBM x BN fp32
  int* tickets;           // one arrival counter per split tile (left at 0)
  int* status;            // device status word
  uint64_t wait_limit_ns;
  int32_t a_mn, b_mn;     // operand majors in the MMA view (1 = MN-major)
  int32_t c_tma = 0;      // 1: row-major C chunks leave by TMA store (tmC is valid)
  int32_t c_vec = 0;      // 1: C's base is 16-byte aligned and its row pitch a multiple of
                          // 16 bytes, so every 4-column group is whole and aligned
  int32_t bias_init = 0;  // 1: each tile's k-block-0 accumulator is seeded with the bias
  int32_t stages = 0;      // ring stages of this launch, 1 ... TcConfig<BN>::kStages (0: all)
  int32_t kgroup = 1;      // k-blocks per TMA copy: the ring's stages are taken kgroup at
                           // a time, one copy per operand (half) each; > 1 needs the
                           // operands' maps encoded for it (3-D for K-major)
  uint32_t idesc;         // tcgen05 instruction descriptor
  uint64_t* trace = nullptr;  // NULL, or kTraceSlots %globaltimer stamps per CTA
  int* sched = nullptr;       // two-SM kernel, whole tiles: NULL for the static schedule,
                              // else {next-tile counter, finished pairs}, both 0 at launch
};

// Phase stamps a traced launch writes per CTA (trace[cta * kTraceSlots + i]).
enum TracePhase : int {
  kTraceStart = 0,      // setup done (barriers, TMEM), roles about to start
  kTraceFirstLoad = 1,  // producer issued its first TMA load
  kTraceFirstData = 2,  // MMA issuer saw its first stage land
  kTraceMmaDone = 3,    // MMA issuer committed its last accumulator
  kTraceLastAccum = 4,  // epilogue received its last accumulator
  kTraceEnd = 5,        // epilogue finished (stores and any split fixup)
  kTraceUnits = 6,      // number of work units (not a time)
  kTraceClusterDone = 7,  // cluster split: the cluster's partials added and stored
  kTraceEntry = 8,      // kernel entry (taken first, written after the prerequisite wait)
  kTraceExit = 9,       // TMEM freed, about to return
  kTraceClusterParked = 10,   // cluster split: every CTA of the cluster parked its partial
  kTraceClusterReduced = 11,  // cluster split: the stamping thread's share of the reduction stored
  kTraceSlots = 12
};

// The thread that stamps the end of the epilogue and everything after it
// (the first epilogue thread).
constexpr int kStampThread = 64;

__device__ __forceinline__ void trace_mark(const TcArgs& a, uint32_t cta, int phase) {
  if (a.trace) a.trace[size_t(cta) * kTraceSlots + phase] = globaltimer_ns();
}

// The bias the output stores add: none when the accumulators were seeded
// with it (it is then already in the sum exactly once per tile).
__device__ __forceinline__ const float* out_bias(const TcArgs& a) {
  return a.bias_init ? nullptr : a.bias;
}

__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// AND of `v` over the 128 epilogue threads (also a barrier among them).
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(uint32_t(v))
      : "memory");
  return out != 0;
}

template <int CW>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[CW]) {
  if constexpr (CW == 32) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_wait_ld32(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  } else {
    static_assert(CW == 16, "chunk width");
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
  }
}

// Seeds one accumulator buffer with the bias before the first MMA of a unit
// that starts at k-block 0 (the reduction then starts from the bias instead
// of zero: the FuseReductionEpilogue reading of the kimm240.github.io/tvm
// series).  `taddr` addresses this warp's 32-lane quarter of the buffer; lane
// `row` of it is output row mm (MMA view), columns nbase ... nbase + BN - 1.
// Not TRANS: every row of column n holds bias[n]; TRANS (C stored
// transposed): every column of row mm holds bias[mm].  0 outside the matrix.
template <int BN, int CW, bool TRANS>
__device__ __forceinline__ void seed_bias(const TcArgs& a, uint32_t taddr, int32_t mm,
                                          int32_t nbase) {
  static_assert(CW == 32 || CW == 16, "chunk width");
  const float rowv = (TRANS && mm < a.Mm) ? __ldg(a.bias + mm) : 0.f;
#pragma unroll 1
  for (int c = 0; c < BN / CW; ++c) {
    uint32_t r[CW];
#pragma unroll
    for (int j = 0; j < CW; ++j) {
      const int32_t n = nbase + c * CW + j;
      const float v = TRANS ? rowv : (n < a.Nm ? __ldg(a.bias + n) : 0.f);
      r[j] = __float_as_uint(v);
    }
    __syncwarp();
    if constexpr (CW == 32)
      tmem_st32(taddr + c * CW, r);
    else
      tmem_st16(taddr + c * CW, r);
  }
  tmem_wait_st();
}

// Writes one chunk of CW accumulator columns held by this thread, for the
// transposed store of swapped operands: C[nn0 + j][mm] = v[j] + bias[mm]
// (thread = output column, so a warp's stores are consecutive in C).
template <int CW, bool OUT_F16>
__device__ __forceinline__ void store_chunk_trans(const TcArgs& a, int32_t mm, int32_t nn0,
                                                  const float (&v)[CW]) {
  if (mm >= a.Mm || nn0 >= a.Nm) return;
  const int32_t ncols = (a.Nm - nn0) < CW ? (a.Nm - nn0) : CW;
  const float* ob = out_bias(a);
  const float bv = ob ? __ldg(ob + mm) : 0.f;
#pragma unroll
  for (int j = 0; j < CW; ++j) {
    if (j < ncols) {
      const int64_t off = int64_t(nn0 + j) * a.ldc + mm;
      if constexpr (OUT_F16)
        reinterpret_cast<__half*>(a.C)[off] = __float2half_rn(v[j] + bv);
      else
        reinterpret_cast<float*>(a.C)[off] = v[j] + bv;
    }
  }
}

// One output element of the cluster split (bounds already checked).
template <bool OUT_F16>
__device__ __forceinline__ void put_elem(const TcArgs& a, int64_t off, float v) {
  if constexpr (OUT_F16)
    reinterpret_cast<__half*>(a.C)[off] = __float2half_rn(v);
  else
    reinterpret_cast<float*>(a.C)[off] = v;
}

// Parked partial layouts of the cluster split (floats): row-major rows of
// BN + 4, or column-major columns of 128 + 4 for the transposed store.  The 4
// extra floats keep 16-byte alignment and spread the column walk over banks.
template <int BN>
constexpr int kParkRowStride = BN + 4;
constexpr int kParkColStride = kBM + 4;

// Four consecutive outputs along C's contiguous direction, `valid` of them
// inside the matrix; one vector store when aligned and whole.
template <bool OUT_F16>
__device__ __forceinline__ void put4(const TcArgs& a, int64_t off, float4 v, int valid) {
  const float f[4] = {v.x, v.y, v.z, v.w};
  if constexpr (OUT_F16) {
    __half* dst = reinterpret_cast<__half*>(a.C) + off;
    if (valid == 4 && (reinterpret_cast<uintptr_t>(dst) & 7) == 0) {
      __half2 h0 = __floats2half2_rn(f[0], f[1]);
      __half2 h1 = __floats2half2_rn(f[2], f[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&h0);
      pk.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(dst) = pk;
      return;
    }
  } else {
    float* dst = reinterpret_cast<float*>(a.C) + off;
    if (valid == 4 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
      *reinterpret_cast<float4*>(dst) = v;
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < valid) put_elem<OUT_F16>(a, off + j, f[j]);
}

// Row-major store of one epilogue warp's 32 rows x CW columns (lane i holds row
// mrow0 + i in v).  Written straight out, each store instruction would touch 32
// rows with 16 bytes each; instead the rows go through the warp's staging block
// sw (rows of CW + 4 floats: conflict-free 16-byte accesses) and come back out
// as runs of CW consecutive columns, 32 / (CW / 4) rows per instruction.  The
// bias is added in fp32 before the single rounding, as in every other store.
template <int CW, bool OUT_F16, int kRows = 32>
__device__ __forceinline__ void store_rows_staged(const TcArgs& a, float* sw, int32_t mrow0,
                                                  int lane, int32_t nn0, const float (&v)[CW]) {
  if (mrow0 >= a.Mm || nn0 >= a.Nm) return;  // the same for the whole warp
  constexpr int LD = CW + 4;
  constexpr int Q = CW / 4;    // float4 per row
  constexpr int RPI = 32 / Q;  // rows per pass
  __syncwarp();                // the previous chunk's reads of sw are done
  float4* mine = reinterpret_cast<float4*>(sw + lane * LD);
#pragma unroll
  for (int j = 0; j < Q; ++j)
    mine[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  __syncwarp();
  const int c4 = lane % Q;
  const int32_t nn = nn0 + 4 * c4;
  const int valid = min(4, a.Nm - nn);
  float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* ob = out_bias(a);
  if (ob && valid > 0) {
    b4.x = __ldg(ob + nn);
    if (valid > 1) b4.y = __ldg(ob + nn + 1);
    if (valid > 2) b4.z = __ldg(ob + nn + 2);
    if (valid > 3) b4.w = __ldg(ob + nn + 3);
  }
  // All shared reads first, then all global stores: a store through the
  // generic C pointer could alias the staging block as far as the compiler
  // knows, so interleaving them would serialise every read behind the store
  // before it.
  constexpr int kPasses = kRows / RPI;  // only the first kRows rows of the block are real
  float4 x[kPasses];
#pragma unroll
  for (int it = 0; it < kPasses; ++it)
    x[it] = *reinterpret_cast<const float4*>(sw + (it * RPI + lane / Q) * LD + 4 * c4);
  if (valid <= 0) return;
#pragma unroll
  for (int it = 0; it < kPasses; ++it) {
    const int32_t mm = mrow0 + it * RPI + lane / Q;
    if (mm >= a.Mm) continue;
    float4 y = x[it];
    y.x += b4.x; y.y += b4.y; y.z += b4.z; y.w += b4.w;
    put4<OUT_F16>(a, int64_t(mm) * a.ldc + nn, y, valid);
  }
}

// The same store when C takes whole, aligned 4-column groups (TcArgs::c_vec):
// the bounds and alignment are settled once per chunk and the row pointer
// advances by a fixed step, so the stores of all passes issue back to back
// instead of one guarded store after another.
template <int CW, bool OUT_F16, int kRows = 32>
__device__ __forceinline__ void store_rows_vec(const TcArgs& a, float* sw, int32_t mrow0,
                                               int lane, int32_t nn0, const float (&v)[CW]) {
  constexpr int LD = CW + 4;
  constexpr int Q = CW / 4;    // float4 per row
  constexpr int RPI = 32 / Q;  // rows per pass
  constexpr int kPasses = kRows / RPI;  // only the first kRows rows of the block are real
  static_assert(kPasses >= 1 && kRows % RPI == 0, "rows per pass");
  __syncwarp();                // the previous chunk's reads of sw are done
  float4* mine = reinterpret_cast<float4*>(sw + lane * LD);
#pragma unroll
  for (int j = 0; j < Q; ++j)
    mine[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  __syncwarp();
  const int c4 = lane % Q;
  const int rsub = lane / Q;
  float4 x[kPasses];
#pragma unroll
  for (int it = 0; it < kPasses; ++it)
    x[it] = *reinterpret_cast<const float4*>(sw + (it * RPI + rsub) * LD + 4 * c4);
  const int32_t nn = nn0 + 4 * c4;
  const int32_t r0 = mrow0 + rsub;
  if (nn >= a.Nm || r0 >= a.Mm) return;  // no warp-wide step follows
  const float* ob = out_bias(a);
  if (ob) {
    const float4 b4 = make_float4(__ldg(ob + nn), __ldg(ob + nn + 1), __ldg(ob + nn + 2),
                                  __ldg(ob + nn + 3));
#pragma unroll
    for (int it = 0; it < kPasses; ++it) {
      x[it].x += b4.x; x[it].y += b4.y; x[it].z += b4.z; x[it].w += b4.w;
    }
  }
  const int32_t rows = a.Mm - r0;  // > 0: rows of this lane's group left in C
  const int64_t step = int64_t(RPI) * a.ldc;
  if constexpr (OUT_F16) {
    __half* p = reinterpret_cast<__half*>(a.C) + int64_t(r0) * a.ldc + nn;
#pragma unroll
    for (int it = 0; it < kPasses; ++it, p += step) {
      const __half2 h0 = __floats2half2_rn(x[it].x, x[it].y);
      const __half2 h1 = __floats2half2_rn(x[it].z, x[it].w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&h0);
      pk.y = *reinterpret_cast<const uint32_t*>(&h1);
      if (it * RPI < rows) *reinterpret_cast<uint2*>(p) = pk;
    }
  } else {
    float* p = reinterpret_cast<float*>(a.C) + int64_t(r0) * a.ldc + nn;
#pragma unroll
    for (int it = 0; it < kPasses; ++it, p += step)
      if (it * RPI < rows) *reinterpret_cast<float4*>(p) = x[it];
  }
}

// Row-major store of one epilogue warp's 32 rows x 32 columns by TMA: lane i
// writes row mrow0 + i (bias added, rounded once to the output type) into the
// warp's 4 KiB box in shared memory, in the layout the tensor map's swizzle
// expects (128-byte rows for fp32, 16-byte piece k at k ^ (row % 8); 64-byte
// rows for fp16, piece k at k ^ ((row / 2) % 4)), which also keeps the shared
// stores free of bank conflicts; lane 0 then issues one bulk store of the box.
// Rows and columns past the matrix are dropped by the TMA unit.  fp16 boxes
// (2 KiB) alternate between the two halves of the warp's 4 KiB, so the next
// chunk is written while the TMA unit still reads the previous one (the unit
// takes a few hundred cycles per copy); a box is reused only after the store
// from it has read it.  `first` (the tile's first chunk, whose box the
// previous tile's last store may still read) waits for every earlier store.
template <bool OUT_F16>
__device__ __forceinline__ void store_rows_tma(const CUtensorMap* tmC, const TcArgs& a,
                                               uint8_t* box, int32_t mrow0, int lane,
                                               int32_t nn0, const float (&v)[32], bool first) {
  if (mrow0 >= a.Mm || nn0 >= a.Nm) return;  // the same for the whole warp
  if constexpr (OUT_F16) box += ((nn0 >> 5) & 1) * 2048;
  if (lane == 0) {
    if (OUT_F16 && !first)
      bulk_wait_read_1();
    else
      bulk_wait_read_all();
  }
  __syncwarp();
  float o[32];
  const float* ob = out_bias(a);
  const float* bp = ob ? ob + nn0 : nullptr;
  if (bp && nn0 + 32 <= a.Nm && (reinterpret_cast<uintptr_t>(bp) & 15) == 0) {
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(bp + j));
      o[j] = v[j] + b4.x; o[j + 1] = v[j + 1] + b4.y;
      o[j + 2] = v[j + 2] + b4.z; o[j + 3] = v[j + 3] + b4.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = v[j] + ((bp && nn0 + j < a.Nm) ? __ldg(bp + j) : 0.f);
  }
  const uint32_t base = smem_u32(box);
  if constexpr (OUT_F16) {
    const uint32_t row = base + uint32_t(lane) * 64u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 p = __floats2half2_rn(o[8 * k + 2 * i], o[8 * k + 2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      st_shared_v4(row + uint32_t((k ^ ((lane >> 1) & 3)) * 16), h[0], h[1], h[2], h[3]);
    }
  } else {
    const uint32_t row = base + uint32_t(lane) * 128u;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      st_shared_v4(row + uint32_t((k ^ (lane & 7)) * 16), __float_as_uint(o[4 * k]),
                   __float_as_uint(o[4 * k + 1]), __float_as_uint(o[4 * k + 2]),
                   __float_as_uint(o[4 * k + 3]));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, base, nn0, mrow0);
    bulk_commit_group();
  }
}

// Any store of an epilogue chunk: transposed stores are already coalesced
// (lanes are consecutive columns of C); row-major ones leave by TMA store when
// the launch set one up (32-column chunks), else through the padded staging
// (with whole aligned 4-column groups where C allows them).
template <int CW, bool OUT_F16, bool TRANS>
__device__ __forceinline__ void store_out(const TcArgs& a, const CUtensorMap* tmC,
                                          uint8_t* stage, int q, int32_t mm, int lane,
                                          int32_t nn0, const float (&v)[CW], bool first) {
  if constexpr (TRANS) {
    store_chunk_trans<CW, OUT_F16>(a, mm, nn0, v);
  } else {
    if constexpr (CW == 32) {
      if (a.c_tma) {
        store_rows_tma<OUT_F16>(tmC, a, stage + q * 4096, mm - lane, lane, nn0, v, first);
        return;
      }
    }
    float* sw = reinterpret_cast<float*>(stage) + q * 32 * (CW + 4);
    if (a.c_vec)
      store_rows_vec<CW, OUT_F16>(a, sw, mm - lane, lane, nn0, v);
    else
      store_rows_staged<CW, OUT_F16>(a, sw, mm - lane, lane, nn0, v);
  }
}

// Cluster split: after every CTA of the cluster parked its fp32 partial of the
// same tile at the start of its shared memory, CTA `rank` adds rows
// [rank*R, (rank+1)*R), R = 128 / s, over all s partials in rank order -- rank
// order is ascending k, so the sum does not depend on timing -- adds the bias
// and writes C.  Work goes in groups of 4 floats along the direction in which
// C is contiguous (output columns, or rows for the transposed store).  All
// `nthreads` threads of the CTA take part, each with the loads of kU groups
// (s 16-byte loads each, the own partial from local shared memory) in flight
// at once: the reduction is bound by the round trip to the peers' memory.
template <int BN, bool OUT_F16, bool TRANS>
__device__ __forceinline__ void csplit_reduce(const TcArgs& a, const uint8_t* smem, int tid,
                                              int nthreads, int32_t tm, int32_t tn) {
  const WorkSpec& W = a.work;
  const int s = W.csplit;
  const int rank = int(blockIdx.x) & (s - 1);
  const int R = kBM / s;  // 64, 32 or 16 rows
  const uint32_t local = smem_u32(smem);
  uint32_t peer[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) peer[j] = j < s ? map_to_rank(local, uint32_t(j)) : 0u;
  const int groups = TRANS ? BN * (R / 4) : R * (BN / 4);
  const float* ob = out_bias(a);
  constexpr int kU = 4;
#pragma unroll 1
  for (int g0 = tid; g0 < groups; g0 += kU * nthreads) {
    float4 part[kU][8];
    int row[kU], col[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int g = g0 + u * nthreads;
      if (TRANS) {
        col[u] = g / (R / 4);
        row[u] = rank * R + (g % (R / 4)) * 4;
      } else {
        row[u] = rank * R + g / (BN / 4);
        col[u] = (g % (BN / 4)) * 4;
      }
      if (g < groups) {
        const uint32_t off =
            4u * uint32_t(TRANS ? col[u] * kParkColStride + row[u] : row[u] * kParkRowStride<BN> + col[u]);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < s)
            part[u][j] = j == rank ? *reinterpret_cast<const float4*>(smem + off)
                                   : ld_dsmem_f32x4(peer[j] + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (g0 + u * nthreads >= groups) break;
      float4 acc = part[u][0];
#pragma unroll
      for (int j = 1; j < 8; ++j)
        if (j < s) {
          acc.x += part[u][j].x; acc.y += part[u][j].y;
          acc.z += part[u][j].z; acc.w += part[u][j].w;
        }
      const int32_t mm = tm * kBM + row[u];  // MMA-view row (first of 4 when TRANS)
      const int32_t nn = tn * BN + col[u];   // MMA-view column (first of 4 otherwise)
      if constexpr (!TRANS) {
        if (mm >= a.Mm || nn >= a.Nm) continue;
        const int valid = min(4, a.Nm - nn);
        if (ob) {
          acc.x += __ldg(ob + nn);
          if (valid > 1) acc.y += __ldg(ob + nn + 1);
          if (valid > 2) acc.z += __ldg(ob + nn + 2);
          if (valid > 3) acc.w += __ldg(ob + nn + 3);
        }
        put4<OUT_F16>(a, int64_t(mm) * a.ldc + nn, acc, valid);
      } else {
        if (mm >= a.Mm || nn >= a.Nm) continue;
        const int valid = min(4, a.Mm - mm);
        if (ob) {
          acc.x += __ldg(ob + mm);
          if (valid > 1) acc.y += __ldg(ob + mm + 1);
          if (valid > 2) acc.z += __ldg(ob + mm + 2);
          if (valid > 3) acc.w += __ldg(ob + mm + 3);
        }
        put4<OUT_F16>(a, int64_t(nn) * a.ldc + mm, acc, valid);
      }
    }
  }
}

// Cluster split with swapped operands and a narrow tile (BN <= 64): every CTA
// pushes the rows of its fp32 partial that rank j adds straight into rank j's
// staging area (idle in this kernel: transposed output needs no staging), as
// slot[src][column][row], R = 128 / s rows per rank, with remote stores that
// need no round trip.  After one cluster barrier each CTA adds the s slots of
// its own rows in source-rank order -- ascending k, so the sum does not depend
// on timing -- adds the bias and writes C; no CTA reads another's memory after
// the barrier, so none has to wait for the others before it exits.
template <int BN>
constexpr bool kPushReduce = BN <= 64;

template <int BN, bool OUT_F16>
__device__ __forceinline__ void csplit_reduce_pushed(const TcArgs& a, const uint8_t* stage,
                                                     int tid, int nthreads, int32_t tm,
                                                     int32_t tn) {
  const WorkSpec& W = a.work;
  const int s = W.csplit;
  const int rank = int(blockIdx.x) & (s - 1);
  const int R = kBM / s;
  const float* slot = reinterpret_cast<const float*>(stage);
  const float* ob = out_bias(a);
  const int groups = BN * (R / 4);  // 4 consecutive rows of one column each
#pragma unroll 1
  for (int g = tid; g < groups; g += nthreads) {
    const int col = g / (R / 4);
    const int r4 = (g % (R / 4)) * 4;
    // all s slots' loads in flight at once, added in source order
    float4 part[8];
#pragma unroll
    for (int src = 0; src < 8; ++src)
      if (src < s) part[src] = *reinterpret_cast<const float4*>(slot + (src * BN + col) * R + r4);
    float4 acc = part[0];
#pragma unroll
    for (int src = 1; src < 8; ++src)
      if (src < s) {
        acc.x += part[src].x; acc.y += part[src].y; acc.z += part[src].z; acc.w += part[src].w;
      }
    const int32_t mm = tm * kBM + rank * R + r4;  // MMA-view row: C column
    const int32_t nn = tn * BN + col;             // MMA-view column: C row
    if (mm >= a.Mm || nn >= a.Nm) continue;
    const int valid = min(4, a.Mm - mm);
    if (ob) {
      acc.x += __ldg(ob + mm);
      if (valid > 1) acc.y += __ldg(ob + mm + 1);
      if (valid > 2) acc.z += __ldg(ob + mm + 2);
      if (valid > 3) acc.w += __ldg(ob + mm + 3);
    }
    put4<OUT_F16>(a, int64_t(nn) * a.ldc + mm, acc, valid);
  }
}

// The same exchange for tiles 32 or 64 columns wide with operands in place
// (row-major output): rank j adds rows [j*R, (j+1)*R) of the tile, and each
// CTA pushes those rows of its partial into rank j's staging area as
// slot[src][row][column], 16 bytes at a time.  A row's float4 c4 sits at
// c4 ^ (row % 8), so the 32 rows a warp pushes at once, and the column groups a
// warp reads back, fall on different banks although rows are a whole number
// of 128-byte lines long.
__device__ __forceinline__ uint32_t push_row_offset(int src, int R, int BN, int r, int c4) {
  return 4u * uint32_t((src * R + r) * BN + 4 * (c4 ^ (r & 7)));
}

template <int BN, bool OUT_F16>
__device__ __forceinline__ void csplit_reduce_pushed_rows(const TcArgs& a, const uint8_t* stage,
                                                          int tid, int nthreads, int32_t tm,
                                                          int32_t tn) {
  static_assert(BN == 32 || BN == 64, "row pushes: 8 or 16 float4 per row");
  const WorkSpec& W = a.work;
  const int s = W.csplit;
  const int rank = int(blockIdx.x) & (s - 1);
  const int R = kBM / s;
  const float* ob = out_bias(a);
  constexpr int G = BN / 4;  // float4 per row
  const int groups = R * G;
#pragma unroll 1
  for (int g = tid; g < groups; g += nthreads) {
    const int r = g / G;
    const int c4 = g % G;
    float4 part[8];
#pragma unroll
    for (int src = 0; src < 8; ++src)
      if (src < s)
        part[src] = *reinterpret_cast<const float4*>(stage + push_row_offset(src, R, BN, r, c4));
    float4 acc = part[0];
#pragma unroll
    for (int src = 1; src < 8; ++src)
      if (src < s) {
        acc.x += part[src].x; acc.y += part[src].y; acc.z += part[src].z; acc.w += part[src].w;
      }
    const int32_t mm = tm * kBM + rank * R + r;
    const int32_t nn = tn * BN + 4 * c4;
    if (mm >= a.Mm || nn >= a.Nm) continue;
    const int valid = min(4, a.Nm - nn);
    if (ob) {
      acc.x += __ldg(ob + nn);
      if (valid > 1) acc.y += __ldg(ob + nn + 1);
      if (valid > 2) acc.z += __ldg(ob + nn + 2);
      if (valid > 3) acc.w += __ldg(ob + nn + 3);
    }
    put4<OUT_F16>(a, int64_t(mm) * a.ldc + nn, acc, valid);
  }
}

// 16-byte store into a cluster CTA's shared memory.
__device__ __forceinline__ void st_dsmem_f32x4(uint32_t cluster_addr, float x, float y, float z,
                                               float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(x),
               "f"(y), "f"(z), "f"(w)
               : "memory");
}

template <int BN, bool OUT_F16, bool TRANS>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcArgs args) {
  using Cfg = TcConfig<BN>;
  // A launch may use fewer stages than the ring can hold: less shared memory,
  // so that the next launch's CTAs fit beside this one's.  The ring's k-block
  // slots are taken J = args.kgroup at a time: one TMA copy per operand (half)
  // brings J consecutive k-blocks (a 3-D box for a K-major operand, a box J
  // k-blocks deep for an MN-major one), as in the 64-row kernel.
  const int J = args.kgroup > 1 ? args.kgroup : 1;
  const int S = (args.stages > 0 ? args.stages : Cfg::kStages) / J;  // stages of J blocks
  constexpr int CW = Cfg::kChunk;

  const uint64_t t_entry = args.trace ? globaltimer_ns() : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                         // S x J x 16 KiB
  uint8_t* sB = smem + S * J * Cfg::kABytes;  // S x J x BN*128 B
  uint8_t* stage = sB + S * J * Cfg::kBBytes; // epilogue staging, 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + Cfg::kEpiStageBytes);
  uint64_t* full = bars;                      // TMA bytes landed in stage s
  uint64_t* empty = bars + S;                 // MMAs reading stage s are done
  uint64_t* acc_full = bars + 2 * S;          // accumulator b finished
  uint64_t* acc_empty = acc_full + 2;         // accumulator b drained by the epilogue
  uint64_t* drain = acc_empty + 2;            // clean-up after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

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
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (args.c_tma) tma_prefetch_map(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Up to here only this CTA's own resources were touched.  Let the next
  // kernel of the stream start its prologue.  Each role then does what needs
  // only this CTA's own resources (work iterators, the first unit's
  // coordinates, the first free stage) and waits for the kernels before this
  // one to complete before it touches global memory (operands, C, workspace,
  // counters, status, trace): with a programmatic launch that preparation
  // overlaps the previous kernel instead of following it.
  pdl_launch_dependents();
  const WaitCtl wc{args.wait_limit_ns, args.status, abort_flag};
  const WorkSpec& W = args.work;
  auto prerequisites_done = [&]() {
    pdl_wait_prerequisites();
    if (threadIdx.x == 0 && args.trace) {
      args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceEntry] = t_entry;
      trace_mark(args, blockIdx.x, kTraceStart);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      WorkIter it;
      it.init_tc(W, blockIdx.x);
      Unit u;
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true;
      bool first = true;
      bool waited = false;
      while (ok && it.next(W, u)) {
        int32_t tm, tn;
        tile_coords(W, u.tile, tm, tn);
        for (int32_t kb = u.kb0; kb < u.kb1; kb += J) {
          if (!wait_bounded(smem_u32(&empty[s]), ph ^ 1, wc, kSiteProducer)) {
            ok = false;
            break;
          }
          if (!waited) {  // the first load: the operands are now final
            prerequisites_done();
            waited = true;
          }
          // whole boxes: zeros past K, or k-blocks past the unit no MMA uses
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, J * Cfg::kStageBytes);
          const uint32_t a_dst = smem_u32(sA + s * J * Cfg::kABytes);
          const uint32_t b_dst = smem_u32(sB + s * J * Cfg::kBBytes);
          const int32_t k0 = kb * kBK;
          if (!args.a_mn) {
            if (J > 1)
              tma_load_3d(a_dst, &tmA, fb, 0, tm * kBM, kb);
            else
              tma_load_2d(a_dst, &tmA, fb, k0, tm * kBM);
          } else {  // two 64-wide halves, J k-blocks deep each
            tma_load_2d(a_dst, &tmA, fb, tm * kBM, k0);
            tma_load_2d(a_dst + J * 8192, &tmA, fb, tm * kBM + 64, k0);
          }
          if (!args.b_mn) {
            if (J > 1)
              tma_load_3d(b_dst, &tmB, fb, 0, tn * BN, kb);
            else
              tma_load_2d(b_dst, &tmB, fb, k0, tn * BN);
          } else {
            if constexpr (BN >= 64) {
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
      if (!waited) prerequisites_done();  // no load at all
      if (!ok) {  // let the copies still in flight land before the CTA exits
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
      // an MN-major operand's 64-wide halves sit J k-blocks (J x 8 KiB) apart
      const uint32_t a_lbo = args.a_mn ? uint32_t(J) * 8192u : 16u;
      const uint32_t b_lbo = args.b_mn ? uint32_t(J) * 8192u : 16u;
      // advance per 16-deep k slice: 32 B along a K-major row, 16 rows (2 KiB) MN-major
      const uint32_t a_step = args.a_mn ? (2048u >> 4) : (32u >> 4);
      const uint32_t b_step = args.b_mn ? (2048u >> 4) : (32u >> 4);
      // k-block j of a group: a whole block K-major, 64 k rows of each half MN-major
      const uint32_t a_blk = args.a_mn ? 8192u : uint32_t(Cfg::kABytes);
      const uint32_t b_blk = args.b_mn ? 8192u : uint32_t(Cfg::kBBytes);
      while (ok && it.next(W, u)) {
        // the epilogue releases each buffer once before its first use (after
        // seeding it, if asked) and once after each drain
        if (!wait_bounded(smem_u32(&acc_empty[b]), aph, wc, kSiteMmaAccum)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(b * BN);
        const bool seeded = args.bias_init && u.kb0 == 0;  // accumulate onto the bias
        for (int32_t kb = u.kb0; kb < u.kb1; kb += J) {
          if (!wait_bounded(smem_u32(&full[s]), ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!any) trace_mark(args, blockIdx.x, kTraceFirstData);
          const uint32_t a0 = smem_u32(sA + s * J * Cfg::kABytes);
          const uint32_t b0 = smem_u32(sB + s * J * Cfg::kBBytes);
          const int nj = u.kb1 - kb < J ? int(u.kb1 - kb) : J;
#pragma unroll 1
          for (int j = 0; j < nj; ++j) {
            const uint64_t adesc = make_sdesc_sw128(a0 + uint32_t(j) * a_blk, a_lbo, 1024);
            const uint64_t bdesc = make_sdesc_sw128(b0 + uint32_t(j) * b_blk, b_lbo, 1024);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_f16(d_tmem, adesc + uint64_t(kk * a_step), bdesc + uint64_t(kk * b_step),
                         args.idesc, (kb > u.kb0 || j > 0 || kk > 0 || seeded) ? 1u : 0u);
          }
          any = true;
          tc_commit(smem_u32(&empty[s]));
          if (++s == S) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        // stamped before the commit, so the epilogue cannot see it first
        trace_mark(args, blockIdx.x, kTraceMmaDone);
        tc_commit(smem_u32(&acc_full[b]));
        if (++b == 2) {
          b = 0;
          aph ^= 1;
        }
      }
      if (!ok && any) {  // every MMA issued so far must finish before TMEM is freed
        tc_commit(smem_u32(drain));
        wait_drain(smem_u32(drain), 0, wc);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;     // accumulator row inside the tile
    const int et = threadIdx.x - 64;   // 0..127
    // `ahead` runs two units ahead of `it`: the unit that will next use the
    // buffer just drained, which is seeded with the bias before its release
    WorkIter it, ahead;
    it.init_tc(W, blockIdx.x);
    ahead.init_tc(W, blockIdx.x);
    pdl_wait_prerequisites();  // the bias (seeding), C and the workspace are global
    Unit u, un;
    auto release = [&](int buf, bool have_next) {
      if (have_next && args.bias_init && un.kb0 == 0) {
        int32_t tm2, tn2;
        tile_coords(W, un.tile, tm2, tn2);
        seed_bias<BN, CW, TRANS>(args, tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN),
                                 tm2 * kBM + row, tn2 * BN);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acc_empty[buf]));
    };
    release(0, ahead.next(W, un));
    release(1, ahead.next(W, un));
    int b = 0;
    uint32_t aph = 0;
    int units = 0;
    while (it.next(W, u)) {
      int32_t tm, tn;
      tile_coords(W, u.tile, tm, tn);  // while the MMAs still run
      const bool got = wait_bounded(smem_u32(&acc_full[b]), aph, wc, kSiteEpilogue);
      if (!epi_all(got)) break;
      tc_fence_after();
      if (et == 0) trace_mark(args, blockIdx.x, kTraceLastAccum);
      ++units;
      const int32_t mm = tm * kBM + row;
      const int32_t nbase = tn * BN;
      const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(b * BN);

      if (TRANS && kPushReduce<BN> && W.csplit > 1) {
        // Cluster split, narrow swapped tile: push each row of the partial to
        // the rank that adds it (csplit_reduce_pushed).
        static_assert(!kPushReduce<BN> || kBM * BN * 4 <= Cfg::kEpiStageBytes, "slots");
        const int s = W.csplit;
        const int R = kBM / s;
        const int owner = row / R;
        const int r_in = row - owner * R;
        const int src = int(blockIdx.x) % s;
        const uint32_t dst = map_to_rank(smem_u32(stage), uint32_t(owner));
#pragma unroll 1
        for (int c = 0; c < BN / CW; ++c) {
          float v[CW];
          __syncwarp();
          tmem_load_chunk<CW>(taddr + c * CW, v);
#pragma unroll
          for (int j = 0; j < CW; ++j)
            st_dsmem_f32(dst + 4u * uint32_t((src * BN + c * CW + j) * R + r_in), v[j]);
        }
      } else if (!TRANS && kPushReduce<BN> && W.csplit > 1) {
        // Cluster split, narrow tile in place: push each row of the partial
        // to the rank that adds it (csplit_reduce_pushed_rows).
        const int s = W.csplit;
        const int R = kBM / s;
        const int owner = row / R;
        const int r_in = row - owner * R;
        const int src = int(blockIdx.x) % s;
        const uint32_t dst = map_to_rank(smem_u32(stage), uint32_t(owner));
#pragma unroll 1
        for (int c = 0; c < BN / CW; ++c) {
          float v[CW];
          __syncwarp();
          tmem_load_chunk<CW>(taddr + c * CW, v);
#pragma unroll
          for (int j = 0; j < CW / 4; ++j)
            st_dsmem_f32x4(dst + push_row_offset(src, R, BN, r_in, c * (CW / 4) + j), v[4 * j],
                           v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      } else if (W.csplit > 1) {
        // Cluster split: park this CTA's fp32 partial in its own (now idle)
        // stage ring, in the layout the reduction walks (csplit_reduce):
        // row-major with rows of BN + 4 floats, or, for the transposed store,
        // column-major with columns of 128 + 4 floats.
        float* park = reinterpret_cast<float*>(smem);
        fence_proxy_async_smem();  // the ring was last touched by TMA and MMA
#pragma unroll 1
        for (int c = 0; c < BN / CW; ++c) {
          float v[CW];
          __syncwarp();
          tmem_load_chunk<CW>(taddr + c * CW, v);
          if constexpr (!TRANS) {
            float4* dst = reinterpret_cast<float4*>(park + row * kParkRowStride<BN> + c * CW);
#pragma unroll
            for (int j = 0; j < CW / 4; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < CW; ++j) park[(c * CW + j) * kParkColStride + row] = v[j];
          }
        }
      } else if (!unit_is_partial(W, u)) {
#pragma unroll 1
        for (int c = 0; c < BN / CW; ++c) {
          float v[CW];
          __syncwarp();
          tmem_load_chunk<CW>(taddr + c * CW, v);
          store_out<CW, OUT_F16, TRANS>(args, &tmC, stage, q, mm, lane, nbase + c * CW, v,
                                        c == 0);
        }
      } else {
        const int32_t st = u.tile - W.dp_tiles;  // split-tile index
        const int32_t me = blockIdx.x;
        const size_t slot_elems = size_t(kBM) * BN;
        float* mine = args.workspace + size_t(split_slot(W, me, st)) * slot_elems;
        // publish this CTA's fp32 partial: float4 j of a row's chunk c at float4
        // index (c * CW/4 + j) * 128 + row, so a warp's stores are contiguous
#pragma unroll 1
        for (int c = 0; c < BN / CW; ++c) {
          float v[CW];
          __syncwarp();
          tmem_load_chunk<CW>(taddr + c * CW, v);
          float4* dst = reinterpret_cast<float4*>(mine) + size_t(c) * (CW / 4) * kBM + row;
#pragma unroll
          for (int j = 0; j < CW / 4; ++j)
            __stcg(dst + j * kBM,
                   make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        }
        __threadfence();
        epi_bar_sync();
        int32_t first, last;
        split_contributors(W, st, first, last);
        if (et == 0) {
          const int old = atomicAdd(&args.tickets[st], 1);
          *last_flag = (old == last - first) ? 1 : 0;
        }
        epi_bar_sync();
        if (*last_flag) {
          __threadfence();
          // Contributors are read kFixBatch at a time (all loads of a batch in
          // flight together) and added strictly in ascending order, so the sum
          // is the same whichever CTA arrives last.
          constexpr int kFixBatch = CW == 32 ? 2 : 4;  // 64 staged floats per thread
#pragma unroll 1
          for (int c = 0; c < BN / CW; ++c) {
            float own[CW], acc[CW];
            __syncwarp();
            tmem_load_chunk<CW>(taddr + c * CW, own);
#pragma unroll 1
            for (int32_t r0 = first; r0 <= last; r0 += kFixBatch) {
              float4 part[kFixBatch][CW / 4];
#pragma unroll
              for (int b = 0; b < kFixBatch; ++b) {
                const int32_t r = r0 + b;
                if (r <= last && r != me) {
                  const float4* src =
                      reinterpret_cast<const float4*>(args.workspace +
                                                      size_t(split_slot(W, r, st)) * slot_elems) +
                      size_t(c) * (CW / 4) * kBM + row;
#pragma unroll
                  for (int j = 0; j < CW / 4; ++j) part[b][j] = __ldcg(src + j * kBM);
                }
              }
#pragma unroll
              for (int b = 0; b < kFixBatch; ++b) {
                const int32_t r = r0 + b;
                if (r > last) break;
                float v[CW];
                if (r == me) {
#pragma unroll
                  for (int j = 0; j < CW; ++j) v[j] = own[j];
                } else {
#pragma unroll
                  for (int j = 0; j < CW / 4; ++j) {
                    v[4 * j] = part[b][j].x; v[4 * j + 1] = part[b][j].y;
                    v[4 * j + 2] = part[b][j].z; v[4 * j + 3] = part[b][j].w;
                  }
                }
                if (r == first) {
#pragma unroll
                  for (int j = 0; j < CW; ++j) acc[j] = v[j];
                } else {
#pragma unroll
                  for (int j = 0; j < CW; ++j) acc[j] += v[j];
                }
              }
            }
            store_out<CW, OUT_F16, TRANS>(args, &tmC, stage, q, mm, lane, nbase + c * CW,
                                          acc, c == 0);
          }
          if (et == 0) atomicExch(&args.tickets[st], 0);  // ready for the next launch
        }
      }
      release(b, ahead.next(W, un));
      if (++b == 2) {
        b = 0;
        aph ^= 1;
      }
    }
    // every bulk store this warp issued has landed before the CTA moves on
    if (args.c_tma && lane == 0) bulk_wait_all();
    __syncwarp();
    if (et == 0) {
      trace_mark(args, blockIdx.x, kTraceEnd);
      if (args.trace) args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceUnits] = uint64_t(units);
    }
  }

  __syncthreads();
  if (W.csplit > 1) {
    // The cluster's tile (s = 2, 4 or 8 CTAs per tile), worked out before
    // the barrier, whose wait hides the divisions.
    int32_t ctm, ctn;
    tile_coords(W, int32_t(blockIdx.x) >> (W.csplit == 8 ? 3 : W.csplit == 4 ? 2 : 1), ctm, ctn);
    // Every thread of every CTA of the cluster reaches the barriers, aborted
    // or not, so none can wait forever.
    cluster_sync_all();  // all partials parked (or pushed to their owners)
    // the tail's stamps come from the thread that stamped the epilogue's end,
    // so they are ordered however the timer reads are scheduled
    if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceClusterParked);
    if constexpr (kPushReduce<BN>) {
      if constexpr (TRANS)
        csplit_reduce_pushed<BN, OUT_F16>(args, stage, threadIdx.x, kTcThreads, ctm, ctn);
      else
        csplit_reduce_pushed_rows<BN, OUT_F16>(args, stage, threadIdx.x, kTcThreads, ctm, ctn);
      if (threadIdx.x == kStampThread) {
        trace_mark(args, blockIdx.x, kTraceClusterReduced);
        trace_mark(args, blockIdx.x, kTraceClusterDone);
      }
    } else {
      csplit_reduce<BN, OUT_F16, TRANS>(args, smem, threadIdx.x, kTcThreads, ctm, ctn);
      if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceClusterReduced);
      cluster_sync_all();  // no CTA still reads another's shared memory
      if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceClusterDone);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
  if (args.trace) {  // the exit stamp after the TMEM is freed
    __syncthreads();
    if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceExit);
  }
}

}  // namespace dg
