// tc2_kernel.cuh: the two-SM tcgen05 GEMM (cta_group::2) for large shapes.
//
// The last rung of the native GEMM ladder in the TIRx "Compiling and inspecting"
// page ("sync -> TMA -> warp specialization -> 2-CTA cluster") on sm_103a:
// a cluster of two CTAs on two SMs owns one 256 x 256 output tile.
//   - Each CTA TMA-loads its own 128 rows of A and its own 128-column half of B
//     into its S-stage ring (32 KiB per stage instead of 48 KiB per SM for the
//     one-SM 128 x 256 tile: each SM fetches half of B).  Both CTAs' bytes
//     complete on the leader CTA's `full` barrier.
//   - One thread of the leader (cluster rank 0) issues
//     tcgen05.mma.cta_group::2 with M = 256, N = 256: the hardware reads A rows
//     0-127 and B columns 0-127 from the leader's shared memory and the other
//     halves from the peer's, at the same offsets, and accumulates rows 0-127 in
//     the leader's TMEM and rows 128-255 in the peer's.
//   - tcgen05.commit with a two-CTA multicast frees the stage in both CTAs and
//     hands both accumulators to their epilogues; each epilogue warp reports a
//     drained accumulator to the leader with a remote mbarrier arrive.
// Persistent over clusters with a grouped raster.  Tiles are whole, except
// for an optional Stream-K region (work.cuh, counted in pair tiles and pairs):
// each CTA of a pair publishes its 128-row half of a partial tile, and per
// half the last pair to arrive adds the halves in ascending k order, so no CTA
// ever waits for another pair.  Every wait is bounded as in the one-SM kernel.
#pragma once

#include "tc_kernel.cuh"

namespace dg {

constexpr int kPairBM = 256;  // rows per cluster tile
constexpr int kPairBN = 256;  // columns per cluster tile
constexpr int kHalfBN = 128;  // B columns each CTA loads

struct Tc2Config {
  static constexpr int kStages = 6;
  static constexpr int kABytes = kBM * kBK * 2;      // 16 KiB: this CTA's 128 rows
  static constexpr int kBBytes = kHalfBN * kBK * 2;  // 16 KiB: this CTA's 128 columns
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 512;  // two 256-column accumulators
  static constexpr int kSchedDepth = 4;  // tile ring of the dynamic schedule
  static constexpr int kBarBytes = 256;
  // epilogue staging (after the stages, so 1024-byte aligned), 4 warps: padded
  // rows of 36 floats, or a 4 KiB swizzled TMA store box each
  static constexpr int kEpiStageBytes = 4 * 32 * (32 + 4) * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kEpiStageBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((2 * kStages + 5 + 2 * kSchedDepth) * 8 + 16 + 4 * kSchedDepth <= kBarBytes,
                "barrier area");
};

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the barrier at this shared-memory offset in both CTAs of the pair
// once every tcgen05 op this thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Same, on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair_self(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on a
// barrier that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// The same for a 3-D box (a group of k-blocks of a K-major operand).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Consumers of one slot of the tile ring: the leader's MMA issuer and four
// epilogue warps, the peer's producer and four epilogue warps.
constexpr int kSchedConsumers = 10;

// The tile ring of the dynamic schedule.  The leader's producer takes tiles
// from a global counter (the first one is the pair's index) and writes each
// into slot d of both CTAs' rings, -1 once the tiles are all taken; every
// other role reads its CTA's copy and reports the slot read on the leader's
// `empty`.  Waits and arrivals are at cluster scope: the two CTAs hand the
// slots to each other.
struct TileRing {
  uint64_t* full;   // this CTA's: one arrival per published tile
  uint64_t* empty;  // the leader's: kSchedConsumers arrivals per slot read
  volatile int32_t* slot;
  uint32_t d = 0, ph = 0;

  __device__ __forceinline__ void advance() {
    if (++d == uint32_t(Tc2Config::kSchedDepth)) {
      d = 0;
      ph ^= 1;
    }
  }
  // Consumer: waits for slot d (bounded), then reads it; false if the wait
  // gave up.  Call done() once every thread that needs the value has it.
  __device__ __forceinline__ bool wait(const WaitCtl& wc, int site) {
    return wait_bounded_cluster(smem_u32(&full[d]), ph, wc, site);
  }
  __device__ __forceinline__ int32_t read() const { return slot[d]; }
  __device__ __forceinline__ void done() {
    mbar_arrive_cluster(map_to_rank(smem_u32(&empty[d]), 0));
    advance();
  }
  // Leader's producer: publishes `tile` in slot d of both CTAs' rings.
  __device__ __forceinline__ bool publish(int32_t tile, const WaitCtl& wc) {
    if (!wait_bounded_cluster(smem_u32(&empty[d]), ph ^ 1, wc, kSiteProducer)) return false;
    const uint32_t sl = smem_u32(const_cast<int32_t*>(&slot[d]));
    const uint32_t fl = smem_u32(&full[d]);
    for (uint32_t r = 0; r < 2; ++r) st_dsmem_u32(map_to_rank(sl, r), uint32_t(tile));
    for (uint32_t r = 0; r < 2; ++r) mbar_arrive_cluster(map_to_rank(fl, r));
    advance();
    return true;
  }
};

// k-block groups: a stage holds G consecutive k-blocks of a unit, brought by
// one copy per operand half (a 3-D box {64, 128, G} for a K-major operand,
// boxes {64, 64 G} for an MN-major one), since the TMA unit of an SM takes
// about the same time per copy up to 32 KiB.  Group g covers k-blocks
// kb0 + gG ... of the unit; the last may be short (its boxes read zeros past
// K, or k-blocks of the next unit, which no MMA uses).
__device__ __forceinline__ int32_t tc2_groups(const Unit& u, int G) {
  return (u.kb1 - u.kb0 + G - 1) / G;
}

// TMA producer (one thread in each CTA): this CTA's A rows and B half per
// group of G k-blocks; the leader's arrive.expect_tx covers both CTAs' bytes.
// Both producers walk the same sequence of (stage, phase) slots; the return
// value is how many of them this one filled (issued loads for), which is all
// of them unless a wait gave up.  Loads still in flight after an abort are
// waited for by tc2_drain_loads once both producers have stopped.
template <int S, int G>
__device__ __forceinline__ uint32_t tc2_producer(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                             const TcArgs& args, uint8_t* sA, uint8_t* sB,
                                             uint64_t* full, uint64_t* empty, const WaitCtl& wc,
                                             uint32_t rank, int32_t cluster_id,
                                             uint64_t t_entry, TileRing& ring) {
  using Cfg = Tc2Config;
  const WorkSpec& W = args.work;
  WorkIter it;
  it.init_tc(W, cluster_id);
  Unit u;
  const int32_t tiles = W.dp_tiles;
  int32_t dyn_next = cluster_id;  // leader, dynamic schedule: the tile to publish next
  int s = 0;
  uint32_t ph = 0, filled = 0;
  bool ok = true;
  bool waited = false;
  auto prerequisites_done = [&]() {  // thread 0 of the CTA
    pdl_wait_prerequisites();
    waited = true;
    if (args.trace) {
      args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceEntry] = t_entry;
      trace_mark(args, blockIdx.x, kTraceStart);
    }
  };
  // The next unit: the static schedule's, or the next tile of the ring (the
  // leader takes it from the global counter and publishes it first).
  auto next_unit = [&]() -> bool {
    if (!args.sched) return it.next(W, u);
    int32_t t;
    if (rank == 0) {
      t = dyn_next < tiles ? dyn_next : -1;
      if (!ring.publish(t, wc)) return ok = false;
      if (!waited) prerequisites_done();  // the counter is global memory
      if (t >= 0) {
        dyn_next = atomicAdd(args.sched, 1) + W.grid;  // the tile after this one
      } else if (atomicAdd(args.sched + 1, 1) == W.grid - 1) {
        // every pair has taken its last tile: ready for the next launch
        atomicExch(args.sched, 0);
        atomicExch(args.sched + 1, 0);
      }
    } else {
      if (!ring.wait(wc, kSiteProducer)) return ok = false;
      t = ring.read();
      ring.done();
    }
    if (t < 0) return false;
    u.tile = t;
    u.kb0 = 0;
    u.kb1 = W.k_iters;
    return true;
  };
  const int32_t row_off = int32_t(rank) * kBM;      // this CTA's rows of the A tile
  const int32_t col_off = int32_t(rank) * kHalfBN;  // this CTA's columns of the B tile
  while (ok && next_unit()) {
    int32_t tm, tn;
    tile_coords(W, u.tile, tm, tn);
    const int32_t a_row = tm * kPairBM + row_off;
    const int32_t b_row = tn * kPairBN + col_off;
    // Every other wave of tiles walks k from the last block to the first: a
    // wave shares the raster group's A row panels with the wave before, and
    // starting from the k-panels that wave loaded last finds them still in
    // L2.  The wave is counted by tile (tiles are taken in order, a wave of
    // `pairs` at a time), not by this pair's units, so that a tile's k order,
    // and with it its fp32 sum, is the same whichever pair computes it.  The
    // MMA issuer consumes the stages in the order they are loaded.
    // Groups are walked last to first on such a wave (and the MMA issuer
    // takes a group's k-blocks last to first), so the k order is exactly the
    // reverse of the forward one, whatever G.
    const bool rev = ((u.tile / W.grid) & 1) != 0;
    const int32_t ng = tc2_groups(u, G);
    for (int32_t i = 0; i < ng; ++i) {
      const int32_t kb = u.kb0 + (rev ? ng - 1 - i : i) * G;  // the group's first k-block
      if (!wait_bounded(smem_u32(&empty[s]), ph ^ 1, wc, kSiteProducer)) {
        ok = false;
        break;
      }
      if (!waited) prerequisites_done();  // the first load: the operands are now final
      const uint32_t fb_local = smem_u32(&full[s]);
      if (rank == 0) mbar_arrive_expect_tx(fb_local, 2 * G * Cfg::kStageBytes);
      const uint32_t fb = map_to_rank(fb_local, 0);
      const uint32_t a_dst = smem_u32(sA + s * G * Cfg::kABytes);
      const uint32_t b_dst = smem_u32(sB + s * G * Cfg::kBBytes);
      const int32_t k0 = kb * kBK;
      // an MN-major operand: two 64-wide halves, each G k-blocks deep
      if (!args.a_mn) {
        if constexpr (G > 1) tma_load_3d_pair(a_dst, &tmA, fb, 0, a_row, kb);
        else tma_load_2d_pair(a_dst, &tmA, fb, k0, a_row);
      } else {
        tma_load_2d_pair(a_dst, &tmA, fb, a_row, k0);
        tma_load_2d_pair(a_dst + G * 8192, &tmA, fb, a_row + 64, k0);
      }
      if (!args.b_mn) {
        if constexpr (G > 1) tma_load_3d_pair(b_dst, &tmB, fb, 0, b_row, kb);
        else tma_load_2d_pair(b_dst, &tmB, fb, k0, b_row);
      } else {
        tma_load_2d_pair(b_dst, &tmB, fb, b_row, k0);
        tma_load_2d_pair(b_dst + G * 8192, &tmB, fb, b_row + 64, k0);
      }
      if (filled++ == 0) trace_mark(args, blockIdx.x, kTraceFirstLoad);
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
  }
  if (!waited) prerequisites_done();  // no load at all
  return filled;
}

// After both producers of the pair have stopped (leader's thread 0, between
// the two closing cluster barriers): waits until every load either producer
// issued has landed, so that neither CTA exits while a copy still writes its
// shared memory.  n0 and n1 count the slots the leader and the peer filled;
// a slot's `full` phase completes once the leader armed it and both halves
// landed.  They differ only after an abort, by less than one ring (a producer
// refills a stage only after the MMA consumed the previous load into it, which
// needed both halves), so for each stage only its last slot can be one-sided:
// filled by the peer alone, the leader arms it for the peer's half; filled by
// the leader alone, the peer's half that will never come is counted as done.
template <int S, int G>
__device__ __forceinline__ void tc2_drain_loads(uint64_t* full, uint32_t n0, uint32_t n1,
                                                const WaitCtl& wc) {
  const uint32_t n = n0 > n1 ? n0 : n1;
#pragma unroll 1
  for (uint32_t s = 0; s < uint32_t(S) && s < n; ++s) {
    const uint32_t q = s + ((n - 1 - s) / S) * S;  // the stage's last filled slot
    const uint32_t bar = smem_u32(&full[s]);
    if (q >= n0)
      mbar_arrive_expect_tx(bar, G * Tc2Config::kStageBytes);  // the peer's half only
    else if (q >= n1)
      mbar_complete_tx(bar, G * Tc2Config::kStageBytes);       // the peer's half never comes
    wait_drain(bar, (q / S) & 1, wc);
  }
}

// MMA issuer (one thread of the leader CTA).
template <int S, int G>
__device__ __forceinline__ void tc2_mma(const TcArgs& args, uint8_t* sA, uint8_t* sB,
                                        uint64_t* full, uint64_t* empty, uint64_t* acc_full,
                                        uint64_t* acc_empty, uint64_t* drain, const WaitCtl& wc,
                                        uint32_t tmem_base, int32_t cluster_id, TileRing& ring) {
  using Cfg = Tc2Config;
  const WorkSpec& W = args.work;
  WorkIter it;
  it.init_tc(W, cluster_id);
  Unit u;
  int s = 0, b = 0;
  uint32_t ph = 0, aph = 0;
  bool ok = true, any = false;
  auto next_unit = [&]() -> bool {
    if (!args.sched) return it.next(W, u);
    if (!ring.wait(wc, kSiteMmaFull)) return ok = false;
    const int32_t t = ring.read();
    ring.done();
    if (t < 0) return false;
    u.tile = t;
    u.kb0 = 0;
    u.kb1 = W.k_iters;
    return true;
  };
  // an MN-major operand's 64-wide halves sit G k-blocks apart; k-block j of
  // a group starts j blocks into the stage (16 KiB K-major, 8 KiB per half
  // MN-major)
  const uint32_t a_lbo = args.a_mn ? uint32_t(G) * 8192u : 16u;
  const uint32_t b_lbo = args.b_mn ? uint32_t(G) * 8192u : 16u;
  const uint32_t a_step = args.a_mn ? (2048u >> 4) : (32u >> 4);
  const uint32_t b_step = args.b_mn ? (2048u >> 4) : (32u >> 4);
  const uint32_t a_blk = args.a_mn ? 8192u : uint32_t(Cfg::kABytes);
  const uint32_t b_blk = args.b_mn ? 8192u : uint32_t(Cfg::kBBytes);
  while (ok && next_unit()) {
    // both CTAs' epilogues release each buffer once before its first use
    // (after seeding it, if asked) and once after each drain
    if (!wait_bounded(smem_u32(&acc_empty[b]), aph, wc, kSiteMmaAccum)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + uint32_t(b * kPairBN);
    const bool seeded = args.bias_init && u.kb0 == 0;  // accumulate onto the bias
    // groups arrive in the producer's order (k ascending, or descending on
    // every other wave of tiles, the k-blocks of a group then taken last to
    // first); the first MMA of the unit starts the sum
    const bool rev = ((u.tile / W.grid) & 1) != 0;
    const int32_t ng = tc2_groups(u, G);
    for (int32_t i = 0; i < ng; ++i) {
      if (!wait_bounded(smem_u32(&full[s]), ph, wc, kSiteMmaFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (!any) trace_mark(args, blockIdx.x, kTraceFirstData);
      const int32_t kb = u.kb0 + (rev ? ng - 1 - i : i) * G;
      const int nj = u.kb1 - kb < G ? int(u.kb1 - kb) : G;
      const uint32_t a0 = smem_u32(sA + s * G * Cfg::kABytes);
      const uint32_t b0 = smem_u32(sB + s * G * Cfg::kBBytes);
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        if (jj < nj) {
          const int j = rev ? nj - 1 - jj : jj;
          const uint64_t adesc = make_sdesc_sw128(a0 + uint32_t(j) * a_blk, a_lbo, 1024);
          const uint64_t bdesc = make_sdesc_sw128(b0 + uint32_t(j) * b_blk, b_lbo, 1024);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_f16_pair(d_tmem, adesc + uint64_t(kk * a_step),
                            bdesc + uint64_t(kk * b_step), args.idesc,
                            (i > 0 || jj > 0 || kk > 0 || seeded) ? 1u : 0u);
        }
      }
      any = true;
      tc_commit_pair_both(smem_u32(&empty[s]));
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
    if (!ok) break;
    // stamped before the commit, so no epilogue can see it first
    trace_mark(args, blockIdx.x, kTraceMmaDone);
    tc_commit_pair_both(smem_u32(&acc_full[b]));
    if (++b == 2) {
      b = 0;
      aph ^= 1;
    }
  }
  if (!ok && any) {  // every MMA issued so far must finish before TMEM is freed
    tc_commit_pair_self(smem_u32(drain));
    wait_drain(smem_u32(drain), 0, wc);
  }
}

// Split unit: this CTA's 128-row half of a partial tile.  The half goes to
// workspace slot 2 * split_slot(pair, tile) + rank (128 x 256 fp32; float4 j of
// a row's 32-column chunk c at float4 index (c * 8 + j) * 128 + row, so each
// warp's accesses are contiguous); the half's arrival counter is
// tickets[2 * tile + rank].  The last of the contributing pairs to arrive adds
// all halves in ascending pair (= k) order, its own from TMEM in place, and
// stores the result: the sum is the same whichever pair arrives last.
template <bool OUT_F16>
__device__ __forceinline__ void tc2_split_half(const TcArgs& args, const CUtensorMap* tmC,
                                               uint8_t* stage, uint32_t taddr, int row,
                                               int32_t mm, int32_t nbase, const Unit& u,
                                               uint32_t rank, int32_t cluster_id,
                                               volatile int* last_flag) {
  const WorkSpec& W = args.work;
  constexpr int CW = 32;
  const int32_t st = u.tile - W.dp_tiles;
  const size_t half_elems = size_t(kBM) * kPairBN;
  auto half_of = [&](int32_t pair) {
    return args.workspace + (size_t(split_slot(W, pair, st)) * 2 + rank) * half_elems;
  };
  float* mine = half_of(cluster_id);
#pragma unroll 1
  for (int c = 0; c < kPairBN / CW; ++c) {
    float v[CW];
    __syncwarp();
    tmem_load_chunk<CW>(taddr + c * CW, v);
    float4* dst = reinterpret_cast<float4*>(mine) + size_t(c) * (CW / 4) * kBM + row;
#pragma unroll
    for (int j = 0; j < CW / 4; ++j)
      __stcg(dst + j * kBM, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
  }
  __threadfence();
  epi_bar_sync();
  int32_t first, last;
  split_contributors(W, st, first, last);
  int* ticket = args.tickets + 2 * st + int32_t(rank);
  if (threadIdx.x == 64) {
    const int old = atomicAdd(ticket, 1);
    *last_flag = (old == last - first) ? 1 : 0;
  }
  epi_bar_sync();
  if (!*last_flag) return;
  __threadfence();
  constexpr int kFixBatch = 2;  // contributors whose loads are in flight together
#pragma unroll 1
  for (int c = 0; c < kPairBN / CW; ++c) {
    float own[CW], acc[CW];
    __syncwarp();
    tmem_load_chunk<CW>(taddr + c * CW, own);
#pragma unroll 1
    for (int32_t r0 = first; r0 <= last; r0 += kFixBatch) {
      float4 part[kFixBatch][CW / 4];
#pragma unroll
      for (int bb = 0; bb < kFixBatch; ++bb) {
        const int32_t r = r0 + bb;
        if (r <= last && r != cluster_id) {
          const float4* src =
              reinterpret_cast<const float4*>(half_of(r)) + size_t(c) * (CW / 4) * kBM + row;
#pragma unroll
          for (int j = 0; j < CW / 4; ++j) part[bb][j] = __ldcg(src + j * kBM);
        }
      }
#pragma unroll
      for (int bb = 0; bb < kFixBatch; ++bb) {
        const int32_t r = r0 + bb;
        if (r > last) break;
        float v[CW];
        if (r == cluster_id) {
#pragma unroll
          for (int j = 0; j < CW; ++j) v[j] = own[j];
        } else {
#pragma unroll
          for (int j = 0; j < CW / 4; ++j) {
            v[4 * j] = part[bb][j].x; v[4 * j + 1] = part[bb][j].y;
            v[4 * j + 2] = part[bb][j].z; v[4 * j + 3] = part[bb][j].w;
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
    store_out<CW, OUT_F16, false>(args, tmC, stage, row >> 5, mm, row & 31, nbase + c * CW, acc,
                                  c == 0);
  }
  if (threadIdx.x == 64) atomicExch(ticket, 0);  // ready for the next launch
}

// Epilogue (warps 2-5 of each CTA): this CTA's 128 rows of the 256 x 256 tile.
template <bool OUT_F16>
__device__ __forceinline__ void tc2_epilogue(const TcArgs& args, uint64_t* acc_full,
                                             uint64_t* acc_empty, const WaitCtl& wc,
                                             uint32_t tmem_base, uint32_t rank,
                                             int32_t cluster_id, volatile int* last_flag,
                                             uint8_t* stage, const CUtensorMap* tmC,
                                             TileRing& ring) {
  const WorkSpec& W = args.work;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int row = q * 32 + lane;
  const uint32_t leader_empty0 = map_to_rank(smem_u32(&acc_empty[0]), 0);
  const uint32_t leader_empty1 = map_to_rank(smem_u32(&acc_empty[1]), 0);
  // `ahead` runs two units ahead of `it`: the unit that will next use the
  // buffer just drained, which is seeded with the bias before its release
  WorkIter it, ahead;
  it.init_tc(W, cluster_id);
  ahead.init_tc(W, cluster_id);
  pdl_wait_prerequisites();  // the bias (seeding), C and the workspace are global
  Unit u, un;
  auto release = [&](int buf, bool have_next) {
    if (have_next && args.bias_init && un.kb0 == 0) {
      int32_t tm2, tn2;
      tile_coords(W, un.tile, tm2, tn2);
      seed_bias<kPairBN, 32, false>(
          args, tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * kPairBN),
          tm2 * kPairBM + int32_t(rank) * kBM + row, tn2 * kPairBN);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(buf == 0 ? leader_empty0 : leader_empty1);
  };
  // (the dynamic schedule runs without the bias seeding, which needs the
  // unit two ahead)
  release(0, !args.sched && ahead.next(W, un));
  release(1, !args.sched && ahead.next(W, un));
  int b = 0;
  uint32_t aph = 0;
  int units = 0;
  // The next unit: the static schedule's, or the next tile of the ring (all
  // four warps read the same slot, so they stop together).
  auto next_unit = [&]() -> bool {
    if (!args.sched) return it.next(W, u);
    if (!epi_all(ring.wait(wc, kSiteEpilogue))) return false;
    const int32_t t = ring.read();
    __syncwarp();
    if (lane == 0) ring.done();
    else ring.advance();
    if (t < 0) return false;
    u.tile = t;
    u.kb0 = 0;
    u.kb1 = W.k_iters;
    return true;
  };
  while (next_unit()) {
    int32_t tm, tn;
    tile_coords(W, u.tile, tm, tn);  // while the MMAs still run
    const bool got = wait_bounded(smem_u32(&acc_full[b]), aph, wc, kSiteEpilogue);
    if (!epi_all(got)) break;
    tc_fence_after();
    if (threadIdx.x == 64) trace_mark(args, blockIdx.x, kTraceLastAccum);
    ++units;
    const int32_t mm = tm * kPairBM + int32_t(rank) * kBM + row;
    const int32_t nbase = tn * kPairBN;
    const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(b * kPairBN);
    if (!unit_is_partial(W, u)) {
#pragma unroll 1
      for (int c = 0; c < kPairBN / 32; ++c) {
        float v[32];
        __syncwarp();
        tmem_load_chunk<32>(taddr + c * 32, v);
        store_out<32, OUT_F16, false>(args, tmC, stage, q, mm, lane, nbase + c * 32, v,
                                      c == 0);
      }
    } else {
      tc2_split_half<OUT_F16>(args, tmC, stage, taddr, row, mm, nbase, u, rank, cluster_id,
                              last_flag);
    }
    release(b, !args.sched && ahead.next(W, un));
    if (++b == 2) {
      b = 0;
      aph ^= 1;
    }
  }
  // every bulk store this warp issued has landed before the CTA moves on
  if (args.c_tma && lane == 0) bulk_wait_all();
  __syncwarp();
  if (threadIdx.x == 64) {
    trace_mark(args, blockIdx.x, kTraceEnd);
    if (args.trace) args.trace[size_t(blockIdx.x) * kTraceSlots + kTraceUnits] = uint64_t(units);
  }
}

// args.work counts cluster tiles (256 x 256) and clusters (work.grid = CTAs / 2).
// G: k-blocks per stage and TMA copy (args.kgroup; the operands' maps are
// encoded for it).
template <bool OUT_F16, int G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const TcArgs args) {
  using Cfg = Tc2Config;
  static_assert(Cfg::kStages % G == 0, "whole groups");
  constexpr int S = Cfg::kStages / G;  // ring stages of G k-blocks

  const uint64_t t_entry = args.trace ? globaltimer_ns() : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * G * Cfg::kABytes;
  uint8_t* stage = sB + S * G * Cfg::kBBytes;  // epilogue staging, 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + Cfg::kEpiStageBytes);
  uint64_t* full = bars;               // leader's counts both CTAs' bytes
  uint64_t* empty = bars + S;          // one multicast commit per phase, in both CTAs
  uint64_t* acc_full = bars + 2 * S;   // one multicast commit per unit, in both CTAs
  uint64_t* acc_empty = acc_full + 2;  // leader's: 4 epilogue warps x 2 CTAs
  uint64_t* drain = acc_empty + 2;
  uint64_t* sched_full = drain + 1;                    // tile ring (dynamic schedule)
  uint64_t* sched_empty = sched_full + Cfg::kSchedDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sched_empty + Cfg::kSchedDepth);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  uint32_t* peer_filled = tmem_slot + 3;  // leader: load slots the peer's producer filled
  int32_t* sched_slot = reinterpret_cast<int32_t*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int32_t cluster_id = int32_t(blockIdx.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 2 * (kEpiThreads / 32));
    }
    mbar_init(smem_u32(drain), 1);
    for (int d = 0; d < Cfg::kSchedDepth; ++d) {
      mbar_init(smem_u32(&sched_full[d]), 1);
      mbar_init(smem_u32(&sched_empty[d]), kSchedConsumers);
    }
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
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Global memory only after the kernels before this one have completed; the
  // producer first prepares its first load (work iterator, coordinates, free
  // stage), which with a programmatic launch overlaps the previous kernel.
  pdl_launch_dependents();
  const WaitCtl wc{args.wait_limit_ns, args.status, abort_flag};
  TileRing ring{sched_full, sched_empty, sched_slot};

  uint32_t filled = 0;  // thread 0: load slots this CTA's producer filled
  if (warp == 0) {
    if (lane == 0) {
      filled = tc2_producer<S, G>(tmA, tmB, args, sA, sB, full, empty, wc, rank, cluster_id,
                               t_entry, ring);
      if (rank != 0) st_dsmem_u32(map_to_rank(smem_u32(peer_filled), 0), filled);
    } else {
      pdl_wait_prerequisites();
    }
  } else if (warp == 1) {
    pdl_wait_prerequisites();
    if (lane == 0 && rank == 0)
      tc2_mma<S, G>(args, sA, sB, full, empty, acc_full, acc_empty, drain, wc, tmem_base,
                 cluster_id, ring);
  } else {
    tc2_epilogue<OUT_F16>(args, acc_full, acc_empty, wc, tmem_base, rank, cluster_id,
                          last_flag, stage, &tmC, ring);
  }

  __syncthreads();
  tc_fence_before();
  // Both CTAs' roles are done: no MMA or remote arrive is still aimed at
  // either CTA, no load will be issued, and the peer's fill count is in.
  cluster_sync_all();
  if (rank == 0 && threadIdx.x == 0) tc2_drain_loads<S, G>(full, filled, *peer_filled, wc);
  cluster_sync_all();  // no copy still lands in either CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
  if (args.trace) {  // the exit stamp after the TMEM is freed, by the end's thread
    __syncthreads();
    if (threadIdx.x == kStampThread) trace_mark(args, blockIdx.x, kTraceExit);
  }
}

}  // namespace dg
