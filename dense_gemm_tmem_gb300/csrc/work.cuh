// work.cuh: how output tiles and their k-blocks are handed to CTAs.
//
// A launch has `grid` persistent CTAs.  Tiles [0, dp_tiles) are computed whole,
// tile c + u*grid by CTA c (data-parallel waves).  The k-blocks of the remaining
// sk_tiles tiles are laid end to end, W = sk_tiles * k_iters iterations, and cut
// into `grid` equal contiguous ranges: CTA r gets [floor(r*W/grid),
// floor((r+1)*W/grid)).  This is the Stream-K work-centric decomposition the
// leiblog.wang Stream-K post describes (split the k axis evenly over the SMs so
// small shapes leave no SM idle).  A range is cut into units at tile
// boundaries; a unit that covers only part of its tile's k-blocks is a partial
// whose fp32 sum goes to the workspace, and the last CTA to finish a tile adds
// the partials in ascending k order (deterministic), then runs the epilogue.
//
// Everything here is __host__ __device__ so the host query functions report
// exactly what the kernel does.
#pragma once

#include <cstdint>

namespace dg {

struct WorkSpec {
  int32_t tiles_m;   // output tiles along the MMA M side
  int32_t tiles_n;   // output tiles along the MMA N side
  int32_t k_iters;   // k-blocks per tile
  int32_t dp_tiles;  // whole tiles, handed out first
  int32_t sk_tiles;  // split tiles, numbered dp_tiles .. dp_tiles + sk_tiles - 1
  int32_t grid;      // CTAs
  int32_t group_m;   // raster group height (tile rows)
  int32_t csplit;    // > 1: cluster split, tile = cta / csplit, k range by rank
};

struct Unit {
  int32_t tile;  // linear tile index
  int32_t kb0;   // first k-block
  int32_t kb1;   // one past the last k-block
};

__host__ __device__ __forceinline__ int64_t split_total(const WorkSpec& w) {
  return int64_t(w.sk_tiles) * w.k_iters;
}

// First iteration of CTA r's share of the split region.
__host__ __device__ __forceinline__ int64_t split_start(const WorkSpec& w, int64_t r) {
  return split_total(w) * r / w.grid;
}

// The CTA whose share holds split iteration x (0 <= x < W): the r with
// start(r) <= x < start(r+1), i.e. r = ceil((x+1)*G/W) - 1.
__host__ __device__ __forceinline__ int32_t split_owner(const WorkSpec& w, int64_t x) {
  const int64_t W = split_total(w);
  return int32_t(((x + 1) * w.grid - 1) / W);
}

struct WorkIter {
  int32_t next_dp;
  int64_t x, end;

  __host__ __device__ __forceinline__ void init(const WorkSpec& w, int32_t cta) {
    next_dp = cta;
    if (w.csplit > 1) {
      // Cluster split (a k-split whose partials are added on chip by the CTAs
      // of one cluster): CTA `cta` owns tile cta / s and the rank-th of s equal
      // contiguous k-block ranges, rank = cta % s.  Encoded as a one-iteration
      // "split region" walk: x = first k-block, end = one past the last.
      const int32_t s = w.csplit;
      const int32_t rank = cta % s;
      next_dp = w.dp_tiles;  // no whole-tile phase
      x = int64_t(cta / s) * w.k_iters + int64_t(rank) * w.k_iters / s;
      end = int64_t(cta / s) * w.k_iters + int64_t(rank + 1) * w.k_iters / s;
      return;
    }
    if (w.sk_tiles > 0) {
      x = split_start(w, cta);
      end = split_start(w, int64_t(cta) + 1);
    } else {
      x = end = 0;
    }
  }

  // The same as init for the tensor-core kernels, whose cluster splits have
  // s = 2, 4 or 8: shifts instead of divisions (a 64-bit division is a long
  // subroutine on the device, paid before the first load).
  __host__ __device__ __forceinline__ void init_tc(const WorkSpec& w, int32_t cta) {
    if (w.csplit == 2 || w.csplit == 4 || w.csplit == 8) {
      const int sh = w.csplit == 8 ? 3 : w.csplit == 4 ? 2 : 1;
      const int32_t rank = cta & (w.csplit - 1);
      const int64_t base = int64_t(cta >> sh) * w.k_iters;
      next_dp = w.dp_tiles;  // no whole-tile phase
      x = base + ((int64_t(rank) * w.k_iters) >> sh);
      end = base + ((int64_t(rank + 1) * w.k_iters) >> sh);
      return;
    }
    init(w, cta);
  }

  __host__ __device__ __forceinline__ bool next(const WorkSpec& w, Unit& u) {
    if (next_dp < w.dp_tiles) {
      u.tile = next_dp;
      u.kb0 = 0;
      u.kb1 = w.k_iters;
      next_dp += w.grid;
      return true;
    }
    if (x < end) {
      const int32_t t = int32_t(x / w.k_iters);
      const int32_t k0 = int32_t(x - int64_t(t) * w.k_iters);
      const int64_t left = end - x;
      const int32_t k1 = (left < int64_t(w.k_iters - k0)) ? int32_t(k0 + left) : w.k_iters;
      u.tile = w.dp_tiles + t;
      u.kb0 = k0;
      u.kb1 = k1;
      x += k1 - k0;
      return true;
    }
    return false;
  }
};

__host__ __device__ __forceinline__ bool unit_is_partial(const WorkSpec& w, const Unit& u) {
  return u.kb0 > 0 || u.kb1 < w.k_iters;
}

// Tile -> (tm, tn) in groups of group_m tile rows, columns sweeping inside a
// group, so CTAs running at the same time share A rows and B columns in L2.
__host__ __device__ __forceinline__ void tile_coords(const WorkSpec& w, int32_t tile,
                                                     int32_t& tm, int32_t& tn) {
  const int32_t per_group = w.group_m * w.tiles_n;
  const int32_t g = tile / per_group;
  const int32_t first_m = g * w.group_m;
  const int32_t rows_left = w.tiles_m - first_m;
  const int32_t gm = rows_left < w.group_m ? rows_left : w.group_m;
  const int32_t r = tile - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

// Contributors of split tile s (0-based inside the split region): CTAs
// first..last, in ascending k order.
__host__ __device__ __forceinline__ void split_contributors(const WorkSpec& w, int32_t s,
                                                            int32_t& first, int32_t& last) {
  first = split_owner(w, int64_t(s) * w.k_iters);
  last = split_owner(w, int64_t(s + 1) * w.k_iters - 1);
}

// Workspace slot holding CTA r's partial of split tile s: each CTA has two,
// one for the tile its range starts in, one for the tile it ends in.
__host__ __device__ __forceinline__ int32_t split_slot(const WorkSpec& w, int32_t r,
                                                       int32_t s) {
  const int32_t start_tile = int32_t(split_start(w, r) / w.k_iters);
  return 2 * r + (start_tile == s ? 0 : 1);
}

}  // namespace dg
