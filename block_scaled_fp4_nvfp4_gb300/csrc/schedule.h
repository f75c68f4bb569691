// Work decomposition shared by the host planner, the device kernel and the
// host-side schedule check: a data-parallel part (whole output tiles, dealt
// round-robin to the persistent CTAs) followed by a stream-K part (the
// remaining tiles' k-tile iterations laid end to end and cut into one equal,
// contiguous range per CTA).
//
// Stream-K: iteration x of the stream-K space belongs to tile x / KT (per
// group), and unit c owns iterations [floor(c*T/G), floor((c+1)*T/G)).  A unit
// is one CTA, or one cluster of two CTAs running tiles 2q and 2q+1 (the same
// B columns) over the same k-range.  A tile covered by several units gets one
// partial result per covering unit ("segment"), numbered in k order; the last
// segment to finish sums them in that order.  In cluster plans (sk_fixup)
// every unit covers at least one whole tile's k-tiles, so a tile has at most
// two segments: segment 1 (the tile's last k-tiles) is the first item of its
// unit and publishes its partial; segment 0 is the last item of the previous
// unit, which adds that partial and stores the tile.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define NVFP4_HD __host__ __device__ __forceinline__
#else
#define NVFP4_HD inline
#endif

namespace nvfp4 {

constexpr int kSchedMaxGroups = 8;

struct Schedule {
  int num_groups;
  int tiles_m[kSchedMaxGroups], tiles_n[kSchedMaxGroups], L[kSchedMaxGroups];
  int ktiles[kSchedMaxGroups];
  int tile_start[kSchedMaxGroups + 1];     // prefix over groups of output tiles
  int sk_tile_first[kSchedMaxGroups];      // first stream-K tile (global index) of group g
  long long sk_iter_start[kSchedMaxGroups + 1];  // prefix over groups of stream-K iterations
  int total_tiles;
  int dp_tiles;     // tiles [0, dp_tiles) run whole, tile c + i*grid on CTA c
  long long sk_iters;  // T: total stream-K iterations (0 = no stream-K part)
  int sk_max_segs;  // workspace slots reserved per stream-K tile
  int cluster;      // CTAs per cluster (1, or 2: the pair runs tiles 2q, 2q+1, sharing B)
  int sk_fixup;     // 1: stream-K tiles of a cluster plan, at most two segments (see above)
};

struct Work {
  int g, l, tm, tn;  // group, batch, m-tile, n-tile
  int kt0, kt1;      // k-tile range [kt0, kt1) of this piece
  int tile;          // global tile index
  int seg, nseg;     // segment index in k order and number of segments of the tile
};

struct WorkCursor {
  int dp_next;  // next data-parallel tile group (one tile per cluster rank)
  int rank;     // rank inside the cluster
  long long x, hi;
};

// CTA owning stream-K iteration y: the largest c with floor(c*T/G) <= y.
NVFP4_HD int sk_owner(long long y, long long T, int G) {
  return static_cast<int>(((y + 1) * G - 1) / T);
}

// `cta` / `grid` count clusters; `rank` is the CTA's rank inside its cluster.
// With clusters of 2 every group has an even number of m-tiles and the
// stream-K part starts at an even tile of each group, so tiles 2q and 2q+1
// (m fastest) share g, l, tn.
NVFP4_HD void work_begin(const Schedule& s, int cta, int grid, WorkCursor& cur, int rank = 0) {
  cur.dp_next = cta;
  cur.rank = rank;
  if (s.sk_iters > 0) {
    cur.x = s.sk_iters * cta / grid;
    cur.hi = s.sk_iters * (cta + 1) / grid;
  } else {
    cur.x = cur.hi = 0;
  }
}

NVFP4_HD void tile_coords(const Schedule& s, int t, Work& w) {
  int g = 0;
  while (g + 1 < s.num_groups && t >= s.tile_start[g + 1]) ++g;
  const int r = t - s.tile_start[g];
  w.g = g;
  w.tile = t;
  w.tm = r % s.tiles_m[g];  // m fastest: concurrent tiles share the same B columns
  const int rest = r / s.tiles_m[g];
  w.tn = rest % s.tiles_n[g];
  w.l = rest / s.tiles_n[g];
}

// Next piece of work of CTA `cta` (of `grid`); false when done.
NVFP4_HD bool work_next(const Schedule& s, int cta, int grid, WorkCursor& cur, Work& w) {
  if (cur.dp_next * s.cluster < s.dp_tiles) {
    tile_coords(s, cur.dp_next * s.cluster + cur.rank, w);
    w.kt0 = 0;
    w.kt1 = s.ktiles[w.g];
    w.seg = 0;
    w.nseg = 1;
    cur.dp_next += grid;
    return true;
  }
  if (cur.x >= cur.hi) return false;
  int g = 0;
  while (g + 1 < s.num_groups && cur.x >= s.sk_iter_start[g + 1]) ++g;
  const long long KT = s.ktiles[g];
  const long long local = cur.x - s.sk_iter_start[g];
  const long long k0 = local % KT;
  const long long t_begin = cur.x - k0;  // first iteration of this tile
  const long long t_end = t_begin + KT;
  const long long end = cur.hi < t_end ? cur.hi : t_end;
  tile_coords(s, s.sk_tile_first[g] + static_cast<int>(local / KT) * s.cluster + cur.rank, w);
  w.kt0 = static_cast<int>(k0);
  w.kt1 = static_cast<int>(end - t_begin);
  const int first = sk_owner(t_begin, s.sk_iters, grid);
  const int last = sk_owner(t_end - 1, s.sk_iters, grid);
  w.seg = cta - first;
  w.nseg = last - first + 1;
  cur.x = end;
  return true;
}

// Workspace slot of a stream-K segment (fp32 partial tile) and its counter.
NVFP4_HD long long sk_slot(const Schedule& s, const Work& w, int seg) {
  return static_cast<long long>(w.tile - s.dp_tiles) * s.sk_max_segs + seg;
}
NVFP4_HD int sk_counter(const Schedule& s, const Work& w) { return w.tile - s.dp_tiles; }

}  // namespace nvfp4
