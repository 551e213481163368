// Persistent tile schedule with a Stream-K tail (host + device).
//
// The output is cut into tiles_m x tiles_n tiles; each tile needs k_steps steps of
// BK = 64 along K.  A persistent grid of `grid` CTAs (one per SM) walks:
//
//   1. Stream-K tiles [0, sk_tiles): their flattened
//      (tile, k-step) space of sk_units = sk_tiles * k_steps units is cut into
//      `grid` contiguous ranges, range c = [c*U/grid, (c+1)*U/grid);
//   2. data-parallel tiles [sk_tiles, sk_tiles + dp_tiles): CTA c takes tiles
//      sk_tiles + c, sk_tiles + c + grid, ...
//      (whole tiles, no partial sums).
//
// The Stream-K pieces come first so that the partial-sum exchange of a split
// tile overlaps the main loop of the CTA's later whole tiles instead of being
// exposed at the end of the launch.  Both phases walk the grouped raster in
// order, so the tiles in flight at any time are neighbours.
//
// This is the schedule of spark-kernels, "stream-k proper": a resident grid, the
// last waves' (tile, k-step) space cut into equal contiguous ranges so that no CTA
// idles at the end, and (UwULLM kernel-dev, budget 4) wave efficiency
// (ctas/SMs)/ceil(ctas/SMs) as the quantity it repairs.
//
// A tile covered by more than one range is finished by whichever of its pieces
// arrives last (an arrival counter per tile); that piece sums every piece's fp32
// partial in increasing k order, so the result does not depend on timing.  The
// counter is reset by the finishing piece, so nothing is cleared between launches.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define SG_HD __host__ __device__ __forceinline__
#else
#define SG_HD inline
#endif

namespace sg {

struct Schedule {
  int32_t tiles_m;   // tiles along the output rows (MMA M side)
  int32_t tiles_n;   // tiles along the output columns (MMA N side)
  int32_t k_steps;   // ceil(K / 64)
  int32_t grid;      // persistent CTAs launched
  int32_t dp_tiles;  // whole tiles handed out round-robin
  int32_t sk_tiles;  // tiles split by Stream-K
  int64_t sk_units;  // sk_tiles * k_steps (< 2^31)
  int32_t group_m;   // raster group height in tiles (L2 locality)
  int32_t sk_q;      // Stream-K units per CTA: sk_units / grid ...
  int32_t sk_r;      // ... and the first sk_r CTAs take one more (sk_units % grid)
  int32_t split;     // > 0: split mode (below); 0: waves + Stream-K
};

// Split mode (split = S > 0): every tile is cut into exactly S pieces of k-steps
// [KS*p/S, KS*(p+1)/S), and CTA c runs piece c % S of tile c / S as its only
// item.  Used where all CTAs are resident at once (memory-bound skinny GEMMs,
// two CTAs per SM): the memory system then shares bandwidth among them, so no
// CTA idles, and each tile's pieces end together.

struct WorkItem {
  int32_t tile;      // linear tile index in raster order
  int32_t k0, k1;    // k-step range [k0, k1) of this piece
  int32_t piece;     // index of this piece among the tile's pieces (k order)
  int32_t npieces;   // 1 = whole tile
  int32_t slot;      // partial-sum slot of this piece (2*cta + which)
  int32_t sk_index;  // tile index inside the Stream-K region (arrival counter)
};

// Stream-K ranges: CTA c takes units [begin(c), begin(c + 1)), the first sk_r
// CTAs sk_q + 1 units each and the rest sk_q.  32-bit arithmetic throughout: the
// scheduler runs in every role of every CTA before its first copy is issued.
SG_HD int32_t sk_range_begin(const Schedule& s, int32_t c) {
  return c * s.sk_q + (c < s.sk_r ? c : s.sk_r);
}

// The CTA whose range holds Stream-K unit u.
SG_HD int32_t sk_owner(const Schedule& s, int32_t u) {
  const int32_t big = s.sk_r * (s.sk_q + 1);  // units held by the sk_r larger ranges
  return u < big ? u / (s.sk_q + 1) : s.sk_r + (u - big) / s.sk_q;
}

// Slot of CTA c's piece of SK tile t: 0 if the piece is the first item of c's
// range (the range starts inside tile t), else 1.
SG_HD int32_t sk_slot(const Schedule& s, int32_t c, int32_t t) {
  const int32_t first_tile = sk_range_begin(s, c) / s.k_steps;
  return 2 * c + (first_tile == t ? 0 : 1);
}

SG_HD int32_t dp_count(const Schedule& s, int32_t c) {
  return c < s.dp_tiles ? (s.dp_tiles - 1 - c) / s.grid + 1 : 0;
}

// Number of Stream-K pieces of CTA c (split mode: its one piece).
SG_HD int32_t sk_count(const Schedule& s, int32_t c) {
  if (s.split > 0) return c < s.tiles_m * s.tiles_n * s.split ? 1 : 0;
  if (s.sk_tiles <= 0) return 0;
  const int32_t u0 = sk_range_begin(s, c), u1 = sk_range_begin(s, c + 1);
  return u1 > u0 ? (u1 - 1) / s.k_steps - u0 / s.k_steps + 1 : 0;
}

// The k-step ranges [k0, k1) of CTA c's work items in get_item's order, for a
// role that needs nothing else (the MMA issuer): the divisions are done once per
// CTA, so an item boundary costs none.
struct KRanges {
  int32_t nsk = 0, u0 = 0, u1 = 0, t0 = 0, k_steps = 0, split_k0 = 0, split_k1 = 0;
  bool split = false;
  SG_HD KRanges(const Schedule& s, int32_t c) : k_steps(s.k_steps) {
    if (s.split > 0) {
      split = true;
      const int32_t pc = c % s.split;
      split_k0 = (s.k_steps * pc) / s.split;
      split_k1 = (s.k_steps * (pc + 1)) / s.split;
      return;
    }
    nsk = sk_count(s, c);
    if (nsk > 0) {
      u0 = sk_range_begin(s, c);
      u1 = sk_range_begin(s, c + 1);
      t0 = u0 / s.k_steps;
    }
  }
  SG_HD void range(int32_t i, int32_t& k0, int32_t& k1) const {
    if (split) {
      k0 = split_k0;
      k1 = split_k1;
    } else if (i >= nsk) {
      k0 = 0;
      k1 = k_steps;
    } else {
      const int32_t tb = (t0 + i) * k_steps, te = tb + k_steps;
      k0 = (u0 > tb ? u0 : tb) - tb;
      k1 = (u1 < te ? u1 : te) - tb;
    }
  }
};

// Number of work items of CTA c.
SG_HD int32_t item_count(const Schedule& s, int32_t c) {
  if (s.split > 0) return c < s.tiles_m * s.tiles_n * s.split ? 1 : 0;
  return sk_count(s, c) + dp_count(s, c);
}

// The i-th work item of CTA c (0 <= i < item_count(s, c)): its Stream-K pieces
// first, then its whole tiles.
SG_HD WorkItem get_item(const Schedule& s, int32_t c, int32_t i) {
  WorkItem w;
  if (s.split > 0) {
    const int32_t t = c / s.split, pc = c - t * s.split;
    w.tile = t;
    w.k0 = (s.k_steps * pc) / s.split;
    w.k1 = (s.k_steps * (pc + 1)) / s.split;
    w.piece = pc;
    w.npieces = s.split;
    w.slot = s.split > 1 ? c : -1;
    w.sk_index = t;
    return w;
  }
  const int32_t nsk = sk_count(s, c);
  if (i >= nsk) {
    w.tile = s.sk_tiles + c + (i - nsk) * s.grid;
    w.k0 = 0;
    w.k1 = s.k_steps;
    w.piece = 0;
    w.npieces = 1;
    w.slot = -1;
    w.sk_index = -1;
    return w;
  }
  const int32_t u0 = sk_range_begin(s, c), u1 = sk_range_begin(s, c + 1);
  const int32_t t = u0 / s.k_steps + i;
  const int32_t tb = t * s.k_steps, te = tb + s.k_steps;
  w.tile = t;
  w.k0 = (u0 > tb ? u0 : tb) - tb;
  w.k1 = (u1 < te ? u1 : te) - tb;
  const int32_t first = sk_owner(s, tb), last = sk_owner(s, te - 1);
  w.piece = c - first;
  w.npieces = last - first + 1;
  w.slot = w.npieces > 1 ? sk_slot(s, c, t) : -1;
  w.sk_index = t;
  return w;
}

// Slot of piece j of Stream-K tile t (t counted inside the Stream-K region).
SG_HD int32_t piece_slot(const Schedule& s, int32_t t, int32_t j) {
  if (s.split > 0) return t * s.split + j;
  const int32_t c = sk_owner(s, t * s.k_steps) + j;
  return sk_slot(s, c, t);
}

// Split-mode schedule: tiles_m x tiles_n tiles, each cut into `split` pieces.
inline Schedule make_split_schedule(int32_t tiles_m, int32_t tiles_n, int32_t k_steps, int32_t split) {
  Schedule s{};
  s.tiles_m = tiles_m;
  s.tiles_n = tiles_n;
  s.k_steps = k_steps;
  s.group_m = 1;
  s.split = split < 1 ? 1 : (split > k_steps ? k_steps : split);
  s.grid = tiles_m * tiles_n * s.split;
  s.dp_tiles = 0;
  s.sk_tiles = tiles_m * tiles_n;
  s.sk_units = static_cast<int64_t>(s.sk_tiles) * k_steps;
  return s;
}

// Grouped raster order: groups of group_m tile-rows, column-major inside a group,
// so the tiles in flight share A rows and B columns in L2.
SG_HD void tile_coords(const Schedule& s, int32_t tile, int32_t& tm, int32_t& tn) {
  const int32_t per_group = s.group_m * s.tiles_n;
  const int32_t g = tile / per_group;
  const int32_t first_m = g * s.group_m;
  const int32_t rows = (s.tiles_m - first_m) < s.group_m ? (s.tiles_m - first_m) : s.group_m;
  const int32_t r = tile - g * per_group;
  tm = first_m + r % rows;
  tn = r / rows;
}

// Wave efficiency (UwULLM kernel-dev, budget 4): (ctas / slots) / ceil(ctas / slots).
SG_HD double wave_efficiency(int64_t ctas, int64_t slots) {
  if (ctas <= 0 || slots <= 0) return 0.0;
  const int64_t waves = (ctas + slots - 1) / slots;
  return static_cast<double>(ctas) / static_cast<double>(slots) / static_cast<double>(waves);
}

// Smallest Stream-K share (k-steps per CTA) for which the remainder tiles alone
// are split; below it the last full wave joins the Stream-K region.
constexpr int64_t kMinSkStepsPerCta = 16;

// What one partial-sum exchange costs, in k-steps of main-loop time (a piece's
// fp32 partial of 128 KB per CTA written, fenced, counted and read back).
// Stream-K is used only when the wave-quantisation time it saves is larger.
constexpr int64_t kSkFixupCostSteps = 24;

// Builds the schedule.
//
// tiles >= CTAs: whole-tile waves; when the tile count is not a multiple of the
//   CTA count, the remainder tiles (plus the last full wave if the remainder is
//   thin) are cut by Stream-K.
// tiles < CTAs, memory-bound (fill_grid): every tile is split along K so that
//   all `num_ctas` CTAs stream an equal share (at least min_units_per_cta k-steps
//   each); the weight stream needs every SM's load bandwidth.
// tiles < CTAs, compute-bound (!fill_grid): Stream-K only pays when a tile can be
//   split at least two ways (s = floor(CTAs / tiles) >= 2): one tile per CTA
//   loses (1 - tiles/CTAs) of a tile's time at most, less than a fixup costs.
inline Schedule make_schedule(int32_t tiles_m, int32_t tiles_n, int32_t k_steps, int32_t num_ctas,
                              int32_t min_units_per_cta, int32_t group_m, bool fill_grid) {
  Schedule s{};
  s.tiles_m = tiles_m;
  s.tiles_n = tiles_n;
  s.k_steps = k_steps;
  s.group_m = group_m < 1 ? 1 : group_m;
  const int64_t T = static_cast<int64_t>(tiles_m) * tiles_n;
  const int64_t G = num_ctas < 1 ? 1 : num_ctas;
  const int64_t per = min_units_per_cta < 1 ? 1 : min_units_per_cta;
  if (T >= G) {
    const int64_t rem = T % G;
    s.grid = static_cast<int32_t>(G);
    // whole-tile waves lose (G - rem) / G of a wave to quantisation
    const bool sk_pays = fill_grid || (G - rem) * k_steps > kSkFixupCostSteps * G;
    if (rem == 0 || k_steps < 2 || !sk_pays) {
      s.dp_tiles = static_cast<int32_t>(T);
      s.sk_tiles = 0;
    } else if (fill_grid || rem * k_steps >= kMinSkStepsPerCta * G) {
      // (memory-bound: small pieces cost no tensor efficiency, and each CTA then
      // ends on a whole tile, so no partial exchange sits at the end)
      // Stream-K over the remainder only: every CTA still gets a piece of at
      // least kMinSkStepsPerCta k-steps, and fewer tiles exchange partial sums.
      s.sk_tiles = static_cast<int32_t>(rem);
      s.dp_tiles = static_cast<int32_t>(T - rem);
    } else {
      // A thin remainder: Stream-K over the last full wave plus the remainder
      // (1 < waves < 2), so no piece is tiny.
      s.sk_tiles = static_cast<int32_t>(rem + G);
      s.dp_tiles = static_cast<int32_t>(T - s.sk_tiles);
    }
  } else {
    const int64_t units = T * k_steps;
    int64_t g;
    if (fill_grid) {
      g = units / per;
      if (g > G) g = G;
    } else {
      // s-way splits save k_steps * (1 - 1/s) per tile, which must beat a fixup
      int64_t split = G / T;  // >= 1
      if (split >= 2 && k_steps - k_steps / split <= kSkFixupCostSteps) split = 1;
      g = split >= 2 ? T * split : T;
      if (g > units / per) g = units / per;
    }
    if (g < T) g = T;
    s.grid = static_cast<int32_t>(g);
    if (g == T) {  // one CTA per tile: plain data-parallel
      s.dp_tiles = static_cast<int32_t>(T);
      s.sk_tiles = 0;
    } else {
      s.dp_tiles = 0;
      s.sk_tiles = static_cast<int32_t>(T);
    }
  }
  s.sk_units = static_cast<int64_t>(s.sk_tiles) * k_steps;
  if (s.sk_units >= (int64_t{1} << 31) - int64_t{2} * s.grid) {  // keep the 32-bit unit math exact
    s.dp_tiles += s.sk_tiles;
    s.sk_tiles = 0;
    s.sk_units = 0;
  }
  s.sk_q = s.sk_units > 0 ? static_cast<int32_t>(s.sk_units / s.grid) : 0;
  s.sk_r = s.sk_units > 0 ? static_cast<int32_t>(s.sk_units % s.grid) : 0;
  return s;
}

}  // namespace sg
