// schedule.cuh: the work list of one persistent unit (a CTA, or a CTA pair).
//
// Stream-K (SK) part: the first sk_tiles tiles (in raster order) are cut
// along K. Their k-blocks, laid end to end (tile-major), are split into
// `units` equal contiguous ranges, one per unit, so that every unit does the
// same number of k-blocks and no unit idles while others finish a partial
// wave. "Two Waves, One Stage Apart" (section "MI300X") sizes a problem so
// that its tile count fills the machine; this removes the need for that.
//
// Data-parallel (DP) part: the remaining tiles go round-robin to the units,
// whole tiles with the whole K range, as in a plain persistent GEMM. The
// planner makes their count a multiple of the unit count.
//
// A unit's range cuts at most two tiles, at its two ends:
//   - its first segment may end a tile that an earlier unit started: this
//     unit is that tile's OWNER and finishes it (adds the other units'
//     partial sums, casts and stores C);
//   - its last segment may start a tile (or, when the range lies inside one
//     tile, cover its middle): this unit is a WRITER and leaves an FP32
//     partial sum in the workspace, with a flag set to the launch id.
// Order of a unit's jobs: the writer segment first (so its partial is ready
// early), then its whole stream-K tiles, then the owner segment, then the DP
// tiles. The owner segment ends at the same point of every unit's timeline
// (every unit has the same stream-K share), after all writer segments, so the
// partials it reads are ready and its fix-up epilogue overlaps the first DP
// tile's main loop; and the DP waves that follow run in lock step, which
// keeps the grouped raster's operand panels shared in L2. Each unit writes at
// most one partial.
//
// The same code runs in the kernel and on the host (the C ABI exports the
// job list so that tests can check it without a GPU).
#pragma once

#include <cstdint>

namespace dtg {

enum : int32_t { JOB_FULL = 0, JOB_WRITER = 1, JOB_OWNER = 2 };

struct Job {
    int32_t tile;
    int32_t kb0, kb1;   // k-blocks [kb0, kb1) of the tile
    int32_t kind;       // JOB_FULL, JOB_WRITER or JOB_OWNER
};

struct UnitSchedule {
    int32_t unit, units, kb;        // this unit, unit count, k-blocks per tile
    int32_t sk_tiles, dp_tiles;     // tiles [0, sk_tiles) SK, [sk_tiles, sk_tiles + dp_tiles) DP
    int32_t n_writer, n_dp, n_full, n_owner;
    int32_t full_first;             // first SK tile this unit does whole
    Job writer, owner;

    // First k-block (linear over the SK tiles) of unit u's range.
    __host__ __device__ static int64_t range_start(int32_t u, int32_t units, int32_t sk_tiles, int32_t kb)
    {
        return static_cast<int64_t>(u) * sk_tiles * kb / units;
    }

    __host__ __device__ UnitSchedule(int32_t u, int32_t units_, int32_t num_tiles, int32_t kb_,
                                     int32_t sk_tiles_)
        : unit(u), units(units_), kb(kb_), sk_tiles(sk_tiles_), dp_tiles(num_tiles - sk_tiles_),
          n_writer(0), n_dp(0), n_full(0), n_owner(0), full_first(0), writer{0, 0, 0, JOB_WRITER},
          owner{0, 0, 0, JOB_OWNER}
    {
        n_dp = u < dp_tiles ? (dp_tiles - 1 - u) / units + 1 : 0;
        if (sk_tiles <= 0)
            return;
        const int64_t g0 = range_start(u, units, sk_tiles, kb);
        const int64_t g1 = range_start(u + 1, units, sk_tiles, kb);
        if (g0 >= g1)
            return;   // no stream-K work for this unit
        const int32_t ta = static_cast<int32_t>(g0 / kb), ka = static_cast<int32_t>(g0 % kb);
        const int32_t tb = static_cast<int32_t>((g1 - 1) / kb), kbe = static_cast<int32_t>((g1 - 1) % kb) + 1;
        int32_t first_full = ta, last_full = tb;   // inclusive range of whole SK tiles
        if (ta == tb) {
            if (ka == 0 && kbe == kb) {
                // one whole tile
            } else if (kbe == kb) {
                n_owner = 1;
                owner = {ta, ka, kb, JOB_OWNER};
                first_full = ta + 1;
            } else {
                n_writer = 1;
                writer = {ta, ka, kbe, JOB_WRITER};
                first_full = ta + 1;
            }
        } else {
            if (ka != 0) {
                n_owner = 1;
                owner = {ta, ka, kb, JOB_OWNER};
                first_full = ta + 1;
            }
            if (kbe != kb) {
                n_writer = 1;
                writer = {tb, 0, kbe, JOB_WRITER};
                last_full = tb - 1;
            }
        }
        n_full = last_full >= first_full ? last_full - first_full + 1 : 0;
        full_first = first_full;
    }

    __host__ __device__ int32_t num_jobs() const { return n_writer + n_dp + n_full + n_owner; }

    __host__ __device__ Job job(int32_t i) const
    {
        if (i < n_writer)
            return writer;
        i -= n_writer;
        if (i < n_full)
            return {full_first + i, 0, kb, JOB_FULL};
        i -= n_full;
        if (i < n_owner)
            return owner;
        i -= n_owner;
        return {sk_tiles + unit + i * units, 0, kb, JOB_FULL};
    }

    // For an owner job: the units whose writer segments hold the rest of the
    // tile are unit - 1, unit - 2, ... down to (and including) first_writer.
    // Units in that span whose stream-K range is empty wrote nothing and are
    // skipped with has_range().
    __host__ __device__ int32_t first_writer() const
    {
        const int64_t tile_start = static_cast<int64_t>(owner.tile) * kb;
        int32_t v = unit - 1;
        while (v > 0 && range_start(v, units, sk_tiles, kb) > tile_start)
            --v;
        return v;
    }

    __host__ __device__ bool has_range(int32_t v) const
    {
        return range_start(v, units, sk_tiles, kb) < range_start(v + 1, units, sk_tiles, kb);
    }
};

} // namespace dtg
