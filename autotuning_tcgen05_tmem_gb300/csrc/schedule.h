// Persistent tile schedule: work unit -> (tile row, tile column, K slice).
//
// "Compilers and Kernel Languages" lists the order in which tiles are scheduled
// among the choices a real kernel adds to the tile shape; "Tiling the hierarchy"
// (permutation interacts with tiling) explains why the order changes which
// panels stay resident.  Units are tile-major with the K slice fastest, so the
// slices of one tile run side by side and meet in L2.  raster 0 walks a band of
// `group` tile-rows column by column (the band's A panels stay hot while B
// panels stream); raster 1 is the transpose.
//
// Shared by the kernel and by the host (gemm_schedule_unit) so that the host
// can report exactly the order the device runs.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__ __forceinline__
#else
#define GEMM_HD inline
#endif

struct SchedUnit {
    int32_t tile_m, tile_n, split, kb_begin, kb_end, tile;
};

GEMM_HD SchedUnit schedule_unit(int64_t unit, int32_t tiles_m, int32_t tiles_n, int32_t split_k,
                                int32_t raster, int32_t group, int32_t num_kb)
{
    SchedUnit r;
    // Units number fewer than 2^31 (tiles x split_k is an int32 of the
    // launch), so 32-bit arithmetic suffices.
    const int32_t u = (int32_t)unit;
    const int32_t tile = u / split_k;
    const int32_t s = u - tile * split_k;
    if (raster == 0) {
        const int32_t per_band = group * tiles_n;
        const int32_t band = tile / per_band;
        const int32_t within = tile - band * per_band;
        const int32_t first = band * group;
        const int32_t height = (tiles_m - first) < group ? (tiles_m - first) : group;
        r.tile_m = first + within % height;
        r.tile_n = within / height;
    } else {
        const int32_t per_band = group * tiles_m;
        const int32_t band = tile / per_band;
        const int32_t within = tile - band * per_band;
        const int32_t first = band * group;
        const int32_t width = (tiles_n - first) < group ? (tiles_n - first) : group;
        r.tile_n = first + within % width;
        r.tile_m = within / width;
    }
    r.split = s;
    // s <= 16 and num_kb <= 2^31 / 32 (K < 2^31, bk >= 32), so s * num_kb < 2^31.
    r.kb_begin = (s * num_kb) / split_k;
    r.kb_end = ((s + 1) * num_kb) / split_k;
    r.tile = r.tile_m * tiles_n + r.tile_n;
    return r;
}
