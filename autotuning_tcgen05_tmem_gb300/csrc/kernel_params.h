// Launch record of the tcgen05 GEMM kernel (host and device agree on it).
#pragma once
#include <stdint.h>

namespace gemmgb {

// Status-word codes written by a kernel whose bounded wait expired.
enum WaitSite : int32_t {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_TMEM_EMPTY = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_EPI_STALL = 5,
    SITE_TEARDOWN = 6,
    SITE_FIXUP = 7,
    SITE_CLUSTER = 8,
};

// Bytes of one reduction block: 128 accumulator rows x 32 fp32 columns.
constexpr uint32_t kRedBlockBytes = 128u * 32u * 4u;

struct KernelParams {
    // Problem in MMA orientation: rows along the MMA M axis, cols along MMA N.
    // Unswapped: rows = M, cols = N.  Swapped (Cᵀ = Bᵀ·Aᵀ): rows = N, cols = M.
    int32_t rows, cols, K;
    int32_t bm, bn, bk, stages;
    int32_t raster, group, split_k;
    int32_t tiles_m, tiles_n, num_kb, num_units;
    int32_t swap_ab, epi;
    int32_t a_mn_major, b_mn_major;   // operand majorness in shared memory
    int32_t a_span3d, b_span3d;       // MMA-A / MMA-B: the tensor map views the operand as
                                       // [spans][rows][one 128-byte span], and one copy takes
                                       // all of a stage's spans (0: one copy per span)
    uint32_t idesc;                    // tcgen05 instruction descriptor
    uint32_t a_stage_bytes, b_stage_bytes, tx_bytes;
    uint32_t a_lbo, b_lbo;             // leading-byte offsets of MN-major operands
    uint32_t acc_cols, n_acc, tmem_cols;
    uint32_t off_b, off_staging, off_bar, staging_buf_bytes;
    const void *bias;                  // nullable iff epi == 0
    const void *residual;              // nullable: C = act(A·B + bias) + residual when set
    float alpha;                       // C = act(alpha·(A·B) + bias): the product's scale
    float *workspace;                  // split-K partial tiles
    int32_t *counters;                 // split-K arrival counters, one per tile (last arriver)
    uint64_t *epochs;                  // one-wave split-K: arrivals per tile share ([tile][S]), never reset
    int32_t *status;                   // device status word (0 = ok)
    int64_t timeout_ns;                // bound of every mbarrier wait
    int32_t debug_stall;               // epilogue waits on a barrier nothing signals
    int32_t early_mask;                // operands not written by the work before this launch
                                       // (bit 0 MMA-A, bit 1 MMA-B): the producer copies them
                                       // before the previous kernel has finished (epilogue
                                       // warps still wait for it)
    int32_t coop_fixup;                // one-wave split-K: every unit has its own CTA, and the
                                       // slices finalise their tile share by share
    int64_t share_poll_cycles;         // how long a share's owner waits for the other slices
                                       // (SM clock cycles) before handing its share over
    int32_t pair;                      // 1: cta_group::2, consecutive CTAs share 256-row tiles
    // Block-scaled FP8 (MX): the packed scale arrays (tensor maps tmSA, tmSB:
    // row atoms x sf_kt K atoms of 512 bytes), their per-stage shared-memory
    // copy and TMEM slot (the block-scaled MMA reads scales from tensor memory).
    int32_t sf_kt;
    uint32_t sf_stage_bytes, off_sf, sc_stage_cols, sc_col0;
    int32_t cluster_k;                 // 0, or S: the S slices of a tile are one thread-block
                                       // cluster and reduce through distributed shared memory
                                       // (one unit per CTA, grid = units)
    uint32_t off_recv;                 // cluster split-K: partials land in an area of their own
                                       // at this offset; 0: in the owner's pipeline ring, once
                                       // the owner has announced that its MMAs are done
};

}  // namespace gemmgb
