/*
 * gemm_gb300.h — C ABI of the autotuned tcgen05 GEMM library for GB300 (sm_103a).
 *
 * The library computes the fused tiled multiply
 *
 *     C[m,n] = act( alpha · sum_k A[m,k] · B[k,n] + bias[n] )  ( + R[m,n] )
 *
 * (alpha = 1 and no R unless asked for) with a tile configuration (BM, BN, BK,
 * pipeline stages, tile order, split-K, CTA pair, operand swap) chosen per
 * problem shape, first by an analytical cost model and then by timing
 * candidates on the device, and cached by shape (and, optionally, in a file).
 *
 * Sources (page title, section):
 *   - "Tile Selection: Cost Models Against Measurement": the search space
 *     ("The structure of the search space"), the analytical model ("Analytical
 *     models and where they break"), measurement controls ("Measurement, and
 *     what it must control"), the hybrid filter → rank → measure arrangement
 *     ("Hybrid strategies"), the cache key (shape, dtype, device, library
 *     version) and per-device selection ("Selection is per device").
 *   - "Compilers and Kernel Languages": tiles run in waves of one per
 *     multiprocessor; the workshop model; real kernels add pipeline depth,
 *     split-K and tile order.
 *   - "Autotuning & cost models": §4 tune on first call and cache by key;
 *     §5 amortisation; §6 cost-model-guided search vs exhaustive.
 *   - "CuTile Autotuning" (tune-once / cache / launch pattern; the search space
 *     includes the original fixed configuration; split buffers while tuning).
 *   - "Tiling the hierarchy": stages hide load latency; the epilogue fused onto
 *     a GEMM is nearly free.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major and dense: A is [M,K], B is [K,N], C is [M,N];
 *     bias is a length-N vector added to every row (the pages do not define
 *     "bias"; this is the plain reading of C = act(A·B + bias)).
 *   - GEMM_BF16: A, B, bias and C are bfloat16; products accumulate in fp32 in
 *     tensor memory; C is rounded to nearest-even once.  GEMM_FP32_TF32: A, B,
 *     bias and C are fp32; the tensor cores read the operands as TF32.
 *     GEMM_FP8_E4M3: A and B are FP8 E4M3 bytes (OCP "E4M3FN": no infinities;
 *     448 is the largest finite value), read by tcgen05.mma kind::f8f6f4; bias,
 *     R and C are bfloat16; the product's scale (the operands' tensor scales)
 *     is gemm_plan_set_scale's alpha.  B is read MN-major in place (as bf16)
 *     when N is a multiple of 16, else from a K-major copy (as fp32).
 *     GEMM_MXFP8_E4M3: block-scaled FP8 in the OCP Microscaling (MX) format
 *     (OCP "Microscaling Formats (MX) Specification" v1.0, MXFP8 E4M3): A and B
 *     are E4M3 bytes as above, and every run of 32 consecutive elements along K
 *     shares one power-of-two scale, an E8M0 byte s meaning 2^(s-127) (255 is
 *     NaN).  C[m,n] = act(alpha·sum_k (A[m,k]·2^(SA[m,k/32]-127))·
 *     (B[k,n]·2^(SB[k/32,n]-127)) + bias[n]) (+ R), read by tcgen05.mma
 *     kind::mxf8f6f4.block_scale with the scales in tensor memory.  The
 *     scales reach the kernel packed by gemm_mx_pack_scales (below); runs go
 *     through gemm_run_mx.  bias, R and C are bfloat16.
 *   - GELU is the erf form 0.5·x·(1 + erf(x/√2)).
 *   - Device pointers are caller-owned, must stay valid until the work queued
 *     on the stream has finished, and must be 16-byte aligned; K·elt and N·elt
 *     must be multiples of 16 bytes (TMA row-stride rule; FP8: K a multiple of
 *     16 and N of 8, the rows of A and of C).
 *   - Every function returns GEMM_OK (0) or a negative gemm_status; the text of
 *     the last error of the calling thread is returned by gemm_last_error().
 *     Nothing aborts, traps or exits the process.
 *   - Extents are int64_t; M, N, K must be >= 0 and < 2^31.  M == 0 or
 *     N == 0 is a no-op; K == 0 gives C = act(bias) (empty sum).
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,  /* null pointer, negative extent, unknown enum */
    GEMM_ERR_MISALIGNED = -2,   /* pointer not 16-byte aligned or row stride not a multiple of 16 B */
    GEMM_ERR_UNSUPPORTED = -3,  /* no feasible configuration / not an sm_100-family GPU */
    GEMM_ERR_INFEASIBLE = -4,   /* an explicit configuration breaks a hardware rule */
    GEMM_ERR_CUDA = -5,         /* a CUDA runtime/driver call failed (text in gemm_last_error) */
    GEMM_ERR_TIMEOUT = -6,      /* a device wait ran past its limit; the kernel returned early */
    GEMM_ERR_NO_DEVICE = -7     /* no CUDA device is visible */
} gemm_status;

typedef enum { GEMM_BF16 = 0, GEMM_FP32_TF32 = 1, GEMM_FP8_E4M3 = 2, GEMM_MXFP8_E4M3 = 3 } gemm_dtype;

typedef enum {
    GEMM_EPI_NONE = 0,       /* C = A·B                 (bias may be NULL) */
    GEMM_EPI_BIAS = 1,       /* C = A·B + bias          */
    GEMM_EPI_BIAS_RELU = 2,  /* C = max(A·B + bias, 0)  */
    GEMM_EPI_BIAS_GELU = 3,  /* C = gelu(A·B + bias)    */
    /* Residual variants: the same, plus R, an [M, N] row-major tensor of C's
     * type passed to gemm_run_ex (the transformer block's "x + f(x)").  The
     * pages name a fused residual add as an epilogue beyond bias and
     * activation; the order (activation, then + R) is the residual
     * connection's. */
    GEMM_EPI_BIAS_RESIDUAL = 4,       /* C = A·B + bias + R          */
    GEMM_EPI_BIAS_RELU_RESIDUAL = 5,  /* C = max(A·B + bias, 0) + R  */
    GEMM_EPI_BIAS_GELU_RESIDUAL = 6,  /* C = gelu(A·B + bias) + R    */
    /* Gated (GLU-style dual output) variants over a fused gate+up weight: B is
     * [K, N] with N a multiple of 64 whose columns come in blocks of 32, gate
     * and up alternating, and bias [N] likewise; C is [M, N/2] with
     *   C[m, o] = act(G[m, o]) · U[m, o],  G = A·B[:, gate(o)] + bias[gate(o)],
     *   U = A·B[:, up(o)] + bias[up(o)],  gate(o) = 64·(o/32) + o%32,  up(o) = gate(o) + 32.
     * One pass over the fused weight, the activation and the product fused
     * into the epilogue ("Tiling the hierarchy", fusion: an elementwise chain
     * fused onto the product that feeds it; "CuTile Autotuning": fused
     * dual-GEMM kernels, Linear + GLU activation).  Unswapped, single-slice
     * configurations only (swap_ab 0, split_k 1), bn a multiple of 64. */
    GEMM_EPI_BIAS_REGLU = 7,          /* act = ReLU                  */
    GEMM_EPI_BIAS_GEGLU = 8,          /* act = GELU (erf form)       */
    GEMM_EPI_BIAS_SWIGLU = 9          /* act = SiLU, x / (1 + e^-x)  */
} gemm_epilogue;

/*
 * One tile configuration ("Tile Selection", "The structure of the search
 * space": block tile, reduction step; "Compilers and Kernel Languages": pipeline
 * depth, split-K, tile order).  bm × bn is the tile of the MMA output: with
 * swap_ab = 0 it tiles C (bm rows of M, bn columns of N); with swap_ab = 1 the
 * kernel computes Cᵀ = Bᵀ·Aᵀ, so bm tiles N and bn tiles M (small-M decode).
 *   bm        128 or 256 (tcgen05 M = 128 per CTA; 256 = two stacked MMAs)
 *   bn        16..256, multiple of 16 (swap) / of 32 and of the 128-byte span
 *             (64 bf16, 32 fp32) when B is the MN-major operand (no swap)
 *   bk        K per pipeline stage: 1..4 spans of 128 bytes (64/128/192/256 bf16)
 *   stages    2..16 shared-memory ring slots
 *   raster    0: tiles walk a band of `group` tile-rows column by column;
 *             1: a band of `group` tile-columns row by row
 *   group     1, 2, 4, 8 or 16
 *   split_k   1..16 slices of K; partial fp32 tiles are summed in slice order
 *             (deterministic: every exchange route gives the same bits)
 *   cta_group 1, or 2: a 256-row tile on a CTA pair (tcgen05 cta_group::2;
 *             bm = 256, no swap; each CTA holds 128 rows and half of B)
 *   swap_ab   0 or 1, as above
 * Block-scaled FP8 (GEMM_MXFP8_E4M3) adds: unswapped bn 128 or 256 (a CTA pair
 * too); swapped (tokens along the MMA's N) bn a multiple of 128 or at least M,
 * so that every tile starts on a 128-column scale atom; bk 128 or 256; and the
 * accumulators plus one TMEM slot of scales per stage within 512 columns.
 */
typedef struct {
    int32_t bm, bn, bk, stages, raster, group, split_k, cta_group, swap_ab;
} gemm_config;

/* Reason codes of gemm_check_config (first rule broken, in this order). */
typedef enum {
    GEMM_FEASIBLE = 0,
    GEMM_REASON_CTA_GROUP = 1,  /* cta_group not 1, or 2 with bm = 256 and no swap */
    GEMM_REASON_UMMA_M = 2,     /* bm not 128/256 (tcgen05 M per CTA is 128) */
    GEMM_REASON_UMMA_N = 3,     /* bn not a multiple of 16 in [16, 256] */
    GEMM_REASON_LAYOUT = 4,     /* swap_ab not 0/1; bn not a multiple of 32 and of the span when unswapped
                                   (MX: bn not 128/256 unswapped; swapped, bn neither a multiple of 128 nor >= M) */
    GEMM_REASON_BK = 5,         /* bk not 1..4 spans of 128 bytes (MX: not 128/256) */
    GEMM_REASON_STAGES = 6,     /* stages outside 2..16 */
    GEMM_REASON_SCHEDULE = 7,   /* raster not 0/1 or group not in {1,2,4,8,16} */
    GEMM_REASON_SPLIT_K = 8,    /* split_k outside 1..16 or above ceil(K/bk) */
    GEMM_REASON_ALIGN = 9,      /* K·elt or N·elt not a multiple of 16 bytes */
    GEMM_REASON_TMEM = 10,      /* one accumulator (MX: plus the scale slots) needs more than 512 TMEM columns */
    GEMM_REASON_SMEM = 11,      /* ring + epilogue staging + barriers exceed the per-block limit */
    GEMM_REASON_REGS = 12       /* kernel registers × 320 threads exceed 65,536 */
} gemm_reason;

/*
 * Device and cost-model parameters ("Tile Selection", "Selection is per device":
 * the SM count and the limits are properties of the device; never hard-coded).
 * gemm_device_params_query fills the device fields from the current device;
 * the model coefficients default to values fitted on a GB300 (least squares in
 * log time over exhaustive tuning tables of the library's own workloads) and may
 * be overridden by the caller.
 */
typedef struct {
    int32_t sm_count;               /* multiprocessors */
    int32_t model_kind;             /* 0 = tcgen05 model; 1 = the workshop model of
                                       "Compilers and Kernel Languages" */
    int64_t smem_per_block;         /* opt-in dynamic shared memory per block, bytes */
    int64_t l2_bytes;
    double  peak_tflops_bf16;       /* dense tensor peak (measured burst on GB300) */
    double  peak_tflops_tf32;
    double  peak_tflops_fp8;        /* FP8 dense peak (measured bf16 x the nominal 2x ratio) */
    double  hbm_gbs;                /* DRAM bandwidth, GB/s */
    double  sm_clock_mhz;
    double  l2_gbs;                 /* aggregate L2 -> shared-memory operand bandwidth, GB/s */
    double  mma_issue_clk;          /* issue cost of one tcgen05.mma, SM clocks */
    double  kblock_clk;             /* per pipeline stage: waits, commits, bookkeeping */
    double  mem_latency_us;         /* load round trip seen by the shared-memory ring */
    double  epi_elems_per_clk;      /* epilogue throughput per CTA, none/bias/ReLU */
    double  epi_gelu_elems_per_clk; /* epilogue throughput per CTA with GELU */
    double  splitk_gbs;             /* per-CTA bandwidth of split-K partial-tile traffic */
    double  launch_us;              /* launch + prologue */
    int32_t kernel_regs;            /* registers/thread of the GEMM kernel (0 = unknown) */
    int32_t threads_per_cta;        /* 320 */
} gemm_device_params;

/* Terms of one cost-model prediction (times in microseconds). */
typedef struct {
    double predicted_us;   /* max(mma, l2, hbm, latency) + epilogue + splitk + launch */
    double mma_us;         /* tensor pipe: max(execute, issue) per K-block, per CTA */
    double l2_us;          /* operand panels streamed from L2 into shared memory */
    double hbm_us;         /* DRAM bytes (compulsory, or per-wave panels past L2) */
    double latency_us;     /* K-blocks x load latency / stages (bytes in flight) */
    double epilogue_us;    /* epilogue not hidden behind a main loop */
    double splitk_us;      /* partial-tile writes and the fix-up reads */
    double launch_us;
    double wave_eff, tile_eff, pad_eff;
    double hbm_bytes, l2_bytes, flops;
    int64_t tiles, units, waves, ctas;
} gemm_model_terms;

/* One row of a tuning table. */
typedef struct {
    gemm_config config;
    double predicted_us;     /* cost model */
    double measured_us;      /* median over interleaved rounds (< 0: not measured) */
    double measured_min_us;  /* fastest round */
    int32_t model_rank;      /* 0-based rank by predicted_us */
    int32_t measured_rank;   /* 0-based rank by measured_us (-1: not measured) */
    int32_t status;          /* GEMM_OK, or the error the candidate returned */
    int32_t reserved;
} gemm_tune_row;

/* How well the model's ordering agreed with measurement over the measured rows
 * ("Autotuning & cost models", §6). */
typedef struct {
    double kendall_tau;      /* τ_b */
    double spearman_rho;
    double regret;           /* measured(model's pick) / measured(best) - 1 */
    double tune_seconds;     /* wall time of the search */
    double best_us;          /* measured time of the winner */
    double fixed_us;         /* measured time of the fixed 128x128 config (< 0 if absent) */
    int32_t top1_hit;        /* model's first choice was the measured fastest */
    int32_t n_measured;
    int32_t n_candidates;
    int32_t reserved;
} gemm_rank_stats;

typedef struct gemm_plan_s *gemm_plan_t;  /* opaque, library-owned */

/* ---------------------------------------------------------------------------
 * Host logic (no GPU needed)
 * ------------------------------------------------------------------------- */

/* Library version string (part of the cache key). */
const char *gemm_version(void);

/* Text of the calling thread's last error ("" if none).  Owned by the library. */
const char *gemm_last_error(void);

/* Nominal GB300 parameters (152 SMs, 227 KB, 126 MB L2, nominal peaks).  Used
 * on machines without a GPU and as the base that _query refines. */
void gemm_device_params_default(gemm_device_params *out);

/* The workshop device of "Compilers and Kernel Languages" (H100: 132 SMs, 228 KB,
 * 989 TFLOP/s BF16, 3.35 TB/s) with model_kind = 1. */
void gemm_device_params_workshop(gemm_device_params *out);

/* Feasibility of `cfg` for the problem: GEMM_FEASIBLE or a gemm_reason (> 0);
 * GEMM_ERR_INVALID_ARG (< 0) for null pointers or bad enums. */
int gemm_check_config(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                      const gemm_config *cfg, const gemm_device_params *dev);

/* The candidate set for the problem ("Tile Selection", "Hybrid strategies":
 * the resource filter).  Writes up to `cap` feasible configs in generation
 * order to out (out may be NULL when cap == 0) and the total count to *n. */
int gemm_enumerate(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                   const gemm_device_params *dev, gemm_config *out, int32_t cap, int32_t *n);

/* The fixed, untuned configuration (128×128 tile, one K span, as many stages as
 * fit, row-major order, no split): the baseline tuning must never lose to. */
int gemm_fixed_config(gemm_dtype dtype, const gemm_device_params *dev, gemm_config *out);

/* Cost-model prediction for one configuration ("Tile Selection", "Analytical
 * models and where they break"; "Compilers and Kernel Languages", workshop). */
int gemm_model_predict(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                       const gemm_config *cfg, const gemm_device_params *dev,
                       gemm_model_terms *out);

/* Rank agreement of two equal-length arrays (n >= 2): τ_b, ρ, top-1, regret. */
int gemm_rank_agreement(const double *predicted, const double *measured, int32_t n,
                        gemm_rank_stats *out);

/* The persistent schedule's map of work unit u to its tile and K slice (the
 * same function the kernel runs).  Outputs may be NULL. */
int gemm_schedule_unit(int64_t unit, int32_t tiles_m, int32_t tiles_n, int32_t split_k,
                       int32_t raster, int32_t group, int32_t num_kb,
                       int32_t *tile_m, int32_t *tile_n, int32_t *split,
                       int32_t *kb_begin, int32_t *kb_end);

/* ---------------------------------------------------------------------------
 * Device entry points (current CUDA device)
 * ------------------------------------------------------------------------- */

/* Parameters of the current device: SM count, shared-memory limit, L2 size,
 * clock and the GEMM kernel's register count, on top of the defaults. */
int gemm_device_params_query(gemm_device_params *out);

/* Apply a text file of cost-model coefficients to *dev: one "name value" pair
 * per line ('#' starts a comment), names being the double fields of
 * gemm_device_params (l2_gbs, mma_issue_clk, kblock_clk, mem_latency_us,
 * epi_elems_per_clk, epi_gelu_elems_per_clk, splitk_gbs, launch_us, peaks,
 * hbm_gbs, sm_clock_mhz), values positive.  A file fitted to one device's
 * timings recalibrates the model for it ("Tile Selection", "Selection is per
 * device").  gemm_device_params_query applies the file named by
 * GEMM_MODEL_PARAMS when that variable is set.  Returns GEMM_ERR_INVALID_ARG
 * (and leaves *dev unchanged) for an unreadable file, an unknown name or a bad
 * value. */
int gemm_model_params_load(const char *path, gemm_device_params *dev);

/* Plan a GEMM: cache lookup by (M, N, K, dtype, epilogue, device name, SM count,
 * library version); on a miss, enumerate → rank by the model → time the top
 * candidates on library-owned buffers → cache the winner ("Autotuning & cost
 * models" §4; "CuTile Autotuning").  Environment: GEMM_DISABLE_AUTOTUNE=1 picks
 * the fixed config without timing; GEMM_TUNE_MODE=exhaustive|topk (default
 * topk); GEMM_TUNE_TOPK=k (default 24).  Synchronises; never touches user
 * memory.  The returned handle is owned by the caller (gemm_plan_destroy) and
 * may be used on one stream at a time.  The synthetic operands the candidates
 * are timed on are normally distributed with standard deviation 1/sqrt(K), the
 * spread of the workloads' N(0,1)/sqrt(K) operands ("Tile Selection",
 * "Measurement, and what it must control": tuning inputs must resemble the real
 * ones in distribution, not merely in shape; gemm_debug_set(6, 0) selects a
 * uniform fill of the same spread); gemm_plan_tuned_on times them on the
 * caller's own operands instead. */
int gemm_plan(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
              gemm_plan_t *out);

/* gemm_plan, but on a cache miss the candidates are timed on copies of the
 * caller's operands (device pointers in the layouts gemm_run / gemm_run_mx
 * take: A [M, K], B [K, N], bias [N] unless GEMM_EPI_NONE, and for block-scaled
 * FP8 the packed scales SA and SB; SA and SB are NULL otherwise) instead of on
 * synthetic ones, so that the values, and the power they draw under the power
 * cap, are the real ones ("Tile Selection", "Measurement, and what it must
 * control").  The operands are only read: the call first synchronises the
 * device (their producers may be on any stream), then copies them into
 * library-owned buffers; it never writes caller memory.  The winner is cached
 * under the same key as gemm_plan's.  GEMM_ERR_INVALID_ARG when an operand the
 * shape needs is NULL. */
int gemm_plan_tuned_on(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const void *A,
                       const void *SA, const void *B, const void *SB, const void *bias, gemm_plan_t *out);

/* Plan with an explicit configuration (no tuning, no cache).  Returns
 * GEMM_ERR_INFEASIBLE, with the reason in gemm_last_error, if it breaks a rule. */
int gemm_plan_with_config(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                          const gemm_config *cfg, gemm_plan_t *out);

/* Scale of the product: C = act(alpha·(A·B) + bias) (+ R).  Default 1; for
 * FP8 operands alpha is scale_A·scale_B.  Applies to launches queued after the
 * call. */
int gemm_plan_set_scale(gemm_plan_t plan, float alpha);

/* Operands named in gemm_plan_set_independent_operands. */
enum { GEMM_OPERAND_A = 1, GEMM_OPERAND_B = 2 };

/* Declare which operands of this plan's launches are never written by the
 * work queued before a launch on its stream: a mask of GEMM_OPERAND_A (A, and
 * SA for block-scaled FP8) and GEMM_OPERAND_B (B, and SB); 0, the default,
 * withdraws the declaration.  Every launch allows programmatic overlap with the
 * previous kernel on the stream, and by default it touches no global memory
 * before that kernel has finished.  In a chain of layers B (the weights) is
 * independent and A (the previous layer's output) is not: declaring B lets
 * the launch copy the first pipeline stages of B while the previous kernel
 * drains, and copy A once it has finished.  Declaring both (independent GEMMs
 * back to back) lets all operand copies and MMAs run ahead; then the
 * producer's bounded waits (the device timeout) also span what remains of the
 * previous kernel, and one that runs longer than the timeout makes the launch
 * report GEMM_ERR_TIMEOUT.  bias and R are always read after the wait, and C,
 * the split-K exchange and the status word are written after it.  B is
 * treated as dependent in plans that first copy it K-major (that copy is the
 * previous kernel).  Applies to launches queued after the call; a caller that
 * breaks the declaration reads operands that may still be being written.
 * GEMM_ERR_INVALID_ARG for a null plan or other bits in the mask. */
int gemm_plan_set_independent_operands(gemm_plan_t plan, int32_t mask);

/* The configuration a plan runs. */
int gemm_plan_config(gemm_plan_t plan, gemm_config *out);

/* How a plan launches its GEMM kernel (library-specific; the pages have no
 * counterpart).  splitk_route: 0 = no split-K; 1 = partial tiles through
 * global memory, the last slice to arrive finalises the tile; 2 = partial
 * tiles through global memory in one wave, each slice finalising its own share
 * of the tile once the others have arrived (an owner whose peers are late, for
 * instance not resident because another kernel holds their SMs, hands its
 * share to whichever slice arrives last, so no slice waits for one that may
 * not run); 3 = the slices of a tile form one thread-block cluster (resident
 * together by construction) and reduce through distributed shared memory. */
typedef struct {
    int32_t grid;          /* CTAs launched */
    int32_t block;         /* threads per CTA */
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t cluster;       /* CTAs per cluster (1 = no cluster) */
    int32_t splitk_route;  /* see above */
    int32_t b_transposed;  /* 1: B is first copied to a K-major layout (one extra kernel) */
    int32_t units;         /* work units: tiles x split_k */
    int32_t tiles;         /* output tiles */
    int32_t span_copies;   /* bit 0: MMA-A, bit 1: MMA-B is copied with one tensor copy per
                              stage over all its 128-byte spans (see gemm_debug_set, what = 7) */
} gemm_launch_info;

int gemm_plan_launch_info(gemm_plan_t plan, gemm_launch_info *out);

/* Enqueue C = act(A·B + bias) on `stream` (asynchronous).  A, B, bias, C are
 * device pointers as described above; bias may be NULL only with
 * GEMM_EPI_NONE.  A split-K plan uses its own workspace, so one plan must not
 * run on two streams at once.  Checked runs (GEMM_CHECK set to anything but 0
 * in the environment when the library loads, or gemm_debug_set(4, 1)): every
 * gemm_run, gemm_run_ex and gemm_run_mx synchronises `stream` and returns
 * GEMM_ERR_TIMEOUT itself when a device wait expired (as gemm_plan_status
 * would). */
int gemm_run(gemm_plan_t plan, const void *A, const void *B, const void *bias, void *C,
             gemm_stream_t stream);

/* gemm_run with a residual: R is a device pointer to [M, N] row-major of C's
 * type, 16-byte aligned, read once per element; it may be C itself (in-place
 * "C += f(A·B + bias)"), and may not overlap C otherwise.  Required (non-NULL)
 * exactly for the residual epilogues, which gemm_run rejects with
 * GEMM_ERR_INVALID_ARG.  Asynchronous on `stream`. */
int gemm_run_ex(gemm_plan_t plan, const void *A, const void *B, const void *bias, const void *R, void *C,
                gemm_stream_t stream);

/* Block-scaled FP8 (GEMM_MXFP8_E4M3 plans, which gemm_run and gemm_run_ex
 * reject): as gemm_run_ex, plus SA and SB, the device pointers of A's and B's
 * scales in the packed layout that gemm_mx_pack_scales writes
 * (gemm_mx_scales_bytes(M, K) and gemm_mx_scales_bytes(N, K) bytes, 16-byte
 * aligned).  R is required exactly for the residual epilogues.  Asynchronous
 * on `stream`. */
int gemm_run_mx(gemm_plan_t plan, const void *A, const void *SA, const void *B, const void *SB, const void *bias,
                const void *R, void *C, gemm_stream_t stream);

/* Bytes of one operand's packed MX scales: the operand's `rows` (M for A, N
 * for B) padded to a multiple of 256 and K padded to a multiple of 256, in
 * atoms of 128 rows x 128 K (512 bytes, four 32-element blocks per row).
 * Returns 0 for a negative extent. */
int64_t gemm_mx_scales_bytes(int64_t rows, int64_t K);

/* Pack one operand's E8M0 scales for gemm_run_mx (asynchronous on `stream`).
 * `scales` is a device pointer to the natural layout: for A (b_side = 0)
 * [rows, ceil(K/32)] row-major (SA[m, j] scales A[m, 32j .. 32j+31]); for B
 * (b_side = 1) [ceil(K/32), rows] row-major (SB[j, n] scales B[32j .. 32j+31,
 * n]).  `packed` receives gemm_mx_scales_bytes(rows, K) bytes: for row r and
 * block j, atom (r/128, j/4) at byte offset ((r/128)·KT + j/4)·512 (KT the
 * padded K over 128), and within it byte (r%32)·16 + ((r%128)/32)·4 + j%4, the
 * order in which tcgen05.cp 32x128b.warpx4 hands a 128-row block's scales to
 * the block-scaled MMA.  Padding bytes are 0 (2^-127; they meet only the zero
 * fill of out-of-range operand elements). */
int gemm_mx_pack_scales(const void *scales, int64_t rows, int64_t K, int32_t b_side, void *packed,
                        gemm_stream_t stream);

/* Same product from HOST buffers (epilogues without residual): copies A, B, bias to plan-owned device
 * buffers, runs, copies C back, and synchronises `stream` before returning.
 * Host buffers should be pinned for full copy bandwidth. */
int gemm_run_host(gemm_plan_t plan, const void *A, const void *B, const void *bias, void *C,
                  gemm_stream_t stream);

/* n independent GEMMs of the plan's shape from HOST buffers (A[i], B[i],
 * bias[i] -> C[i]; bias may be NULL with GEMM_EPI_NONE; epilogues without
 * residual), pipelined so that host<->device copies overlap the kernels: GEMM
 * i runs on `stream` when i is even and on a second, plan-owned stream when i
 * is odd, with a second plan of the same configuration (its own device
 * buffers and split-K state, made on the first call with n > 1, so make that
 * call before any stream capture).  The second stream starts after the work
 * already queued on `stream`.  Returns after every C is in host memory and
 * both plans' device status words have been read: GEMM_ERR_TIMEOUT if a device
 * wait expired.  The copies overlap only when the host buffers are pinned
 * (page-locked); pageable buffers give correct results without overlap.  Like
 * gemm_run_host, this is the library's end-to-end entry point: the pages
 * measure kernels, and this measures what a caller holding host data sees.
 * "Tiling the hierarchy", double buffering (a copy overlaps compute only when
 * it is asynchronous), applied one level up, to the host link. */
int gemm_run_host_many(gemm_plan_t plan, int32_t n, const void *const *A, const void *const *B,
                       const void *const *bias, void *const *C, gemm_stream_t stream);

/* Synchronise and read the plan's device status word: GEMM_OK or
 * GEMM_ERR_TIMEOUT (a bounded wait expired; the status is cleared and the
 * split-K counters reset so the plan can run again). */
int gemm_plan_status(gemm_plan_t plan);

void gemm_plan_destroy(gemm_plan_t plan);

/* Exhaustively time every feasible candidate (or the model's top `topk` when
 * topk > 0) and fill `rows` (up to cap, ordered by measured time, unmeasured
 * rows last) and `stats`.  *n_rows receives the number of rows written. */
int gemm_tune(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
              int32_t topk, gemm_tune_row *rows, int32_t cap, int32_t *n_rows,
              gemm_rank_stats *stats);

/* gemm_tune on copies of the caller's operands (as gemm_plan_tuned_on takes
 * them) instead of synthetic ones; never touches the cache. */
int gemm_tune_on(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const void *A, const void *SA,
                 const void *B, const void *SB, const void *bias, int32_t topk, gemm_tune_row *rows, int32_t cap,
                 int32_t *n_rows, gemm_rank_stats *stats);

/* Search strategies at a given measurement budget ("Autotuning & cost models"
 * §6): time every candidate; the cost model's top k (plus the fixed tile, so
 * tuning never loses to it — "CuTile Autotuning"); or k candidates drawn
 * uniformly at random from the seeded splitmix64 stream `seed`. */
typedef enum { GEMM_SEARCH_EXHAUSTIVE = 0, GEMM_SEARCH_MODEL_TOPK = 1, GEMM_SEARCH_RANDOM_K = 2 } gemm_search;

/* gemm_tune with an explicit strategy and budget k (ignored for exhaustive). */
int gemm_tune_search(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, gemm_search mode,
                     int32_t k, uint64_t seed, gemm_tune_row *rows, int32_t cap, int32_t *n_rows,
                     gemm_rank_stats *stats);

/* Tune-once cache: number of searches run, lookups served, entries held. */
int gemm_cache_stats(int64_t *tunes, int64_t *hits, int64_t *entries);
void gemm_cache_clear(void);

/* Tuning database ("Tile Selection", "Measurement, and what it must control":
 * results shipped with the artifact or kept in a database that persists across
 * deployments; "Autotuning & cost models" §5: ahead-of-time tuning log).  A text
 * file, one entry per line: the cache key (M|N|K|dtype|epilogue|device name|SM
 * count|library version), a tab, and the nine config fields.  Save writes the
 * whole cache atomically (temporary file + rename); load merges entries into
 * the cache (an entry serves only its own device and library version; one that
 * the current limits reject is re-tuned).  With GEMM_TUNING_DB=<path>, gemm_plan
 * loads that file on first use and appends every new winner to it. */
int gemm_cache_save(const char *path, int64_t *n_written);
int gemm_cache_load(const char *path, int64_t *n_loaded);

/* Shipped configuration set ("Tile Selection": a kernel ships a short list of
 * configurations; "Autotuning & cost models": tune ahead of time, not per
 * call).  From a measured table times[s * n_configs + c] (microseconds; <= 0
 * where configuration c does not run shape s), picks at most max_set
 * configurations greedily: each step adds the one that most raises the sum
 * over shapes of (shape's best time) / (fastest chosen time), the lowest
 * index among equal gains, and stops early when nothing gains.  That sum is
 * monotone and submodular, so the set is within (1 - 1/e) of the best set of
 * its size.  Writes the chosen column indices in order and the mean and worst
 * slowdown (chosen / best; +inf for a shape no chosen configuration runs).
 * Host only. */
int gemm_select_config_set(const double *times, int32_t n_shapes, int32_t n_configs, int32_t max_set,
                           int32_t *chosen, int32_t *n_chosen, double *mean_slowdown, double *worst_slowdown);

/* Plan by timing only the members of `list` (n configurations) that the
 * rules accept for this shape, on library-owned buffers; the fastest wins.
 * The cache is neither read nor written.  GEMM_ERR_UNSUPPORTED if no member
 * runs the shape. */
int gemm_plan_from_list(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                        const gemm_config *list, int32_t n, gemm_plan_t *out);

/* Ahead-of-time tuning: gemm_plan for each of the n shapes mnk[3i..3i+2]
 * (M, N, K), so that every one is in the cache; then, if db_path is not NULL,
 * gemm_cache_save(db_path).  *n_tuned (nullable) = shapes newly tuned (the
 * others were cached already). */
int gemm_tune_batch(const int64_t *mnk, int32_t n, gemm_dtype dtype, gemm_epilogue epi, const char *db_path,
                    int32_t *n_tuned);

/* Debug controls.  what = 0: wait limit in nanoseconds (default 2e9; every
 * mbarrier wait in the kernel gives up after it, sets the status word and
 * returns); what = 1: make the epilogue wait on a barrier that nothing signals
 * (1 = on, 0 = off) so that the timeout path can be tested; what = 2: how B
 * reaches the tensor cores in plans made afterwards (0 = by dtype: bf16 is read
 * MN-major in place, FP8 too when N is a multiple of 16, fp32 is first
 * transposed into a plan-owned K-major copy; 1 = always transposed; 2 = always
 * MN-major); what = 3: how split-K slices exchange partial tiles in plans made
 * afterwards (0 = through distributed shared memory when all units fit in one
 * wave and the slices of a tile can form a thread-block cluster, else through
 * global memory; 1 = always through global memory); what = 4: checked runs
 * (1 = every run synchronises and reports a device timeout, 0 = off; the
 * initial value comes from GEMM_CHECK); what = 5: how many SM clock cycles the
 * owner of a one-wave split-K share (splitk_route 2) waits for the other
 * slices before handing its share over (default 50000, about 25 us; 0 = hand
 * over at once, which tests use to drive that path); what = 6: the value
 * distribution of the tuner's synthetic operands (1 = normal, the default; 0 =
 * uniform of the same standard deviation); what = 7: how the producer copies
 * an operand's stage (1 = the default: one tensor copy for all of the stage's
 * 128-byte spans where the operand's contiguous extent is a whole number of
 * spans; 0 = one copy per span; the results are the same bits either way).
 * Affects launches (what 0, 1, 4, 5), plans (what 2, 3, 7) or tunings (what 6)
 * made after the call, from any thread. */
int gemm_debug_set(int32_t what, int64_t value);

/* ---------------------------------------------------------------------------
 * Allocation-free entry point.  The pages have no counterpart: this is a
 * deployment aid, not part of the method.
 * ------------------------------------------------------------------------- */

/* Size of the fixed scratch behind gemm_run_noalloc: split-K partial tiles
 * (16 MiB of fp32) and one arrival counter per output tile (at most 4096 tiles). */
#define GEMM_NOALLOC_WORKSPACE_BYTES (16u * 1024u * 1024u)
#define GEMM_NOALLOC_MAX_TILES 4096

/* C = act(A·B + bias) for bf16 operands with the explicit configuration *cfg,
 * for callers that cannot call cudaMalloc: code running under a framework whose
 * caching allocator owns the device memory (a raw cudaMalloc escapes its
 * accounting and may synchronise the device), or services that reserve all
 * device memory up front and must not fail or stall on an allocation while
 * serving.  It allocates nothing, host or device: its scratch (status word,
 * split-K counters and partial tiles) is one fixed array compiled into the
 * library, which every GPU that loads the library holds until the process exits.
 * Arguments are those of gemm_plan_with_config + gemm_run (bf16 only; epilogues
 * without residual; single-CTA tiles, cta_group 1, else GEMM_ERR_UNSUPPORTED);
 * the call is asynchronous on `stream` and returns after the launch.
 *   - The first call on a device sets that device up (looks up the scratch's
 *     device address, reads the device's limits, sets the kernel's shared-memory
 *     limit); make that first call before any stream capture.
 *   - Returns GEMM_ERR_INVALID_ARG, with the limits in gemm_last_error, when the
 *     problem needs more than GEMM_NOALLOC_MAX_TILES output tiles or, with
 *     split_k > 1, more than GEMM_NOALLOC_WORKSPACE_BYTES of partial tiles.
 *   - All calls share the scratch and it keeps the previous call's contents;
 *     each call first clears, on `stream`, the status word and the counters it
 *     uses.  Calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on the scratch and must be serialised by the caller.
 *   - A device wait that expires is recorded in the scratch's status word.  In
 *     checked-run mode (GEMM_CHECK, or gemm_debug_set(4, 1)) the call
 *     synchronises `stream`, reads that word (without allocating) and returns
 *     GEMM_ERR_TIMEOUT, like gemm_run; otherwise it is not reported, and the
 *     next call clears it. */
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_epilogue epi, const gemm_config *cfg,
                     const void *A, const void *B, const void *bias, void *C, gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
