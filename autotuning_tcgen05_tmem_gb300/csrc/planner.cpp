// Selection-layer host logic: device parameters, the feasibility filter, the
// candidate generator, the analytical cost model and rank agreement.
//
// Sources (page title, section):
//  * "Tile Selection: Cost Models Against Measurement": hardware limits that are
//    checkable before any code runs ("The structure of the search space");
//    the roofline model with its pipeline-fill, occupancy and tail corrections
//    ("Analytical models and where they break"); the hybrid filter -> rank ->
//    measure arrangement ("Hybrid strategies"); per-device selection.
//  * "Compilers and Kernel Languages": waves of one tile per multiprocessor,
//    the workshop model (HBM traffic divided by g = √(tiles sharing panels in
//    one wave), compute divided by wave and tile efficiency, time = max).
//  * "Tiling the hierarchy": shared memory holds the reuse tile, the pipeline
//    stages and the epilogue scratch together; stages convert load + compute
//    into max(load, compute) once enough bytes are in flight; the threshold
//    regime when the working set fits in a cache level.
//  * "Autotuning & cost models" §6: the model ranks, measurement decides; rank
//    agreement (Kendall τ, Spearman ρ) says how far the ranking can be trusted.
#include <math.h>
#include <stdarg.h>
#include <string.h>

#include <algorithm>
#include <numeric>

#include "gemm_internal.h"

namespace gemmgb {

// GB300 values.  Peaks: a measured copy bandwidth and cuBLAS bf16 burst rate on
// this part; model coefficients: least-squares fit (log time) to exhaustive
// tuning tables of 34 workloads on a GB300 (gemm_tune, every candidate timed).
void params_default(gemm_device_params *d)
{
    memset(d, 0, sizeof(*d));
    d->sm_count = 152;
    d->model_kind = 0;
    d->smem_per_block = 232448;
    d->l2_bytes = 129LL * 1024 * 1024;
    d->peak_tflops_bf16 = 1889.6;
    d->peak_tflops_tf32 = 944.8;
    d->peak_tflops_fp8 = 3779.2;     // the nominal 2x of bf16
    d->hbm_gbs = 6675.8;
    d->sm_clock_mhz = 2070.0;
    d->l2_gbs = 14888.0;
    d->mma_issue_clk = 39.53;
    d->kblock_clk = 483.2;
    d->mem_latency_us = 1.375;
    d->epi_elems_per_clk = 3.632;
    d->epi_gelu_elems_per_clk = 5.109;
    d->splitk_gbs = 15.99;
    d->launch_us = 7.50;
    d->kernel_regs = 0;
    d->threads_per_cta = kThreadsPerCta;
}

void params_workshop(gemm_device_params *d)
{
    params_default(d);
    d->sm_count = 132;
    d->model_kind = 1;
    d->smem_per_block = 228 * 1024;
    d->peak_tflops_bf16 = 989.0;
    d->peak_tflops_tf32 = 494.5;
    d->peak_tflops_fp8 = 1978.0;
    d->hbm_gbs = 3350.0;
}

static int staging_bytes(int dt, int swap_ab)
{
    const int rows = swap_ab ? 16 : 32;   // store chunk: 32 rows x 32 cols, or 16 token rows x 32 cols
    return 8 * 2 * rows * 32 * out_elt_bytes(dt);   // 8 epilogue warps x 2 buffers of C
}

Layout layout_of(const gemm_config &c, int dt)
{
    Layout L;
    const int e = elt_bytes(dt);
    // A CTA pair (cta_group 2) splits the tile: each CTA stages 128 rows of A
    // and half of B's columns, and accumulates its 128 rows x bn.
    const bool pair = c.cta_group == 2;
    L.a_stage_bytes = (uint32_t)((pair ? 128 : c.bm) * c.bk * e);
    L.b_stage_bytes = (uint32_t)((pair ? c.bn / 2 : c.bn) * c.bk * e);
    L.stage_bytes = L.a_stage_bytes + L.b_stage_bytes;
    L.staging_total = (uint32_t)staging_bytes(dt, c.swap_ab);
    L.staging_buf_bytes = L.staging_total / 16;
    // MX: each stage also stages the scale atoms of its A rows (bm/128) and B
    // columns (bn/128), bk/128 atoms along K each, and gives them a TMEM slot
    // of 4 columns per atom (tcgen05.cp 32x128b.warpx4 fills 4 columns).
    const int mx_atoms =
        dt == GEMM_MXFP8_E4M3 ? ((pair ? 1 : c.bm / 128) + std::max(1, c.bn / 128)) * (c.bk / 128) : 0;
    L.sf_stage_bytes = (uint32_t)(mx_atoms * kMxAtomBytes);
    L.sc_stage_cols = (uint32_t)(mx_atoms * 4);
    L.off_b = (uint32_t)c.stages * L.a_stage_bytes;
    L.off_sf = L.off_b + (uint32_t)c.stages * L.b_stage_bytes;
    L.off_staging = L.off_sf + (((uint32_t)c.stages * L.sf_stage_bytes + 1023u) & ~1023u);
    L.off_bar = L.off_staging + L.staging_total;
    L.smem_total = L.off_bar + (uint32_t)kAuxSmem;
    L.acc_cols = (uint32_t)((pair ? 1 : c.bm / 128) * c.bn);
    const uint32_t sc_total = (uint32_t)c.stages * L.sc_stage_cols;
    L.n_acc = (2 * L.acc_cols + sc_total <= (uint32_t)kTmemColumns) ? 2u : 1u;
    L.sc_col0 = L.acc_cols * L.n_acc;
    uint32_t need = L.sc_col0 + sc_total, cols = 32;
    while (cols < need) cols <<= 1;
    L.tmem_cols = cols;
    return L;
}

KernelParams kernel_params_of(int64_t M, int64_t N, int64_t K, int dt, int act, const gemm_config &c,
                              bool b_kmajor)
{
    const Layout L = layout_of(c, dt);
    KernelParams k;
    memset(&k, 0, sizeof(k));
    k.rows = (int32_t)(c.swap_ab ? N : M);
    k.cols = (int32_t)(c.swap_ab ? M : N);
    k.K = (int32_t)K;
    k.bm = c.bm;
    k.bn = c.bn;
    k.bk = c.bk;
    k.stages = c.stages;
    k.raster = c.raster;
    k.group = c.group;
    k.split_k = c.split_k;
    k.tiles_m = (int32_t)cdiv(k.rows, c.bm);
    k.tiles_n = (int32_t)cdiv(k.cols, c.bn);
    k.num_kb = (int32_t)cdiv(K, c.bk);
    k.num_units = (int32_t)((int64_t)k.tiles_m * k.tiles_n * c.split_k);
    k.swap_ab = c.swap_ab;
    k.epi = act;
    // User B is N-contiguous (MN-major) unless it is first transposed.  It is
    // MMA-A when swapped and MMA-B otherwise; A is always K-major.
    k.a_mn_major = (c.swap_ab && !b_kmajor) ? 1 : 0;
    k.b_mn_major = (!c.swap_ab && !b_kmajor) ? 1 : 0;
    // Operand formats: BF16 = 1 of kind::f16, TF32 = 2 of kind::tf32, E4M3 = 0 of kind::f8f6f4
    // and of kind::mxf8f6f4.
    const uint32_t fmt = dt == GEMM_BF16 ? 1u : dt == GEMM_FP32_TF32 ? 2u : 0u;
    k.pair = c.cta_group == 2 ? 1 : 0;
    k.alpha = 1.0f;
    const uint32_t mma_m = k.pair ? 256u : 128u;  // a pair's MMA spans both CTAs' 128 rows
    // Instruction descriptor: bits 4-5 the accumulator format (fp32 = 1), 7-9 and
    // 10-12 A's and B's formats, 15 and 16 their majorness, 17-22 N/8, 24-28 M/16.
    // The block-scaled kind has an fp32 accumulator implied and uses bits 4-5
    // (and 29-30) for B's (A's) scale ID, set per MMA; bit 23 = 1 names the
    // scales E8M0.
    const bool mx = dt == GEMM_MXFP8_E4M3;
    k.idesc = (mx ? (1u << 23) : (1u << 4)) | (fmt << 7) | (fmt << 10) | ((uint32_t)k.a_mn_major << 15) |
              ((uint32_t)k.b_mn_major << 16) | ((uint32_t)(c.bn >> 3) << 17) | ((mma_m >> 4) << 24);
    k.a_stage_bytes = L.a_stage_bytes;
    k.b_stage_bytes = L.b_stage_bytes;
    k.tx_bytes = L.stage_bytes + L.sf_stage_bytes;
    k.sf_kt = mx ? (int32_t)mx_k_atoms(K) : 0;
    k.sf_stage_bytes = L.sf_stage_bytes;
    k.off_sf = L.off_sf;
    k.sc_stage_cols = L.sc_stage_cols;
    k.sc_col0 = L.sc_col0;
    k.a_lbo = k.a_mn_major ? (uint32_t)(c.bk * 128) : 16u;
    k.b_lbo = k.b_mn_major ? (uint32_t)(c.bk * 128) : 16u;
    k.acc_cols = L.acc_cols;
    k.n_acc = L.n_acc;
    k.tmem_cols = L.tmem_cols;
    k.off_b = L.off_b;
    k.off_staging = L.off_staging;
    k.off_bar = L.off_bar;
    k.staging_buf_bytes = L.staging_buf_bytes;
    return k;
}

// Whether split-K slices of a tile can reduce through distributed shared
// memory: cluster of S in {2, 4, 8} CTAs, unswapped, and the partials an owner
// receives (its blocks x (S - 1) x 16 KB) fit in its pipeline ring.  Blocks
// (128 rows x 32 columns) are owned in groups of two when there are at least
// 2S of them, else one by one; group j belongs to slice j mod S.
uint32_t cluster_recv_bytes(const gemm_config &c)
{
    const int S = c.split_k;
    // Blocks of 128 rows x 32 columns, or x 16 when swapped, each in a 16 KB
    // slot; a CTA of a pair holds 128 rows of the tile.
    const int halves = c.cta_group == 2 ? 1 : c.bm / 128;
    const int nblocks = halves * (c.swap_ab ? c.bn / 16 : c.bn / 32);
    const int gsz = nblocks >= 2 * S ? 2 : 1;
    const int ngroups = (nblocks + gsz - 1) / gsz;
    const int64_t owned = (int64_t)gsz * ((ngroups + S - 1) / S);
    return (uint32_t)(owned * (S - 1) * (int64_t)kRedBlockBytes);
}

bool cluster_reduce_fits(const gemm_config &c, int dt)
{
    const int S = c.split_k;
    // A cluster holds S CTAs, or S pairs: at most 8 CTAs (the portable size).
    if (!(S == 2 || S == 4 || S == 8) || S * c.cta_group > 8) return false;
    if (c.swap_ab && c.bn > 128) return false;   // up to 8 chunks per half
    const Layout L = layout_of(c, dt);
    return cluster_recv_bytes(c) <= L.off_staging;
}

// The most stages (at most kMaxStages) whose layout fits in shared memory, by
// the same count as the feasibility rule (the MX scale area rounded up to 1 KB).
int max_stages_for(int bm, int bn, int bk, int dt, int swap_ab, int64_t smem_per_block, int cta_group)
{
    for (int s = kMaxStages; s >= 1; --s) {
        const gemm_config c{bm, bn, bk, s, 0, 1, 1, cta_group, swap_ab};
        if ((int64_t)layout_of(c, dt).smem_total <= smem_per_block) return s;
    }
    return 0;
}

const char *reason_text(int r)
{
    switch (r) {
    case GEMM_FEASIBLE: return "feasible";
    case GEMM_REASON_CTA_GROUP: return "cta_group must be 1, or 2 with bm = 256 and no swap";
    case GEMM_REASON_UMMA_M: return "bm must be 128 or 256 (tcgen05 M per CTA is 128)";
    case GEMM_REASON_UMMA_N: return "bn must be a multiple of 16 in [16, 256]";
    case GEMM_REASON_LAYOUT:
        return "bn must be a multiple of 32 and of the 128-byte span when B is MN-major (a CTA pair: bn/2 a "
               "multiple of the span; block-scaled FP8: bn 128 or 256, or swapped a multiple of 128 or >= M; "
               "gated epilogues: unswapped, split_k 1, bn and N multiples of 64)";
    case GEMM_REASON_BK: return "bk must be 1..4 spans of 128 bytes (block-scaled FP8: 128 or 256)";
    case GEMM_REASON_STAGES: return "stages must be in 2..16";
    case GEMM_REASON_SCHEDULE: return "raster must be 0/1 and group one of 1,2,4,8,16";
    case GEMM_REASON_SPLIT_K: return "split_k must be in 1..16 and at most ceil(K/bk)";
    case GEMM_REASON_ALIGN: return "K*elt and N*elt must be multiples of 16 bytes (TMA row stride)";
    case GEMM_REASON_TMEM: return "one accumulator (block-scaled FP8: plus the scale slots) needs more than 512 TMEM columns";
    case GEMM_REASON_SMEM: return "ring + staging + barriers exceed the shared-memory limit";
    case GEMM_REASON_REGS: return "kernel registers x threads exceed the register file";
    default: return "unknown reason";
    }
}

int check_config(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &c,
                 const gemm_device_params &d)
{
    const int e = elt_bytes(dt);
    const int span = span_elems(dt);
    if (c.cta_group != 1 && c.cta_group != 2) return GEMM_REASON_CTA_GROUP;
    if (c.cta_group == 2 && (c.bm != 256 || c.swap_ab != 0)) return GEMM_REASON_CTA_GROUP;
    if (c.bm != 128 && c.bm != 256) return GEMM_REASON_UMMA_M;
    if (c.bn % 16 != 0 || c.bn < 16 || c.bn > 256) return GEMM_REASON_UMMA_N;
    if (c.swap_ab != 0 && c.swap_ab != 1) return GEMM_REASON_LAYOUT;
    // B columns come in units of the MN-major swizzle span when B is read in
    // place; a K-major copy of B needs only the epilogue's 32-column chunks.
    const int b_unit = b_in_place(dt, N) ? span : 32;
    if (c.swap_ab == 0 && (c.bn % b_unit != 0 || c.bn % 32 != 0)) return GEMM_REASON_LAYOUT;
    if (c.cta_group == 2 && (c.bn / 2) % b_unit != 0) return GEMM_REASON_LAYOUT;
    // MX: the scales of a tile's MMA-N columns come in whole 128-column atoms, so
    // an unswapped tile has bn 128 or 256, and a swapped one (tokens along N)
    // starts every tile on an atom: bn a multiple of 128, or all of M in one tile.
    if (dt == GEMM_MXFP8_E4M3 && c.swap_ab == 0 && c.bn != 128 && c.bn != 256) return GEMM_REASON_LAYOUT;
    if (dt == GEMM_MXFP8_E4M3 && c.swap_ab == 1 && c.bn % 128 != 0 && M > c.bn) return GEMM_REASON_LAYOUT;
    // Gated epilogues: a tile holds whole 64-column gate+up block pairs of the
    // fused weight and drains them in one pass (unswapped, no split-K).
    if (is_glu(epi) && (c.swap_ab != 0 || c.split_k != 1 || c.bn % 64 != 0 || N % 64 != 0))
        return GEMM_REASON_LAYOUT;
    if (c.bk % span != 0 || c.bk / span < 1 || c.bk / span > 4) return GEMM_REASON_BK;
    if (dt == GEMM_MXFP8_E4M3 && c.bk != 128 && c.bk != 256) return GEMM_REASON_BK;
    if (c.stages < 2 || c.stages > kMaxStages) return GEMM_REASON_STAGES;
    if ((c.raster != 0 && c.raster != 1) ||
        !(c.group == 1 || c.group == 2 || c.group == 4 || c.group == 8 || c.group == 16))
        return GEMM_REASON_SCHEDULE;
    const int64_t num_kb = cdiv(K, c.bk);
    if (c.split_k < 1 || c.split_k > kMaxSplitK || c.split_k > std::max<int64_t>(1, num_kb))
        return GEMM_REASON_SPLIT_K;
    if ((K * e) % 16 != 0 || (N * out_elt_bytes(dt)) % 16 != 0 || (b_in_place(dt, N) && (N * e) % 16 != 0))
        return GEMM_REASON_ALIGN;
    const Layout L = layout_of(c, dt);
    if (L.sc_col0 + (uint32_t)c.stages * L.sc_stage_cols > (uint32_t)kTmemColumns) return GEMM_REASON_TMEM;
    if ((int64_t)L.smem_total > d.smem_per_block) return GEMM_REASON_SMEM;
    if (d.kernel_regs > 0 && (int64_t)d.kernel_regs * d.threads_per_cta > 65536) return GEMM_REASON_REGS;
    return GEMM_FEASIBLE;
}

std::vector<gemm_config> enumerate(int64_t M, int64_t N, int64_t K, int dt, int epi,
                                   const gemm_device_params &d)
{
    static const int kSplits[] = {2, 3, 4, 6, 8, 12, 16};
    static const int kGroups[] = {1, 4, 8, 16};
    std::vector<gemm_config> out;
    const int span = span_elems(dt);
    const int nswap = (M <= 256) ? 2 : 1;
    for (int swap = 0; swap < nswap; ++swap) {
        const int64_t rows = swap ? N : M, cols = swap ? M : N;
        // (bm, cta_group): single-CTA tiles of 128 or 256 rows, and 256-row tiles
        // on a CTA pair (unswapped only).
        const std::pair<int, int> shapes[] = {{128, 1}, {256, 1}, {256, 2}};
        for (const auto &shape : shapes) {
            const int bm = shape.first, cg = shape.second;
            if (cg == 2 && swap) continue;
            std::vector<int> bns;
            if (swap) bns = {16, 32, 64, 128, 256};
            else if (cg == 2) bns = dt == GEMM_BF16                  ? std::vector<int>{128, 256}
                                    : (is_fp8(dt) && b_in_place(dt, N)) ? std::vector<int>{256}
                                    : dt == GEMM_MXFP8_E4M3             ? std::vector<int>{128, 256}
                                                                        : std::vector<int>{64, 128, 256};
            else if (dt == GEMM_BF16) bns = {64, 128, 192, 256};
            else if (dt == GEMM_FP8_E4M3) bns = b_in_place(dt, N) ? std::vector<int>{128, 256}
                                                                  : std::vector<int>{64, 128, 192, 256};
            else if (dt == GEMM_MXFP8_E4M3) bns = {128, 256};
            else bns = {32, 64, 128, 192, 256};
            for (int bn : bns) {
                for (int bk : {span, 2 * span}) {
                    const int st_max = max_stages_for(bm, bn, bk, dt, swap, d.smem_per_block, cg);
                    if (st_max < 2) continue;
                    std::vector<int> stage_list = {std::min(4, st_max)};
                    if (st_max != stage_list[0]) stage_list.push_back(st_max);
                    // CTAs per tile: cg.  Split-K and raster variants are judged by CTA counts.
                    const int64_t tiles = cdiv(rows, bm) * cdiv(cols, bn);
                    const int64_t num_kb = cdiv(K, bk);
                    std::vector<int> splits;
                    if (tiles * cg < 4LL * d.sm_count)
                        for (int s : kSplits)
                            if (2LL * s <= num_kb && tiles * s * cg <= 16LL * d.sm_count) splits.push_back(s);
                    std::vector<std::pair<int, int>> scheds = {{0, 1}};
                    if (tiles * cg > d.sm_count) {
                        scheds.clear();
                        for (int r = 0; r < 2; ++r)
                            for (int g : kGroups) scheds.push_back({r, g});
                    }
                    struct Combo { int raster, group, split; };
                    std::vector<Combo> combos;
                    for (auto &s : scheds) combos.push_back({s.first, s.second, 1});
                    for (int s : splits) combos.push_back({0, 1, s});
                    for (int st : stage_list) {
                        for (const Combo &cb : combos) {
                            gemm_config c{bm, bn, bk, st, cb.raster, cb.group, cb.split, cg, swap};
                            if (check_config(M, N, K, dt, epi, c, d) == GEMM_FEASIBLE) out.push_back(c);
                        }
                    }
                }
            }
        }
    }
    return out;
}

gemm_config fixed_config(int dt, const gemm_device_params &d)
{
    const int span = span_elems(dt);
    gemm_config c{128, 128, span, max_stages_for(128, 128, span, dt, 0, d.smem_per_block, 1), 0, 1, 1, 1, 0};
    return c;
}

// ---------------------------------------------------------------------------
// Cost model
// ---------------------------------------------------------------------------

static gemm_model_terms predict_workshop(int64_t M, int64_t N, int64_t K, int dt, const gemm_config &c,
                                         const gemm_device_params &d)
{
    // "Compilers and Kernel Languages", workshop paragraph.  The tile-efficiency
    // law 0.5 + 0.5·min(1, bm·bn/128²) is the reading that reproduces the page's
    // printed ratios; g = √min(tiles, SMs).
    gemm_model_terms t;
    memset(&t, 0, sizeof(t));
    const double e = elt_bytes(dt);
    const int64_t tiles = cdiv(M, c.bm) * cdiv(N, c.bn);
    const int64_t waves = cdiv(tiles, d.sm_count);
    const double weff = (double)tiles / ((double)waves * d.sm_count);
    const double teff = 0.5 + 0.5 * std::min(1.0, (double)c.bm * c.bn / (128.0 * 128.0));
    const double flops = 2.0 * (double)M * (double)N * (double)K;
    const double compute = flops / (d.peak_tflops_bf16 * 1e12) / weff / teff;
    const double g = sqrt((double)std::min<int64_t>(tiles, d.sm_count));
    const double panel = (double)tiles * K * (c.bm + c.bn) * e / g + (double)M * N * e;
    const double floor_b = ((double)M * K + (double)K * N + (double)M * N) * e;
    const double bytes = std::max(panel, floor_b);
    const double memory = bytes / (d.hbm_gbs * 1e9);
    t.mma_us = compute * 1e6;
    t.hbm_us = memory * 1e6;
    t.predicted_us = std::max(compute, memory) * 1e6;
    t.wave_eff = weff;
    t.tile_eff = teff;
    t.pad_eff = 1.0;
    t.hbm_bytes = bytes;
    t.flops = flops;
    t.tiles = tiles;
    t.units = tiles;
    t.waves = waves;
    t.ctas = std::min<int64_t>(tiles, d.sm_count);
    return t;
}

gemm_model_terms predict(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &c,
                         const gemm_device_params &d)
{
    if (d.model_kind == 1) return predict_workshop(M, N, K, dt, c, d);
    gemm_model_terms t;
    memset(&t, 0, sizeof(t));
    const double e = elt_bytes(dt);
    const int64_t rows = c.swap_ab ? N : M, cols = c.swap_ab ? M : N;
    const int64_t tiles_m = cdiv(rows, c.bm), tiles_n = cdiv(cols, c.bn);
    const int64_t tiles = tiles_m * tiles_n;
    const int64_t S = c.split_k;
    const int64_t num_kb = cdiv(K, c.bk);
    const int64_t units = tiles * S;
    const int64_t sms = d.sm_count;
    // A CTA pair (cta_group 2) runs each unit on two CTAs, each holding 128 rows
    // of the tile and loading half of B's columns.
    const int64_t cg = c.cta_group == 2 ? 2 : 1;
    const int64_t rows_cta = cg == 2 ? 128 : c.bm;
    const int64_t bcols_cta = cg == 2 ? c.bn / 2 : c.bn;
    const int64_t cta_units = units * cg;
    int64_t ctas = std::max<int64_t>(cg, std::min(cta_units, sms));
    if (cg == 2) ctas &= ~(int64_t)1;
    const int64_t waves = cdiv(cta_units, sms);
    const int64_t upc = cdiv(units, ctas / cg);      // units of the busiest CTA
    const int64_t kbu = cdiv(num_kb, S);             // K-blocks of the longest slice
    const double clk = d.sm_clock_mhz * 1e6;
    const double flops = 2.0 * (double)M * (double)N * (double)K;

    // Tensor pipe, per K-block of one CTA: the MMAs execute at the per-SM share
    // of the peak, and the issuing warp spends mma_issue_clk per MMA plus
    // kblock_clk per stage; the slower of the two sets the pace.
    const double peak =
        (dt == GEMM_BF16 ? d.peak_tflops_bf16 : is_fp8(dt) ? d.peak_tflops_fp8 : d.peak_tflops_tf32) * 1e12;
    const double halves = cg == 2 ? 1 : c.bm / 128, ksteps = (double)c.bk * e / 32.0, kslice = 32.0 / e;
    const double mma_flop = 2.0 * 128.0 * c.bn * kslice;
    const double t_exec = halves * ksteps * mma_flop / (peak / (double)sms);
    const double t_issue = (halves * ksteps * d.mma_issue_clk + d.kblock_clk) / clk;
    const double t_mma = (double)upc * (double)kbu * std::max(t_exec, t_issue);

    // L2 -> shared memory: every unit streams (bm + bn)·bk·elt bytes per K-block
    // ("Tile Selection": per-block panel traffic; reuse across blocks is in L2).
    // (MX: plus 4 scale bytes per row and column per 128 K.)
    const double sf_per_k = dt == GEMM_MXFP8_E4M3 ? 4.0 / 128.0 : 0.0;
    const double l2_bytes =
        (double)cta_units * (double)kbu * (double)(rows_cta + bcols_cta) * (double)c.bk * (e + sf_per_k);
    const double t_l2 = l2_bytes / (d.l2_gbs * 1e9);

    // HBM: operands either fit in half of L2 (threshold regime: compulsory bytes
    // only) or are re-read once per wave of concurrent tiles, with the wave's
    // footprint shaped by the tile order (group-G band).
    const double in_bytes = ((double)M * K + (double)K * N) * (e + sf_per_k);
    const int64_t wave_tiles = std::min<int64_t>(tiles, std::max<int64_t>(1, ctas / cg / S));
    int64_t rows_w, cols_w;
    if (c.raster == 0) {
        rows_w = std::min<int64_t>(std::min<int64_t>(c.group, tiles_m), wave_tiles);
        cols_w = std::min<int64_t>(cdiv(wave_tiles, rows_w), tiles_n);
    } else {
        cols_w = std::min<int64_t>(std::min<int64_t>(c.group, tiles_n), wave_tiles);
        rows_w = std::min<int64_t>(cdiv(wave_tiles, cols_w), tiles_m);
    }
    const double panel = ((double)tiles / (double)wave_tiles) * (double)K *
                         ((double)rows_w * c.bm + (double)cols_w * c.bn) * (e + sf_per_k);
    const double operand = (in_bytes <= (double)d.l2_bytes / 2.0) ? in_bytes : std::max(in_bytes, panel);
    // C (half the fused width for the gated epilogues), bias, and the residual
    // R of the "+ R" epilogues.
    const double eo = out_elt_bytes(dt);
    const double c_cols = is_glu(epi) ? (double)(N / 2) : (double)N;
    const double hbm = operand + (double)M * c_cols * eo + (epi != GEMM_EPI_NONE ? (double)N * eo : 0.0) +
                       (is_residual(epi) ? (double)M * N * eo : 0.0);
    const double t_hbm = hbm / (d.hbm_gbs * 1e9);

    // Bytes in flight ("Tiling the hierarchy", double buffering): the ring
    // covers one load latency per `stages` K-blocks.
    const double t_lat = (double)upc * (double)kbu * d.mem_latency_us * 1e-6 / c.stages;
    const double t_main = std::max(std::max(t_mma, t_l2), std::max(t_hbm, t_lat));

    // Epilogue and split-K exchange.
    const bool gelu = epi == GEMM_EPI_BIAS_GELU || epi == GEMM_EPI_BIAS_GELU_RESIDUAL ||
                      epi == GEMM_EPI_BIAS_GEGLU || epi == GEMM_EPI_BIAS_SWIGLU;
    const double rate = (gelu ? d.epi_gelu_elems_per_clk : d.epi_elems_per_clk) * clk;
    const double elems = (double)rows_cta * c.bn;   // one CTA's share of a tile
    const double part = elems * 4.0;
    double exposed, t_split;
    if (S == 1) {
        // Double-buffered accumulators hide the epilogue behind the next unit's
        // main loop unless it is the slower of the two.
        const double epi_t = elems / rate;
        const bool two_acc = layout_of(c, dt).n_acc == 2;
        const double main_unit = t_main / (double)upc;
        exposed = epi_t + (double)(upc - 1) * (two_acc ? std::max(0.0, epi_t - main_unit) : epi_t);
        t_split = 0.0;
    } else if (cta_units <= sms) {
        // Cooperative fix-up: each slice keeps its own share of the tile in TMEM,
        // writes the other (S-1)/S and reads (S-1) partials of its share.
        exposed = elems / (double)S / rate;
        t_split = 2.0 * part * (double)(S - 1) / (double)S / (d.splitk_gbs * 1e9);
    } else {
        // Last arriver: the CTA finishing a tile reads all S partials.
        const double fix_tiles = (double)cdiv(tiles * cg, ctas);
        exposed = fix_tiles * elems / rate;
        t_split = ((double)upc + fix_tiles * (double)S) * part / (d.splitk_gbs * 1e9);
    }
    const double total = t_main + exposed + t_split + d.launch_us * 1e-6;

    t.predicted_us = total * 1e6;
    t.mma_us = t_mma * 1e6;
    t.l2_us = t_l2 * 1e6;
    t.hbm_us = t_hbm * 1e6;
    t.latency_us = t_lat * 1e6;
    t.epilogue_us = exposed * 1e6;
    t.splitk_us = t_split * 1e6;
    t.launch_us = d.launch_us;
    t.wave_eff = (double)cta_units / ((double)waves * (double)sms);
    t.tile_eff = t_exec / std::max(t_exec, t_issue);
    t.pad_eff = K > 0 ? ((double)rows * cols * K) /
                            ((double)tiles_m * c.bm * (double)tiles_n * c.bn * (double)num_kb * c.bk)
                      : 1.0;
    t.hbm_bytes = hbm;
    t.l2_bytes = l2_bytes;
    t.flops = flops;
    t.tiles = tiles;
    t.units = units;
    t.waves = waves;
    t.ctas = ctas;
    return t;
}

// ---------------------------------------------------------------------------
// Shipped configuration set
// ---------------------------------------------------------------------------

// Greedy choice of a small configuration set from a measured table
// t[shape * n_configs + config] (<= 0: the configuration does not run the
// shape).  The set's quality is the sum over shapes of best_s / (the set's
// fastest time on s), zero where no member runs s; each step adds the
// configuration with the largest gain (the lowest index among equal gains)
// until max_set members are chosen or nothing gains.  The quality is monotone
// and submodular in the set, so the greedy set is within (1 - 1/e) of the best
// set of its size.
int select_config_set(const double *t, int ns, int nc, int max_set, int32_t *chosen, int32_t *n_chosen,
                      double *mean_slowdown, double *worst_slowdown)
{
    std::vector<double> best(ns, 0.0), cur(ns, 0.0);
    for (int s = 0; s < ns; ++s) {
        double b = 0.0;
        for (int c = 0; c < nc; ++c) {
            const double v = t[(size_t)s * nc + c];
            if (v > 0.0 && (b == 0.0 || v < b)) b = v;
        }
        best[s] = b;
    }
    auto quality = [&](int s, int c) {
        const double v = t[(size_t)s * nc + c];
        return (v > 0.0 && best[s] > 0.0) ? best[s] / v : 0.0;
    };
    std::vector<char> used(nc, 0);
    int k = 0;
    while (k < max_set) {
        double best_gain = 0.0;
        int pick = -1;
        for (int c = 0; c < nc; ++c) {
            if (used[c]) continue;
            double gain = 0.0;
            for (int s = 0; s < ns; ++s) gain += std::max(0.0, quality(s, c) - cur[s]);
            if (gain > best_gain) {
                best_gain = gain;
                pick = c;
            }
        }
        if (pick < 0) break;
        used[pick] = 1;
        chosen[k++] = pick;
        for (int s = 0; s < ns; ++s) cur[s] = std::max(cur[s], quality(s, pick));
    }
    *n_chosen = k;
    double sum = 0.0, worst = 0.0;
    int counted = 0;
    for (int s = 0; s < ns; ++s) {
        if (best[s] <= 0.0) continue;
        const double slow = cur[s] > 0.0 ? 1.0 / cur[s] : HUGE_VAL;
        sum += slow;
        worst = std::max(worst, slow);
        ++counted;
    }
    if (mean_slowdown) *mean_slowdown = counted ? sum / counted : 1.0;
    if (worst_slowdown) *worst_slowdown = counted ? worst : 1.0;
    return GEMM_OK;
}

// ---------------------------------------------------------------------------
// Rank agreement
// ---------------------------------------------------------------------------

static std::vector<double> average_ranks(const double *v, int n)
{
    std::vector<int> idx(n);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return v[a] < v[b]; });
    std::vector<double> r(n);
    for (int i = 0; i < n;) {
        int j = i;
        while (j + 1 < n && v[idx[j + 1]] == v[idx[i]]) ++j;
        const double avg = 0.5 * (i + j) + 1.0;
        for (int t = i; t <= j; ++t) r[idx[t]] = avg;
        i = j + 1;
    }
    return r;
}

gemm_rank_stats rank_agreement(const double *x, const double *y, int n)
{
    gemm_rank_stats s;
    memset(&s, 0, sizeof(s));
    int64_t conc = 0, disc = 0, tx = 0, ty = 0;
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j) {
            const int dx = (x[i] > x[j]) - (x[i] < x[j]);
            const int dy = (y[i] > y[j]) - (y[i] < y[j]);
            if (dx == 0 && dy == 0) continue;
            if (dx == 0) ++tx;
            else if (dy == 0) ++ty;
            else if (dx == dy) ++conc;
            else ++disc;
        }
    const double den = sqrt((double)(conc + disc + tx) * (double)(conc + disc + ty));
    s.kendall_tau = den > 0 ? (double)(conc - disc) / den : NAN;
    const std::vector<double> rx = average_ranks(x, n), ry = average_ranks(y, n);
    double mx = 0, my = 0;
    for (int i = 0; i < n; ++i) {
        mx += rx[i];
        my += ry[i];
    }
    mx /= n;
    my /= n;
    double sxy = 0, sxx = 0, syy = 0;
    for (int i = 0; i < n; ++i) {
        sxy += (rx[i] - mx) * (ry[i] - my);
        sxx += (rx[i] - mx) * (rx[i] - mx);
        syy += (ry[i] - my) * (ry[i] - my);
    }
    s.spearman_rho = (sxx > 0 && syy > 0) ? sxy / sqrt(sxx * syy) : NAN;
    int pick = 0, best = 0;
    for (int i = 1; i < n; ++i) {
        if (x[i] < x[pick]) pick = i;
        if (y[i] < y[best]) best = i;
    }
    s.top1_hit = y[pick] == y[best] ? 1 : 0;
    s.regret = y[pick] / y[best] - 1.0;
    s.best_us = y[best];
    s.n_measured = n;
    s.fixed_us = -1.0;
    return s;
}

}  // namespace gemmgb
