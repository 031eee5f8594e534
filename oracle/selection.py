"""Oracle for the selection layer: candidate spaces, wave arithmetic, cost models,
schedule order and rank agreement — plain Python, one function per idea.

TEST INFRASTRUCTURE ONLY: imported by tests/ (and nothing in the product).

Sources (page title, section / equation):
  * "Tile Selection: Cost Models Against Measurement"
      - "The structure of the search space": the candidate enumerator, the
        48 KB shared-memory cap of 12,288 fp32 panel elements.
      - "Analytical models and where they break": per-block traffic
        4K(BM+BN) bytes, 2·BM·BN·K operations, intensity BM·BN/(2(BM+BN)).
  * "Compilers and Kernel Languages" (workshop paragraph and "A different tile
    for every shape"): waves of one tile per multiprocessor, the H100 workshop
    model and its printed results.
  * "Tiling the hierarchy", square-tile derivation: traffic 2N³/T with
    T = √(C/3); the double-buffering discussion (stages hide latency).
  * "Autotuning & cost models", §6: cost-model-guided search vs measurement;
    rank agreement is how the model's ordering is judged against measurement.

Parity status of each function is stated in its docstring.  The GB300 rules
(`gb300_*`) restate the library's documented feasibility rules, enumeration and
cost model independently of the library source.  What the pages fix in them is
pinned (tests/test_oracle_gb300_pins.py, each pin with a planted mistake it
catches): gb300_model's panel bytes equal the per-block traffic law of "Tile
Selection" ("Analytical models and where they break") summed over tiles; its
waves and wave efficiency equal the wave arithmetic of "Compilers and Kernel
Languages" on CTAs (tiles x slices x CTAs per tile); no prediction beats the
roofline floor; its HBM bytes are the compulsory bytes when A and B fit in half
of L2; gb300_candidates equals a brute-force filter of its documented grid and
holds the fixed tile ("CuTile Autotuning").  The rest is "parity unpinned"
against the pages, which say nothing about TMEM or tcgen05: the feasibility
rules themselves (pinned only by brute force and by set-equality with the
library) and the fitted coefficients of the GB300 cost model (judged by rank
agreement with measurement; the model also reduces to the workshop model).
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

# ---------------------------------------------------------------------------
# "Tile Selection", "The structure of the search space": the fp32 SIMT enumerator
# ---------------------------------------------------------------------------

P1_BLOCK = (32, 64, 128, 256)
P1_KSTEP = (8, 16, 32, 64)
P1_THREAD = (2, 4, 8)


def p1_candidates(M, N, K, smem_bytes=48 * 1024, max_threads=1024):
    """All (BM, BN, KS, TM, TN) the page's enumerator accepts, in its loop order.

    Rules (page: "The structure of the search space"): both fp32 panels fit in
    shared memory, 4·(BM·KS + KS·BN) <= smem; the block has between 32 and
    max_threads threads, (BM/TM)·(BN/TN); whole warps; TM·TN <= 128 accumulators.
    The problem extents do not enter the rules (the page's listing ignores them).
    Pinned by: the 12,288-element cap the page prints for 48 KB, the "few hundred
    to a few thousand" count it states, and brute-force rule checks in tests."""
    del M, N, K
    out = []
    for bm, bn, ks, tm, tn in itertools.product(P1_BLOCK, P1_BLOCK, P1_KSTEP,
                                                P1_THREAD, P1_THREAD):
        panel_bytes = 4 * ks * (bm + bn)
        nthreads = (bm // tm) * (bn // tn)
        ok = (panel_bytes <= smem_bytes
              and 32 <= nthreads <= max_threads
              and nthreads % 32 == 0
              and tm * tn <= 128)
        if ok:
            out.append((bm, bn, ks, tm, tn))
    return out


def p1_panel_cap_elements(smem_bytes=48 * 1024):
    """Largest BM·KS + KS·BN that fits as fp32: smem / 4 (12,288 at 48 KB)."""
    return smem_bytes // 4


# ---------------------------------------------------------------------------
# Wave arithmetic ("Compilers and Kernel Languages": tiles run in waves of one
# per multiprocessor; 133 tiles on 132 take two waves)
# ---------------------------------------------------------------------------

def ceil_div(a, b):
    return -(-a // b)


def tile_count(M, N, bm, bn):
    return ceil_div(M, bm) * ceil_div(N, bn)


def waves(units, sms):
    return ceil_div(units, sms)


def wave_efficiency(units, sms):
    """Fraction of multiprocessor-slots busy over the waves the units need."""
    return units / (waves(units, sms) * sms)


# ---------------------------------------------------------------------------
# "Tile Selection", "Analytical models and where they break"
# ---------------------------------------------------------------------------

def block_traffic_bytes(bm, bn, K, elt=4):
    """Bytes one block moves over the full depth: K·(BM+BN)·elt (4K(BM+BN) for fp32)."""
    return K * (bm + bn) * elt


def block_ops(bm, bn, K):
    return 2 * bm * bn * K


def block_intensity(bm, bn, K, elt=4):
    """Operations per byte of one block; for fp32 it equals BM·BN/(2(BM+BN))."""
    return block_ops(bm, bn, K) / block_traffic_bytes(bm, bn, K, elt)


def roofline_time(M, N, K, bm, bn, peak_flops, bw, elt=4):
    """The page's simplest model: max(ops/peak, grid traffic/bandwidth) with no
    panel sharing between blocks."""
    grid_bytes = tile_count(M, N, bm, bn) * block_traffic_bytes(bm, bn, K, elt)
    return max(2 * M * N * K / peak_flops, grid_bytes / bw)


# ---------------------------------------------------------------------------
# "Tiling the hierarchy": square tiles at one level of capacity C (elements)
# ---------------------------------------------------------------------------

def square_tile_side(capacity_elems):
    """Three resident T×T tiles: 3T² <= C, so T = √(C/3)."""
    return math.sqrt(capacity_elems / 3.0)


def square_tile_traffic_law(Nn, T):
    """Closed form 2N³/T (elements read)."""
    return 2 * Nn ** 3 / T


def square_tile_traffic_count(Nn, T):
    """Explicit count: walk the (N/T)³ tile triples, each reading one A tile and
    one B tile of T² elements."""
    assert Nn % T == 0
    nt = Nn // T
    total = 0
    for _i in range(nt):
        for _j in range(nt):
            for _k in range(nt):
                total += T * T  # A[i,k]
                total += T * T  # B[k,j]
    return total


def double_buffer_load_ns(tile_bytes, bw_bytes_per_s, capacity_factor=1.0):
    """Bandwidth time of one tile load; halving reuse capacity multiplies traffic
    by √2 ("Tiling the hierarchy", double-buffering discussion)."""
    return tile_bytes / bw_bytes_per_s * 1e9 * capacity_factor


# ---------------------------------------------------------------------------
# "Compilers and Kernel Languages": the H100 workshop model
# ---------------------------------------------------------------------------

@dataclass
class WorkshopDevice:
    sms: int = 132
    smem_bytes: int = 228 * 1024
    peak_flops: float = 989e12
    bw: float = 3.35e12
    elt: int = 2          # BF16 operands
    bk: int = 64


WORKSHOP_TILES = (32, 64, 128, 256)


def workshop_tile_efficiency(bm, bn):
    """Reading: the page says only that tile efficiency "falls for tiles smaller
    than 128 × 128"; the simplest law that reproduces both printed ratios
    (1.83× and 1.50×) is 0.5 + 0.5·min(1, bm·bn/128²)."""
    return 0.5 + 0.5 * min(1.0, bm * bn / (128 * 128))


def workshop_time(M, N, K, bm, bn, dev: WorkshopDevice = WorkshopDevice()):
    """Modelled time (seconds) of one bm × bn tile shape.

    compute = 2MNK / peak / wave efficiency / tile efficiency;
    memory  = max(panel traffic / g + C bytes, compulsory bytes) / bandwidth, where
              g = √(tiles sharing panels in one wave) = √min(tiles, SMs);
    time    = max(compute, memory).
    Pinned by the page's printed results (tests/golden/workshop_h100.json)."""
    t = tile_count(M, N, bm, bn)
    compute = 2.0 * M * N * K / dev.peak_flops / wave_efficiency(t, dev.sms) \
        / workshop_tile_efficiency(bm, bn)
    g = math.sqrt(min(t, dev.sms))
    panel = t * K * (bm + bn) * dev.elt / g + M * N * dev.elt
    floor = (M * K + K * N + M * N) * dev.elt
    memory = max(panel, floor) / dev.bw
    return max(compute, memory)


def workshop_sweep(M, N, K, dev: WorkshopDevice = WorkshopDevice()):
    """Every (bm, bn) with its time; best = first minimum in bm-outer, bn-inner
    order (reading: the page's tie-break between equal times)."""
    times = {}
    for bm in WORKSHOP_TILES:
        for bn in WORKSHOP_TILES:
            times[(bm, bn)] = workshop_time(M, N, K, bm, bn, dev)
    best = None
    for key, val in times.items():
        if best is None or val < times[best]:
            best = key
    worst = max(times, key=lambda k: times[k])
    return {"times": times, "best": best, "worst": worst,
            "best_s": times[best], "worst_s": times[worst],
            "fixed_128": times[(128, 128)]}


# ---------------------------------------------------------------------------
# GB300 restatement of the library's documented rules.  The generator is pinned
# by a brute-force filter of its grid; the TMEM/tcgen05 rules themselves are
# parity unpinned against the pages, which say nothing about them.
# ---------------------------------------------------------------------------

DT_BF16, DT_FP32, DT_FP8, DT_MXFP8 = 0, 1, 2, 3
EPI_NONE, EPI_BIAS, EPI_RELU, EPI_GELU = 0, 1, 2, 3
EPI_BIAS_RES, EPI_RELU_RES, EPI_GELU_RES = 4, 5, 6   # the same plus a residual R
EPI_REGLU, EPI_GEGLU, EPI_SWIGLU = 7, 8, 9          # gated: act(gate) ⊙ up over a fused [K, N] weight, C [M, N/2]


def is_glu(epi):
    return epi in (EPI_REGLU, EPI_GEGLU, EPI_SWIGLU)

R_OK, R_CTA_GROUP, R_UMMA_M, R_UMMA_N, R_LAYOUT, R_BK, R_STAGES, R_SCHEDULE, \
    R_SPLIT_K, R_ALIGN, R_TMEM, R_SMEM, R_REGS = range(13)

THREADS_PER_CTA = 320
TMEM_COLUMNS = 512
AUX_SMEM = 2048            # barriers/flags (1 KB) + 1 KB alignment slack
MAX_STAGES = 16
SPLITS = (2, 3, 4, 6, 8, 12, 16)
GROUPS = (1, 2, 4, 8, 16)


@dataclass
class Config:
    bm: int
    bn: int
    bk: int
    stages: int
    raster: int = 0
    group: int = 1
    split_k: int = 1
    cta_group: int = 1
    swap_ab: int = 0

    def astuple(self):
        return (self.bm, self.bn, self.bk, self.stages, self.raster, self.group,
                self.split_k, self.cta_group, self.swap_ab)


@dataclass
class Device:
    """Mirror of the library's device-parameter record, field by field."""
    sm_count: int = 152
    model_kind: int = 0
    smem_per_block: int = 232448
    l2_bytes: int = 129 * 1024 * 1024
    peak_tflops_bf16: float = 1889.6
    peak_tflops_tf32: float = 944.8
    peak_tflops_fp8: float = 3779.2
    hbm_gbs: float = 6675.8
    sm_clock_mhz: float = 2070.0
    l2_gbs: float = 14888.0
    mma_issue_clk: float = 39.53
    kblock_clk: float = 483.2
    mem_latency_us: float = 1.375
    epi_elems_per_clk: float = 3.632
    epi_gelu_elems_per_clk: float = 5.109
    splitk_gbs: float = 15.99
    launch_us: float = 7.50
    kernel_regs: int = 0
    threads_per_cta: int = THREADS_PER_CTA
    extra: dict = field(default_factory=dict)


def is_fp8(dtype):
    """FP8 E4M3 operands, with one tensor scale or block-scaled (MX)."""
    return dtype in (DT_FP8, DT_MXFP8)


def elt_bytes(dtype):
    """Operand element size: bf16 2, FP8 E4M3 (plain or MX) 1, fp32 4."""
    return 2 if dtype == DT_BF16 else 1 if is_fp8(dtype) else 4


def b_in_place(dtype, N):
    """B read MN-major in place: bf16 always, FP8 when its rows (N bytes) meet
    the 16-byte stride rule; otherwise from a K-major copy (fp32 always)."""
    return dtype == DT_BF16 or (is_fp8(dtype) and N % 16 == 0)


MX_ATOM_BYTES = 512     # 128 rows x four 32-element scale blocks


def mx_atoms(cfg: Config, dtype):
    """Scale atoms one MX stage stages: A's bm/128 row atoms and B's bn/128
    column atoms, bk/128 of each along K (zero for other dtypes)."""
    if dtype != DT_MXFP8:
        return 0
    a_atoms = 1 if cfg.cta_group == 2 else cfg.bm // 128     # a pair: each CTA holds 128 rows
    return (a_atoms + max(1, cfg.bn // 128)) * (cfg.bk // 128)


def out_elt_bytes(dtype):
    """Size of C, bias and R: FP8 operands produce bf16."""
    return 4 if dtype == DT_FP32 else 2


def span_elems(dtype):
    """Elements of one 128-byte swizzle span along the contiguous dimension."""
    return 128 // elt_bytes(dtype)


def staging_bytes(dtype, swap_ab):
    """Epilogue staging: 8 epilogue warps × 2 buffers × one store chunk
    (32 rows × 32 columns, or 16 token rows × 32 columns when swapped)."""
    rows = 16 if swap_ab else 32
    return 8 * 2 * rows * 32 * out_elt_bytes(dtype)


def cta_share(cfg: Config):
    """(A rows, B columns) one CTA stages: a CTA pair (cta_group 2) splits a
    256-row tile into 128 rows of A per CTA and halves B's columns."""
    if cfg.cta_group == 2:
        return 128, cfg.bn // 2
    return cfg.bm, cfg.bn


def stage_bytes(cfg: Config, dtype):
    a_rows, b_cols = cta_share(cfg)
    return (a_rows + b_cols) * cfg.bk * elt_bytes(dtype)


def smem_bytes(cfg: Config, dtype):
    """Ring (operands, then the MX scale atoms rounded up to 1 KB) + epilogue
    staging + barriers."""
    scales = cfg.stages * mx_atoms(cfg, dtype) * MX_ATOM_BYTES
    scales = -(-scales // 1024) * 1024
    return cfg.stages * stage_bytes(cfg, dtype) + scales + staging_bytes(dtype, cfg.swap_ab) + AUX_SMEM


def max_stages(bm, bn, bk, dtype, swap_ab, smem_per_block, cta_group=1):
    """The most stages (at most MAX_STAGES) whose shared-memory footprint, as
    smem_bytes counts it, fits; 0 when not even one does."""
    for st in range(MAX_STAGES, 0, -1):
        if smem_bytes(Config(bm, bn, bk, st, cta_group=cta_group, swap_ab=swap_ab), dtype) <= smem_per_block:
            return st
    return 0


def tmem_columns(cfg: Config, dtype=None):
    """Columns of one accumulator (fp32, one column per output column per 128
    rows), how many accumulators fit (2 = epilogue overlaps the next tile), and
    the MX scale columns (4 per atom, one slot per stage) that share the 512."""
    acc = (1 if cfg.cta_group == 2 else cfg.bm // 128) * cfg.bn
    scales = cfg.stages * 4 * mx_atoms(cfg, dtype)
    nbuf = 2 if 2 * acc + scales <= TMEM_COLUMNS else 1
    return acc, nbuf, scales


def gb300_check(M, N, K, dtype, epi, cfg: Config, dev: Device):
    """First violated rule, in the documented order, or R_OK."""
    elt = elt_bytes(dtype)
    span = span_elems(dtype)
    if cfg.cta_group not in (1, 2):
        return R_CTA_GROUP
    if cfg.cta_group == 2 and (cfg.bm != 256 or cfg.swap_ab != 0):
        return R_CTA_GROUP
    if cfg.bm not in (128, 256):
        return R_UMMA_M
    if cfg.bn % 16 != 0 or not (16 <= cfg.bn <= 256):
        return R_UMMA_N
    if cfg.swap_ab not in (0, 1):
        return R_LAYOUT
    # B in place comes in MN-major swizzle spans; a K-major copy of B only
    # needs the epilogue's 32-column chunks.
    b_unit = span if b_in_place(dtype, N) else 32
    if cfg.swap_ab == 0 and (cfg.bn % b_unit != 0 or cfg.bn % 32 != 0):
        return R_LAYOUT
    if cfg.cta_group == 2 and (cfg.bn // 2) % b_unit != 0:
        return R_LAYOUT
    # MX: scales of the MMA-N columns come in 128-column atoms; a swapped tile
    # (tokens along N) must start on one: bn a multiple of 128 or M in one tile.
    if dtype == DT_MXFP8 and cfg.swap_ab == 0 and cfg.bn not in (128, 256):
        return R_LAYOUT
    if dtype == DT_MXFP8 and cfg.swap_ab == 1 and cfg.bn % 128 != 0 and M > cfg.bn:
        return R_LAYOUT
    # Gated epilogues: a tile holds whole 64-column gate+up block pairs of the
    # fused weight and drains them in one pass (unswapped, no split-K).
    if is_glu(epi) and (cfg.swap_ab != 0 or cfg.split_k != 1 or cfg.bn % 64 != 0 or N % 64 != 0):
        return R_LAYOUT
    if cfg.bk % span != 0 or not (1 <= cfg.bk // span <= 4):
        return R_BK
    if dtype == DT_MXFP8 and cfg.bk not in (128, 256):
        return R_BK
    if not (2 <= cfg.stages <= MAX_STAGES):
        return R_STAGES
    if cfg.raster not in (0, 1) or cfg.group not in GROUPS:
        return R_SCHEDULE
    num_kb = ceil_div(K, cfg.bk)
    if cfg.split_k < 1 or cfg.split_k > 16 or cfg.split_k > max(1, num_kb):
        return R_SPLIT_K
    if (K * elt) % 16 != 0 or (N * out_elt_bytes(dtype)) % 16 != 0 or \
            (b_in_place(dtype, N) and (N * elt) % 16 != 0):
        return R_ALIGN
    acc, nbuf, scales = tmem_columns(cfg, dtype)
    if acc * nbuf + scales > TMEM_COLUMNS:
        return R_TMEM
    if smem_bytes(cfg, dtype) > dev.smem_per_block:
        return R_SMEM
    if dev.kernel_regs > 0 and dev.kernel_regs * dev.threads_per_cta > 65536:
        return R_REGS
    return R_OK


def gb300_candidates(M, N, K, dtype, epi, dev: Device):
    """The documented GB300 candidate generator (nested in this order): swap_ab,
    (bm, cta_group) in (128, 1), (256, 1), (256, 2) (pairs unswapped only), bn,
    bk, stages, then the schedule/split combinations, judged by CTA counts
    (tiles × cta_group); infeasible combinations are dropped."""
    span = span_elems(dtype)
    out = []
    swaps = (0, 1) if M <= 256 else (0,)
    for swap in swaps:
        rows, cols = (N, M) if swap else (M, N)
        for bm, cg in ((128, 1), (256, 1), (256, 2)):
            if cg == 2 and swap:
                continue
            if swap:
                bns = (16, 32, 64, 128, 256)
            elif cg == 2:
                bns = (128, 256) if dtype == DT_BF16 else \
                    (256,) if (is_fp8(dtype) and b_in_place(dtype, N)) else \
                    (128, 256) if dtype == DT_MXFP8 else (64, 128, 256)
            elif dtype == DT_BF16:
                bns = (64, 128, 192, 256)
            elif dtype == DT_FP8:
                bns = (128, 256) if b_in_place(dtype, N) else (64, 128, 192, 256)
            elif dtype == DT_MXFP8:
                bns = (128, 256)
            else:
                bns = (32, 64, 128, 192, 256)
            for bn in bns:
                for bk in (span, 2 * span):
                    st_max = max_stages(bm, bn, bk, dtype, swap, dev.smem_per_block, cg)
                    if st_max < 2:
                        continue
                    stage_list = sorted({min(4, st_max), st_max})
                    tiles = ceil_div(rows, bm) * ceil_div(cols, bn)
                    num_kb = ceil_div(K, bk)
                    splits = []
                    if tiles * cg < 4 * dev.sm_count:
                        splits = [s for s in SPLITS
                                  if 2 * s <= num_kb and tiles * s * cg <= 16 * dev.sm_count]
                    scheds = [(0, 1)]
                    if tiles * cg > dev.sm_count:
                        scheds = [(r, g) for r in (0, 1) for g in (1, 4, 8, 16)]
                    combos = [(r, g, 1) for (r, g) in scheds] + [(0, 1, s) for s in splits]
                    for st in stage_list:
                        for (r, g, s) in combos:
                            cfg = Config(bm, bn, bk, st, r, g, s, cg, swap)
                            if gb300_check(M, N, K, dtype, epi, cfg, dev) == R_OK:
                                out.append(cfg)
    return out


def gb300_fixed_config(dtype, dev: Device):
    """The untuned default: 128 × 128 tiles, one span of K, as many stages as fit,
    row-major tile order, no split, no swap."""
    span = span_elems(dtype)
    st = max_stages(128, 128, span, dtype, 0, dev.smem_per_block)
    return Config(128, 128, span, st, 0, 1, 1, 1, 0)


# ---------------------------------------------------------------------------
# Persistent tile schedule (grouped raster), restated
# ---------------------------------------------------------------------------

def schedule_unit(u, tiles_m, tiles_n, split_k, raster, group, num_kb):
    """Work unit u -> (tile_m, tile_n, split, kb_begin, kb_end).

    Units are tile-major (the split index varies fastest).  raster 0 walks a band
    of `group` tile-rows column by column; raster 1 walks a band of `group`
    tile-columns row by row ("Compilers and Kernel Languages": the order in which
    tiles are scheduled is one of the choices a real kernel adds)."""
    tile, s = divmod(u, split_k)
    if raster == 0:
        per_band = group * tiles_n
        band, r = divmod(tile, per_band)
        first = band * group
        height = min(group, tiles_m - first)
        tm, tn = first + r % height, r // height
    else:
        per_band = group * tiles_m
        band, r = divmod(tile, per_band)
        first = band * group
        width = min(group, tiles_n - first)
        tn, tm = first + r % width, r // width
    return tm, tn, s, (s * num_kb) // split_k, ((s + 1) * num_kb) // split_k


# ---------------------------------------------------------------------------
# GB300 cost model, restated from its documented terms.  Its panel traffic,
# waves, roofline floor and compulsory bytes are pinned against the pages; its
# fitted coefficients are parity unpinned.  With model_kind = 1 it is the
# workshop model above.
# ---------------------------------------------------------------------------

def gb300_model(M, N, K, dtype, epi, cfg: Config, dev: Device):
    """Predicted time and its terms (a dict, times in microseconds).

    Terms (documented model): the busiest CTA's K-blocks times the slower of MMA
    execution (per-SM share of the peak) and MMA issue (issue clocks per MMA +
    clocks per stage); L2 -> shared-memory panel bytes over the L2 bandwidth;
    HBM bytes (compulsory when A+B fit in half of L2, otherwise per-wave panels)
    over the HBM bandwidth; K-blocks × latency / stages; their maximum, plus the
    epilogue time no main loop hides, the split-K partial-tile traffic and the
    launch cost."""
    if dev.model_kind == 1:
        wd = WorkshopDevice(sms=dev.sm_count, peak_flops=dev.peak_tflops_bf16 * 1e12,
                            bw=dev.hbm_gbs * 1e9, elt=elt_bytes(dtype))
        t = tile_count(M, N, cfg.bm, cfg.bn)
        return {"predicted_us": workshop_time(M, N, K, cfg.bm, cfg.bn, wd) * 1e6,
                "tiles": t, "units": t, "waves": waves(t, dev.sm_count),
                "wave_eff": wave_efficiency(t, dev.sm_count),
                "tile_eff": workshop_tile_efficiency(cfg.bm, cfg.bn)}
    elt = elt_bytes(dtype)
    rows, cols = (N, M) if cfg.swap_ab else (M, N)
    tiles_m, tiles_n = ceil_div(rows, cfg.bm), ceil_div(cols, cfg.bn)
    tiles = tiles_m * tiles_n
    S = cfg.split_k
    num_kb = ceil_div(K, cfg.bk)
    units = tiles * S
    sms = dev.sm_count
    # A CTA pair runs each unit on two CTAs (128 tile rows and half of B each).
    cg = 2 if cfg.cta_group == 2 else 1
    rows_cta, bcols_cta = cta_share(cfg)
    cta_units = units * cg
    ctas = max(cg, min(cta_units, sms))
    if cg == 2:
        ctas -= ctas % 2
    nw = waves(cta_units, sms)
    per_cta_units = ceil_div(units, ctas // cg)
    slice_kb = ceil_div(num_kb, S)
    clock = dev.sm_clock_mhz * 1e6
    flops = 2.0 * M * N * K

    peak = (dev.peak_tflops_bf16 if dtype == DT_BF16 else
            dev.peak_tflops_fp8 if is_fp8(dtype) else dev.peak_tflops_tf32) * 1e12
    halves = 1 if cg == 2 else cfg.bm // 128
    ksteps = cfg.bk * elt / 32
    one_mma = 2.0 * 128 * cfg.bn * (32 / elt)
    execute = halves * ksteps * one_mma / (peak / sms)
    issue = (halves * ksteps * dev.mma_issue_clk + dev.kblock_clk) / clock
    mma_s = per_cta_units * slice_kb * max(execute, issue)

    # MX scales add 4 bytes per row (and per column) for every 128 of K.
    per_k = elt + (4 / 128 if dtype == DT_MXFP8 else 0.0)
    l2_bytes = cta_units * slice_kb * (rows_cta + bcols_cta) * cfg.bk * per_k
    l2_s = l2_bytes / (dev.l2_gbs * 1e9)

    in_bytes = (M * K + K * N) * per_k
    wave_tiles = min(tiles, max(1, ctas // cg // S))
    if cfg.raster == 0:
        rows_w = min(cfg.group, tiles_m, wave_tiles)
        cols_w = min(ceil_div(wave_tiles, rows_w), tiles_n)
    else:
        cols_w = min(cfg.group, tiles_n, wave_tiles)
        rows_w = min(ceil_div(wave_tiles, cols_w), tiles_m)
    panel = (tiles / wave_tiles) * K * (rows_w * cfg.bm + cols_w * cfg.bn) * per_k
    operand = in_bytes if in_bytes <= dev.l2_bytes / 2 else max(in_bytes, panel)
    eo = out_elt_bytes(dtype)
    c_cols = N // 2 if is_glu(epi) else N                     # a gated C is half the fused width
    hbm = (operand + M * c_cols * eo + (N * eo if epi != EPI_NONE else 0)
           + (M * N * eo if epi in (EPI_BIAS_RES, EPI_RELU_RES, EPI_GELU_RES) else 0))   # C, bias, residual R
    hbm_s = hbm / (dev.hbm_gbs * 1e9)

    latency_s = per_cta_units * slice_kb * dev.mem_latency_us * 1e-6 / cfg.stages
    main = max(mma_s, l2_s, hbm_s, latency_s)

    per_clock = dev.epi_gelu_elems_per_clk if epi in (EPI_GELU, EPI_GELU_RES, EPI_GEGLU, EPI_SWIGLU) \
        else dev.epi_elems_per_clk
    rate = per_clock * clock
    elems = rows_cta * cfg.bn          # one CTA's share of a tile
    partial = elems * 4
    if S == 1:
        one = elems / rate
        two_buffers = tmem_columns(cfg, dtype)[1] == 2
        unit_main = main / per_cta_units
        hidden_excess = max(0.0, one - unit_main) if two_buffers else one
        epi_s = one + (per_cta_units - 1) * hidden_excess
        split_s = 0.0
    elif cta_units <= sms:
        epi_s = (elems / S) / rate
        split_s = 2 * partial * (S - 1) / S / (dev.splitk_gbs * 1e9)
    else:
        fix = ceil_div(tiles * cg, ctas)
        epi_s = fix * elems / rate
        split_s = (per_cta_units + fix * S) * partial / (dev.splitk_gbs * 1e9)
    total = main + epi_s + split_s + dev.launch_us * 1e-6
    if K > 0:
        pad = (rows * cols * K) / (tiles_m * cfg.bm * tiles_n * cfg.bn * num_kb * cfg.bk)
    else:
        pad = 1.0
    return {"predicted_us": total * 1e6, "mma_us": mma_s * 1e6, "l2_us": l2_s * 1e6,
            "hbm_us": hbm_s * 1e6, "latency_us": latency_s * 1e6, "epilogue_us": epi_s * 1e6,
            "splitk_us": split_s * 1e6, "launch_us": dev.launch_us,
            "wave_eff": cta_units / (nw * sms), "tile_eff": execute / max(execute, issue), "pad_eff": pad,
            "hbm_bytes": hbm, "l2_bytes": l2_bytes, "flops": flops,
            "tiles": tiles, "units": units, "waves": nw, "ctas": ctas}


# ---------------------------------------------------------------------------
# Rank agreement between predicted and measured times
# ---------------------------------------------------------------------------

def average_ranks(values):
    """1-based ranks, ties sharing the mean of their positions."""
    order = sorted(range(len(values)), key=lambda i: values[i])
    ranks = [0.0] * len(values)
    i = 0
    while i < len(order):
        j = i
        while j + 1 < len(order) and values[order[j + 1]] == values[order[i]]:
            j += 1
        avg = (i + j) / 2.0 + 1.0
        for t in range(i, j + 1):
            ranks[order[t]] = avg
        i = j + 1
    return ranks


def kendall_tau_b(x, y):
    """τ_b = (concordant − discordant) / √((n0 − ties_x)(n0 − ties_y)), by
    looking at every pair."""
    n = len(x)
    conc = disc = tx = ty = 0
    for i in range(n):
        for j in range(i + 1, n):
            dx = (x[i] > x[j]) - (x[i] < x[j])
            dy = (y[i] > y[j]) - (y[i] < y[j])
            if dx == 0 and dy == 0:
                continue
            if dx == 0:
                tx += 1
            elif dy == 0:
                ty += 1
            elif dx == dy:
                conc += 1
            else:
                disc += 1
    denom = math.sqrt((conc + disc + tx) * (conc + disc + ty))
    return (conc - disc) / denom if denom > 0 else float("nan")


def spearman_rho(x, y):
    """Pearson correlation of the average ranks."""
    rx, ry = average_ranks(x), average_ranks(y)
    n = len(x)
    mx, my = sum(rx) / n, sum(ry) / n
    sxy = sum((a - mx) * (b - my) for a, b in zip(rx, ry))
    sxx = sum((a - mx) ** 2 for a in rx)
    syy = sum((b - my) ** 2 for b in ry)
    return sxy / math.sqrt(sxx * syy) if sxx > 0 and syy > 0 else float("nan")


def rank_agreement(predicted, measured):
    """τ_b, ρ, whether the model's first choice is the measured fastest, and the
    regret of following the model (its pick's measured time / best − 1)."""
    pick = min(range(len(predicted)), key=lambda i: predicted[i])
    best = min(range(len(measured)), key=lambda i: measured[i])
    return {"kendall_tau": kendall_tau_b(predicted, measured),
            "spearman_rho": spearman_rho(predicted, measured),
            "top1_hit": int(measured[pick] == measured[best]),
            "regret": measured[pick] / measured[best] - 1.0}


# ---------------------------------------------------------------------------
# Shipped configuration set ("Tile Selection": a small list of configurations
# per kernel; "Autotuning & cost models": tune ahead of time)
# ---------------------------------------------------------------------------

def shipped_set_value(times, chosen):
    """Sum over shapes of best / (fastest chosen time); 0 for a shape that no
    chosen configuration runs (times <= 0 mean "does not run")."""
    total = 0.0
    for row in times:
        runs = [v for v in row if v > 0]
        if not runs:
            continue
        best = min(runs)
        got = [row[c] for c in chosen if row[c] > 0]
        total += best / min(got) if got else 0.0
    return total


def shipped_set_greedy(times, max_set):
    """Adds, one at a time, the configuration that most raises the value (the
    lowest column among equal gains); stops at max_set or when nothing gains.
    Returns (chosen, mean slowdown, worst slowdown) over shapes that some
    configuration runs."""
    n_shapes = len(times)
    n_cfg = len(times[0]) if n_shapes else 0
    best = []
    for row in times:
        runs = [v for v in row if v > 0]
        best.append(min(runs) if runs else 0.0)
    covered = [0.0] * n_shapes          # current best / fastest-chosen per shape
    chosen = []
    while len(chosen) < min(max_set, n_cfg):
        pick, pick_gain = None, 0.0
        for c in range(n_cfg):
            if c in chosen:
                continue
            gain = 0.0
            for s in range(n_shapes):
                q = best[s] / times[s][c] if (times[s][c] > 0 and best[s] > 0) else 0.0
                gain += max(0.0, q - covered[s])
            if gain > pick_gain:
                pick, pick_gain = c, gain
        if pick is None:
            break
        chosen.append(pick)
        for s in range(n_shapes):
            q = best[s] / times[s][pick] if (times[s][pick] > 0 and best[s] > 0) else 0.0
            covered[s] = max(covered[s], q)
    slow = [1.0 / covered[s] if covered[s] > 0 else math.inf for s in range(n_shapes) if best[s] > 0]
    mean = sum(slow) / len(slow) if slow else 1.0
    worst = max(slow) if slow else 1.0
    return chosen, mean, worst


def shipped_set_optimal(times, size):
    """Brute force over every set of `size` columns: the largest value."""
    n_cfg = len(times[0]) if times else 0
    best_v, best_set = -1.0, ()
    for subset in itertools.combinations(range(n_cfg), min(size, n_cfg)):
        v = shipped_set_value(times, subset)
        if v > best_v:
            best_v, best_set = v, subset
    return list(best_set), best_v
