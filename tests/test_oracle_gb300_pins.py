"""Pins of the GB300 selection oracle (oracle/selection.py: gb300_model,
gb300_candidates) against what the pages and plain arithmetic fix, each with a
planted mistake that the pin must catch.

What the pages fix, and the pin for each:
  * "Tile Selection: Cost Models Against Measurement", "Analytical models and
    where they break": a block moves K·(BM+BN) elements of its panels over the
    full depth (4K(BM+BN) bytes in fp32), and with no panel shared through
    shared memory the grid moves that times the tile count.  gb300_model's
    l2_bytes (panel bytes staged into shared memory) must equal it, for single
    CTAs, CTA pairs (two CTAs holding one 256-row tile) and split-K alike.
  * "Compilers and Kernel Languages", workshop paragraph: tiles run in waves of
    one per multiprocessor, 133 tiles on 132 take two waves; 64 tiles on 132
    leave half of them idle.  gb300_model's waves and wave efficiency must equal
    a round-by-round dispatch of the CTAs (tiles x slices x CTAs per tile).
  * The same page, "A different tile for every shape": the roofline floor (the
    larger of operations at peak and compulsory bytes at bandwidth) bounds every
    prediction from below.
  * "Tiling the hierarchy", capacity discussion: when A and B fit in (half of)
    L2 the operands cost their compulsory bytes once; the model's HBM bytes must
    then be exactly the compulsory bytes of A, B, bias, C (and R).
  * The GB300 candidate generator must equal a brute-force filter of its
    documented grid ("CuTile Autotuning": the space holds the original fixed
    configuration).

The mistakes are planted in the oracle (on the CPU, through monkeypatch) and
each test asserts that its pin fails on them."""
import inspect
import itertools
import textwrap

import pytest

from oracle import selection as sel

ELT = {sel.DT_BF16: 2, sel.DT_FP32: 4, sel.DT_FP8: 1, sel.DT_MXFP8: 1}     # operand bytes
OUT = {sel.DT_BF16: 2, sel.DT_FP32: 4, sel.DT_FP8: 2, sel.DT_MXFP8: 2}     # C, bias, R bytes

# Shapes of the workloads (the under-filled 1000x1000x8192, the square 8192^3,
# the 16-token decode, the 256^3 fp32 case, sweep projections) plus ragged ones.
SHAPES = [
    (1000, 1000, 8192, sel.DT_BF16, sel.EPI_GELU),
    (8192, 8192, 8192, sel.DT_BF16, sel.EPI_RELU),
    (16, 28672, 8192, sel.DT_BF16, sel.EPI_NONE),
    (256, 256, 256, sel.DT_FP32, sel.EPI_RELU),
    (4096, 4096, 4096, sel.DT_FP32, sel.EPI_NONE),
    (128, 4096, 14336, sel.DT_BF16, sel.EPI_GELU),
    (512, 6144, 4096, sel.DT_BF16, sel.EPI_GELU_RES),
    (1000, 1000, 8192, sel.DT_FP8, sel.EPI_GELU),
    (2048, 1024, 4096, sel.DT_MXFP8, sel.EPI_BIAS),
    (300, 320, 1032, sel.DT_BF16, sel.EPI_BIAS),
    (512, 28672, 4096, sel.DT_BF16, sel.EPI_GEGLU),      # gated: fused gate+up weight, C of half its width
]


def _plant(monkeypatch, name, old, new):
    """Replaces `old` by `new` in the source of oracle function `name` and
    installs the result in its place: a planted mistake, for this test only."""
    src = textwrap.dedent(inspect.getsource(getattr(sel, name)))
    assert src.count(old) == 1, old
    scope = dict(vars(sel))
    exec(compile(src.replace(old, new), sel.__file__, "exec"), scope)
    monkeypatch.setattr(sel, name, scope[name])


def _page_law_panel_bytes(M, N, K, dt, cfg):
    """Per-block panel bytes over the full depth, K·(BM+BN)·element size, times
    the number of blocks (in the MMA orientation: a swapped tile is bm rows of
    Bᵀ by bn columns of Aᵀ)."""
    rows, cols = (N, M) if cfg.swap_ab else (M, N)
    blocks = -(-rows // cfg.bm) * -(-cols // cfg.bn)
    return blocks * K * (cfg.bm + cfg.bn) * ELT[dt]


def _law_cases():
    dev = sel.Device()
    for (M, N, K, dt, epi) in SHAPES:
        if dt == sel.DT_MXFP8:
            continue            # MX adds scale bytes the page's law does not know
        for c in sel.gb300_candidates(M, N, K, dt, epi, dev):
            # the law counts K exactly: every slice a whole number of K-blocks
            if K % (c.bk * c.split_k) == 0:
                yield M, N, K, dt, epi, c


def test_fp32_law_is_the_pages_four_k_bm_plus_bn():
    # the page prints the fp32 form 4K(BM+BN): the helper reads the same number
    assert _page_law_panel_bytes(256, 256, 256, sel.DT_FP32, sel.Config(128, 64, 32, 4)) == \
        2 * 4 * 4 * 256 * (128 + 64)


def test_panel_traffic_equals_the_per_block_law():
    dev = sel.Device()
    n = kinds = 0
    seen = set()
    for M, N, K, dt, epi, c in _law_cases():
        got = sel.gb300_model(M, N, K, dt, epi, c, dev)["l2_bytes"]
        assert got == pytest.approx(_page_law_panel_bytes(M, N, K, dt, c), rel=1e-12), (M, N, K, dt, c)
        seen.add((c.cta_group, c.split_k > 1, c.swap_ab))
        n += 1
    kinds = len(seen)
    assert n > 500 and kinds >= 5      # pairs, split-K and swapped tiles all covered


def test_panel_law_catches_a_pair_that_loads_the_whole_tile(monkeypatch):
    monkeypatch.setattr(sel, "cta_share", lambda cfg: (cfg.bm, cfg.bn))
    with pytest.raises(AssertionError):
        test_panel_traffic_equals_the_per_block_law()


def test_panel_law_catches_a_wrong_element_size(monkeypatch):
    real = sel.elt_bytes
    monkeypatch.setattr(sel, "elt_bytes", lambda dt: 4 if dt == sel.DT_BF16 else real(dt))
    with pytest.raises(AssertionError):
        test_panel_traffic_equals_the_per_block_law()


# --- waves -------------------------------------------------------------------

def _dispatch_rounds(ctas, sms):
    """Round-by-round dispatch: each round puts one CTA on every free SM."""
    rounds, left = 0, ctas
    while left > 0:
        left -= sms
        rounds += 1
    return rounds


def test_waves_printed_examples_through_the_model():
    dev = sel.Device(sm_count=132)
    # 133 tiles of 128 x 128 on 132 multiprocessors: two waves, the second almost empty
    r = sel.gb300_model(133 * 128, 128, 1024, sel.DT_BF16, sel.EPI_NONE, sel.Config(128, 128, 64, 4), dev)
    assert r["tiles"] == 133 and r["waves"] == 2
    assert r["wave_eff"] == pytest.approx(133 / 264)
    # 1000 x 1000 on 128 x 128 tiles: 64 tiles, under half of the 132 busy
    r = sel.gb300_model(1000, 1000, 8192, sel.DT_BF16, sel.EPI_GELU, sel.Config(128, 128, 64, 4), dev)
    assert r["tiles"] == 64 and r["waves"] == 1 and r["wave_eff"] < 0.5


def test_waves_equal_a_round_by_round_dispatch():
    n = 0
    for sms in (132, 148, 152):
        dev = sel.Device(sm_count=sms)
        for (M, N, K, dt, epi) in SHAPES:
            for c in sel.gb300_candidates(M, N, K, dt, epi, dev)[::3]:
                r = sel.gb300_model(M, N, K, dt, epi, c, dev)
                rows, cols = (N, M) if c.swap_ab else (M, N)
                ctas = -(-rows // c.bm) * -(-cols // c.bn) * c.split_k * c.cta_group
                w = _dispatch_rounds(ctas, sms)
                assert r["waves"] == w, (M, N, K, c)
                assert r["wave_eff"] == pytest.approx(ctas / (w * sms), rel=1e-12)
                n += 1
    assert n > 300


def test_wave_pin_catches_an_off_by_one(monkeypatch):
    monkeypatch.setattr(sel, "waves", lambda units, sms: units // sms + 1)
    with pytest.raises(AssertionError):
        test_waves_equal_a_round_by_round_dispatch()


def test_wave_pin_catches_pairs_counted_as_one_cta(monkeypatch):
    _plant(monkeypatch, "gb300_model", "nw = waves(cta_units, sms)", "nw = waves(units, sms)")
    with pytest.raises(AssertionError):
        test_waves_equal_a_round_by_round_dispatch()


def test_panel_law_catches_slices_counted_once(monkeypatch):
    _plant(monkeypatch, "gb300_model", "l2_bytes = cta_units * slice_kb", "l2_bytes = tiles * cg * slice_kb")
    with pytest.raises(AssertionError):
        test_panel_traffic_equals_the_per_block_law()


# --- roofline floor and compulsory bytes ----------------------------------------

def _compulsory_bytes(M, N, K, dt, epi):
    e, eo = ELT[dt], OUT[dt]
    gated = epi in (sel.EPI_REGLU, sel.EPI_GEGLU, sel.EPI_SWIGLU)
    b = (M * K + K * N) * e + M * (N // 2 if gated else N) * eo      # A, B, C (a gated C: N/2 wide)
    if epi != sel.EPI_NONE:
        b += N * eo                                                  # bias (fused, N wide when gated)
    if epi in (sel.EPI_BIAS_RES, sel.EPI_RELU_RES, sel.EPI_GELU_RES):
        b += M * N * eo                                              # R
    return b


def _peak_flops(dt, dev):
    return 1e12 * (dev.peak_tflops_bf16 if dt == sel.DT_BF16 else
                   dev.peak_tflops_fp8 if dt in (sel.DT_FP8, sel.DT_MXFP8) else dev.peak_tflops_tf32)


def test_no_prediction_beats_the_roofline_floor():
    dev = sel.Device()
    n = 0
    for (M, N, K, dt, epi) in SHAPES:
        floor_s = max(2.0 * M * N * K / _peak_flops(dt, dev), _compulsory_bytes(M, N, K, dt, epi) / (dev.hbm_gbs * 1e9))
        for c in sel.gb300_candidates(M, N, K, dt, epi, dev):
            r = sel.gb300_model(M, N, K, dt, epi, c, dev)
            # no part of the model may beat its own bound either
            assert r["mma_us"] * 1e-6 >= 2.0 * M * N * K / _peak_flops(dt, dev) * (1 - 1e-12), c
            assert r["hbm_us"] * 1e-6 >= _compulsory_bytes(M, N, K, dt, epi) / (dev.hbm_gbs * 1e9) * (1 - 1e-12), c
            assert r["predicted_us"] * 1e-6 >= floor_s, c
            n += 1
    assert n > 1000


def test_floor_pin_catches_half_the_operand_bytes(monkeypatch):
    real = sel.elt_bytes
    monkeypatch.setattr(sel, "elt_bytes", lambda dt: 1 if dt == sel.DT_BF16 else real(dt))
    with pytest.raises(AssertionError):
        test_no_prediction_beats_the_roofline_floor()


def test_floor_pin_catches_a_dropped_unit_count(monkeypatch):
    # the busiest CTA's MMA time counted for one unit only
    _plant(monkeypatch, "gb300_model", "mma_s = per_cta_units * slice_kb", "mma_s = slice_kb")
    with pytest.raises(AssertionError):
        test_no_prediction_beats_the_roofline_floor()


def test_floor_pin_catches_a_peak_for_the_wrong_dtype(monkeypatch):
    # bf16 priced at the FP8 rate
    _plant(monkeypatch, "gb300_model", "peak = (dev.peak_tflops_bf16 if", "peak = (dev.peak_tflops_fp8 if")
    with pytest.raises(AssertionError):
        test_no_prediction_beats_the_roofline_floor()


def test_hbm_bytes_are_compulsory_when_operands_fit_in_half_of_l2():
    dev = sel.Device()
    n = 0
    for (M, N, K, dt, epi) in SHAPES:
        fits = (M * K + K * N) * ELT[dt] <= dev.l2_bytes / 2
        for c in sel.gb300_candidates(M, N, K, dt, epi, dev)[::2]:
            hbm = sel.gb300_model(M, N, K, dt, epi, c, dev)["hbm_bytes"]
            # block-scaled FP8 also reads one E8M0 scale byte per 32 elements of K
            scales = (M + N) * K / 32 if dt == sel.DT_MXFP8 else 0
            want = _compulsory_bytes(M, N, K, dt, epi) + scales
            if fits:
                assert hbm == pytest.approx(want, rel=1e-12), (M, N, K, c)
            else:
                assert hbm >= want * (1 - 1e-12), (M, N, K, c)
            n += 1
    assert n > 500


def test_hbm_pin_catches_a_dropped_output_term(monkeypatch):
    monkeypatch.setattr(sel, "out_elt_bytes", lambda dt: 0)
    with pytest.raises(AssertionError):
        test_hbm_bytes_are_compulsory_when_operands_fit_in_half_of_l2()


def test_hbm_pin_catches_a_dropped_c_term(monkeypatch):
    _plant(monkeypatch, "gb300_model", "hbm = (operand + M * c_cols * eo +", "hbm = (operand +")
    with pytest.raises(AssertionError):
        test_hbm_bytes_are_compulsory_when_operands_fit_in_half_of_l2()


def test_gated_shapes_only_generate_unswapped_unsplit_tiles_of_whole_block_pairs():
    dev = sel.Device()
    cands = sel.gb300_candidates(512, 28672, 4096, sel.DT_BF16, sel.EPI_GEGLU, dev)
    assert cands and all(c.swap_ab == 0 and c.split_k == 1 and c.bn % 64 == 0 for c in cands)
    assert sel.gb300_check(512, 28672 + 32, 4096, sel.DT_BF16, sel.EPI_GEGLU, sel.Config(128, 128, 64, 4),
                           dev) == sel.R_LAYOUT


def test_hbm_pin_catches_a_wrong_output_size(monkeypatch):
    monkeypatch.setattr(sel, "out_elt_bytes", lambda dt: 4)
    with pytest.raises(AssertionError):
        test_hbm_bytes_are_compulsory_when_operands_fit_in_half_of_l2()


# --- the candidate generator against a brute-force filter of its grid -------------

# The documented grid: every field's full range.
GRID_BM_CG = ((128, 1), (256, 1), (256, 2))
GRID_BN = tuple(range(16, 257, 16))
GRID_STAGES = tuple(range(2, 17))
GRID_RASTER = (0, 1)
GRID_GROUP = (1, 2, 4, 8, 16)
GRID_SPLIT = tuple(range(1, 17))
# The documented generation rules, written as predicates on one configuration.
DOC_SPLITS = (2, 3, 4, 6, 8, 12, 16)
DOC_RASTER_GROUPS = (1, 4, 8, 16)


def _doc_bn_list(dt, cg, swap, N):
    """bn per case, as documented: swapped {16..256 powers of 2}; pairs: bf16
    {128, 256}, FP8/MX in place {256}, MX from a K-major copy {128, 256}, else
    {64, 128, 256}; single CTA: bf16 {64, 128, 192, 256}, FP8 in place
    {128, 256} else {64, 128, 192, 256}, MX {128, 256}, fp32 {32, 64, 128, 192, 256}."""
    in_place = dt == sel.DT_BF16 or (dt in (sel.DT_FP8, sel.DT_MXFP8) and N % 16 == 0)
    if swap:
        return {16, 32, 64, 128, 256}
    if cg == 2:
        if dt == sel.DT_BF16:
            return {128, 256}
        if dt in (sel.DT_FP8, sel.DT_MXFP8) and in_place:
            return {256}
        if dt == sel.DT_MXFP8:
            return {128, 256}
        return {64, 128, 256}
    if dt == sel.DT_BF16:
        return {64, 128, 192, 256}
    if dt == sel.DT_FP8:
        return {128, 256} if in_place else {64, 128, 192, 256}
    if dt == sel.DT_MXFP8:
        return {128, 256}
    return {32, 64, 128, 192, 256}


def _brute_force_candidates(M, N, K, dt, epi, dev):
    span = 128 // ELT[dt]
    out = set()
    for swap in (0, 1):
        if swap and M > 256:
            continue
        rows, cols = (N, M) if swap else (M, N)
        for (bm, cg), bn in itertools.product(GRID_BM_CG, GRID_BN):
            if (cg == 2 and swap) or bn not in _doc_bn_list(dt, cg, swap, N):
                continue
            for bk in (span * j for j in (1, 2, 3, 4)):
                if bk not in (span, 2 * span):
                    continue
                # the most stages whose shared-memory footprint fits
                ok_st = [s for s in GRID_STAGES
                         if sel.smem_bytes(sel.Config(bm, bn, bk, s, 0, 1, 1, cg, swap), dt) <= dev.smem_per_block]
                if not ok_st:
                    continue
                smax = max(ok_st)
                tiles = -(-rows // bm) * -(-cols // bn)
                nkb = -(-K // bk)
                for st, r, g, s in itertools.product(GRID_STAGES, GRID_RASTER, GRID_GROUP, GRID_SPLIT):
                    if st not in (min(4, smax), smax):
                        continue
                    if s == 1:
                        sched_ok = (r, g) == (0, 1) or (tiles * cg > dev.sm_count and g in DOC_RASTER_GROUPS)
                    else:
                        sched_ok = ((r, g) == (0, 1) and s in DOC_SPLITS and tiles * cg < 4 * dev.sm_count
                                    and 2 * s <= nkb and tiles * s * cg <= 16 * dev.sm_count)
                    if not sched_ok:
                        continue
                    c = sel.Config(bm, bn, bk, st, r, g, s, cg, swap)
                    if sel.gb300_check(M, N, K, dt, epi, c, dev) == sel.R_OK:
                        out.add(c.astuple())
    return out


GEN_SHAPES = [
    (1000, 1000, 8192, sel.DT_BF16, sel.EPI_GELU),
    (16, 28672, 8192, sel.DT_BF16, sel.EPI_NONE),
    (256, 256, 256, sel.DT_FP32, sel.EPI_RELU),
    (8192, 8192, 8192, sel.DT_BF16, sel.EPI_RELU),
    (1000, 1000, 8192, sel.DT_FP8, sel.EPI_GELU),
    (16, 8192, 8192, sel.DT_MXFP8, sel.EPI_NONE),
    (300, 320, 1032, sel.DT_BF16, sel.EPI_BIAS),
    (512, 28672, 4096, sel.DT_BF16, sel.EPI_SWIGLU),
]


@pytest.mark.parametrize("M,N,K,dt,epi", GEN_SHAPES)
def test_generator_equals_the_brute_force_filter(M, N, K, dt, epi):
    dev = sel.Device()
    got = [c.astuple() for c in sel.gb300_candidates(M, N, K, dt, epi, dev)]
    assert len(got) == len(set(got))
    want = _brute_force_candidates(M, N, K, dt, epi, dev)
    assert set(got) == want
    fixed = sel.gb300_fixed_config(dt, dev).astuple()
    assert fixed in want      # the original fixed tile is always a candidate
    # the fixed tile: 128 x 128, one span of K, as many stages as the rules allow
    span = 128 // ELT[dt]
    assert fixed[:3] == (128, 128, span) and fixed[4:] == (0, 1, 1, 1, 0)
    assert sel.gb300_check(M, N, K, dt, epi, sel.Config(128, 128, span, fixed[3] + 1), dev) in \
        (sel.R_SMEM, sel.R_STAGES, sel.R_TMEM) or fixed[3] == 16


def test_generator_pin_catches_a_missing_split_class(monkeypatch):
    monkeypatch.setattr(sel, "SPLITS", tuple(s for s in sel.SPLITS if s != 3))
    with pytest.raises(AssertionError):
        test_generator_equals_the_brute_force_filter(1000, 1000, 8192, sel.DT_BF16, sel.EPI_GELU)


def test_generator_pin_catches_one_stage_short(monkeypatch):
    real = sel.max_stages
    monkeypatch.setattr(sel, "max_stages", lambda *a, **k: max(0, real(*a, **k) - 1))
    with pytest.raises(AssertionError):
        test_generator_equals_the_brute_force_filter(8192, 8192, 8192, sel.DT_BF16, sel.EPI_RELU)


def test_generator_pin_catches_a_wrong_swizzle_span(monkeypatch):
    monkeypatch.setattr(sel, "span_elems", lambda dt: 64 // ELT[dt])
    with pytest.raises(AssertionError):
        test_generator_equals_the_brute_force_filter(1000, 1000, 8192, sel.DT_BF16, sel.EPI_GELU)
