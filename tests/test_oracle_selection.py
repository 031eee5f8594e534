"""Pins for the selection-layer oracle (oracle/selection.py): the pages' printed
numbers and closed forms, brute force on small cases, and library routines
(scipy.stats) for the rank statistics."""
import itertools
import math
import random

import numpy as np
import pytest

from oracle import selection as sel


# --- "Tile Selection", "The structure of the search space" -------------------

def test_p1_panel_cap_is_the_printed_12288(golden):
    g = golden("p1_enumerator.json")
    assert sel.p1_panel_cap_elements(g["smem_bytes"]) == g["panel_cap_elements"]


def _rule_smem(bm, bn, ks, smem):      # each rule as its own predicate
    return 4 * bm * ks + 4 * ks * bn <= smem


def _rule_threads(bm, bn, tm, tn, max_threads):
    t = (bm // tm) * (bn // tn)
    return 32 <= t <= max_threads


def _rule_warps(bm, bn, tm, tn):
    return ((bm // tm) * (bn // tn)) % 32 == 0


def _rule_acc(tm, tn):
    return tm * tn <= 128


@pytest.mark.parametrize("smem", [48 * 1024, 228 * 1024, 16 * 1024])
def test_p1_candidates_equal_rule_by_rule_brute_force(smem):
    got = sel.p1_candidates(256, 256, 256, smem_bytes=smem)
    brute = [t for t in itertools.product((32, 64, 128, 256), (32, 64, 128, 256),
                                          (8, 16, 32, 64), (2, 4, 8), (2, 4, 8))
             if _rule_smem(t[0], t[1], t[2], smem) and _rule_threads(t[0], t[1], t[3], t[4], 1024)
             and _rule_warps(t[0], t[1], t[3], t[4]) and _rule_acc(t[3], t[4])]
    assert got == brute
    assert len(set(got)) == len(got)


def test_p1_count_in_the_stated_range(golden):
    g = golden("p1_enumerator.json")
    got = sel.p1_candidates(256, 256, 256, smem_bytes=g["smem_bytes"])
    lo, hi = g["count_range_stated"]
    assert lo <= len(got) <= hi
    assert len(got) == g["count_derived_from_listing"]
    assert len({t[:3] for t in got}) == g["distinct_block_tiles_derived_from_listing"]
    assert len(sel.p1_candidates(1, 1, 1, smem_bytes=228 * 1024)) == g["count_derived_at_228KB"]


# --- "Compilers and Kernel Languages": waves and the workshop model ----------

def test_waves_printed_example(golden):
    w = golden("workshop_h100.json")["waves_example"]
    assert sel.waves(w["tiles"], w["sms"]) == w["waves"]
    assert sel.waves(132, 132) == 1


def test_underfilled_fixed_tile_is_under_half_a_wave(golden):
    g = golden("workshop_h100.json")["underfilled"]
    M, N, _K = g["shape"]
    t = sel.tile_count(M, N, 128, 128)
    assert t == g["fixed_128_tiles"]
    assert sel.wave_efficiency(t, 132) < 0.5


def test_workshop_large_square(golden):
    g = golden("workshop_h100.json")["large_square"]
    r = sel.workshop_sweep(*g["shape_reading"])
    assert list(r["best"]) == g["best_tile"]
    assert round(r["best_s"] * 1e6) == g["best_us"]
    assert round(r["worst_s"] / r["best_s"], 2) == g["worst_over_best"]
    assert round(r["fixed_128"] / r["best_s"], 2) == g["fixed_128_over_best"]


def test_workshop_underfilled(golden):
    g = golden("workshop_h100.json")["underfilled"]
    M, N, K = g["shape"]
    r = sel.workshop_sweep(M, N, K)
    assert list(r["best"]) == g["best_tile"]
    t = sel.tile_count(M, N, *r["best"])
    assert round(100 * sel.wave_efficiency(t, 132)) == g["best_wave_efficiency_percent"]
    assert round(r["fixed_128"] / r["best_s"], 2) == g["fixed_128_over_best"]


def test_workshop_decode_all_tie_at_the_weight_floor(golden):
    g = golden("workshop_h100.json")["decode_16_tokens"]
    r = sel.workshop_sweep(*g["shape_reading"])
    times = list(r["times"].values())
    assert len(times) == g["tile_shapes"]
    assert max(times) == min(times)
    assert round(times[0] * 1e6, 1) == g["all_tie_us"]


def test_workshop_mistakes_change_the_printed_numbers(golden):
    """Dropping a term of the model moves a printed number."""
    g = golden("workshop_h100.json")
    dev = sel.WorkshopDevice()
    # without the tile-efficiency term the worst/best ratio collapses to ~1
    M = N = K = 8192
    no_teff = [2.0 * M * N * K / dev.peak_flops / sel.wave_efficiency(sel.tile_count(M, N, a, b), 132)
               for a in sel.WORKSHOP_TILES for b in sel.WORKSHOP_TILES]
    assert round(max(no_teff) / min(no_teff), 2) != g["large_square"]["worst_over_best"]
    # without the X/Y bytes in the floor the decode tie is 35.06 us, not 35.2
    Md, Nd, Kd = g["decode_16_tokens"]["shape_reading"]
    assert round(Kd * Nd * 2 / dev.bw * 1e6, 1) != g["decode_16_tokens"]["all_tie_us"]


# --- "Tiling the hierarchy" ---------------------------------------------------

@pytest.mark.parametrize("Nn,T", [(8, 1), (8, 2), (8, 4), (16, 4), (16, 8), (32, 8), (32, 16)])
def test_square_tile_traffic_law_matches_explicit_count(Nn, T):
    assert sel.square_tile_traffic_count(Nn, T) == sel.square_tile_traffic_law(Nn, T)


def test_square_tile_side_and_capacity_form():
    C = 3 * 64 * 64
    assert sel.square_tile_side(C) == 64
    Nn = 4096
    T = sel.square_tile_side(C)
    assert sel.square_tile_traffic_law(Nn, T) == pytest.approx(2 * Nn ** 3 * math.sqrt(3) / math.sqrt(C))


def test_l2_tile_example(golden):
    g = golden("page_arithmetic.json")["l2_tile_example"]
    assert g["factor"] * g["multiple"] == g["factored"]
    extra = sel.square_tile_traffic_law(1, g["factored"]) / sel.square_tile_traffic_law(1, g["optimal"]) - 1
    assert round(100 * extra) == g["extra_traffic_percent"]


def test_double_buffer_example(golden):
    g = golden("page_arithmetic.json")["double_buffer_example"]
    t = sel.double_buffer_load_ns(g["tile_bytes"], g["bw_bytes_per_s"])
    assert round(t) == g["load_ns"]
    assert round(sel.double_buffer_load_ns(g["tile_bytes"], g["bw_bytes_per_s"], math.sqrt(2))) == g["penalised_ns"]


def test_amortisation_and_search_space_examples(golden):
    a = golden("page_arithmetic.json")["amortisation_example"]
    assert round(a["t_search_s"] / (a["saved_us"] * 1e-6)) == a["break_even_calls"]
    s = golden("page_arithmetic.json")["search_space_example"]
    assert math.prod(s["factors"]) == s["configs"]
    assert round(s["configs"] * s["seconds_each"] / 60) == s["minutes"]


@pytest.mark.parametrize("bm,bn", [(32, 32), (64, 256), (128, 128), (256, 64)])
def test_block_intensity_is_independent_of_K(bm, bn):
    vals = {sel.block_intensity(bm, bn, K) for K in (1, 8, 64, 4096)}
    assert len(vals) == 1
    assert vals.pop() == pytest.approx(bm * bn / (2 * (bm + bn)))


# --- tile schedule ------------------------------------------------------------

@pytest.mark.parametrize("tm,tn,S,raster,group,nkb", [
    (7, 5, 1, 0, 1, 4), (7, 5, 1, 0, 4, 4), (7, 5, 3, 1, 4, 9), (1, 9, 2, 0, 16, 2),
    (16, 16, 1, 1, 8, 1), (3, 11, 4, 1, 2, 8), (8, 8, 16, 0, 8, 16)])
def test_schedule_is_a_bijection_with_balanced_k_ranges(tm, tn, S, raster, group, nkb):
    seen = set()
    for u in range(tm * tn * S):
        a, b, s, k0, k1 = sel.schedule_unit(u, tm, tn, S, raster, group, nkb)
        assert 0 <= a < tm and 0 <= b < tn and 0 <= s < S
        assert (s * nkb) // S == k0 and k1 - k0 in (nkb // S, nkb // S + 1)
        seen.add((a, b, s))
    assert len(seen) == tm * tn * S
    # the k ranges of one tile cover [0, nkb) exactly
    cover = sorted(sel.schedule_unit(u, tm, tn, S, raster, group, nkb)[3:] for u in range(S))
    assert cover[0][0] == 0 and cover[-1][1] == nkb
    assert all(cover[i][1] == cover[i + 1][0] for i in range(len(cover) - 1))


def test_schedule_group_one_is_row_major():
    order = [sel.schedule_unit(u, 3, 4, 1, 0, 1, 1)[:2] for u in range(12)]
    assert order == [(m, n) for m in range(3) for n in range(4)]
    order = [sel.schedule_unit(u, 3, 4, 1, 1, 1, 1)[:2] for u in range(12)]
    assert order == [(m, n) for n in range(4) for m in range(3)]


def test_schedule_group_band_walks_columns():
    order = [sel.schedule_unit(u, 4, 3, 1, 0, 2, 1)[:2] for u in range(12)]
    assert order[:6] == [(0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2)]


# --- rank agreement -------------------------------------------------------------

def test_rank_agreement_hand_cases():
    r = sel.rank_agreement([1, 2, 3, 4], [10, 20, 30, 40])
    assert r["kendall_tau"] == 1 and r["spearman_rho"] == 1 and r["top1_hit"] == 1 and r["regret"] == 0
    r = sel.rank_agreement([4, 3, 2, 1], [10, 20, 30, 40])
    assert r["kendall_tau"] == -1 and r["spearman_rho"] == -1 and r["top1_hit"] == 0
    assert r["regret"] == pytest.approx(3.0)


def test_rank_agreement_against_scipy():
    stats = pytest.importorskip("scipy.stats")
    rng = random.Random(11)
    for n in (5, 17, 60):
        x = [rng.choice([1.0, 2.0, 3.0, 4.5, rng.random()]) for _ in range(n)]
        y = [rng.choice([0.5, rng.random(), rng.random()]) for _ in range(n)]
        assert sel.kendall_tau_b(x, y) == pytest.approx(stats.kendalltau(x, y).statistic, abs=1e-12)
        assert sel.spearman_rho(x, y) == pytest.approx(stats.spearmanr(x, y).statistic, abs=1e-12)


# --- GB300 restatement: invariants only (parity unpinned against the pages) ----

def test_gb300_model_kind_one_is_the_workshop_model(golden):
    g = golden("workshop_h100.json")["large_square"]
    dev = sel.Device(sm_count=132, model_kind=1, peak_tflops_bf16=989.0, hbm_gbs=3350.0)
    best = min(((bm, bn) for bm in sel.WORKSHOP_TILES for bn in sel.WORKSHOP_TILES),
               key=lambda t: sel.gb300_model(8192, 8192, 8192, 0, 2,
                                             sel.Config(t[0], t[1], 64, 4), dev)["predicted_us"])
    assert list(best) == g["best_tile"]


def test_gb300_candidates_are_feasible_unique_and_hold_the_fixed_tile():
    dev = sel.Device()
    for (M, N, K, dt) in [(256, 256, 256, 1), (1000, 1000, 8192, 0), (16, 28672, 8192, 0),
                          (8192, 8192, 8192, 0), (128, 4096, 14336, 0)]:
        cands = sel.gb300_candidates(M, N, K, dt, 3, dev)
        tup = [c.astuple() for c in cands]
        assert len(set(tup)) == len(tup) > 0
        assert all(sel.gb300_check(M, N, K, dt, 3, c, dev) == sel.R_OK for c in cands)
        assert sel.gb300_fixed_config(dt, dev).astuple() in tup
        for c in cands:
            assert sel.smem_bytes(c, dt) <= dev.smem_per_block


def test_gb300_check_reasons():
    dev = sel.Device()
    ok = sel.Config(128, 128, 64, 4)
    assert sel.gb300_check(1024, 1024, 1024, 0, 2, ok, dev) == sel.R_OK
    bad = [(sel.Config(64, 128, 64, 4), sel.R_UMMA_M), (sel.Config(128, 120, 64, 4), sel.R_UMMA_N),
           (sel.Config(128, 96, 64, 4), sel.R_LAYOUT), (sel.Config(128, 128, 48, 4), sel.R_BK),
           (sel.Config(128, 128, 64, 1), sel.R_STAGES), (sel.Config(128, 128, 64, 4, 0, 3), sel.R_SCHEDULE),
           (sel.Config(128, 128, 64, 4, 0, 1, 17), sel.R_SPLIT_K), (sel.Config(128, 128, 64, 12), sel.R_SMEM),
           (sel.Config(128, 128, 64, 4, cta_group=2), sel.R_CTA_GROUP)]
    for cfg, why in bad:
        assert sel.gb300_check(1024, 1024, 1024, 0, 2, cfg, dev) == why, cfg
    assert sel.gb300_check(1024, 1023, 1024, 0, 2, ok, dev) == sel.R_ALIGN
    assert sel.gb300_check(1024, 1024, 1024, 0, 2, sel.Config(256, 256, 64, 2), dev) == sel.R_OK
    assert sel.gb300_check(1024, 1024, 1024, 0, 2, sel.Config(256, 256, 64, 2), dev) == sel.R_OK


def test_gb300_model_terms_behave():
    dev = sel.Device()
    # split-K on an under-filled shape raises wave efficiency and shortens the main loop
    a = sel.gb300_model(1000, 1000, 8192, 0, 3, sel.Config(128, 128, 64, 4), dev)
    b = sel.gb300_model(1000, 1000, 8192, 0, 3, sel.Config(128, 128, 64, 4, split_k=2), dev)
    assert b["wave_eff"] > a["wave_eff"] and b["mma_us"] < a["mma_us"] and b["splitk_us"] > 0
    # the decode shape is bound by HBM, and its bytes are at least the compulsory ones
    d = sel.gb300_model(16, 28672, 8192, 0, 0, sel.Config(256, 16, 128, 3, split_k=1, swap_ab=1), dev)
    assert d["hbm_us"] > d["mma_us"]
    assert d["hbm_bytes"] >= (16 * 8192 + 8192 * 28672 + 16 * 28672) * 2
    # a multi-wave split-K pays the last arriver's reads of every slice
    e = sel.gb300_model(1000, 1000, 8192, 0, 3, sel.Config(128, 256, 64, 4, split_k=8), dev)
    f = sel.gb300_model(1000, 1000, 8192, 0, 3, sel.Config(128, 256, 64, 4, split_k=4), dev)
    assert e["units"] > dev.sm_count >= f["units"] and e["splitk_us"] > 4 * f["splitk_us"]


def test_shipped_set_hand_example():
    # best per shape: 10 (c0), 25 (c1), 4.5 (c2).  Step 1 gains: c0 1+25/30+4.5/5,
    # c1 10/12+1+4.5/9, c2 25/40+1, c3 10/20+4.5/6 -> c0.  Step 2: c1 gains
    # 1-25/30, c2 gains 1-4.5/5 -> c1.  Slowdowns 1, 1, 5/4.5.
    t = [[10, 12, 0, 20], [30, 25, 40, 0], [5, 9, 4.5, 6]]
    chosen, mean, worst = sel.shipped_set_greedy(t, 2)
    assert chosen == [0, 1]
    assert mean == pytest.approx((1 + 1 + 5 / 4.5) / 3, rel=1e-15)
    assert worst == pytest.approx(5 / 4.5, rel=1e-15)
    assert sel.shipped_set_greedy(t, 4)[0] == [0, 1, 2]      # c3 adds nothing
    assert sel.shipped_set_optimal(t, 2) == ([0, 1], pytest.approx(1 + 1 + 4.5 / 5))


def test_shipped_set_greedy_is_within_the_submodular_bound_of_the_optimum():
    rng = np.random.default_rng(5)
    bound = 1 - 1 / math.e
    for trial in range(60):
        ns, nc = rng.integers(2, 7), rng.integers(3, 8)
        t = rng.uniform(1, 10, size=(ns, nc))
        t[rng.uniform(size=(ns, nc)) < 0.2] = 0.0
        for size in range(1, min(4, nc) + 1):
            chosen, _, _ = sel.shipped_set_greedy(t.tolist(), size)
            _, opt = sel.shipped_set_optimal(t.tolist(), size)
            got = sel.shipped_set_value(t.tolist(), chosen)
            assert got >= bound * opt - 1e-12
            assert got <= opt + 1e-12
        # enough members to hold every shape's best: slowdown 1 everywhere
        full, mean, worst = sel.shipped_set_greedy(t.tolist(), nc)
        if all((row > 0).any() for row in t):
            assert mean == pytest.approx(1.0) and worst == pytest.approx(1.0)


def test_shipped_set_single_shape_picks_its_fastest_configuration():
    t = [[7.0, 3.0, 0.0, 5.0]]
    assert sel.shipped_set_greedy(t, 1) == ([1], 1.0, 1.0)
