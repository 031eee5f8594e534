"""Host logic of the library, called through the C ABI on a machine without a
GPU: symbol exports, and parity of the feasibility filter, candidate
generator, cost model, tile schedule and rank statistics with the oracle's
independent restatements (integer results bit-exact, model times to 1e-12)."""
import math
import os
import random
import re

import numpy as np
import pytest

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import _build
from oracle import selection as sel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def to_oracle_device(d) -> sel.Device:
    return sel.Device(**{k: v for k, v in d.asdict().items()})


def to_oracle_config(c) -> sel.Config:
    return sel.Config(*c.astuple())


SHAPES = [(256, 256, 256, 1, 2), (1000, 1000, 8192, 0, 3), (8192, 8192, 8192, 0, 2),
          (16, 28672, 8192, 0, 0), (128, 4096, 14336, 0, 3), (512, 1024, 4096, 0, 3),
          (2048, 28672, 4096, 0, 3), (8192, 4096, 14336, 0, 3), (17, 96, 40, 1, 1),
          (1, 8, 8, 0, 0), (300, 200, 72, 0, 2), (64, 64, 0, 0, 1),
          # FP8 E4M3 operands (bf16 C): K-major copy of B, 128-byte spans of 128 elements
          (1000, 1000, 8192, 2, 3), (8192, 8192, 8192, 2, 2), (16, 28672, 8192, 2, 0), (300, 200, 128, 2, 2),
          (512, 1024, 4096, 2, 6), (100, 104, 48, 2, 1),
          # block-scaled FP8 (MX): no swap, no pairs, bn 128/256, bk 128/256, scale slots in TMEM
          (1000, 1000, 8192, 3, 3), (8192, 8192, 8192, 3, 2), (16, 28672, 8192, 3, 0), (300, 200, 128, 3, 2),
          (512, 1024, 4096, 3, 6), (100, 104, 48, 3, 1),
          # gated epilogues (ReGLU, GeGLU, SwiGLU) over a fused gate+up weight
          (512, 28672, 4096, 0, 8), (16, 28672, 4096, 0, 9), (1000, 1024, 8192, 2, 7), (256, 256, 256, 1, 8),
          (300, 192, 72, 0, 7)]


def test_library_exports_every_declared_symbol():
    with open(os.path.join(ROOT, "include", "gemm_gb300.h")) as f:
        header = f.read()
    declared = set(re.findall(r"^(?:const\s+)?(?:int64_t|int|void|char)\s*\*?\s*(gemm_[a-z_]+)\s*\(",
                              header, flags=re.M))
    assert declared == set(g.EXPORTS)
    L = g.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_version_and_defaults():
    assert g.version().startswith("gb300-tcgen05-gemm")
    d = g.device_params_default()
    assert d.sm_count == 152 and d.threads_per_cta == 320 and d.model_kind == 0
    w = g.device_params_workshop()
    assert (w.sm_count, w.model_kind, w.peak_tflops_bf16, w.hbm_gbs) == (132, 1, 989.0, 3350.0)


@pytest.mark.parametrize("M,N,K,dt,epi", SHAPES)
def test_enumeration_equals_oracle(M, N, K, dt, epi):
    d = g.device_params_default()
    lib_c = [c.astuple() for c in g.enumerate_configs(M, N, K, dt, epi, d)]
    orc_c = [c.astuple() for c in sel.gb300_candidates(M, N, K, dt, epi, to_oracle_device(d))]
    assert lib_c == orc_c


def test_enumeration_on_other_devices():
    for sms, smem in [(132, 232448), (148, 232448), (80, 101376), (152, 166912)]:
        d = g.device_params_default()
        d.sm_count, d.smem_per_block = sms, smem
        for (M, N, K, dt, epi) in SHAPES[:6]:
            lib_c = [c.astuple() for c in g.enumerate_configs(M, N, K, dt, epi, d)]
            orc_c = [c.astuple() for c in sel.gb300_candidates(M, N, K, dt, epi, to_oracle_device(d))]
            assert lib_c == orc_c


def test_check_config_equals_oracle_on_a_grid():
    d = g.device_params_default()
    od = to_oracle_device(d)
    rng = random.Random(5)
    grid = list(__import__("itertools").product(
        (64, 128, 192, 256), (8, 16, 32, 48, 64, 96, 128, 192, 256, 272), (16, 32, 48, 64, 128, 256, 320),
        (1, 2, 3, 8, 16, 17), (0, 1, 2), (1, 3, 4, 16), (1, 2, 16, 17), (1, 2), (0, 1, 2)))
    sample = rng.sample(grid, 6000)
    for (M, N, K, dt) in [(1000, 1000, 8192, 0), (256, 256, 256, 1), (16, 28672, 8192, 0), (100, 36, 12, 0),
                          (100, 36, 12, 1), (5, 5, 5, 1), (1000, 1008, 8192, 3), (16, 28672, 8192, 3),
                          (100, 104, 48, 3)]:
        for t in sample:
            c = g.make_config(*t)
            for epi in (2, 8):
                assert g.check_config(M, N, K, dt, epi, c, d) == sel.gb300_check(M, N, K, dt, epi, sel.Config(*t), od), \
                    (M, N, K, dt, epi, t)


def test_check_config_register_rule():
    d = g.device_params_default()
    d.kernel_regs = 400
    c = g.make_config(128, 128, 64, 4)
    assert g.check_config(1024, 1024, 1024, 0, 2, c, d) == g.REASONS.index("REGS")
    d.kernel_regs = 145
    assert g.check_config(1024, 1024, 1024, 0, 2, c, d) == 0


def test_fixed_config_equals_oracle_and_is_128x128():
    d = g.device_params_default()
    for dt in (0, 1):
        f = g.fixed_config(dt, d)
        assert f.astuple() == sel.gb300_fixed_config(dt, to_oracle_device(d)).astuple()
        assert (f.bm, f.bn, f.split_k, f.swap_ab) == (128, 128, 1, 0)


@pytest.mark.parametrize("M,N,K,dt,epi", SHAPES)
def test_cost_model_equals_oracle(M, N, K, dt, epi):
    d = g.device_params_default()
    od = to_oracle_device(d)
    for c in g.enumerate_configs(M, N, K, dt, epi, d):
        t = g.model_predict(M, N, K, dt, epi, c, d).asdict()
        o = sel.gb300_model(M, N, K, dt, epi, to_oracle_config(c), od)
        for key in ("predicted_us", "mma_us", "l2_us", "hbm_us", "latency_us", "epilogue_us", "splitk_us",
                    "launch_us", "wave_eff", "tile_eff", "pad_eff", "hbm_bytes", "l2_bytes", "flops"):
            assert t[key] == pytest.approx(o[key], rel=1e-12, abs=1e-12), (key, c)
        for key in ("tiles", "units", "waves", "ctas"):
            assert t[key] == o[key]


def test_cost_model_workshop_mode_reproduces_the_printed_numbers(golden):
    w = g.device_params_workshop()
    gl = golden("workshop_h100.json")
    tiles = [(a, b) for a in (32, 64, 128, 256) for b in (32, 64, 128, 256)]

    def times(M, N, K):
        return {t: g.model_predict(M, N, K, 0, 0, g.make_config(t[0], t[1], 64, 4), w).predicted_us
                for t in tiles}
    sq = times(*gl["large_square"]["shape_reading"])
    best = min(tiles, key=lambda t: sq[t])        # first minimum in bm-outer order
    assert list(best) == gl["large_square"]["best_tile"]
    assert round(sq[best]) == gl["large_square"]["best_us"]
    assert round(max(sq.values()) / sq[best], 2) == gl["large_square"]["worst_over_best"]
    assert round(sq[(128, 128)] / sq[best], 2) == gl["large_square"]["fixed_128_over_best"]
    uf = times(*gl["underfilled"]["shape"])
    best = min(tiles, key=lambda t: uf[t])
    assert list(best) == gl["underfilled"]["best_tile"]
    assert round(uf[(128, 128)] / uf[best], 2) == gl["underfilled"]["fixed_128_over_best"]
    te = g.model_predict(*gl["underfilled"]["shape"], 0, 0, g.make_config(32, 256, 64, 4), w)
    assert round(100 * te.wave_eff) == gl["underfilled"]["best_wave_efficiency_percent"]
    dc = times(*gl["decode_16_tokens"]["shape_reading"])
    assert len(set(dc.values())) == 1
    assert round(next(iter(dc.values())), 1) == gl["decode_16_tokens"]["all_tie_us"]


def test_schedule_equals_oracle():
    rng = random.Random(9)
    for _ in range(300):
        tm, tn = rng.randint(1, 40), rng.randint(1, 40)
        S = rng.choice([1, 2, 3, 4, 8, 16])
        raster, group = rng.randint(0, 1), rng.choice([1, 2, 4, 8, 16])
        nkb = rng.randint(S, 300)
        for u in rng.sample(range(tm * tn * S), min(50, tm * tn * S)):
            assert g.schedule_unit(u, tm, tn, S, raster, group, nkb) == \
                sel.schedule_unit(u, tm, tn, S, raster, group, nkb)


def test_rank_agreement_equals_oracle():
    rng = random.Random(13)
    for n in (2, 3, 7, 40):
        for _ in range(20):
            x = [rng.choice([1.0, 2.0, rng.random()]) for _ in range(n)]
            y = [rng.choice([0.5, rng.random(), rng.random()]) + 0.01 for _ in range(n)]
            s = g.rank_agreement(x, y)
            o = sel.rank_agreement(x, y)
            for key in ("kendall_tau", "spearman_rho", "regret"):
                a, b = getattr(s, key), o[key]
                assert (math.isnan(a) and math.isnan(b)) or a == pytest.approx(b, abs=1e-12)
            assert s.top1_hit == o["top1_hit"]


def test_argument_errors_are_status_codes():
    d = g.device_params_default()
    with pytest.raises(g.GemmError) as e:
        g.check_config(-1, 4, 4, 0, 0, g.make_config(128, 128, 64, 4), d)
    assert e.value.code == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError):
        g.schedule_unit(10, 2, 2, 1, 0, 1, 4)
    with pytest.raises(g.GemmError):
        g.rank_agreement([1.0], [2.0])
    with pytest.raises(g.GemmError):
        g.debug_set(0, 0)
    with pytest.raises(g.GemmError):
        g.debug_set(7, 2)
    with pytest.raises(g.GemmError):
        g.debug_set(8, 1)


def test_device_calls_without_a_gpu_fail_loudly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(g.GemmError) as e:
        g.plan(128, 128, 128, "bf16", "relu")
    assert e.value.code in (g.ERR_NO_DEVICE, g.ERR_UNSUPPORTED)
    with pytest.raises(g.GemmError):
        g.device_params_query()


def test_tuning_database_round_trip(tmp_path):
    """The database file is parsed and rewritten without a GPU: comments and
    malformed lines are skipped, entries keep their key and nine fields."""
    g.cache_clear()
    src = tmp_path / "db.txt"
    src.write_text("# comment\n"
                   "1000|1000|8192|0|3|NVIDIA GB300|152|v\t256 128 64 4 0 1 4 1 0\n"
                   "16|28672|8192|0|0|NVIDIA GB300|152|v\t128 16 128 5 0 8 1 1 1\n"
                   "broken line without a tab\n")
    assert g.cache_load(str(src)) == 2
    assert g.cache_stats()["entries"] == 2
    out = tmp_path / "out.txt"
    assert g.cache_save(str(out)) == 2
    body = [l for l in out.read_text().splitlines() if not l.startswith("#")]
    assert sorted(body) == sorted(l for l in src.read_text().splitlines() if "\t" in l)
    g.cache_clear()
    assert g.cache_stats()["entries"] == 0
    with pytest.raises(g.GemmError):
        g.cache_load(str(tmp_path / "missing.txt"))


def test_shipped_set_selection_equals_oracle():
    rng = np.random.default_rng(11)
    for trial in range(40):
        ns, nc = int(rng.integers(1, 9)), int(rng.integers(1, 12))
        t = rng.uniform(1, 50, size=(ns, nc))
        t[rng.uniform(size=(ns, nc)) < 0.25] = 0.0
        for k in (1, 2, 3, 5, 12):
            got = g.select_config_set(t, k)
            want = sel.shipped_set_greedy(t.tolist(), k)
            assert got[0] == want[0]
            assert got[1] == pytest.approx(want[1], rel=1e-12) and got[2] == pytest.approx(want[2], rel=1e-12)
    assert g.lib().gemm_select_config_set(None, 2, 2, 1, None, None, None, None) == g.ERR_INVALID_ARG


def test_operand_declaration_argument_checks():
    # A null plan is refused without a device; unknown operand letters never
    # reach the library.
    assert g.lib().gemm_plan_set_independent_operands(None, g.OPERAND_B) == g.ERR_INVALID_ARG

    class NoPlan:
        _h = None

    with pytest.raises(ValueError):
        g.Plan.set_independent_operands(NoPlan(), "AC")
