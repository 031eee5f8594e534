"""The selection layer on the GPU: tune-once cache, the fixed-tile switch,
selection exactness (the chosen configuration is the measured fastest within
3%), the tune report, and the bounded-wait timeout path."""
import ctypes
import os

import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import alloc_out, normalised_error, operands

pytestmark = pytest.mark.gpu


def test_tune_once_cache_by_shape_and_dtype():
    g.cache_clear()
    M, N, K = 256, 512, 1024
    p1 = g.plan(M, N, K, "bf16", "relu")
    s1 = g.cache_stats()
    assert (s1["tunes"], s1["hits"], s1["entries"]) == (1, 0, 1)
    p2 = g.plan(M, N, K, "bf16", "relu")            # same key: served from the cache
    s2 = g.cache_stats()
    assert (s2["tunes"], s2["hits"], s2["entries"]) == (1, 1, 1)
    assert p1.config.astuple() == p2.config.astuple()
    g.plan(M, N, K, "fp32", "relu").close()         # dtype is part of the key
    g.plan(M, N, K, "bf16", "gelu").close()         # so is the epilogue
    s3 = g.cache_stats()
    assert (s3["tunes"], s3["entries"]) == (3, 3)
    p1.close()
    p2.close()


def test_disable_autotune_gives_the_fixed_tile():
    dev = g.device_params_query()
    os.environ["GEMM_DISABLE_AUTOTUNE"] = "1"
    try:
        before = g.cache_stats()["tunes"]
        with g.plan(640, 768, 2048, "bf16", "gelu") as p:
            assert p.config.astuple() == g.fixed_config("bf16", dev).astuple()
            A, B, bias = operands(640, 768, 2048, "bf16", "scaled_normal", seed=3)
            C, _ = alloc_out(640, 768, g.BF16)
            p.run(A.cuda(), B.cuda(), bias.cuda(), C)
            assert p.status() == 0
        assert g.cache_stats()["tunes"] == before
    finally:
        del os.environ["GEMM_DISABLE_AUTOTUNE"]
    assert normalised_error(C.cpu(), A, B, bias, "gelu") <= 2e-3


def test_tune_report_is_complete_and_ranked():
    w = inputs.WORKLOADS["bf16_gelu_out_t512"]
    r = g.tune(w.M, w.N, w.K, w.dtype, w.epi, topk=0)
    st = r.stats
    assert st.n_candidates == st.n_measured == len(r.rows) > 50
    meas = [row.measured_us for row in r.rows]
    assert all(m > 0 for m in meas) and meas == sorted(meas)
    assert [row.measured_rank for row in r.rows] == list(range(len(r.rows)))
    assert sorted(row.model_rank for row in r.rows) == list(range(len(r.rows)))
    assert -1 <= st.kendall_tau <= 1 and -1 <= st.spearman_rho <= 1
    assert st.best_us == meas[0] and st.fixed_us >= st.best_us
    assert st.regret >= 0 and st.tune_seconds > 0
    fixed = g.fixed_config(w.dtype, g.device_params_query()).astuple()
    assert fixed in [row.config.astuple() for row in r.rows]


def _time_configs(w, cfgs, rounds=7, reps=20):
    """Median microseconds per config: interleaved rounds over rotating inputs."""
    sets = []
    for s in range(4):
        A, B, bias = inputs.make_workload(w, seed=40 + s, device="cuda")
        sets.append((A, B, bias, torch.empty(w.M, w.N, dtype=A.dtype, device="cuda")))
    plans = [g.plan_with_config(w.M, w.N, w.K, w.dtype, w.epi, c) for c in cfgs]
    for p in plans:
        for (A, B, bias, C) in sets:
            p.run(A, B, bias, C)
    torch.cuda.synchronize()
    times = [[] for _ in cfgs]
    for r in range(rounds):
        for i in [(j + r) % len(cfgs) for j in range(len(cfgs))]:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for k in range(reps):
                A, B, bias, C = sets[k % len(sets)]
                plans[i].run(A, B, bias, C)
            e1.record()
            torch.cuda.synchronize()
            times[i].append(e0.elapsed_time(e1) * 1e3 / reps)
    for p in plans:
        assert p.status() == 0
        p.close()
    return [float(np.median(t)) for t in times]


@pytest.mark.parametrize("name", ["bf16_gelu_out_t512", "bf16_gelu_1000x1000x8192"])
def test_selection_is_the_measured_fastest_within_3_percent(name):
    w = inputs.WORKLOADS[name]
    g.cache_clear()
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
        chosen = p.config
    r = g.tune(w.M, w.N, w.K, w.dtype, w.epi, topk=0)
    rivals = [row.config for row in r.rows[:6] if row.config.astuple() != chosen.astuple()]
    for attempt in range(2):       # one re-measure if clocks moved during the first
        t = _time_configs(w, [chosen] + rivals)
        if t[0] <= 1.03 * min(t):
            break
    assert t[0] <= 1.03 * min(t), (chosen, t)


def test_bounded_wait_returns_timeout_and_the_context_survives():
    A, B, bias = operands(256, 256, 512, "bf16", "int", seed=5)
    Ad, Bd, bd = A.cuda(), B.cuda(), bias.cuda()
    C, _ = alloc_out(256, 256, g.BF16)
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 2)
    with g.plan_with_config(256, 256, 512, "bf16", "relu", cfg) as p:
        g.debug_set(0, 50_000_000)           # 50 ms wait limit
        g.debug_set(1, 1)                    # the epilogue waits on a barrier nothing signals
        try:
            p.run(Ad, Bd, bd, C)
            assert p.status() == g.ERR_TIMEOUT
            assert "wait expired" in g.last_error()
        finally:
            g.debug_set(1, 0)
            g.debug_set(0, 2_000_000_000)
        p.run(Ad, Bd, bd, C)                 # the same plan, and the context, still work
        assert p.status() == 0
    from gpu_util import device_bits, oracle_rounded_bits
    assert np.array_equal(device_bits(C.cpu()), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


def test_zero_extents_through_the_tuned_path():
    with g.plan(0, 64, 64, "bf16", "none") as p:
        p.run(None, None, None, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
        assert p.status() == 0
    bias = torch.linspace(-1, 1, 64).to(torch.bfloat16).cuda()
    C = torch.empty(40, 64, dtype=torch.bfloat16, device="cuda")
    with g.plan(40, 64, 0, "bf16", "relu") as p:
        p.run(None, None, bias, C)
        assert p.status() == 0
    assert torch.equal(C.cpu(), torch.relu(bias.float()).to(torch.bfloat16).cpu().expand(40, 64))


def test_tuning_database_serves_a_later_process_and_persists_new_winners(tmp_path):
    g.cache_clear()
    w = inputs.WORKLOADS["bf16_gelu_kv_t512"]
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
        chosen = p.config.astuple()
    db = tmp_path / "tuning.db"
    assert g.cache_save(str(db)) == 1
    g.cache_clear()
    assert g.cache_load(str(db)) == 1
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:     # served from the loaded entry
        assert p.config.astuple() == chosen
    st = g.cache_stats()
    assert st["tunes"] == 0 and st["hits"] == 1
    # just-in-time persistence: a new winner is appended to GEMM_TUNING_DB
    g.cache_clear()
    jit = tmp_path / "jit.db"
    os.environ["GEMM_TUNING_DB"] = str(jit)
    try:
        g.plan(384, 512, 1024, "bf16", "relu").close()
    finally:
        del os.environ["GEMM_TUNING_DB"]
    lines = [l for l in jit.read_text().splitlines() if "\t" in l]
    assert len(lines) == 1 and lines[0].startswith("384|512|1024|0|2|")


def test_search_strategies_measure_their_budget():
    w = inputs.WORKLOADS["bf16_gelu_out_t512"]
    rnd = g.tune_search(w.M, w.N, w.K, w.dtype, w.epi, g.SEARCH_RANDOM_K, k=8, seed=7)
    assert rnd.stats.n_measured == 8
    again = g.tune_search(w.M, w.N, w.K, w.dtype, w.epi, g.SEARCH_RANDOM_K, k=8, seed=7)
    pick = sorted(r.config.astuple() for r in rnd.rows if r.measured_us > 0)
    assert pick == sorted(r.config.astuple() for r in again.rows if r.measured_us > 0)  # seeded
    top = g.tune_search(w.M, w.N, w.K, w.dtype, w.epi, g.SEARCH_MODEL_TOPK, k=8)
    assert top.stats.n_measured in (8, 9)                # + the fixed tile when it is not in the top 8
    measured = [r for r in top.rows if r.measured_us > 0]
    assert sorted(r.model_rank for r in measured)[:8] == list(range(8))


def test_plan_from_list_times_only_the_list_and_picks_its_fastest():
    w = inputs.WORKLOADS["bf16_gelu_out_t512"]
    C = g.make_config
    shipped = [C(128, 128, 64, 4), C(256, 128, 128, 4, 0, 1, 1, 2), C(128, 64, 64, 6), C(256, 256, 64, 6, 0, 1, 1, 2),
               C(256, 256, 64, 12)]                            # the last breaks the shared-memory rule
    before = g.cache_stats()
    with g.plan_from_list(w.M, w.N, w.K, w.dtype, w.epi, shipped) as p:
        chosen = p.config.astuple()
    assert g.cache_stats() == before                        # the cache is neither read nor written
    feasible = shipped[:4]
    assert chosen in [c.astuple() for c in feasible]
    for attempt in range(2):
        t = _time_configs(w, feasible)
        mine = t[[c.astuple() for c in feasible].index(chosen)]
        if mine <= 1.03 * min(t):
            break
    assert mine <= 1.03 * min(t), (chosen, t)
    with pytest.raises(g.GemmError) as e:
        g.plan_from_list(w.M, w.N, w.K, w.dtype, w.epi, [C(256, 256, 64, 12)])
    assert e.value.code == g.ERR_UNSUPPORTED


def test_tune_batch_fills_the_cache_and_the_database(tmp_path):
    g.cache_clear()
    db = tmp_path / "aot.db"
    shapes = [(256, 512, 1024), (384, 512, 1024), (512, 1024, 2048)]
    assert g.tune_batch(shapes, "bf16", "relu", str(db)) == 3
    assert g.cache_stats()["entries"] == 3
    assert g.tune_batch(shapes, "bf16", "relu") == 0         # all cached now
    lines = [l for l in db.read_text().splitlines() if "\t" in l]
    assert len(lines) == 3
    g.cache_clear()
    assert g.cache_load(str(db)) == 3
    for M, N, K in shapes:
        g.plan(M, N, K, "bf16", "relu").close()
    assert g.cache_stats()["tunes"] == 0


def test_checked_runs_report_a_device_timeout_from_the_run_itself():
    A, B, bias = operands(256, 256, 512, "bf16", "int", seed=6)
    Ad, Bd, bd = A.cuda(), B.cuda(), bias.cuda()
    C, _ = alloc_out(256, 256, g.BF16)
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 2)
    with g.plan_with_config(256, 256, 512, "bf16", "relu", cfg) as p:
        g.debug_set(4, 1)                    # checked runs: every run synchronises and reads the status
        try:
            p.run(Ad, Bd, bd, C)             # a normal run returns OK
            g.debug_set(0, 50_000_000)
            g.debug_set(1, 1)                # the epilogue waits on a barrier nothing signals
            with pytest.raises(g.GemmError) as e:
                p.run(Ad, Bd, bd, C)
            assert e.value.code == g.ERR_TIMEOUT
        finally:
            g.debug_set(1, 0)
            g.debug_set(0, 2_000_000_000)
            g.debug_set(4, 0)
        p.run(Ad, Bd, bd, C)
        assert p.status() == 0
    from gpu_util import device_bits, oracle_rounded_bits
    assert np.array_equal(device_bits(C.cpu()), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


def test_tuning_on_the_callers_operands():
    """gemm_tune_on / gemm_plan_tuned_on time the candidates on copies of the
    caller's operands: the caller's buffers are left as they were, the plan
    runs correctly, and the winner is cached under gemm_plan's key."""
    M, N, K = 256, 384, 1024
    A, B, bias = operands(M, N, K, "bf16", "int", seed=31)
    Ad, Bd, bd = A.cuda(), B.cuda(), bias.cuda()
    before = [t.clone() for t in (Ad, Bd, bd)]
    r = g.tune_on(M, N, K, "bf16", "relu", Ad, Bd, bd, topk=6)
    assert r.stats.n_measured >= 6 and all(row.status == 0 for row in r.rows if row.measured_us > 0)
    g.cache_clear()
    with g.plan_tuned_on(M, N, K, "bf16", "relu", Ad, Bd, bd) as p:
        Cd, _ = alloc_out(M, N, g.BF16)
        p.run(Ad, Bd, bd, Cd)
        assert p.status() == 0
        cfg = p.config.astuple()
    for t, b in zip((Ad, Bd, bd), before):
        assert torch.equal(t, b)
    from gpu_util import device_bits, oracle_rounded_bits
    assert np.array_equal(device_bits(Cd.cpu()), oracle_rounded_bits(A, B, bias, "relu", g.BF16))
    st = g.cache_stats()
    with g.plan(M, N, K, "bf16", "relu") as p2:          # served from the cache
        assert p2.config.astuple() == cfg
    assert g.cache_stats()["hits"] == st["hits"] + 1
    # a missing operand is an argument error
    rc = g.lib().gemm_tune_on(M, N, K, g.BF16, 2, None, None, g._ptr(Bd), None, g._ptr(bd), 4, None, 0,
                              ctypes.byref(ctypes.c_int32(0)), None)
    assert rc == g.ERR_INVALID_ARG


def test_uniform_and_normal_tuning_fills_both_run():
    M, N, K = 256, 256, 512
    try:
        g.debug_set(6, 0)
        a = g.tune(M, N, K, "bf16", "gelu", topk=4)
    finally:
        g.debug_set(6, 1)
    b = g.tune(M, N, K, "bf16", "gelu", topk=4)
    assert a.stats.n_measured >= 4 and b.stats.n_measured >= 4
