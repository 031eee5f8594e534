"""Host-side parts of bench.py: the replica aggregation over ranks (two gloo
processes on the CPU) and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 1.0 + rank          # rank 1 is the slower replica
    worst = bench.combine_ranks(elapsed, dist)
    value = bench.job_value(2e9, 8, 10, world, worst)
    q.put((rank, worst, value))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_report_the_max_time_and_the_whole_job_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in out:
        assert worst == 2.0
        assert value == pytest.approx(2e9 * 8 * 10 * 2 / 2.0 / 1e12)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--cpu-budget", "1", "--workload", "fp32_relu_256"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["steps"] == 2


def test_expected_random_best_closed_form_against_enumeration():
    import itertools
    sys.path.insert(0, ROOT)
    import bench
    vals = [5.0, 3.0, 9.0, 4.0, 7.0, 3.5]
    for k in range(1, 7):
        subsets = list(itertools.combinations(vals, k))
        brute = sum(min(vals) / min(s) for s in subsets) / len(subsets)
        assert bench.expected_random_best(vals, k) == pytest.approx(brute, rel=1e-12)


def test_shipped_set_report_on_a_small_table():
    sys.path.insert(0, ROOT)
    import bench
    c = [(128, 128, 64, 4, 0, 1, 1, 1, 0), (256, 256, 64, 3, 0, 1, 1, 1, 0), (256, 128, 64, 4, 0, 1, 1, 2, 0)]
    tables = {"a": {c[0]: 10.0, c[1]: 20.0}, "b": {c[0]: 30.0, c[1]: 15.0, c[2]: 14.0}, "c": {c[2]: 5.0}}
    r = bench.shipped_set_report(tables, sizes=(1, 3))
    assert r["workloads"] == 3 and r["configurations"] == 3
    assert r["1"]["in_sample_worst"] is None            # one member cannot run every workload
    assert r["3"]["in_sample_mean"] == 1.0 and r["3"]["in_sample_worst"] == 1.0
    # c2 first (gain 2), then c0 (gain 1 on "a"); c1 then gains nothing, so the set stops at two
    assert [tuple(x) for x in r["3"]["configs"]] == [c[2], c[0]]


def test_peak_choice_follows_the_sampled_clocks():
    sys.path.insert(0, ROOT)
    import bench
    assert not bench.power_capped({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert bench.power_capped({"sm_mhz": 1515.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert bench.power_capped({"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert not bench.power_capped(None)


def test_clock_samples_are_placed_by_their_own_timestamps():
    sys.path.insert(0, ROOT)
    import bench
    import datetime
    c = bench.ClockSampler(0)
    c.proc = object()                       # as if nvidia-smi were running
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    for i, mhz in enumerate((2070, 1500, 1500, 2070)):
        t = base + datetime.timedelta(milliseconds=100 * i)
        c.samples.append((t.timestamp(), [t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], str(mhz), "2070", "900",
                                          "0x0", "Not Active", "Not Active", "Not Active",
                                          "Active" if mhz < 2000 else "Not Active"]))
    s = c.summary_between(base.timestamp() + 0.05, base.timestamp() + 0.25)
    assert s["samples_in_timed_region"] == 2 and s["sm_mhz"] == 1500 and s["reasons"] == ["sw_power_cap"]


def test_captured_traffic_matches_workload_config_and_build():
    """The roofline's traffic comes from the committed ncu summaries only for the
    same workload, configuration and source digest; anything else reads None."""
    sys.path.insert(0, ROOT)
    import bench
    from autotuning_tcgen05_tmem_gb300 import _build
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    name, ents = next(iter(table.items()))
    ent = ents[0] if isinstance(ents, list) else ents
    got = bench.captured_traffic(name, ent["config"])
    if ent["source_digest"] == _build._sources_digest():
        assert got == ent["dram_bytes_per_launch"]
    else:
        assert got is None
    assert bench.captured_traffic(name, [1] * 9) is None
    assert bench.captured_traffic("no_such_workload", ent["config"]) is None
