"""The multi-GPU bookkeeping of bench.py on CPU ranks (gloo, world size 2).

With several GPUs the layer runs as independent replicas (tokens are
independent without a global capacity): the job's time is the slowest
rank's and its throughput counts every rank's tokens.  These checks run the
same helpers bench.py uses, over two gloo processes on this host.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r reports step times (10 + r, 3 - r) ms
    got = bench.max_over_ranks([10.0 + rank, 3.0 - rank])
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_slowest_rank_sets_the_time_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == [11.0, 3.0]


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_tokens_per_s(16384, 4, 2.0) == pytest.approx(16384 * 4 / 2e-3)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]     # no process group: identity


def _clock_rows(rows):
    """nvidia-smi CSV rows in the sampler's field order: (time, sm MHz,
    reasons active?) per row, the same GPU."""
    lines = []
    for t, sm, slow in rows:
        act = "Active" if slow else "Not Active"
        lines.append(f"2026/01/02 03:04:{t:06.3f}, 0, GPU-x, {sm}, 2032, 900.00 W, 0x0, "
                     f"Not Active, Not Active, {act}, Not Active")
    return "\n".join(lines)


def test_clock_summary_keeps_only_the_timed_region():
    sys.path.insert(0, ROOT)
    import datetime
    import bench
    base = datetime.datetime(2026, 1, 2, 3, 4, 0).timestamp()
    # idle samples (345 MHz) before and after; loaded ones inside [10, 10.3]
    text = _clock_rows([(9.90, 345, False), (10.05, 2032, False), (10.10, 2017, False),
                        (10.25, 2032, False), (10.40, 345, True)])
    got = bench.ClockSampler.summarise(text, "GPU-x", (base + 10.0, base + 10.3))
    assert got["in_region"] == 3 and got["samples"] == 3
    assert got["sm_mhz"] == 2032 and got["sm_max_mhz"] == 2032
    assert got["reasons"] == []                    # the slowdown came after the region
    # another GPU's rows are ignored
    assert bench.ClockSampler.summarise(text, "GPU-y", None) is None


def test_clock_summary_of_a_region_between_two_samples():
    sys.path.insert(0, ROOT)
    import datetime
    import bench
    base = datetime.datetime(2026, 1, 2, 3, 4, 0).timestamp()
    text = _clock_rows([(9.0, 345, False), (10.00, 2032, False), (10.05, 2010, True),
                        (11.0, 345, False)])
    got = bench.ClockSampler.summarise(text, None, (base + 10.01, base + 10.04))
    assert got["in_region"] == 0 and got["samples"] == 2
    assert got["sm_mhz"] == (2032 + 2010) / 2
    assert got["reasons"] == ["sw_thermal_slowdown"]


def test_reference_arm_prints_one_contract_line(capsys):
    """bench.py --impl reference (the oracle on this host) prints one JSON
    line with the keys of the measurement contract."""
    sys.path.insert(0, ROOT)
    import json
    import bench
    bench.main(["--impl", "reference", "--workload", "toy_top2_fp32", "--steps", "2",
                "--warmup", "3", "--cpu-seconds", "0.5"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "toy_top2_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["single_thread_value"] > 0 and cb["host"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_bench_rejects_too_few_warmup_steps():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--warmup", "2"])


def _build_main(out, i):
    sys.path.insert(0, ROOT)
    import bench
    out[i] = bench.build_library()


def test_ranks_started_together_build_the_library_in_turn():
    """bench.py under torchrun: every rank calls the build step at once; the
    file lock lets them through one at a time and all get the library."""
    sys.path.insert(0, ROOT)
    from routing_dispatch_expert_05_b300 import build as B
    B.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_build_main, args=(out, i)) for i in range(3)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(600)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1, 2] and set(res.values()) == {B.LIB_PATH}
