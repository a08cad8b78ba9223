"""Host logic of bench.py without a GPU: the N>1 replica path's max-over-ranks
timing (world size 2 over gloo), argument handling and peak lookup."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    w, r, loc = bench.dist_env()
    got = bench.reduce_max(10.0 * (rank + 1), w, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, loc, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1, "cpu") == 3.5


def test_warmup_must_be_at_least_three():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peaks_lookup_has_the_denominators():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 500


def test_clock_summary_keeps_the_timed_window():
    import datetime
    cs = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)

    def line(dt_ms, mhz, cap):
        ts = (base + datetime.timedelta(milliseconds=dt_ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"

    # samples every 50 ms from 0 to 1000 ms; the timed window is 410..490 ms
    cs.lines = [line(t, 1000 + t, "Active" if t == 450 else "Not Active") for t in range(0, 1001, 50)]
    t0 = (base + datetime.timedelta(milliseconds=410)).timestamp()
    t1 = (base + datetime.timedelta(milliseconds=490)).timestamp()
    s = cs.summary(t0, t1)
    assert s["samples"] == 3  # 360 .. 540 ms: one interval of slack on each side
    assert s["sm_mhz"] == 1450
    assert s["reasons"] == ["sw_power_cap"]
    assert cs.summary(t1 + 10, t1 + 20) is None


def test_clock_sampler_drains_its_pipe_while_running():
    # a sampler that writes far more than a pipe buffer before it is stopped
    # must neither stall nor lose lines: the reader thread keeps up
    import sys

    class Fake(bench.ClockSampler):
        def command(self):
            code = ("import sys, time\n"
                    "for i in range(4000):\n"
                    "    sys.stdout.write('%06d' % i + ',' + 'x' * 120 + '\\n')\n"
                    "sys.stdout.flush()\n"
                    "time.sleep(30)\n")
            return [sys.executable, "-c", code]

    cs = Fake(0)
    cs.start()
    import time
    deadline = time.time() + 20
    while len(cs.lines) < 4000 and time.time() < deadline:
        time.sleep(0.05)
    cs.stop()
    assert len(cs.lines) == 4000  # ~500 KB went through while the process kept running
    assert cs.lines[0].startswith("000000,") and cs.lines[-1].startswith("003999,")
    assert cs.summary(0.0, 1.0) is None  # not nvidia-smi lines: nothing to summarise


def test_reference_arm_prints_one_contract_line():
    # the reference arm times the oracle on the host cores: one JSON line with
    # the same metric and config as the GPU arm, and no GPU work at all
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    import time
    t0 = time.time()
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--cpu-budget-s", "2"], cwd=root, capture_output=True,
                       text=True, timeout=600)
    elapsed = time.time() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["gpu_launches"] == 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    # ms_per_step is a measured sample time, not an extrapolation: the steps it
    # claims fit inside the process's own run
    assert 0 < d["steps"] * d["ms_per_step"] / 1e3 <= d["wall_s_timed_region"] <= elapsed
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("pages-benchmark-shaped")
