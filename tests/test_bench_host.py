"""Host logic of bench.py on the CPU: rank aggregation over gloo (world size 2) and the clock summary."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, str(ROOT))
    import bench
    d = bench.Dist()
    try:
        # Rank r processed (r + 1) * 100 units in (r + 1) seconds.
        value, slowest = bench.aggregate((rank + 1) * 100.0, float(rank + 1), d)
        d.barrier()
        q.put((rank, value, slowest))
    finally:
        d.close()


def _reference_rank_main(rank, world, port, q):
    import contextlib
    import io
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, str(ROOT))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
                         "--reference-budget", "2"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_under_two_ranks_prints_once():
    """Launched as N ranks, the reference arm runs and prints on rank 0 only; the others exit 0."""
    import json
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reference_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rc0, out0), (r1, rc1, out1) = results
    assert rc0 == 0 and rc1 == 0
    lines = [x for x in out0.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"
    assert not [x for x in out1.splitlines() if x.startswith("{")]


def test_replica_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, slowest in results:
        assert slowest == 2.0                 # the slowest rank's time
        assert value == pytest.approx(300.0 / 2.0)  # all ranks' units / that time


def test_clock_summary_windows_and_reasons():
    sys.path.insert(0, str(ROOT))
    import datetime as dt
    import bench

    def row(t, mhz, slow="Not Active", cap="Not Active"):
        stamp = dt.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return [stamp, "0", str(mhz), "2070", "900.0", "0x0", slow, "Not Active", "Not Active", cap]

    t0 = 1_800_000_000.0
    rows = [row(t0 - 1, 300), row(t0 + 0.1, 1900), row(t0 + 0.2, 1950, cap="Active"), row(t0 + 0.3, 2000),
            row(t0 + 5, 300, slow="Active")]
    s = bench.ClockSampler.summarize(rows, t0, t0 + 1)
    assert s["samples"] == 3 and s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    s2 = bench.ClockSampler.summarize(rows, t0 + 10, t0 + 11)
    assert s2["samples"] == 5 and "hw_slowdown" in s2["reasons"]
    assert bench.ClockSampler.summarize([], 0, 1) is None


def test_reference_arm_line_on_cpu():
    sys.path.insert(0, str(ROOT))
    import bench
    args = bench.argparse.Namespace(workload="tiny", steps=3, warmup=3, gpus=1, reference_budget=2.0)
    d = bench.Dist()
    line = bench.run_reference(args, d)
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["metric"] == bench.METRIC


def test_e2e_is_the_pipelined_drive_whichever_is_faster():
    """The end-to-end figure is fixed in advance to the pipelined drive; the serial one is reported
    beside it and never replaces it, also when it is the faster (a short step)."""
    import bench
    long_step = bench.e2e_line(6.1e12 * 100, 0.0206, 5.4e12 * 100, 0.0234, 100, 1705472, 1048576, 91)
    assert long_step["mode"] == "pipelined" and long_step["value"] == round(6.1e12 * 100 / 1e9, 2)
    assert long_step["serial"]["value"] < long_step["value"] and long_step["passes"] == 91
    short_step = bench.e2e_line(2.3e12, 0.07, 3.1e12, 0.05, 1000, 10, 20, 5)
    assert short_step["mode"] == "pipelined" and short_step["value"] == round(2.3e12 / 1e9, 2)
    assert short_step["serial"]["value"] > short_step["value"]
    assert short_step["h2d_bytes_per_step"] == 10 and short_step["d2h_bytes_per_step"] == 20


def test_bf16_peak_burst_and_sustained(tmp_path, monkeypatch):
    """A kernel timed alone is compared with the burst GEMM rate, one timed in a second-long loop with the
    sustained one; without the measured file the fallbacks are used and said to be."""
    import json
    import bench
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1913.6, "bf16_tflops_sustained": 1696.8}))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.bf16_peak_tflops() == (1913.6, "measured")
    assert bench.bf16_peak_tflops(sustained=True) == (1696.8, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1913.6}))
    assert bench.bf16_peak_tflops(sustained=True) == (1913.6, "measured")   # no sustained figure measured
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.bf16_peak_tflops()[1] == "fallback" and bench.bf16_peak_tflops(True)[1] == "fallback"
