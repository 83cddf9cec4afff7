"""Benchmark of the paged KV-cache hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload llama3_8b]

One step = one pass of the whole hot path over one batch: kv_append of this
step's token for every sequence, then paged decode attention (partition
kernel + merge kernel) over the block-table KV cache.  The default workload
is one LLaMA-3-8B-shaped layer (B 128, 32 q / 8 kv heads, head_dim 128,
context lengths uniform in 512..4096, block 16, ~1.2 GB of K+V): synthetic
bf16 N(0, 1) data from a seeded generator.

Reported (one JSON line on rank 0):
  value       algorithmic GB/s of the step (attention + append bytes) with the
              inputs resident in HBM, device-timed with CUDA events: the median
              of repeated timed passes of K steps (at least --passes, and about
              --min-seconds of timed work, so the clock samples cover it);
  e2e         the same metric through the public API with every step's inputs
              copied from pinned host memory and its output read back, inside
              the timed region; the copies run on their own streams, double-
              buffered, overlapping the neighbouring steps' kernels (the serial
              form, copies and kernels one after another, is reported beside it
              and never replaces it);
  roofline    the partition kernel (dominant): algorithmic bytes per launch /
              its mean duration (CUDA events on the launching stream, taken in
              passes interleaved with the value passes) against the measured
              HBM copy bandwidth;
  cpu_baseline  the fp64 CPU oracle on the host cores, on the same workload.
``--impl reference`` times that oracle as the reference arm.

Multi-GPU: ``torchrun --nproc-per-node N bench.py --gpus N``: every rank runs
an independent replica of the step on its own GPU (no collective on the
path; weak scaling); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

from workloads import SPECS, algorithmic_bytes, append_bytes, make_decode_case  # noqa: E402

METRIC = "paged decode attention achieved HBM GB/s (% of GB300 peak); seq·layer/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2 ** 20


KERNEL_SOURCES = {
    "paged_decode_partition_kernel": ("paged_kv_cache_275_gb300/csrc/paged_decode.cu",
                                      "paged_kv_cache_275_gb300/csrc/pkv_internal.h"),
    "paged_prefill_kernel": ("paged_kv_cache_275_gb300/csrc/paged_prefill.cu",
                             "paged_kv_cache_275_gb300/csrc/paged_prefill.h",
                             "paged_kv_cache_275_gb300/csrc/pkv_internal.h"),
    "kv_append_kernel": ("paged_kv_cache_275_gb300/csrc/kv_append.cu",
                         "paged_kv_cache_275_gb300/csrc/pkv_internal.h"),
}


def source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from profiles/traffic.txt, if measured on the current kernel source."""
    path = ROOT / "profiles" / "traffic.txt"
    if not path.exists():
        return None
    want = source_hash(kernel)
    for line in path.read_text().splitlines():
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload and f[2] == want:
            return float(f[3])
    return None


def prefill_compulsory_bytes(c) -> int:
    """Bytes a prefill launch must move at least: q and out, plus every cached K/V row its queries see
    (each (sequence, kv head) row read once) and the block-table entries."""
    lens = c.context_lens.cpu().tolist()
    hkv, d = c.spec.num_kv_heads, c.spec.head_dim
    qo = 2 * c.q.numel() * c.q.element_size()
    kv = sum(2 * L * hkv * d * 2 for L in lens)
    tables = sum(4 * ((L + 15) // 16) for L in lens)
    return int(qo + kv + tables)


def bf16_peak_tflops(sustained: bool = False) -> tuple[float, str]:
    """The measured cuBLAS bf16 dense rate: the burst figure for a kernel timed alone, the sustained one
    (seconds of back-to-back GEMMs at the power cap) for a kernel timed in a loop that long."""
    try:
        peaks_json = json.loads((ROOT / "MEASURED_PEAKS.json").read_text())
        if sustained and "bf16_tflops_sustained" in peaks_json:
            return float(peaks_json["bf16_tflops_sustained"]), "measured"
        return float(peaks_json["bf16_tflops"]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def peaks() -> tuple[float, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if not self.pg:
            return x
        dev = f"cuda:{self.local_rank}" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(per_rank_units: float, per_rank_seconds: float, dist: Dist) -> tuple[float, float]:
    """Whole-job throughput: units summed over ranks / the slowest rank's time."""
    total_units = dist.sum(per_rank_units)
    slowest = dist.max(per_rank_seconds)
    return total_units / slowest, slowest


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.proc = None
        self.gpu = gpu_index
        self.windows: list[tuple[float, float]] = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> list[list[str]]:
        if not self.proc:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        return rows

    @staticmethod
    def summarize(rows, t0: float, t1: float) -> dict | None:
        import datetime as _dt
        if not rows:
            return None

        def ts(r):
            try:
                return _dt.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except Exception:
                return None

        inside = [r for r in rows if ts(r) is not None and t0 <= ts(r) <= t1]
        window = "timed region"
        if not inside:
            inside, window = rows, "warm-up + timed region (timed region shorter than one sample)"

        def num(x):
            try:
                return float(x)
            except Exception:
                return None

        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        mx = [num(r[3]) for r in inside if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        power = [num(r[4]) for r in inside if num(r[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


def nvidia_smi_id(dev: torch.device) -> str:
    """nvidia-smi --id for a torch device (its PCI bus id; CUDA_VISIBLE_DEVICES may renumber)."""
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(dev.index or 0)


# ---------------------------------------------------------------------------
# CPU side: the oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_step_seconds(case_cpu, threads: int) -> float:
    import oracle
    kc, vc = case_cpu.k_cache, case_cpu.v_cache
    t = time.perf_counter()
    st = oracle.kv_append(case_cpu.new_k, case_cpu.new_v, case_cpu.slot_mapping, kc, vc)
    _, st2 = oracle.paged_decode_attention(case_cpu.q, kc, vc, case_cpu.block_tables, case_cpu.context_lens,
                                           case_cpu.scale, num_threads=threads)
    dt = time.perf_counter() - t
    if st != 0 or st2 != 0:
        raise RuntimeError("oracle failed on the benchmark workload")
    return dt


def step_bytes(case) -> int:
    s = case.spec
    return (algorithmic_bytes(case.context_lens.cpu(), s.num_q_heads, s.num_kv_heads, s.head_dim)
            + append_bytes(int(case.slot_mapping.numel()), s.num_kv_heads, s.head_dim))


def cpu_baseline(case_cpu, target_s: float = 10.0, max_s: float = 30.0) -> dict:
    threads = os.cpu_count() or 1
    b = step_bytes(case_cpu)
    times = []
    t_start = time.perf_counter()
    while True:
        times.append(oracle_step_seconds(case_cpu, threads))
        el = time.perf_counter() - t_start
        if el >= target_s or el + times[-1] > max_s:
            break
    total = sum(times)
    # One thread as well, on a bounded sample of the same step (the first n sequences, ~3 s).
    lens = case_cpu.context_lens.tolist()
    probe = make_decode_case(case_cpu.spec.name, seed=0, lengths=lens[:8])
    per_seq = oracle_step_seconds(probe, 1) / 8
    n = max(1, min(len(lens), int(3.0 / max(per_seq, 1e-9))))
    one = make_decode_case(case_cpu.spec.name, seed=0, lengths=lens[:n])
    t1 = oracle_step_seconds(one, 1)
    return {"value": round(b * len(times) / total / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the full {case_cpu.spec.name} step (append + attention, all {case_cpu.spec.num_seqs} "
                      f"sequences x {case_cpu.spec.num_q_heads} q heads) repeated {len(times)} times, fp64, "
                      f"{threads} threads, {total:.1f} s",
            "seconds_per_step": round(total / len(times), 4),
            "single_thread": {"value": round(step_bytes(one) / t1 / 1e9, 4), "unit": UNIT, "cores": 1,
                              "sample": f"the first {n} sequences of the same step (all q heads), one thread, "
                                        f"{t1:.1f} s"}}


def trace_cpu_baseline(sampled=(0, 50, 99)) -> dict:
    """The fp64 oracle on the continuous-batching trace, on its sampled steps: every layer of each
    sampled step with all host threads, and one layer of each with one thread.  The oracle replays
    a step's work (the joins' prompt appends, the step's appends, attention) on one CPU pool pair
    of the trace's shape; the values are random, the schedule (slots, tables, lengths) the trace's."""
    import oracle
    from workloads import TRACE, TraceGenerator, make_generator, randn_bf16
    from workloads import algorithmic_bytes as ab
    spec = TRACE
    tg = TraceGenerator(spec, seed=0)
    H, Hkv, D, NL = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.num_layers
    g = make_generator(2)
    kc = randn_bf16((tg.num_blocks, Hkv, 16, D), g)
    vc = randn_bf16((tg.num_blocks, Hkv, 16, D), g)
    threads = os.cpu_count() or 1
    res = {"all": [0.0, 0, 0], "one": [0.0, 0, 0]}   # seconds, seq-layers, bytes
    for st in tg.steps():
        if st.step not in sampled:
            continue
        B = len(st.seq_ids)
        js = torch.cat([st.join_slots[x] for x in st.joined]) if st.joined else None
        nbytes = ab(st.context_lens, H, Hkv, D) + append_bytes(B + (0 if js is None else js.numel()), Hkv, D)
        for layer in range(NL + 1):
            kind, nt = ("all", threads) if layer < NL else ("one", 1)
            q = randn_bf16((B, H, D), g)
            nk, nv = randn_bf16((B, Hkv, D), g), randn_bf16((B, Hkv, D), g)
            pk = randn_bf16((js.numel(), Hkv, D), g) if js is not None else None
            pv = randn_bf16((js.numel(), Hkv, D), g) if js is not None else None
            t = time.perf_counter()
            if js is not None and oracle.kv_append(pk, pv, js, kc, vc) != oracle.OK:
                raise RuntimeError("oracle prompt append failed on the trace")
            if oracle.kv_append(nk, nv, st.slot_mapping, kc, vc) != oracle.OK:
                raise RuntimeError("oracle append failed on the trace")
            _, status = oracle.paged_decode_attention(q, kc, vc, st.block_tables, st.context_lens, D ** -0.5,
                                                      num_threads=nt)
            res[kind][0] += time.perf_counter() - t
            if status != oracle.OK:
                raise RuntimeError("oracle attention failed on the trace")
            res[kind][1] += B
            res[kind][2] += nbytes

    def line(kind, cores, sample):
        sec, n, b = res[kind]
        return {"value": round(n / sec, 2), "unit": "seq·layer/s", "gbs": round(b / sec / 1e9, 4), "cores": cores,
                "kind": "oracle", "sample": sample, "seconds": round(sec, 2)}

    out = line("all", threads, f"steps {list(sampled)} x all {NL} layers, fp64, {threads} threads")
    out["single_thread"] = line("one", 1, f"steps {list(sampled)} x one layer, fp64, one thread")
    return out


def run_reference(args, dist: Dist) -> dict | None:
    """Reference arm: the fp64 CPU oracle on the host cores, rank 0 only."""
    if dist.rank != 0:
        return None
    threads = os.cpu_count() or 1
    spec = SPECS[args.workload]
    # A bounded sample of the workload per step: the first n sequences (all q heads), with n sized so
    # that the whole --warmup + --steps run stays near --reference-budget seconds (at most 1 s a step).
    case = make_decode_case(args.workload, seed=0, num_seqs=spec.num_seqs)
    probe = make_decode_case(args.workload, seed=0, lengths=case.context_lens[:8].tolist())
    per_seq = oracle_step_seconds(probe, threads) / 8
    budget = min(1.0, args.reference_budget / (args.steps + args.warmup))
    n = max(1, min(spec.num_seqs, int(budget / max(per_seq, 1e-9))))
    sample = make_decode_case(args.workload, seed=0, lengths=case.context_lens[:n].tolist())
    for _ in range(args.warmup):
        oracle_step_seconds(sample, threads)
    secs = [oracle_step_seconds(sample, threads) for _ in range(args.steps)]
    total = sum(secs)
    b = step_bytes(sample)
    value = b * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "sample_seqs": n, "num_q_heads": spec.num_q_heads,
                   "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim, "block_size": 16},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"first {n} of {spec.num_seqs} {args.workload} sequences (all q heads) per step"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "seq_layer_per_s": round(n * args.steps / total, 2),
    }
    return line


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
def fused_step_timing(pkv, g, spec, out, ws, stream, K: int, W: int, bytes_step: int) -> dict:
    """The same step through pkv_decode_step (RoPE + append + attention in two launches), timed with
    CUDA events as launched and as a replayed CUDA graph."""
    from workloads import rope_cos_sin
    table = rope_cos_sin(spec.max_blocks_per_seq * 16, spec.head_dim, 5e5).to(g.q.device)

    def step():
        pkv.decode_step(g.q, g.new_k, g.new_v, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                        table, workspace=ws, stream=stream)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
        sec = timed(step, K)
    res = {"value": round(bytes_step / sec / 1e9, 2), "unit": "GB/s", "ms_per_step": round(sec * 1e3, 4),
           "launches_per_step": 2, "rope": "rotate-half, theta 5e5"}
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(W):
                graph.replay()
            gsec = timed(graph.replay, K)
        res["graph"] = {"value": round(bytes_step / gsec / 1e9, 2), "ms_per_step": round(gsec * 1e3, 4)}
    except Exception as e:  # report, do not fail the headline
        res["graph"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    if pkv.get_and_clear_device_error(stream) != 0:
        raise RuntimeError("device error during the fused-step timing")
    return res


def e2e_line(pipe_value: float, pipe_s: float, serial_value: float, serial_s: float, K: int, h2d: int,
             d2h: int, passes: int) -> dict:
    """The end-to-end figure is the pipelined drive, fixed in advance: the way a serving loop would
    overlap its transfers with the neighbouring steps' kernels.  The serial drive (copy in, kernels,
    copy out on one stream) is reported beside it and never replaces it."""
    return {"value": round(pipe_value / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * pipe_s / K, 4), "mode": "pipelined",
            "copies": "two device slots; step i+1's inputs in and step i-1's output out on two copy streams "
                      "while step i computes",
            "passes": passes, "timing": "median of the passes, each K steps",
            "serial": {"value": round(serial_value / 1e9, 2), "ms_per_step": round(1e3 * serial_s / K, 4),
                       "copies": "in, kernels, out, one after another on the compute stream"}}


def run_ours(args, dist: Dist) -> dict | None:
    import numpy as np

    import paged_kv_cache_275_gb300 as pkv
    from paged_kv_cache_275_gb300 import build as _build
    _build.build(quiet=True)
    pkv.load()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device for --impl ours")
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)

    case_cpu = make_decode_case(args.workload, seed=0)
    spec = case_cpu.spec
    B, hq, hkv, D = spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    g = case_cpu.to(dev)
    out = torch.empty_like(g.q)
    parts = args.partitions or pkv.default_partitions(B, hq, hkv, D, spec.max_blocks_per_seq)
    ws = torch.empty(pkv.workspace_size(B, hq, hkv, D, spec.max_blocks_per_seq, parts), dtype=torch.uint8,
                     device=dev)
    pool_bytes = 2 * g.k_cache.numel() * 2

    def append():
        pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache, stream=stream)

    def attend(phases):
        pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                                   num_partitions=parts, phases=phases, workspace=ws, stream=stream)

    # Parity on the same inputs before timing (sampled outputs against the oracle).
    with torch.cuda.stream(stream):
        append()
        attend(pkv.PHASE_ALL)
    stream.synchronize()
    if pkv.get_and_clear_device_error(stream) != 0:
        raise RuntimeError("device error during the parity run")
    parity = None
    if dist.rank == 0:
        import oracle
        kc, vc = case_cpu.k_cache.clone(), case_cpu.v_cache.clone()
        oracle.kv_append(case_cpu.new_k, case_cpu.new_v, case_cpu.slot_mapping, kc, vc)
        append_exact = bool(torch.equal(g.k_cache.cpu().view(torch.int16), kc.view(torch.int16))
                            and torch.equal(g.v_cache.cpu().view(torch.int16), vc.view(torch.int16)))
        rng = np.random.default_rng(0)
        si = rng.integers(0, B, 256).astype(np.int32)
        hi = rng.integers(0, hq, 256).astype(np.int32)
        ref, st = oracle.paged_decode_sampled(case_cpu.q, kc, vc, case_cpu.block_tables, case_cpu.context_lens,
                                              case_cpu.scale, si, hi)
        got = out.cpu().to(torch.float64).numpy()[si, hi]
        diff = got - ref
        parity = {"append_bit_exact": append_exact, "sampled_outputs": int(si.size),
                  "max_abs": float(np.abs(diff).max()),
                  "rel_rms": float(np.sqrt(np.mean(diff ** 2)) / np.sqrt(np.mean(ref ** 2)))}
        if not append_exact or st != 0 or parity["max_abs"] > 1e-2 or parity["rel_rms"] > 5e-3:
            raise RuntimeError(f"parity check failed before timing: {parity}")
        del kc, vc

    bytes_attn = algorithmic_bytes(case_cpu.context_lens, hq, hkv, D)
    bytes_step = bytes_attn + append_bytes(B, hkv, D)

    def step(ev=None, i=0):
        append()
        if ev is not None:
            ev[0][i].record(stream)
        attend(pkv.PHASE_PARTITION)
        if ev is not None:
            ev[1][i].record(stream)
        attend(pkv.PHASE_MERGE)

    K, W = args.steps, args.warmup
    sampler = ClockSampler(nvidia_smi_id(dev))
    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
    stream.synchronize()
    ev_part = ([torch.cuda.Event(enable_timing=True) for _ in range(K)],
               [torch.cuda.Event(enable_timing=True) for _ in range(K)])
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def value_pass() -> float:
        """K steps bracketed by a barrier and a device synchronisation on both sides.  The step loop
        carries no events between its kernels: an event recorded between two launches would stand
        between them in the stream and end their programmatic overlap."""
        dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_begin.record(stream)
            for _ in range(K):
                step()
            t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        dist.barrier()
        return t_begin.elapsed_time(t_end) / 1e3

    def roofline_pass() -> list[float]:
        """The same K steps with events around each partition launch on its stream (the roofline)."""
        with torch.cuda.stream(stream):
            for i in range(K):
                step(ev_part, i)
        stream.synchronize()
        return [ev_part[0][i].elapsed_time(ev_part[1][i]) for i in range(K)]

    # Repeated passes: at least --passes, and enough for about --min-seconds of timed steps, so that
    # the clock sampler sees the timed region many times; the median pass is the reported one.
    first = value_pass()
    passes = max(args.passes, math.ceil(args.min_seconds / max(first, 1e-6)))
    passes = int(dist.max(float(min(passes, args.max_passes))))
    launches0 = pkv.kernel_launch_count()
    wall0 = time.time()
    pass_s, part_ms = [], []
    for _ in range(passes):
        pass_s.append(value_pass())
        part_ms.extend(roofline_pass())
    wall1 = time.time()
    launches = pkv.kernel_launch_count() - launches0
    if pkv.get_and_clear_device_error(stream) != 0:
        raise RuntimeError("device error during the timed region")
    elapsed = statistics.median(pass_s)

    # End to end through the public API: this step's inputs staged in one pinned host buffer and sent
    # with one copy, the kernels reading views of its device twin, the output read back to pinned memory.
    # Measured twice: serially on the compute stream, and pipelined, with two device slots for the
    # inputs and the output so that step i+1's inputs go in (and step i-1's output comes back) on their
    # own copy streams while step i computes.  Every step makes both copies in either form.
    names = ("q", "new_k", "new_v", "slot_mapping", "block_tables", "context_lens")
    offsets, total = {}, 0
    for name in names:
        t = getattr(case_cpu, name)
        offsets[name] = total
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    stage_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_dev = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, name):
        t = getattr(case_cpu, name)
        n = t.numel() * t.element_size()
        return buf[offsets[name]:offsets[name] + n].view(t.dtype).view(t.shape)

    for name in names:
        view(stage_host, name).copy_(getattr(case_cpu, name))
    e2e = {name: view(stage_dev, name) for name in names}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        stage_dev.copy_(stage_host, non_blocking=True)
        pkv.kv_append(e2e["new_k"], e2e["new_v"], e2e["slot_mapping"], g.k_cache, g.v_cache, stream=stream)
        pkv.paged_decode_attention(e2e["q"], g.k_cache, g.v_cache, e2e["block_tables"], e2e["context_lens"],
                                   g.scale, out, num_partitions=parts, workspace=ws, stream=stream)
        out_host.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(W):
            e2e_step()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def serial_pass() -> float:
        dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(K):
                e2e_step()
            e1.record(stream)
        stream.synchronize()
        dist.barrier()
        return e0.elapsed_time(e1) / 1e3

    e2e_passes = int(dist.max(float(max(5, min(passes, math.ceil(args.min_seconds / 4 / max(first, 1e-6)))))))
    serial_elapsed = statistics.median([serial_pass() for _ in range(e2e_passes)])
    if not torch.equal(out_host, out.cpu()):
        raise RuntimeError("e2e output read-back mismatch")

    # Pipelined: slot s = i % 2 holds step i's inputs and output on the device.
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    slots_in = [stage_dev, torch.empty_like(stage_dev)]
    slots_view = [e2e, {name: view(slots_in[1], name) for name in names}]
    slots_out = [out, torch.empty_like(out)]
    hosts_out = [out_host, torch.empty_like(out_host).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # slot's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # slot's kernels finished (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # slot's output is back on the host (output free)

    def pipelined_step(i):
        sl = i % 2
        v = slots_view[sl]
        h2d_stream.wait_event(ev_done[sl])
        with torch.cuda.stream(h2d_stream):
            slots_in[sl].copy_(stage_host, non_blocking=True)
        ev_in[sl].record(h2d_stream)
        stream.wait_event(ev_in[sl])
        stream.wait_event(ev_out[sl])
        pkv.kv_append(v["new_k"], v["new_v"], v["slot_mapping"], g.k_cache, g.v_cache, stream=stream)
        pkv.paged_decode_attention(v["q"], g.k_cache, g.v_cache, v["block_tables"], v["context_lens"], g.scale,
                                   slots_out[sl], num_partitions=parts, workspace=ws, stream=stream)
        ev_done[sl].record(stream)
        d2h_stream.wait_event(ev_done[sl])
        with torch.cuda.stream(d2h_stream):
            hosts_out[sl].copy_(slots_out[sl], non_blocking=True)
        ev_out[sl].record(d2h_stream)

    def pipelined(n, e_start=None, e_end=None):
        if e_start is not None:
            e_start.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        for i in range(n):
            pipelined_step(i)
        stream.wait_stream(d2h_stream)
        if e_end is not None:
            e_end.record(stream)

    for h in hosts_out:
        h.zero_()
    pipelined(max(W, 2))
    stream.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def pipelined_pass() -> float:
        dist.barrier()
        torch.cuda.synchronize()
        pipelined(K, p0, p1)
        stream.synchronize()
        dist.barrier()
        return p0.elapsed_time(p1) / 1e3

    e2e_elapsed = statistics.median([pipelined_pass() for _ in range(e2e_passes)])
    for h, o in zip(hosts_out[:min(K, 2)], slots_out):
        if not torch.equal(h, o.cpu()):
            raise RuntimeError("pipelined e2e output read-back mismatch")
    fused = fused_step_timing(pkv, g, spec, out, ws, stream, K, W, bytes_step)
    rows = sampler.stop() if sampler else []

    value, slowest = aggregate(bytes_step * K, elapsed, dist)
    e2e_value, _ = aggregate(bytes_step * K, e2e_elapsed, dist)
    serial_value, _ = aggregate(bytes_step * K, serial_elapsed, dist)
    seqs, _ = aggregate(B * K, elapsed, dist)
    if dist.rank != 0:
        return None

    peak, peak_kind = peaks()
    part_mean_s = statistics.fmean(part_ms) / 1e3
    achieved = bytes_attn / part_mean_s / 1e9
    clocks = ClockSampler.summarize(rows, wall0, wall1)
    cpu = cpu_baseline(case_cpu, target_s=args.cpu_seconds) if args.cpu_seconds > 0 else None
    line = {
        "metric": METRIC, "value": round(value / 1e9, 2), "unit": UNIT, "n_gpus": dist.world, "steps": K,
        "warmup": W, "ms_per_step": round(1e3 * slowest / K, 4), "higher_is_better": True, "scaling": "weak",
        "passes": passes, "timing": "median of the passes, each K steps bracketed by a barrier and a device "
                                    "synchronisation; ms_per_step of the fastest and slowest pass beside it",
        "ms_per_step_min_max": [round(1e3 * min(pass_s) / K, 4), round(1e3 * max(pass_s) / K, 4)],
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{spec.name}: {spec.description}", "num_seqs": B, "num_q_heads": hq,
                   "num_kv_heads": hkv, "head_dim": D, "block_size": 16,
                   "mean_context_len": round(float(case_cpu.context_lens.float().mean()), 1),
                   "kv_pool_bytes": pool_bytes, "num_partitions": parts,
                   "l2": f"inputs larger than L2: the {pool_bytes / 1e9:.2f} GB K/V pool streams through the "
                         f"{L2_BYTES >> 20} MiB L2 every step; no flush",
                   "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU"},
        "pct_of_peak": {"measured": round(100 * value / 1e9 / peak, 2), "nominal_8TBps": round(
            100 * value / 1e9 / NOMINAL_HBM_GBS, 2), "peak_kind": peak_kind},
        "seq_layer_per_s": round(seqs, 1),
        "step_bytes": bytes_step,
        "roofline": {"kernel": "paged_decode_partition_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of": f"{peak_kind} HBM copy bandwidth", "frac_nominal_8TBps": round(
                         achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": args.traffic if args.traffic is not None else recorded_traffic(
                         "paged_decode_partition_kernel", args.workload),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/traffic.txt "
                                       f"(kernel source {source_hash('paged_decode_partition_kernel')})",
                     "algorithmic_bytes_per_launch": bytes_attn,
                     "mean_launch_us": round(part_mean_s * 1e6, 2),
                     "launches_timed": len(part_ms),
                     "launch_us_min_median_max": [round(1e3 * min(part_ms), 2),
                                                  round(1e3 * statistics.median(part_ms), 2),
                                                  round(1e3 * max(part_ms), 2)]},
        "e2e": e2e_line(e2e_value, e2e_elapsed, serial_value, serial_elapsed, K, h2d, d2h, e2e_passes),
        "gpu_launches": launches,
        "clocks": clocks,
        "parity": parity,
        "fused_step": fused,
        "cpu_baseline": cpu,
    }
    return line


# ---------------------------------------------------------------------------
# Component measurements (not the headline step): block copy, block manager
# ---------------------------------------------------------------------------
def append_component(args, pkv, peak: float, peak_kind: str) -> dict:
    """kv_append at prompt size: 16 prompts of 4096 tokens (65536 tokens, LLaMA-3 kv layout: 8 kv heads,
    D 128) written into randomly permuted blocks of a 1.2 GB pool; plus the decode size (one token for
    each of 128 sequences), which launch latency bounds."""
    from workloads import make_generator, randn_bf16
    dev = torch.device("cuda", 0)
    hkv, d, nb = 8, 128, 18432
    n_seq, per_seq = 16, 4096
    n = n_seq * per_seq
    kc = torch.zeros((nb, hkv, 16, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    blocks = torch.randperm(nb, generator=make_generator(11))[:n // 16]
    tok = torch.arange(n)
    slots = (blocks[tok // 16] * 16 + tok % 16).to(torch.int64).to(dev)
    k = randn_bf16((n, hkv, d), make_generator(12, "cuda"), "cuda")
    v = randn_bf16((n, hkv, d), make_generator(13, "cuda"), "cuda")
    pkv.kv_append(k, v, slots, kc, vc)
    torch.cuda.synchronize()
    b_idx, off = slots // 16, slots % 16
    if (pkv.get_and_clear_device_error() != 0 or not torch.equal(kc[b_idx, :, off].view(torch.int16), k.view(torch.int16))
            or not torch.equal(vc[b_idx, :, off].view(torch.int16), v.view(torch.int16))):
        raise RuntimeError("kv_append parity failed before timing")
    stream = torch.cuda.current_stream()

    def timed(kk, vv, ss, steps):
        for _ in range(args.warmup):
            pkv.kv_append(kk, vv, ss, kc, vc)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            pkv.kv_append(kk, vv, ss, kc, vc)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps

    steps = min(args.steps, 500)
    sec = timed(k, v, slots, steps)
    moved = 2 * (2 * n * hkv * d * 2) + 8 * n    # K and V rows read and written, and the slot ids
    gbs = moved / sec / 1e9
    # Decode size, replayed from a CUDA graph of 64 calls: one Python call takes longer than the kernel.
    dec_slots = slots[::per_seq // 8][:128].contiguous()
    dk, dv = k[:128].contiguous(), v[:128].contiguous()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            pkv.kv_append(dk, dv, dec_slots, kc, vc, stream=side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(64):
            pkv.kv_append(dk, dv, dec_slots, kc, vc, stream=side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, steps // 64)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    dec_sec = e0.elapsed_time(e1) / 1e3 / (64 * reps)
    if pkv.get_and_clear_device_error() != 0:
        raise RuntimeError("device error during the kv_append timing")
    return {"component": "kv_append", "metric": "kv_append HBM GB/s (K/V rows read + written, slot ids)",
            "value": round(gbs, 1), "unit": "GB/s", "steps": steps, "warmup": args.warmup,
            "us_per_launch": round(sec * 1e6, 2),
            "config": {"workload": "16 prompts x 4096 tokens, 8 kv heads, D 128, into permuted blocks of an "
                                   "18432-block (1.2 GB) pool", "tokens": n,
                       "l2": "536 MB moved per launch, over 4x the L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "frac_of": f"{peak_kind} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": moved,
                         "traffic": recorded_traffic("kv_append_kernel", "append_16x4096"),
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/traffic.txt "
                                           f"(kernel source {source_hash('kv_append_kernel')})"},
            "decode_size": {"tokens": 128, "us_per_launch": round(dec_sec * 1e6, 2),
                            "bytes_per_launch": 2 * (2 * 128 * hkv * d * 2) + 8 * 128,
                            "timing": "CUDA graph of 64 calls, replayed",
                            "note": "one token per sequence: launch latency, not bandwidth"}}


def chain_component(args, pkv, peak: float, peak_kind: str) -> dict:
    """Decode calls back to back: per-call time of chains of partition-only, partition + merge, and
    append + partition + merge calls on --workload (CUDA events at each end of a chain of --steps calls,
    the median of 5 chains), for each partition count in --chain-partitions (0 = the default)."""
    dev = torch.device("cuda", 0)
    c = make_decode_case(args.workload, seed=0).to(dev)
    s = c.spec
    B, hq, hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    nbytes = algorithmic_bytes(c.context_lens.cpu(), hq, hkv, D)
    out = torch.empty_like(c.q)
    stream = torch.cuda.Stream(dev)
    default = pkv.default_partitions(B, hq, hkv, D, s.max_blocks_per_seq)
    rows = []
    for parts in [int(x) or default for x in args.chain_partitions.split(",")]:
        ws = torch.empty(pkv.workspace_size(B, hq, hkv, D, s.max_blocks_per_seq, parts), dtype=torch.uint8,
                         device=dev)

        def attend(ph):
            pkv.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, out,
                                       num_partitions=parts, phases=ph, workspace=ws, stream=stream)

        def append():
            pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache, stream=stream)

        row = {"num_partitions": parts}
        for label, fn in (("partition_us", lambda: attend(pkv.PHASE_PARTITION)),
                          ("partition_merge_us", lambda: attend(pkv.PHASE_ALL)),
                          ("append_partition_merge_us", lambda: (append(), attend(pkv.PHASE_ALL)))):
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    fn()
                ts = []
                for _ in range(5):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(args.steps):
                        fn()
                    e1.record(stream)
                    stream.synchronize()
                    ts.append(e0.elapsed_time(e1) / args.steps * 1e3)
            row[label] = round(statistics.median(ts), 2)
        row["partition_frac"] = round(nbytes / (row["partition_us"] * 1e-6) / 1e9 / peak, 4)
        row["partition_merge_frac"] = round(nbytes / (row["partition_merge_us"] * 1e-6) / 1e9 / peak, 4)
        if pkv.get_and_clear_device_error(stream) != 0:
            raise RuntimeError("device error during the chain timing")
        rows.append(row)
    return {"component": "chain", "metric": "decode calls back to back: microseconds per call",
            "workload": f"{s.name}: {s.description}", "algorithmic_bytes_per_call": nbytes, "chain_length": args.steps,
            "frac_of": f"{peak_kind} HBM copy bandwidth ({peak} GB/s)", "rows": rows}


def run_component(args) -> dict:
    import numpy as np

    import paged_kv_cache_275_gb300 as pkv
    from paged_kv_cache_275_gb300 import build as _build
    from workloads import make_generator, randn_bf16
    _build.build(quiet=True)
    peak, peak_kind = peaks()
    if args.component == "block_manager":
        # Host allocator throughput on a decode trace: 256 sequences, 1000 append steps.
        longest = 1000 + 3 * 255 + args.warmup + args.steps
        bm = pkv.BlockManager(256 * (longest // 16 + 2))
        ids = np.arange(256, dtype=np.int64)
        for i in range(256):
            bm.add_sequence(i, 1000 + 3 * i)
        for _ in range(args.warmup):
            bm.append_slots(ids)
        t = time.perf_counter()
        for _ in range(args.steps):
            bm.append_slots(ids)
        dt = time.perf_counter() - t
        return {"component": "block_manager", "metric": "append slots per second (host, one thread)",
                "value": round(256 * args.steps / dt, 1), "unit": "slot/s", "steps": args.steps,
                "us_per_batch_of_256": round(1e6 * dt / args.steps, 2), "kind": "C ABI through ctypes"}
    if args.component == "trace":
        # Continuous-batching trace (Qwen3-0.6B shape, 28 layers, up to 256 sequences, 100 decode steps):
        # every input of every step is generated and staged on the device first; the timed region is
        # the library calls only (prompt appends of joining sequences, the step's appends, attention).
        from workloads import TRACE, TraceGenerator, make_generator, randn_bf16, algorithmic_bytes as ab
        spec = TRACE
        tg = TraceGenerator(spec, seed=0)
        gen = make_generator(1, "cuda")
        H, Hkv, D, NL = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.num_layers
        kp = [randn_bf16((tg.num_blocks, Hkv, 16, D), gen, "cuda") for _ in range(NL)]
        vp = [randn_bf16((tg.num_blocks, Hkv, 16, D), gen, "cuda") for _ in range(NL)]
        steps = []
        seq_layers = 0
        bytes_total = 0
        for st in tg.steps():
            B = len(st.seq_ids)
            js = torch.cat([st.join_slots[x] for x in st.joined]).cuda() if st.joined else None
            nj = 0 if js is None else js.numel()
            steps.append(dict(bt=st.block_tables.cuda(), cl=st.context_lens.cuda(), slots=st.slot_mapping.cuda(),
                              js=js, q=randn_bf16((NL, B, H, D), gen, "cuda"),
                              k=randn_bf16((NL, B, Hkv, D), gen, "cuda"), v=randn_bf16((NL, B, Hkv, D), gen, "cuda"),
                              pk=randn_bf16((nj, Hkv, D), gen, "cuda") if nj else None,
                              pv=randn_bf16((nj, Hkv, D), gen, "cuda") if nj else None,
                              out=torch.empty(B, H, D, dtype=torch.bfloat16, device="cuda")))
            seq_layers += B * NL
            bytes_total += NL * (ab(st.context_lens, H, Hkv, D) + append_bytes(B + nj, Hkv, D))
        W = tg.width
        ws = torch.empty(pkv.workspace_size(256, H, Hkv, D, W), dtype=torch.uint8, device="cuda")

        def run():
            for x in steps:
                for layer in range(NL):
                    if x["js"] is not None:
                        pkv.kv_append(x["pk"], x["pv"], x["js"], kp[layer], vp[layer])
                    pkv.kv_append(x["k"][layer], x["v"][layer], x["slots"], kp[layer], vp[layer])
                    pkv.paged_decode_attention(x["q"][layer], kp[layer], vp[layer], x["bt"], x["cl"], D ** -0.5,
                                               x["out"], workspace=ws)

        run()  # warm-up pass (also the parity-tested path)
        torch.cuda.synchronize()
        launches0 = pkv.kernel_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        sec = e0.elapsed_time(e1) / 1e3
        if pkv.get_and_clear_device_error() != 0:
            raise RuntimeError("device error during the trace")
        peak_gbs = bytes_total / sec / 1e9
        return {"component": "trace", "metric": "continuous-batching trace seq·layer/s", "value": round(
            seq_layers / sec, 1), "unit": "seq·layer/s", "gbs": round(peak_gbs, 1),
                "frac_of_measured_hbm": round(peak_gbs / peak, 4), "frac_of_nominal_8TBps": round(
                    peak_gbs / NOMINAL_HBM_GBS, 4),
                "seconds": round(sec, 4), "host_wall_seconds": round(wall, 4),
                "gpu_launches": pkv.kernel_launch_count() - launches0,
                "cpu_baseline": trace_cpu_baseline() if args.cpu_seconds > 0 else None,
                "config": {"workload": f"{spec.name}: {NL} layers, <= {spec.max_seqs} sequences, {spec.steps} "
                                       f"decode steps, Poisson({spec.join_rate}) joins / finishes",
                           "seq_layers": seq_layers, "algorithmic_bytes": bytes_total}}
    if args.component == "prefill":
        from workloads import make_prefill_case, prefill_flops
        c = make_prefill_case(args.prefill_workload, seed=0).to("cuda")
        pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache)
        out = torch.empty_like(c.q)
        max_q = max(c.spec.chunk_lens)

        if args.prefill_splits == 0:  # the library's one-wave choice
            args.prefill_splits = pkv.prefill_default_splits(c.context_lens.shape[0], max_q, c.spec.num_q_heads,
                                                             c.spec.num_kv_heads)
        ws = None
        if args.prefill_splits > 1:
            ws = torch.empty(pkv.prefill_workspace_size(c.context_lens.shape[0], max_q, c.spec.num_q_heads,
                                                        c.spec.num_kv_heads, c.spec.head_dim, args.prefill_splits),
                             dtype=torch.uint8, device="cuda")

        def call():
            pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.query_start,
                                        max_q, c.scale, out, num_splits=args.prefill_splits, workspace=ws)

        for _ in range(args.warmup):
            call()
        stream = torch.cuda.current_stream()
        # Passes of `steps` launches, each bracketed by events, repeated for at least --min-seconds so
        # that the clock sampler sees the timed region; the median pass is reported.
        sampler = ClockSampler(nvidia_smi_id(torch.device("cuda", 0)))
        torch.cuda.synchronize()
        t_start = time.time()
        pass_sec = []
        while len(pass_sec) < max(1, args.passes) or (time.time() - t_start < args.min_seconds
                                                       and len(pass_sec) < args.max_passes):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            pass_sec.append(e0.elapsed_time(e1) / 1e3 / args.steps)
        t_stop = time.time()
        clocks = ClockSampler.summarize(sampler.stop(), t_start, t_stop)
        if pkv.get_and_clear_device_error() != 0:
            raise RuntimeError("device error during the prefill timing")
        sec = sorted(pass_sec)[len(pass_sec) // 2]
        flops = prefill_flops(c.context_lens.cpu(), c.query_start.cpu(), c.spec.num_q_heads, c.spec.head_dim)
        tf = flops / sec / 1e12
        # The passes run back to back for at least a second: the GPU settles at its power cap, so the
        # sustained peak is the denominator; the burst one is reported beside it.
        sustained = t_stop - t_start >= 1.0
        bf16_peak, kind = bf16_peak_tflops(sustained)
        burst_peak, _ = bf16_peak_tflops(False)
        return {"component": "prefill", "metric": "chunked paged prefill attention TFLOP/s (causal flops)",
                "value": round(tf, 2), "unit": "TFLOP/s", "steps": args.steps, "warmup": args.warmup,
                "us_per_launch": round(sec * 1e6, 2), "passes": len(pass_sec),
                "us_per_launch_min_max": [round(min(pass_sec) * 1e6, 2), round(max(pass_sec) * 1e6, 2)],
                "timing": "median of the passes, each `steps` launches between CUDA events", "clocks": clocks,
                "config": {"workload": c.spec.description, "tokens": int(c.q.shape[0]),
                           "num_splits": args.prefill_splits,
                           "context_lens": c.context_lens.tolist()},
                "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                             "frac": round(tf / bf16_peak, 4),
                             "frac_of": f"{kind} bf16 dense (cuBLAS, {'sustained' if sustained else 'burst'})",
                             "frac_of_burst": round(tf / burst_peak, 4), "timed_seconds": round(t_stop - t_start, 2),
                             "fastest_pass_tflops": round(flops / min(pass_sec) / 1e12, 2),
                             "algorithmic_flops_per_launch": flops,
                             "traffic": recorded_traffic("paged_prefill_kernel", args.prefill_workload),
                             "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/traffic.txt "
                                               f"(kernel source {source_hash('paged_prefill_kernel')})",
                             "compulsory_bytes_per_launch": prefill_compulsory_bytes(c)}}
    if args.component == "kv_append":
        return append_component(args, pkv, peak, peak_kind)
    if args.component == "chain":
        return chain_component(args, pkv, peak, peak_kind)
    # copy_blocks: copy-on-write of 4096 distinct block pairs of the Qwen3/LLaMA-3 kv layout.
    dev = torch.device("cuda", 0)
    g = make_generator(7)
    nb, hkv, d, n = 16384, 8, 128, 4096
    kc = randn_bf16((nb, hkv, 16, d), make_generator(8, "cuda"), "cuda")
    vc = randn_bf16((nb, hkv, 16, d), make_generator(9, "cuda"), "cuda")
    perm = torch.randperm(nb, generator=g)
    pairs = torch.stack([perm[:n], perm[n:2 * n]], dim=1).to(torch.int64).to(dev)
    ref_k = kc[pairs[:, 0]].clone()
    pkv.copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    if not torch.equal(kc[pairs[:, 1]], ref_k) or pkv.get_and_clear_device_error() != 0:
        raise RuntimeError("copy_blocks parity failed before timing")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        pkv.copy_blocks(kc, vc, pairs)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        pkv.copy_blocks(kc, vc, pairs)
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / args.steps
    moved = n * 2 * (hkv * 16 * d * 2) * 2          # K and V blocks, read + written
    gbs = moved / sec / 1e9
    return {"component": "copy_blocks", "metric": "block copy HBM GB/s (read + write)", "value": round(gbs, 1),
            "unit": "GB/s", "steps": args.steps, "warmup": args.warmup, "us_per_launch": round(sec * 1e6, 2),
            "config": {"pairs": n, "block_bytes_k_plus_v": 2 * hkv * 16 * d * 2, "pool_blocks": nb},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "frac_of": f"{peak_kind} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": moved, "traffic": None}}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--passes", type=int, default=25, help="least number of timed passes of --steps steps")
    ap.add_argument("--min-seconds", type=float, default=1.5,
                    help="timed passes continue until about this much timed GPU work")
    ap.add_argument("--max-passes", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(SPECS), default="llama3_8b")
    ap.add_argument("--partitions", type=int, default=0, help="num_partitions (0 = the library default)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline budget (0 skips it)")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="seconds the reference arm's warm-up + timed steps should take")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per partition launch from an ncu capture of the current kernel")
    ap.add_argument("--prefill-workload", choices=("prefill_llama3_8b", "prefill_qwen3_0.6b", "prefill_llama3_8b_one"),
                    default="prefill_llama3_8b", help="chunked-prefill workload of --component prefill")
    ap.add_argument("--prefill-splits", type=int, default=1,
                    help="split each tile pair's key steps over this many CTAs (merge pass after); 0: the "
                         "library's choice (one wave)")
    ap.add_argument("--component", choices=("copy_blocks", "block_manager", "prefill", "trace", "kv_append", "chain"),
                    default=None, help="measure one component instead of the decode step")
    ap.add_argument("--chain-partitions", default="0",
                    help="chain component: comma-separated num_partitions values (0 = the library default)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.component:
        print(json.dumps(run_component(args)), flush=True)
        return 0
    dist = Dist()
    try:
        line = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
