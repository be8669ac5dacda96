#!/usr/bin/env python3
"""Benchmark of split-KV decode attention on one GB300 (or N, one process each).

One step = one ``fd_decode`` call (plan, split, merge: a single kernel launch)
over the batch-1 128k-context GQA workload (B=1, Hq=32, Hkv=8, D=128,
T=131072, bf16 K/V, fp32 q/out), inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {fdecode,reference}] [--workload 1..5]

``--impl reference`` times the float64 CPU oracle (the only reference this
method has) on the host cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import ctypes
import dataclasses
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step; KV-read HBM GB/s as % of GB300 peak (1 GPU)"
L2_BYTES = 129 * 1000 * 1000    # GB300 L2
FLUSH_BYTES = 256 << 20         # written between launches when the inputs would stay in L2
DEFAULT_WORKLOAD = 3
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fdecode", "reference"], default="fdecode")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this batch size instead of its own (smaller profiling captures)")
    ap.add_argument("--append", action="store_true",
                    help="fused append-KV + decode (fd_append_decode): each step writes the last token's k/v")
    ap.add_argument("--unfused", type=int, default=0, metavar="S",
                    help="time fd_split_partial with S splits + fd_combine (two launches per step)")
    ap.add_argument("--rows", type=int, default=1,
                    help="query rows per sequence (causal window through fd_decode_rows); 1 = fd_decode")
    ap.add_argument("--graph", action="store_true",
                    help="time one CUDA graph of K launches instead of K stream launches (the stream launches "
                         "are enqueued while a short sleep kernel holds the GPU before the start event)")
    ap.add_argument("--prefill", type=int, default=0, metavar="N",
                    help="time fd_prefill on an N-token causal prompt (B=1, Hq=32, Hkv=8, D=128): TFLOP/s")
    ap.add_argument("--prefill-kv-heads", type=int, default=8, metavar="HKV",
                    help="KV heads of the --prefill prompt (32 = MHA; 32 must be a multiple)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
KERNEL_SOURCES = ("fd_split.cuh", "fd_split_mma.cuh", "fd_device.cuh", "fd_plan.h", "fd_split_launch.cuh", "fd_split_bf16.cu",
                  "fd_split_f32.cu")
PREFILL_SOURCES = ("fd_prefill.cu", "fd_prefill.h", "fd_device.cuh")


def source_hash(sources=KERNEL_SOURCES) -> str:
    """Hash of a kernel's device code (host-only files excluded); the split kernel by default."""
    h = hashlib.sha256()
    for name in sources:
        h.update(open(os.path.join(ROOT, "split_kv_decode_fd_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:12]


def prefill_l2_note(N: int, hkv: int) -> str:
    """What one prefill step touches (q, K/V, output) against the L2 size: each step re-reads q and K/V."""
    q = 32 * N * 128 * 4
    kv = 2 * hkv * N * 128 * 2
    total = 2 * q + kv
    if total > L2_BYTES:
        return (f"q {q / 1e6:.0f} MB + K/V {kv / 1e6:.0f} MB + output {q / 1e6:.0f} MB = {total / 1e6:.0f} MB per step "
                f"> {L2_BYTES / 1e6:.0f} MB L2; no flush")
    return f"q, K/V and output {total / 1e6:.1f} MB per step fit in L2 (warm: no flush)"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def measured_tensor_peak():
    """Dense bf16 tensor peak: MEASURED_PEAKS.json (burst figure: a kernel timed alone), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        for key in ("bf16_tflops", "bf16_tflops_burst"):
            if key in d and float(d[key]) > 0:
                return float(d[key]), f"measured (MEASURED_PEAKS.json {key}, cuBLAS bf16 GEMM)"
    except (OSError, ValueError, TypeError):
        pass
    return 1900.0, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


def recorded_traffic(workload_name: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel sources."""
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        txt = open(p).read()
        if f"workload: {workload_name}" not in txt:
            continue
        vals = {}
        for line in txt.splitlines():
            line = line.strip().lstrip("-* ").strip()
            if ":" in line and line.startswith(("traffic_bytes_per_launch", "source_sha")):
                k, v = line.split(":", 1)
                v = v.strip(" `").split()
                vals[k.strip(" `")] = v[0].strip("`") if v else ""
        if vals.get("source_sha") == source_hash(sources) and "traffic_bytes_per_launch" in vals:
            try:
                return int(float(vals["traffic_bytes_per_launch"]))
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [ln for t, ln in self.lines if t0 <= t <= t1] or [ln for _, ln in self.lines[-1:]]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(inside)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_bytes(case) -> int:
    """Algorithmic bytes of one step: valid K+V rows, q in, out written (as the metric counts them)."""
    s = case.spec
    return case.kv_bytes() + s.B * s.Hq * s.D * 4 * 2


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", cpu_cores()))


class OracleSampler:
    """Host-side copy of a workload for timing the float64 oracle on bounded samples."""

    def __init__(self, case):
        import numpy as np
        self.np = np
        self.case = case
        s = case.spec
        self.g = s.Hq // s.Hkv
        self.q = case.q.detach().cpu().numpy().astype(np.float64)
        self.lens = case.lengths
        self.k = case.k.detach().cpu()
        self.v = case.v.detach().cpu()
        self.table = None if case.block_table is None else case.block_table.cpu().numpy()
        self.es = case.k.element_size()

    def group(self, b, kvh, n_tok=None):
        """Oracle on the first n_tok keys of (b, kv head) for its g query heads: (seconds, kv bytes)."""
        import oracle
        np, s = self.np, self.case.spec
        L = self.lens[b] if n_tok is None else min(n_tok, self.lens[b])
        qb = self.q[b:b + 1, kvh * self.g:(kvh + 1) * self.g]
        if self.table is None:
            kb = self.k[b:b + 1, kvh:kvh + 1, :L].float().numpy()
            vb = self.v[b:b + 1, kvh:kvh + 1, :L].float().numpy()
            t0 = time.perf_counter()
            oracle.decode(qb, kb, vb, s.scale, seq_lens=[L], max_seq_len=L)
        else:
            npg = -(-L // s.page_size)
            pages = self.table[b, :npg]
            kb = self.k[pages][:, kvh:kvh + 1].float().numpy()
            vb = self.v[pages][:, kvh:kvh + 1].float().numpy()
            t0 = time.perf_counter()
            oracle.decode(qb, kb, vb, s.scale, seq_lens=[L], block_table=np.arange(npg)[None],
                          page_size=s.page_size)
        return time.perf_counter() - t0, L * s.D * 2 * self.es

    def whole_groups(self, seconds):
        """Whole (b, kv head) groups in order until `seconds` of oracle time: (GB/s, note, seconds)."""
        s = self.case.spec
        done, el, n = 0, 0.0, 0
        for b in range(s.B):
            for kvh in range(s.Hkv):
                if self.lens[b] == 0:
                    continue
                t, nb = self.group(b, kvh)
                el, done, n = el + t, done + nb, n + 1
                if el >= seconds:
                    break
            if el >= seconds:
                break
        note = (f"{n} of {s.B * s.Hkv} whole (batch, kv-head) groups, {self.g} query heads each; "
                "float64 NumPy oracle")
        return done / el / 1e9, note, el


# ------------------------------------------------------------------ arms
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    from workloads import CONFIGS, make_case
    spec = CONFIGS[args.workload]
    smp = OracleSampler(make_case(spec, "cpu"))
    b0 = next(b for b, L in enumerate(smp.lens) if L > 0)
    # each step: the oracle on the first n_tok keys of one (b, kv-head) group, sized so
    # that warm-up plus timed steps take about two minutes of host time
    budget = max(0.01, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    t_probe, _ = smp.group(b0, 0, 4096)
    n_tok = int(min(smp.lens[b0], max(128, 4096 * budget / max(t_probe, 1e-6))))
    for _ in range(args.warmup):
        smp.group(b0, 0, n_tok)
    secs, nbytes = [], 0
    for i in range(args.steps):
        t, nb = smp.group(b0, i % spec.Hkv, n_tok)
        secs.append(t)
        nbytes += nb
    value = nbytes / sum(secs) / 1e9
    cores = blas_threads()
    note = (f"per step: first {n_tok} keys of one (batch, kv-head) group ({smp.g} query heads), "
            "float64 NumPy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": spec.name, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv,
                                        "D": spec.D, "T": spec.T_cap, "kv_dtype": spec.kv_dtype},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": note},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fdecode(args):
    world, rank, local = dist_env()
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libfdecode has no CPU path)")
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    import split_kv_decode_fd_gb300 as fd
    from workloads import CONFIGS, make_case
    fd.load_library()

    spec = CONFIGS[args.workload]
    if args.batch > 0:
        spec = dataclasses.replace(spec, B=args.batch, name=f"{spec.name}_batch{args.batch}")
    n_q = args.rows
    if n_q > 1 and args.append:
        raise SystemExit("--rows and --append are separate variants")
    if n_q > 1:
        spec = dataclasses.replace(spec, name=f"{spec.name}_rows{n_q}_causal")
    if args.append:
        spec = dataclasses.replace(spec, name=f"{spec.name}_append")
    case = make_case(spec, device)
    kv_bytes = case.kv_bytes()
    step_bytes = kv_bytes + spec.B * spec.Hq * n_q * spec.D * 4 * 2
    rows_shape = (spec.B, spec.Hq, n_q) if n_q > 1 else (spec.B, spec.Hq)
    out = torch.empty(rows_shape + (spec.D,), dtype=torch.float32, device=device)
    lse = torch.empty(rows_shape, dtype=torch.float32, device=device)
    ws = fd.Workspace()
    stream = torch.cuda.current_stream(device)
    if n_q > 1:
        gen = torch.Generator(device=device).manual_seed(spec.seed + 17)
        q_rows = torch.randn(rows_shape + (spec.D,), generator=gen, device=device, dtype=torch.float32)

        def step():
            fd.decode_rows(q_rows, case.k, case.v, causal=True, seq_lens=case.seq_lens,
                           max_seq_len=case.max_seq_len, block_table=case.block_table, scale=spec.scale,
                           n_splits=spec.n_splits, out=out, lse=lse, workspace=ws)
    elif args.unfused:
        spec = dataclasses.replace(spec, name=f"{spec.name}_unfused{args.unfused}")
        o_part = torch.empty((spec.B, spec.Hq, args.unfused, spec.D), dtype=torch.float32, device=device)
        m_part = torch.empty((spec.B, spec.Hq, args.unfused), dtype=torch.float32, device=device)
        l_part = torch.empty_like(m_part)
        lib = fd.load_library()
        kvd = fd.fdecode._kv_desc(case.k, case.v, case.block_table)

        def step():
            s_ = torch.cuda.current_stream(device).cuda_stream
            lib.fd_split_partial(case.q.data_ptr(), ctypes.byref(kvd), spec.B, spec.Hq, spec.Hkv,
                                 case.seq_lens.data_ptr() if case.seq_lens is not None else None,
                                 case.max_seq_len, spec.D, float(spec.scale), args.unfused, o_part.data_ptr(),
                                 m_part.data_ptr(), l_part.data_ptr(), s_)
            lib.fd_combine(o_part.data_ptr(), m_part.data_ptr(), l_part.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           spec.B, spec.Hq, spec.D, args.unfused, s_)
    elif args.append:
        # the sequences' last token is the one appended: lengths before the append are L_b - 1
        lens_full = torch.tensor(case.lengths, dtype=torch.int32, device=device)
        seq_before = (lens_full - 1).contiguous()
        gen = torch.Generator(device=device).manual_seed(spec.seed + 29)
        k_new = torch.randn((spec.B, spec.Hkv, spec.D), generator=gen, device=device).to(case.k.dtype)
        v_new = torch.randn((spec.B, spec.Hkv, spec.D), generator=gen, device=device).to(case.k.dtype)
        step_bytes += 2 * k_new.numel() * k_new.element_size()  # the new rows, read and stored

        def step():
            fd.append_decode(case.q, case.k, case.v, k_new, v_new, seq_lens=seq_before,
                             max_seq_len=case.max_seq_len - 1, block_table=case.block_table, scale=spec.scale,
                             n_splits=spec.n_splits, out=out, lse=lse, workspace=ws)
    else:
        def step():
            fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                      block_table=case.block_table, scale=spec.scale, n_splits=spec.n_splits, out=out, lse=lse,
                      workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fd.workspace_status(ws) != 0:
        raise SystemExit("kernel reported an error during warm-up")

    # ---- per-launch spread (diagnostic, outside the timed region): events around single launches
    n_ev = min(200, max(20, args.steps))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    launch_us = [a.elapsed_time(b) * 1e3 for a, b in ev]

    # ---- timed region: K steps back to back, CUDA events on the launching stream around the whole
    # region, clocks sampled meanwhile.  By default K stream launches, enqueued while a sleep kernel
    # holds the GPU before the start event (host launch latency stays outside the region and
    # consecutive launches overlap through programmatic dependent launch); --graph: one CUDA graph.
    K = args.steps
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(K):
                step()
        torch.cuda.synchronize()
        graph.replay()  # one untimed replay: the graph's first launch uploads it
        torch.cuda.synchronize()
        if fd.workspace_status(ws) != 0:
            raise SystemExit("kernel reported an error in the captured steps")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if graph is None:
        torch.cuda._sleep(4_000_000)  # ~2 ms at 2 GHz, before the start event: the launches queue up meanwhile
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(K):
            step()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop(t0, t1)
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / K
    value = world * step_bytes * K / (total_ms * 1e-3) / 1e9
    # one launch per step, back to back: the average launch duration is the region / K
    mean_launch_us = ms_per_step * 1e3
    achieved = step_bytes / (mean_launch_us * 1e-6) / 1e9
    peak, peak_src = measured_peak()

    # ---- inputs that fit in L2: the back-to-back figure above is warm (L2-resident).  The cold
    # figure flushes L2 with a 256 MB write before every launch (outside the events) and times
    # each launch with events on its stream; it becomes the line's value.
    l2_note = f"inputs {kv_bytes / 1e6:.0f} MB > 129 MB L2; no flush"
    warm = None
    timed_launches = K * (2 if args.unfused else 1)
    if kv_bytes < L2_BYTES:
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        n_cold = max(20, min(200, K))
        cold_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cold)]
        for i, (a, b) in enumerate(cold_ev):
            flush.fill_(i & 0xFF)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        cold_us = [a.elapsed_time(b) * 1e3 for a, b in cold_ev]
        timed_launches = n_cold * (2 if args.unfused else 1)
        del flush
        warm = {"us_per_step": ms_per_step * 1e3, "value": value, "unit": "GB/s",
                "method": "one CUDA graph of K back-to-back launches, inputs L2-resident"}
        ms_per_step = statistics.mean(cold_us) * 1e-3
        value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
        mean_launch_us = ms_per_step * 1e3
        achieved = step_bytes / (mean_launch_us * 1e-6) / 1e9
        l2_note = (f"inputs {kv_bytes / 1e6:.1f} MB < 129 MB L2: L2 flushed by a {FLUSH_BYTES >> 20} MB write "
                   f"before each of {n_cold} launches, each timed with events on its stream "
                   f"(~3 us of event overhead included); p10/p50/p90 "
                   f"{[round(x, 2) for x in statistics.quantiles(cold_us, n=10)[0::4]]} us")

    # ---- end to end: host q in, host out/lse back (fd_decode_host; with rows, copies around fd_decode_rows)
    q_host = (q_rows if n_q > 1 else case.q).cpu().pin_memory()
    lens_host = None if case.seq_lens is None else case.seq_lens.cpu().pin_memory()
    out_h = torch.empty(rows_shape + (spec.D,), dtype=torch.float32, pin_memory=True)
    lse_h = torch.empty(rows_shape, dtype=torch.float32, pin_memory=True)
    ws_h = fd.Workspace()
    e2e_api = "fd_decode_host" if not args.unfused else "fd_decode_host (the fused path: the split + combine pair has no host-buffer entry)"
    if args.append:
        e2e_api = "pinned copies + fd_append_decode"
        q_dev = torch.empty_like(case.q)
        out_d, lse_d = torch.empty_like(out), torch.empty_like(lse)

        def e2e_step():
            q_dev.copy_(q_host, non_blocking=True)
            fd.append_decode(q_dev, case.k, case.v, k_new, v_new, seq_lens=seq_before,
                             max_seq_len=case.max_seq_len - 1, block_table=case.block_table, scale=spec.scale,
                             n_splits=spec.n_splits, out=out_d, lse=lse_d, workspace=ws_h)
            out_h.copy_(out_d, non_blocking=True)
            lse_h.copy_(lse_d, non_blocking=True)
            torch.cuda.current_stream(device).synchronize()
    elif n_q > 1:
        e2e_api = "pinned copies + fd_decode_rows"
        q_dev = torch.empty_like(q_rows)
        lens_dev = None if lens_host is None else torch.empty_like(case.seq_lens)
        lens_pinned = None if lens_host is None else lens_host.pin_memory()
        out_d, lse_d = torch.empty_like(out), torch.empty_like(lse)

        def e2e_step():
            q_dev.copy_(q_host, non_blocking=True)
            if lens_dev is not None:
                lens_dev.copy_(lens_pinned, non_blocking=True)
            fd.decode_rows(q_dev, case.k, case.v, causal=True, seq_lens=lens_dev, max_seq_len=case.max_seq_len,
                           block_table=case.block_table, scale=spec.scale, n_splits=spec.n_splits, out=out_d,
                           lse=lse_d, workspace=ws_h)
            out_h.copy_(out_d, non_blocking=True)
            lse_h.copy_(lse_d, non_blocking=True)
            torch.cuda.current_stream(device).synchronize()
    else:
        # a decode loop's view: the same pinned host buffers every step, arguments marshalled once
        e2e_api = ("fd_decode_host via HostDecoder (pinned q, lengths, out, lse: read and written by the kernels "
                   "over the host link every step)") if not args.unfused else e2e_api
        e2e_step = fd.HostDecoder(q_host, case.k, case.v, seq_lens_host=lens_host, max_seq_len=case.max_seq_len,
                                  block_table=case.block_table, scale=spec.scale, n_splits=spec.n_splits,
                                  out_host=out_h, lse_host=lse_h, workspace=ws_h)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    k_e2e = max(10, min(K, 2000))
    barrier(world)
    te0 = time.perf_counter()
    for _ in range(k_e2e):
        e2e_step()
    te1 = time.perf_counter()
    e2e_s = max_over_ranks(te1 - te0, world, device)
    e2e_value = world * step_bytes * k_e2e / e2e_s / 1e9
    h2d = q_host.numel() * 4 + (0 if lens_host is None or args.append else lens_host.numel() * 4)
    d2h = out_h.numel() * 4 + lse_h.numel() * 4

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    # ---- CPU baseline: the oracle on a bounded sample, host cores, rank 0 at N=1
    cpu = None
    if world == 1 and not args.no_cpu_baseline and n_q == 1 and not args.append and not args.unfused:
        v, note, el = OracleSampler(case).whole_groups(args.cpu_seconds)
        cpu = {"value": v, "unit": "GB/s", "cores": blas_threads(), "cpu_model": cpu_model(), "kind": "oracle",
               "sample": note, "seconds": round(el, 2)}

    gpd = fd.workspace_status(ws)
    g = spec.Hq * n_q // spec.Hkv
    gpad = 1
    while gpad < g and gpad < (16 if spec.kv_dtype == "bf16" else 8):
        gpad *= 2
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv, "D": spec.D,
                   "T": spec.T_cap, "kv_dtype": spec.kv_dtype, "q_dtype": "f32", "layout": spec.layout,
                   "rows": n_q, "append": bool(args.append),
                   "kv_bytes_per_step": kv_bytes, "bytes_per_step": step_bytes,
                   "l2": l2_note,
                   "plan": "balanced" if spec.n_splits == 0 else f"n_splits={spec.n_splits}",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "kernel": f"fd_split_kernel<D={spec.D},{spec.kv_dtype},G={gpad}> (fused LSE merge)",
                   "launch": ("single launches after an L2 flush, events around each" if warm is not None else
                              "one CUDA graph of K fd_decode-family calls" if graph is not None else
                              "K stream launches, enqueued behind a sleep kernel before the start event"),
                   "single_launch_event_us_p10_p50_p90": [round(x, 2) for x in
                                                          statistics.quantiles(launch_us, n=10)[0::4]]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(spec.name),
                     "peak_source": peak_src, "kernel": "fd_split_kernel", "launches_per_step": 1,
                     "mean_launch_us": mean_launch_us},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": k_e2e, "api": e2e_api},
        "warm": warm,
        "gpu_launches": timed_launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "kernel_status": gpd,
        "source_sha": source_hash(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_prefill(args):
    """fd_prefill on an N-token causal prompt whose keys fill the cache: a tensor-bound step."""
    world, rank, local = dist_env()
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libfdecode has no CPU path)")
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    import split_kv_decode_fd_gb300 as fd
    from workloads import make_case, small_spec
    fd.load_library()
    N, hkv = args.prefill, args.prefill_kv_heads
    if hkv < 1 or 32 % hkv:
        raise SystemExit("--prefill-kv-heads must divide 32")
    spec = small_spec(f"prefill_causal_B1_Hq32_Hkv{hkv}_N{N}", 1, 32, hkv, 128, N, seed=1003)
    case = make_case(spec, device)
    gen = torch.Generator(device=device).manual_seed(spec.seed + 31)
    q = torch.randn((1, 32, N, 128), generator=gen, device=device)
    out = torch.empty_like(q)
    lse = torch.empty((1, 32, N), device=device)
    ws = fd.Workspace()

    def step():
        fd.prefill(q, case.k, case.v, causal=True, max_seq_len=N, scale=spec.scale, out=out, lse=lse, workspace=ws)

    # useful flops: q.k and p.v over each row's causal keys (row i sees i + 1 keys), 2 per multiply-add
    flops = 4.0 * 128 * 32 * (N * (N + 1) / 2)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fd.workspace_status(ws) != 0:
        raise SystemExit("kernel reported an error during warm-up")
    K = args.steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(K):
            step()
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop(t0, t1)
    total_ms = max_over_ranks(start.elapsed_time(end), world, device)
    ms_per_step = total_ms / K
    tflops = flops / (ms_per_step * 1e-3) / 1e12
    peak, peak_src = measured_tensor_peak()
    # end to end: host q in, host out + lse back, copies around fd_prefill
    q_host = q.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=torch.float32, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=torch.float32, pin_memory=True)
    q_dev = torch.empty_like(q)

    def e2e_step():
        q_dev.copy_(q_host, non_blocking=True)
        fd.prefill(q_dev, case.k, case.v, causal=True, max_seq_len=N, scale=spec.scale, out=out, lse=lse,
                   workspace=ws)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    k_e2e = max(5, min(K, 50))
    te0 = time.perf_counter()
    for _ in range(k_e2e):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - te0, world, device)
    if rank != 0:
        return 0
    line = {
        "metric": "prefill attention TFLOP/s (useful causal flops)", "value": world * tflops, "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16x2 (hi+lo) -> f32",
        "data": "synthetic",
        "config": {"workload": spec.name, "B": 1, "Hq": 32, "Hkv": hkv, "D": 128, "n_q": N, "keys": N,
                   "causal": True, "kv_dtype": "bf16", "q_dtype": "f32", "flops_per_step": flops,
                   "launch": "one CUDA graph of K fd_prefill calls", "l2": prefill_l2_note(N, hkv),
                   "kernel": "fd_prefill_kernel (tcgen05.mma M=128; q and p as bf16 hi+lo: 2 MMAs per product)"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "traffic": recorded_traffic(spec.name, PREFILL_SOURCES), "peak_source": peak_src,
                     "kernel": "fd_prefill_kernel",
                     "launches_per_step": 1, "mean_launch_us": ms_per_step * 1e3},
        "e2e": {"value": world * flops * k_e2e / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": q_host.numel() * 4, "d2h_bytes_per_step": (out_h.numel() + lse_h.numel()) * 4,
                "steps": k_e2e, "api": "pinned copies + fd_prefill"},
        "gpu_launches": K, "clocks": clocks, "cpu_baseline": None, "kernel_status": fd.workspace_status(ws),
        "source_sha": source_hash(PREFILL_SOURCES),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.prefill:
        return run_prefill(args)
    return run_fdecode(args)


if __name__ == "__main__":
    sys.exit(main())
