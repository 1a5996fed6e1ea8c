"""Throughput benchmark of the fused attention forward + backward on GB300.

One step = one pass of the whole hot path over one batch: fa_fwd (O, LSE)
then fa_bwd (Delta + dQ-accumulator zeroing, the fused backward kernel, dQ
conversion) on the long-context workload B=1, H=16, S=32768, D=128, bf16,
non-causal (the causal variant is measured in the same run and reported
under "causal").  Metric: TFLOPS counted as 4*B*H*S^2*D for the forward and
2.5x that for the backward (halved when causal).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank processes its own batch (independent
heads; no collective on the data path), value = total FLOPs / max time.
--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
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

import torch  # noqa: E402

METRIC = ("attention fwd/bwd TFLOPS (bf16, hdim128, S=32k) and % of 2.25 PF dense BF16 peak")
WORKLOAD = dict(name="B1_H16_S32768_D128", B=1, H=16, S=32768, D=128)
NOMINAL_PEAK_TFLOPS = 2250.0


def flops(B, H, S, D, causal):
    f = 4.0 * B * H * S * S * D
    if causal:
        f /= 2
    return f, 2.5 * f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # csv lines: timestamp, then the clock fields
        self.regions = {}  # name -> (t0, t1), host wall-clock seconds

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def _parse(line):
        """(wall-clock seconds, [fields after the timestamp]) of one sample, or None."""
        import datetime

        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            return None
        try:
            t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None
        return t, parts[1:]

    def mark(self, name, t0, t1):
        """Record the wall-clock span (time.time()) of a timed region, so that
        its own samples can be told apart from the others'."""
        self.regions[name] = (t0, t1)

    def region_mhz(self, name):
        """Median SM clock of the samples taken inside region `name` (None if none)."""
        if name not in self.regions:
            return None
        t0, t1 = self.regions[name]
        sm = []
        for line in self.lines:
            rec = self._parse(line)
            if rec is None or not (t0 <= rec[0] <= t1):
                continue
            try:
                sm.append(float(rec[1][0]))
            except ValueError:
                pass
        return statistics.median(sm) if sm else None

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        """Median SM clock, max clock and throttle reasons over the samples
        taken inside the marked timed regions (all samples if none marked)."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        spans = list(self.regions.values())
        for line in self.lines:
            rec = self._parse(line)
            if rec is None:
                continue
            if spans and not any(t0 <= rec[0] <= t1 for t0, t1 in spans):
                continue
            parts = rec[1]
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU) sample


def oracle_sample(q, k, v, dout, causal, scale, rows):
    """Time the fp64 CPU oracle on a bounded sample of the workload: head
    (0, 0), the listed query rows: forward rows (O, LSE), the backward row
    statistics (LSE, Delta) and the dQ rows.  The dK/dV pass is not in the
    sample (each key column needs every row's statistics, i.e. the whole
    head).  Returns (seconds, FLOPs of the work that ran), counted the
    metric's way per query row: 4*S*D forward, and of the backward's 10*S*D
    the three products the dQ rows need (S recomputed, dP, dQ: 6*S*D);
    halved under the causal mask."""
    import numpy as np

    import oracle

    qh, kh, vh, dh = (t[0, :, 0].double().numpy() for t in (q, k, v, dout))
    S, D = qh.shape
    t0 = time.perf_counter()
    oracle.forward_head(qh, kh, vh, causal, scale, rows=rows)
    lse, delta = oracle.row_stats_head(qh, kh, vh, dh, causal, scale, rows)
    lf = np.zeros(S)
    df = np.zeros(S)
    lf[rows] = lse
    df[rows] = delta
    oracle.dq_rows_head(qh, kh, vh, dh, lf, df, causal, scale, rows)
    dt = time.perf_counter() - t0
    per_row = (4.0 + 6.0) * S * D * (0.5 if causal else 1.0)
    return dt, per_row * len(rows)


SAMPLE_WHAT = ("forward, backward row statistics and dQ (not the dK/dV pass) for {n} of {S} "
               "query rows of head (0,0)")


def pick_rows(S, n, seed=0):
    g = torch.Generator().manual_seed(seed)
    return sorted(torch.randperm(S, generator=g)[:n].tolist())


def cpu_sample(q, k, v, dout, causal, scale, target_s=12.0):
    """Size the oracle sample to about target_s seconds, run it, and describe it."""
    import oracle

    S = q.shape[1]
    n = 32
    dt, fl = oracle_sample(q, k, v, dout, causal, scale, pick_rows(S, n, seed=2))
    # grow the sample until it is about target_s of CPU work (fixed per-call
    # costs make the first estimate low)
    for _ in range(3):
        if dt >= 0.6 * target_s or n >= S:
            break
        n = int(min(S, max(2 * n, n * target_s / max(dt, 1e-3))))
        dt, fl = oracle_sample(q, k, v, dout, causal, scale, pick_rows(S, n, seed=2))
    return {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": oracle.threads(), "kind": "oracle",
            "sample": (f"fp64 CPU oracle on {WORKLOAD['name']} "
                       f"{'causal' if causal else 'non-causal'}: "
                       + SAMPLE_WHAT.format(n=n, S=S)
                       + f" ({dt:.1f} s); FLOPs: 4*S*D forward + 6*S*D (S, dP, dQ products) "
                       "per sampled row, the metric's count for the work that ran")}


# ---------------------------------------------------------------- GPU timing


class Buffers:
    """Device buffers of one fwd+bwd step (inputs resident in HBM)."""

    def __init__(self, q, k, v, dout, dev):
        from exact_attention_36_gb300 import fa

        B, S, H, D = q.shape
        self.q, self.k, self.v, self.dout = (t.to(dev) for t in (q, k, v, dout))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        n = B * H * S
        ws = torch.empty(fa.bwd_workspace_size(B, H, S, D), dtype=torch.uint8, device=dev)
        acc_bytes = (n * D * 4 + 255) // 256 * 256
        self.dq_acc = ws[:acc_bytes].view(torch.float32)
        self.delta = ws[acc_bytes:acc_bytes + n * 4].view(torch.float32)
        self.ws = ws
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.sem = None
        if BWD_MODE.get("deterministic"):
            self.sem = torch.empty(fa.bwd_semaphore_bytes(B, H, S, D) // 4, dtype=torch.int32,
                                   device=dev)


# forward numerics knobs of profiling runs (library defaults unless given)
FWD_KNOBS = {}
# backward variant of measurement runs: {"deterministic": True} times the
# fixed-order dQ mode, {"pair_mode": 1} the CTA-pair kernel (defaults unless given)
BWD_MODE = {}


def run_step(buf, causal, scale, ev=None):
    from exact_attention_36_gb300 import fa

    if ev is not None:
        ev[0].record()
    fa.fwd(buf.q, buf.k, buf.v, buf.o, buf.lse, causal, scale, **FWD_KNOBS)
    if ev is not None:
        ev[1].record()
    if buf.sem is not None:
        fa.bwd_deterministic(buf.q, buf.k, buf.v, buf.o, buf.dout, buf.lse, buf.dq_acc,
                             buf.delta, buf.sem, buf.dq, buf.dk, buf.dv, causal, scale)
    else:
        fa.bwd(buf.q, buf.k, buf.v, buf.o, buf.dout, buf.lse, buf.dq_acc, buf.delta,
               buf.dq, buf.dk, buf.dv, causal, scale, pair_mode=BWD_MODE.get("pair_mode", -1))
    if ev is not None:
        ev[2].record()


def barrier(dist_on):
    """All ranks meet, and this rank's GPU work is finished."""
    if dist_on:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x, dist_on):
    """The largest value of x over all ranks (the step time that counts)."""
    if not dist_on:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank, ms_max):
    """Whole-job throughput: every rank processes its own batch (weak
    scaling), so the job does world x the per-rank FLOPs in the slowest
    rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def time_device(buf, causal, scale, steps, warmup, dist_on):
    """Device-time K steps (CUDA events on the launching stream).  Returns
    (ms per step, fwd ms per launch, bwd ms per call, (wall t0, wall t1) of
    the timed region)."""
    for _ in range(warmup):
        run_step(buf, causal, scale)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    t0 = time.time()
    start.record()
    for i in range(steps):
        run_step(buf, causal, scale, evs[i])
    stop.record()
    barrier(dist_on)
    t1 = time.time()
    total = start.elapsed_time(stop)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    return max_over_ranks(total, dist_on) / steps, fwd_ms, bwd_ms, (t0, t1)


def time_e2e(q, k, v, dout, buf, causal, scale, steps, warmup, dist_on):
    """The same step through the C ABI with host buffers.  Every step copies
    its Q, K, V, dO from pinned host memory and reads its dQ, dK, dV back;
    the copies are double-buffered, so step k+1's inputs arrive while step k
    computes, and uploads and read-backs run on two streams of their own (the
    host link carries both directions at once).  Returns (ms per step, H2D
    bytes, D2H bytes, (wall t0, wall t1) of the timed region)."""
    dev = buf.q.device
    hin = [t.pin_memory() for t in (q, k, v, dout)]
    hout = [[torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
            for _ in range(2)]
    bufs = [buf, Buffers(q, k, v, dout, dev)]
    comp = torch.cuda.current_stream()
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]  # inputs of buffer b copied
    done = [torch.cuda.Event() for _ in range(2)]   # step on buffer b computed
    fetched = [torch.cuda.Event() for _ in range(2)]  # outputs of buffer b read back

    def upload(b):
        with torch.cuda.stream(copy_in):
            copy_in.wait_event(done[b])  # the previous step on this buffer finished with it
            for d, h in zip((bufs[b].q, bufs[b].k, bufs[b].v, bufs[b].dout), hin):
                d.copy_(h, non_blocking=True)
            ready[b].record(copy_in)

    def run(nsteps):
        for b in range(2):
            done[b].record(comp)
            fetched[b].record(comp)
        upload(0)
        for s in range(nsteps):
            b = s & 1
            if s + 1 < nsteps:
                upload(b ^ 1)
            comp.wait_event(ready[b])
            comp.wait_event(fetched[b])  # its previous outputs were read back
            run_step(bufs[b], causal, scale)
            done[b].record(comp)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(done[b])
                for h, d in zip(hout[b], (bufs[b].dq, bufs[b].dk, bufs[b].dv)):
                    h.copy_(d, non_blocking=True)
                fetched[b].record(copy_out)
        comp.wait_stream(copy_in)
        comp.wait_stream(copy_out)

    run(warmup)
    barrier(dist_on)
    t0 = time.time()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    run(steps)
    stop.record(comp)
    barrier(dist_on)
    t1 = time.time()
    ms = max_over_ranks(start.elapsed_time(stop), dist_on) / steps
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout[0])
    return ms, h2d, d2h, (t0, t1)


# ---------------------------------------------------------------- main


# Translation units (and headers) that build each timed call; a traffic
# figure recorded from an ncu capture is reported only while these files are
# byte-for-byte what they were when it was captured.
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cu", "fa_api.cu", "fa_common.cuh", "sm100_ptx.cuh",
                      "exp2_poly.cuh", "exp2_poly_coeffs.h"],
    "fa_bwd": ["fa_bwd.cu", "fa_api.cu", "fa_common.cuh", "sm100_ptx.cuh"],
}
# ncu kernel names (prefix before the template arguments) of each call
CALL_KERNELS = {
    "fa_fwd_kernel": ["fa_fwd_kernel"],
    "fa_bwd": ["fa_bwd_prep", "fa_bwd_kernel", "fa_bwd_dq_cvt"],
}
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def source_hash(call):
    """sha256 (first 16 hex digits) of the sources that build `call`."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_36_gb300", "csrc")
    for name in KERNEL_SOURCES[call]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(call):
    """DRAM bytes per call from the last ncu capture, or None when the
    capture is missing or its kernels' sources have changed since."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    with open(TRAFFIC_JSON) as f:
        rec = json.load(f)
    ent = rec.get(call)
    if not ent or ent.get("source_hash") != source_hash(call):
        return None
    return ent.get("bytes_per_launch")


def record_traffic(csv_path, hashes_path, workload, command):
    """Write profiles/traffic.json from an ncu --csv capture of
    dram__bytes_read.sum / dram__bytes_write.sum over one bench step
    (one launch of each kernel).  `hashes_path` holds the source hashes
    printed by --source-hashes on the box in the same call as the capture;
    a call whose sources differ here is refused."""
    import csv

    with open(hashes_path) as f:
        box_hashes = json.load(f)
    by_kernel = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        name = row["Kernel Name"]
        base = name.split("(")[0].split("<")[0].split("::")[-1].strip()
        val = float(row["Metric Value"].replace(",", ""))
        unit = row.get("Metric Unit", "byte").strip().lower()
        mult = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9}.get(unit, 1)
        key = (row["ID"], base)
        by_kernel.setdefault(key, 0.0)
        by_kernel[key] += val * mult
    per_base = {}
    for (_, base), b in by_kernel.items():
        per_base.setdefault(base, []).append(b)
    out = {}
    for call, kernels in CALL_KERNELS.items():
        if box_hashes.get(call) != source_hash(call):
            raise SystemExit(f"{call}: sources differ from the captured ones; not recorded")
        if not all(k in per_base for k in kernels):
            continue
        per = {k: int(statistics.median(per_base[k])) for k in kernels}
        out[call] = {"source_hash": source_hash(call), "sources": KERNEL_SOURCES[call],
                     "bytes_per_launch": sum(per.values()), "per_kernel_bytes": per,
                     "launches_seen": {k: len(per_base[k]) for k in kernels},
                     "workload": workload, "command": command}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    return out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for quick runs)")
    ap.add_argument("--seq", type=int, default=WORKLOAD["S"],
                    help="sequence length override (profiling runs on a smaller case)")
    ap.add_argument("--dim", type=int, default=WORKLOAD["D"],
                    help="head dim override (profiling runs)")
    ap.add_argument("--batch", type=int, default=WORKLOAD["B"],
                    help="batch override (profiling runs)")
    ap.add_argument("--poly-groups", type=int, default=-1,
                    help="forward: columns of every 8 whose exp2 takes the FMA polynomial "
                         "(profiling runs; -1 = library default)")
    ap.add_argument("--poly-degree", type=int, default=-1,
                    help="forward: degree of that polynomial, 3 or 5 (profiling runs)")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the fixed-order (bitwise repeatable) backward (measurement runs)")
    ap.add_argument("--pair", action="store_true",
                    help="time the CTA-pair backward kernel, D = 128 (measurement runs)")
    ap.add_argument("--only-noncausal", action="store_true",
                    help="skip the causal measurement and the e2e loop (profiling runs)")
    ap.add_argument("--source-hashes", action="store_true",
                    help="print the source hash of each timed call and exit")
    ap.add_argument("--record-traffic", nargs=2, metavar=("NCU_CSV", "HASHES_JSON"),
                    help="write profiles/traffic.json from an ncu DRAM-bytes capture and exit")
    ap.add_argument("--traffic-command", default="",
                    help="with --record-traffic: the capture command, recorded beside it")
    return ap.parse_args()


def reference_arm(args, rank):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample (a fixed set of query rows of one head) of the workload."""
    if rank != 0:
        return
    from exact_attention_36_gb300.inputs import make_qkvdo

    import oracle

    W = WORKLOAD
    q, k, v, do = make_qkvdo(W["B"], W["H"], W["S"], W["D"], seed=0)
    scale = 1.0 / math.sqrt(W["D"])
    probe = pick_rows(W["S"], 16, seed=1)
    dt0, _ = oracle_sample(q, k, v, do, False, scale, probe)
    n = int(max(16, min(W["S"], 16 * 4.0 / max(dt0, 1e-3))))  # ~4 s per step
    rows = pick_rows(W["S"], n, seed=2)
    for _ in range(args.warmup):
        oracle_sample(q, k, v, do, False, scale, rows)
    times, fl = [], 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample(q, k, v, do, False, scale, rows)
        times.append(dt)
    t = sum(times) / len(times)
    value = fl / t / 1e12
    sample = (f"fp64 CPU oracle on {W['name']} non-causal, per step: "
              + SAMPLE_WHAT.format(n=n, S=W["S"])
              + "; FLOPs: 4*S*D forward + 6*S*D (S, dP, dQ products) per sampled row")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": W["name"], "B": 1, "H": 16, "S": W["S"], "D": W["D"],
                       "causal": False, "sample_rows": n},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.source_hashes:
        print(json.dumps({call: source_hash(call) for call in KERNEL_SOURCES}))
        return
    if args.record_traffic:
        out = record_traffic(args.record_traffic[0], args.record_traffic[1],
                             f"B{args.batch}_H16_S{args.seq}_D{args.dim} non-causal, one bench step",
                             args.traffic_command)
        print(json.dumps(out, indent=1))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local_rank)
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    from exact_attention_36_gb300 import build as fa_build
    from exact_attention_36_gb300 import fa
    from exact_attention_36_gb300.inputs import make_qkvdo

    fa_build.build()
    W = dict(WORKLOAD)
    W.update(B=args.batch, S=args.seq, D=args.dim)
    W["name"] = f"B{W['B']}_H{W['H']}_S{W['S']}_D{W['D']}"
    is_headline = (W["B"], W["S"], W["D"]) == (WORKLOAD["B"], WORKLOAD["S"], WORKLOAD["D"])
    if args.poly_groups >= 0:
        FWD_KNOBS["poly_exp2_groups"] = args.poly_groups
    if args.poly_degree >= 0:
        FWD_KNOBS["poly_exp2_degree"] = args.poly_degree
    if args.deterministic:
        BWD_MODE["deterministic"] = True
    if args.pair:
        BWD_MODE["pair_mode"] = 1
    B, H, S, D = W["B"], W["H"], W["S"], W["D"]
    scale = 1.0 / math.sqrt(D)
    # every rank draws its own batch (weak scaling over independent heads)
    q, k, v, do = make_qkvdo(B, H, S, D, seed=rank)
    dev = torch.device("cuda", local_rank)
    buf = Buffers(q, k, v, do, dev)
    peaks, peak_src = load_peaks()

    with ClockSampler(local_rank) as clk:
        ms, fwd_ms, bwd_ms, span = time_device(buf, False, scale, args.steps, args.warmup,
                                               dist_on)
        clk.mark("noncausal", *span)
        if args.only_noncausal:
            ms_c = fwd_ms_c = bwd_ms_c = float("nan")
            e2e_ms, h2d, d2h = float("nan"), 0, 0
        else:
            ms_c, fwd_ms_c, bwd_ms_c, span = time_device(buf, True, scale, args.steps,
                                                         args.warmup, dist_on)
            clk.mark("causal", *span)
            e2e_ms, h2d, d2h, span = time_e2e(q, k, v, do, buf, False, scale, args.steps,
                                              args.warmup, dist_on)
            clk.mark("e2e", *span)
    clocks = clk.summary()
    assert fa.device_error() == 0, "a bounded device wait ran out"

    ff, fb = flops(B, H, S, D, False)
    ffc, fbc = flops(B, H, S, D, True)
    value = job_tflops(world, ff + fb, ms)
    fwd_tf, bwd_tf = ff / (fwd_ms * 1e-3) / 1e12, fb / (bwd_ms * 1e-3) / 1e12
    # The calls are timed one at a time inside a sub-second region, so the
    # burst peak (a GEMM timed alone) is the denominator; the sustained one
    # (a seconds-long GEMM loop, taken at a lower clock under the power cap)
    # is reported beside it with the clock it was measured at.
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained")
    if bwd_ms >= fwd_ms:
        dom, dom_ms, dom_fl, call = "fa_bwd (preprocess + main + dQ convert)", bwd_ms, fb, "fa_bwd"
    else:
        dom, dom_ms, dom_fl, call = "fa_fwd_kernel", fwd_ms, ff, "fa_fwd_kernel"
    traffic = recorded_traffic(call) if is_headline else None
    achieved = dom_fl / (dom_ms * 1e-3) / 1e12

    def per_clock(fl, ms_call, mhz):
        # clock-normalised: FLOP per SM cycle (of 8192 for the dense bf16
        # tensor pipe) at the median SM clock sampled during the call's region
        if mhz is None or not (ms_call == ms_call):
            return None
        cycles = ms_call * 1e-3 * mhz * 1e6
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        return {"sm_mhz": mhz, "kcycles": cycles / 1e3,
                "flop_per_sm_cycle": fl / cycles / n_sm,
                "frac_of_8192": fl / cycles / n_sm / 8192.0}

    mhz_n, mhz_c = clk.region_mhz("noncausal"), clk.region_mhz("causal")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": W["name"], "B": B, "H": H, "S": S, "D": D, "causal": False,
                   "scale": scale, "inputs": "seeded N(0,1) bf16",
                   "l2": (f"inputs larger than L2 (Q,K,V,dO = {4 * B * S * H * D * 2 >> 20} MiB "
                          "per step)"),
                   "parallelism": f"independent batch per GPU x{world}"},
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "fwd_pct_of_2250": 100 * fwd_tf / NOMINAL_PEAK_TFLOPS,
        "bwd_pct_of_2250": 100 * bwd_tf / NOMINAL_PEAK_TFLOPS,
        "pct_of_2250": 100 * value / world / NOMINAL_PEAK_TFLOPS,
        "fwd_frac_of_burst": fwd_tf / peak, "bwd_frac_of_burst": bwd_tf / peak,
        "clock_normalised": {"fwd": per_clock(ff, fwd_ms, mhz_n),
                             "bwd": per_clock(fb, bwd_ms, mhz_n),
                             "causal_fwd": per_clock(ffc, fwd_ms_c, mhz_c),
                             "causal_bwd": per_clock(fbc, bwd_ms_c, mhz_c)},
        "causal": {"tflops": job_tflops(world, ffc + fbc, ms_c), "ms_per_step": ms_c,
                   "fwd_tflops": ffc / (fwd_ms_c * 1e-3) / 1e12,
                   "bwd_tflops": fbc / (bwd_ms_c * 1e-3) / 1e12,
                   "fwd_frac_of_burst": ffc / (fwd_ms_c * 1e-3) / 1e12 / peak,
                   "bwd_frac_of_burst": fbc / (bwd_ms_c * 1e-3) / 1e12 / peak},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_sustained": peak_sus,
                     "peak_sustained_sm_mhz": peaks.get("clocks_under_load", {}).get(
                         "sm_mhz_median"),
                     "frac_of_sustained": achieved / peak_sus if peak_sus else None,
                     "sm_mhz_during_call": mhz_n},
        "e2e": {"value": job_tflops(world, ff + fb, e2e_ms), "unit": "TFLOPS",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "sm_mhz": clk.region_mhz("e2e")},
        # fa_fwd 1 + fa_bwd 3 (4 in the fixed-order mode) per step of the value's region
        "gpu_launches": (5 if args.deterministic else 4) * args.steps,
        "clocks": clocks,
    }
    if FWD_KNOBS:
        line["config"]["forward_knobs"] = dict(FWD_KNOBS)
    if BWD_MODE:
        line["config"]["backward_mode"] = dict(BWD_MODE)
    if args.only_noncausal:
        line["causal"] = None
        line["e2e"] = None
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_sample(q, k, v, do, False, scale)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
