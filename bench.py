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

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

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

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
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
    statistics (LSE, Delta) and the dQ rows.  Returns (seconds, metric FLOPs)
    where the FLOPs are the metric's count for those rows: 4*S*D per row
    forward and 2.5x that backward (halved under the causal mask)."""
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
    per_row = 4.0 * S * D * (0.5 if causal else 1.0)
    return dt, per_row * len(rows) * 3.5


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
            "sample": (f"fp64 CPU oracle, head (0,0) of {WORKLOAD['name']} "
                       f"{'causal' if causal else 'non-causal'}: forward, backward row "
                       f"statistics and dQ for {n} of {S} query rows ({dt:.1f} s); FLOPs "
                       "counted as the metric counts them for those rows")}


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


def run_step(buf, causal, scale, ev=None):
    from exact_attention_36_gb300 import fa

    if ev is not None:
        ev[0].record()
    fa.fwd(buf.q, buf.k, buf.v, buf.o, buf.lse, causal, scale)
    if ev is not None:
        ev[1].record()
    fa.bwd(buf.q, buf.k, buf.v, buf.o, buf.dout, buf.lse, buf.dq_acc, buf.delta,
           buf.dq, buf.dk, buf.dv, causal, scale)
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
    (ms per step, fwd ms per launch, bwd ms per call)."""
    for _ in range(warmup):
        run_step(buf, causal, scale)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    start.record()
    for i in range(steps):
        run_step(buf, causal, scale, evs[i])
    stop.record()
    barrier(dist_on)
    total = start.elapsed_time(stop)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    return max_over_ranks(total, dist_on) / steps, fwd_ms, bwd_ms


def time_e2e(q, k, v, dout, buf, causal, scale, steps, warmup, dist_on):
    """The same step through the C ABI with host buffers.  Every step copies
    its Q, K, V, dO from pinned host memory and reads its dQ, dK, dV back;
    the copies run on a second stream, double-buffered, so step k+1's inputs
    arrive while step k computes.  Returns (ms per step, H2D bytes, D2H bytes)."""
    dev = buf.q.device
    hin = [t.pin_memory() for t in (q, k, v, dout)]
    hout = [[torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
            for _ in range(2)]
    bufs = [buf, Buffers(q, k, v, dout, dev)]
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]  # inputs of buffer b copied
    done = [torch.cuda.Event() for _ in range(2)]   # step on buffer b computed
    fetched = [torch.cuda.Event() for _ in range(2)]  # outputs of buffer b read back

    def upload(b):
        with torch.cuda.stream(copy):
            copy.wait_event(done[b])  # the previous step on this buffer finished with it
            for d, h in zip((bufs[b].q, bufs[b].k, bufs[b].v, bufs[b].dout), hin):
                d.copy_(h, non_blocking=True)
            ready[b].record(copy)

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
            with torch.cuda.stream(copy):
                copy.wait_event(done[b])
                for h, d in zip(hout[b], (bufs[b].dq, bufs[b].dk, bufs[b].dv)):
                    h.copy_(d, non_blocking=True)
                fetched[b].record(copy)
        comp.wait_stream(copy)

    run(warmup)
    barrier(dist_on)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    run(steps)
    stop.record(comp)
    barrier(dist_on)
    ms = max_over_ranks(start.elapsed_time(stop), dist_on) / steps
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout[0])
    return ms, h2d, d2h


# ---------------------------------------------------------------- main


def kernel_source_hash():
    """Hash of the CUDA sources: traffic figures recorded from an ncu capture
    are only reported while the kernels they describe are unchanged."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_36_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


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
    ap.add_argument("--only-noncausal", action="store_true",
                    help="skip the causal measurement and the e2e loop (profiling runs)")
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
    sample = (f"fp64 CPU oracle on head (0,0) of {W['name']} non-causal: forward, backward "
              f"row statistics and dQ for {n} of {W['S']} query rows per step")
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
    if args.seq != W["S"]:
        W["S"] = args.seq
        W["name"] = f"B1_H16_S{args.seq}_D128"
    B, H, S, D = W["B"], W["H"], W["S"], W["D"]
    scale = 1.0 / math.sqrt(D)
    # every rank draws its own batch (weak scaling over independent heads)
    q, k, v, do = make_qkvdo(B, H, S, D, seed=rank)
    dev = torch.device("cuda", local_rank)
    buf = Buffers(q, k, v, do, dev)
    peaks, peak_src = load_peaks()

    with ClockSampler(local_rank) as clk:
        ms, fwd_ms, bwd_ms = time_device(buf, False, scale, args.steps, args.warmup, dist_on)
        if args.only_noncausal:
            ms_c = fwd_ms_c = bwd_ms_c = float("nan")
            e2e_ms, h2d, d2h = float("nan"), 0, 0
        else:
            ms_c, fwd_ms_c, bwd_ms_c = time_device(buf, True, scale, args.steps, args.warmup,
                                                   dist_on)
            e2e_ms, h2d, d2h = time_e2e(q, k, v, do, buf, False, scale, args.steps,
                                        args.warmup, dist_on)
    clocks = clk.summary()
    assert fa.device_error() == 0, "a bounded device wait ran out"

    ff, fb = flops(B, H, S, D, False)
    ffc, fbc = flops(B, H, S, D, True)
    value = job_tflops(world, ff + fb, ms)
    fwd_tf, bwd_tf = ff / (fwd_ms * 1e-3) / 1e12, fb / (bwd_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    if bwd_ms >= fwd_ms:
        dom, dom_ms, dom_fl = "fa_bwd (preprocess + main + dQ convert)", bwd_ms, fb
        traffic = recorded_traffic("fa_bwd") if S == WORKLOAD["S"] else None
    else:
        dom, dom_ms, dom_fl = "fa_fwd_kernel", fwd_ms, ff
        traffic = recorded_traffic("fa_fwd_kernel") if S == WORKLOAD["S"] else None
    achieved = dom_fl / (dom_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": W["name"], "B": B, "H": H, "S": S, "D": D, "causal": False,
                   "scale": scale, "inputs": "seeded N(0,1) bf16",
                   "l2": "inputs larger than L2 (Q,K,V,dO = 512 MiB per step)",
                   "parallelism": f"independent batch per GPU x{world}"},
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_pct_of_2250": 100 * fwd_tf / NOMINAL_PEAK_TFLOPS,
        "bwd_pct_of_2250": 100 * bwd_tf / NOMINAL_PEAK_TFLOPS,
        "pct_of_2250": 100 * value / world / NOMINAL_PEAK_TFLOPS,
        "causal": {"tflops": job_tflops(world, ffc + fbc, ms_c), "ms_per_step": ms_c,
                   "fwd_tflops": ffc / (fwd_ms_c * 1e-3) / 1e12,
                   "bwd_tflops": fbc / (bwd_ms_c * 1e-3) / 1e12},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_src} bf16_tflops_sustained", "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic},
        "e2e": {"value": job_tflops(world, ff + fb, e2e_ms), "unit": "TFLOPS",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 4 * args.steps,  # fa_fwd 1 + fa_bwd 3 per step of the value's region
        "clocks": clocks,
    }
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
