"""Benchmark of the VC-Attention hot path on GB300.

One step = the whole path over one batch: vca_group (k-means + permutation) ->
vca_prep_quant (fused V-Smooth prep) -> vca_attention (FP8 attention with
ExpCast and the mean restore), on the Wan2.2-14B-shaped video self-attention
workload (B=1, H=40, N=70,656, d=128, k=64, 8 k-means rounds).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload wan|wan_exp|nvfp4|tiny] [--N n] [--table]

`value` = attention FLOP (4 B H N^2 d) per second of the whole step, inputs
resident in device memory; `e2e` = the same with every step's inputs copied
from pinned host memory and its output copied back inside the timed region,
the copies on their own streams overlapping the neighbouring steps' kernels.
`--impl reference` times the CPU oracle on the host cores instead (a bounded
sample of the same workload per step, extrapolated).  Under torchrun every rank
runs its own replica of the workload (the path shards by (batch, head) with no
exchange); the max time over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wan")
    ap.add_argument("--N", type=int, default=0, help="override the sequence length")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the attention timings of the exp-path and NVFP4 configurations")
    ap.add_argument("--table", action="store_true",
                    help="one line per configuration (tiny, Wan + ExpCast, Wan exp path, NVFP4, the N sweep): "
                         "each kernel's time against its roofline and the error against exact attention")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = self.smi_id(device_index)
        self.proc = None
        self.lines = []

    @staticmethod
    def smi_id(device_index: int) -> str:
        """nvidia-smi's name for CUDA device `device_index`: CUDA numbers the
        devices CUDA_VISIBLE_DEVICES lists, nvidia-smi all of them."""
        vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        if device_index < len(vis) and (vis[device_index].isdigit() or vis[device_index].startswith("GPU-")):
            return vis[device_index]
        return str(device_index)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


# The attention kernel of each V format, and the sources it is built from.
ATTN_KERNELS = {
    "e4m3": ("attention_e4m3_kernel", ["vca_attention.cu", "vca_attention_common.cuh", "vca_device.cuh"]),
    "nvfp4": ("attention_nvfp4_kernel", ["vca_attention_fp4.cu", "vca_attention_common.cuh", "vca_device.cuh"]),
}


def kernel_sources_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "bit_attention_video_smooth_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def attention_traffic(w):
    """DRAM bytes per attention launch from the committed ncu summary, scaled
    linearly in B*H*N to this workload; None when the kernel's sources changed
    since the capture."""
    name, files = ATTN_KERNELS[w.vmode]
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "attention_traffic.json")))[name]
        if rec.get("sources_sha256") != kernel_sources_sha(files):
            return None
        c = rec["captured_on"]
        return rec["dram_bytes_per_launch"] * (w.B * w.H * w.N) / (c["B"] * c["H"] * c["N"])
    except (OSError, ValueError, KeyError):
        return None


# Nominal dense tensor rates of a GB300 (TFLOP/s), for the fraction of nominal
# reported beside the measured one.
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0, "fp4": 13500.0}
# The rate each attention kernel's two contractions run at (QK, PV): the
# E4M3 kernel runs both as FP8 MMAs; the NVFP4 kernel runs QK as FP8 and PV as
# the block-scaled FP4 MMA.
ATTN_RATES = {"e4m3": ("fp8", "fp8"), "nvfp4": ("fp8", "fp4")}


def _bound(rates, tflops):
    """Bound of a kernel whose FLOPs split evenly between QK and PV."""
    return 1.0 / (0.5 / tflops[rates[0]] + 0.5 / tflops[rates[1]])


def attention_peak(vmode, peaks):
    """Tensor peak of the attention kernel in TFLOP/s, and its source.

    From the measured burst cuBLAS bf16 rate b, scaled by the nominal ratios
    (FP8 = 2 b, FP4 = 6 b): the kernels run at the full SM clock without
    reaching the power cap, so the burst figure applies (the sustained figure
    was taken at a power-capped clock well below the kernel's)."""
    if peaks and "bf16_tflops" in peaks:
        b, src = peaks["bf16_tflops"], "measured burst cuBLAS bf16"
    else:
        b, src = 1900.0, "fallback 1.9 PF burst bf16"
    measured = {k: b * v / NOMINAL_TFLOPS["bf16"] for k, v in NOMINAL_TFLOPS.items()}
    qk, pv = ATTN_RATES[vmode]
    return _bound(ATTN_RATES[vmode], measured), f"{src} x nominal ratios; QK at the {qk} rate, PV at the {pv} rate"


def attention_nominal(vmode):
    return _bound(ATTN_RATES[vmode], NOMINAL_TFLOPS)


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(w, seed: int = 0):
    """Time the oracle on a bounded sample of workload `w`; returns (seconds
    extrapolated to one whole step, cores, description)."""
    import numpy as np
    import oracle
    from bit_attention_video_smooth_gb300 import inputs as I

    oracle.build()
    cores = oracle.threads()
    # 1024 query rows per head (always the first and last blocks' edge rows) on
    # eight heads: about 11 s of oracle work on 16 cores at the Wan shape
    heads = max(1, min(w.BH, 8))
    rows_per_head = 1024
    sub = I.with_n(w, w.N, H=heads, B=1)
    q, k, v = (I.to_u16(t).reshape(heads, w.N, 128) for t in I.make_qkv(sub, seed=seed))
    rows = I.sample_rows(w.N, rows_per_head, seed=seed).numpy()
    t0 = time.perf_counter()
    _, perm, _, _ = oracle.group(v, w.k, w.iters)
    t1 = time.perf_counter()
    vmode = oracle.V_NVFP4 if w.vmode == "nvfp4" else oracle.V_E4M3
    pre = oracle.prep(q, k, v, perm, vmode=vmode)
    t2 = time.perf_counter()
    mode = oracle.P_NVFP4 if w.vmode == "nvfp4" else (oracle.P_EXPCAST if w.expcast else oracle.P_EXP)
    oracle.attention(pre, mode, rows=rows)
    t3 = time.perf_counter()
    reps = w.BH / heads
    full = (t1 - t0) * reps + (t2 - t1) * reps + (t3 - t2) * reps * (w.N / rows.size)
    desc = (f"oracle on {heads} of {w.BH} heads: group+prep in full, attention on {rows.size} of {w.N} "
            f"query rows per head; extrapolated x{reps:.2f} heads, x{w.N / rows.size:.1f} rows")
    return full, cores, desc, (t3 - t0)


# ---------------------------------------------------------------------------
# distributed helpers (replicas: barrier + max over ranks only)
# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def dist_max(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
def workload_config(w, n_gpus):
    """The `config` of a bench line (both arms print the same one)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "k": w.k, "iters": w.iters,
            "vmode": w.vmode, "expcast": w.expcast, "parallelism": f"replicas x{n_gpus}",
            "l2": f"inputs (3 x {w.BH * w.N * 256 / 1e6:.0f} MB) exceed L2; no flush"}


def run_reference(args, w, ws, rank):
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(w, seed=1)
    times, cores, desc = [], 1, ""
    for i in range(args.steps):
        full, cores, desc, _ = oracle_sample(w, seed=2 + i)
        times.append(full)
    t = statistics.mean(times)
    value = w.flops / t / 1e12
    line = {
        "impl": "reference", "metric": "VC-attention TFLOP/s (group + prep + attention step)",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64/f32 (oracle)", "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, ws, rank, local):
    import torch
    from bit_attention_video_smooth_gb300 import inputs as I
    from bit_attention_video_smooth_gb300 import vca

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    vmode = vca.VCA_V_NVFP4 if w.vmode == "nvfp4" else vca.VCA_V_E4M3
    Q, K, V = I.make_qkv(w, seed=1234 + rank, device=dev)
    g = vca.alloc_group(w.B, w.H, w.N, w.k, dev)
    p = vca.alloc_prep(w.B, w.H, w.N, vmode, dev)
    O = torch.empty((w.B, w.H, w.N, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(marks=None):
        if marks:
            marks[0].record(stream)
        vca.vca_group(V, w.k, w.iters, g.labels, g.perm, g.counts, g.centroids, g.ws)
        if marks:
            marks[1].record(stream)
        vca.vca_prep_quant(Q, K, V, g.perm, vmode, p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale,
                           p.v_mean, p.ws)
        if marks:
            marks[2].record(stream)
        vca.vca_attention(p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean, w.B, w.H, w.N, 128,
                          0.0, int(w.expcast), vmode, O, status)
        if marks:
            marks[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    # inputs (Q, K, V: 3 x BH N d bf16) exceed the 129 MB L2, so no flush is needed between steps
    marks = [[ev() for _ in range(4)] for _ in range(args.steps)]
    start, stop = ev(), ev()
    dist_barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            step(marks[i])
        stop.record(stream)
        torch.cuda.synchronize()
    dist_barrier(ws)
    ms_total = start.elapsed_time(stop)
    t_group = statistics.mean(m[0].elapsed_time(m[1]) for m in marks)
    t_prep = statistics.mean(m[1].elapsed_time(m[2]) for m in marks)
    t_attn = statistics.mean(m[2].elapsed_time(m[3]) for m in marks)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    ms_step = dist_max(ms_total / args.steps, ws)
    value = ws * w.flops / (ms_step * 1e-3) / 1e12

    # End to end through the public API: every step copies its inputs from
    # pinned host memory and its output back, inside the timed region.  The
    # copies run on their own streams and overlap the neighbouring steps'
    # kernels, as a serving pipeline would: E2E_SETS sets of device inputs
    # and outputs, a step's inputs travelling up to E2E_SETS - 1 steps ahead.
    # Three sets, not two: on the Grace host, host<->device copies stall now
    # and then for 30-130 ms (about every 0.5 s once much memory has been
    # freed, as after a test run), longer than one step; a second step of
    # lead absorbs that.
    e2e = None
    if not args.no_e2e:
        E2E_SETS = 3
        hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
        hO = [torch.empty(O.shape, dtype=O.dtype, pin_memory=True) for _ in range(E2E_SETS)]
        d_in = [tuple(torch.empty_like(t) for t in (Q, K, V)) for _ in range(E2E_SETS)]
        d_out = [torch.empty_like(O) for _ in range(E2E_SETS)]
        copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(E2E_SETS)]
        in_free = [torch.cuda.Event() for _ in range(E2E_SETS)]
        out_ready = [torch.cuda.Event() for _ in range(E2E_SETS)]
        out_free = [torch.cuda.Event() for _ in range(E2E_SETS)]

        def e2e_step(i):
            sl = i % E2E_SETS
            dq, dk, dv = d_in[sl]
            copy_in.wait_event(in_free[sl])           # step i-E2E_SETS has finished reading this set
            with torch.cuda.stream(copy_in):
                dq.copy_(hQ, non_blocking=True)
                dk.copy_(hK, non_blocking=True)
                dv.copy_(hV, non_blocking=True)
                in_ready[sl].record(copy_in)
            stream.wait_event(in_ready[sl])
            stream.wait_event(out_free[sl])           # step i-E2E_SETS's output has left this buffer
            vca.vca_group(dv, w.k, w.iters, g.labels, g.perm, g.counts, g.centroids, g.ws)
            vca.vca_prep_quant(dq, dk, dv, g.perm, vmode, p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale,
                               p.v_mean, p.ws)
            in_free[sl].record(stream)
            vca.vca_attention(p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean, w.B, w.H, w.N, 128,
                              0.0, int(w.expcast), vmode, d_out[sl], status)
            out_ready[sl].record(stream)
            copy_out.wait_event(out_ready[sl])
            with torch.cuda.stream(copy_out):
                hO[sl].copy_(d_out[sl], non_blocking=True)
                out_free[sl].record(copy_out)

        for i in range(max(3, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        es, ee = ev(), ev()
        dist_barrier(ws)
        es.record(copy_in)
        for i in range(args.steps):
            e2e_step(i)
        copy_out.wait_stream(stream)
        ee.record(copy_out)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the end-to-end run")
        ms_e2e = dist_max(es.elapsed_time(ee) / args.steps, ws)
        h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV))
        e2e = {"value": ws * w.flops / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hO[0].numel() * hO[0].element_size(),
               "copies": f"own streams, overlapping the neighbouring steps' kernels ({E2E_SETS} buffer sets)"}

    peak, peak_note = attention_peak(w.vmode, load_peaks())
    achieved = w.flops / (t_attn * 1e-3) / 1e12
    traffic = attention_traffic(w)
    line = {
        "metric": "VC-attention TFLOP/s (group + prep + attention step)", "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if vmode == 0 else "e4m3/e2m1",
        "data": "synthetic",
        "config": workload_config(w, ws),
        "breakdown_ms": {"group": t_group, "prep": t_prep, "attention": t_attn},
        "attention_tflops": achieved,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_note,
                     "kernel": ATTN_KERNELS[w.vmode][0], "nominal_peak": attention_nominal(w.vmode),
                     "frac_of_nominal": achieved / attention_nominal(w.vmode)},
        "gpu_launches": args.steps * (1 + 2 * w.iters + 1 + 3 + 1),
        "clocks": clocks.summary(),
    }
    if e2e:
        line["e2e"] = e2e
    if not args.no_extra and w.name == "wan":
        line["other_configs"] = other_configs(args, p, w, status, stream)
    if rank == 0 and not args.no_cpu_baseline:
        full, cores, desc, wall = oracle_sample(w)
        line["cpu_baseline"] = {"value": w.flops / full / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "sample_wall_s": wall}
    if rank == 0:
        print(json.dumps(line), flush=True)


def other_configs(args, p, w, status, stream):
    """Attention alone on the other single-GPU configurations, timed in the
    same process after the step: the Wan shape with ExpCast off (the exp path,
    on the step's prepared operands), the NVFP4 workload and the sequence-length
    sweep's other points (each with its own inputs, grouped and prepared
    once)."""
    import torch
    from bit_attention_video_smooth_gb300 import inputs as I
    from bit_attention_video_smooth_gb300 import vca

    reps = max(3, args.steps)
    peaks = load_peaks()

    def timed(fn):
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the other configurations")
        return e0.elapsed_time(e1) / reps

    def entry(wl, ms):
        peak, _ = attention_peak(wl.vmode, peaks)
        tf = wl.flops / (ms * 1e-3) / 1e12
        return {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "vmode": wl.vmode, "expcast": wl.expcast,
                "attention_ms": ms, "attention_tflops": tf, "frac": tf / peak, "peak": peak,
                "frac_of_nominal": tf / attention_nominal(wl.vmode), "kernel": ATTN_KERNELS[wl.vmode][0],
                "reps": reps}

    out = {}
    we = I.WORKLOADS["wan_exp"]
    O = torch.empty((w.B, w.H, w.N, 128), dtype=torch.bfloat16, device=p.q8.device)
    out["wan_exp"] = entry(we, timed(lambda: vca.vca_attention(
        p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean, w.B, w.H, w.N, 128, 0.0, 0, 0, O, status)))
    del O
    w4 = I.WORKLOADS["nvfp4"]
    Q, K, V = I.make_qkv(w4, seed=4321, device=p.q8.device)
    g = vca.group(V, w4.k, w4.iters)
    p4 = vca.prep_quant(Q, K, V, g.perm, vca.VCA_V_NVFP4)
    O4 = torch.empty((w4.B, w4.H, w4.N, 128), dtype=torch.bfloat16, device=p.q8.device)
    out["nvfp4"] = entry(w4, timed(lambda: vca.attention(p4, w4.B, w4.H, w4.N, expcast=False, out=O4,
                                                         dev_status=status)))
    del Q, K, V, g, p4, O4
    torch.cuda.empty_cache()
    # the N sweep at B=1, H=40 (N = 70,656 is the step itself)
    for n in (4096, 16384, 32768, 131072):
        ws = I.with_n(I.WORKLOADS["sweep"], n)
        Q, K, V = I.make_qkv(ws, seed=4321 + n, device=p.q8.device)
        g = vca.group(V, ws.k, ws.iters)
        ps = vca.prep_quant(Q, K, V, g.perm, vca.VCA_V_E4M3)
        del Q, K, V, g
        Os = torch.empty((ws.B, ws.H, ws.N, 128), dtype=torch.bfloat16, device=p.q8.device)
        out[ws.name] = entry(ws, timed(lambda: vca.attention(ps, ws.B, ws.H, ws.N, expcast=ws.expcast, out=Os,
                                                             dev_status=status)))
        del ps, Os
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# per-configuration table: kernels against their rooflines
# ---------------------------------------------------------------------------
def group_bytes(w) -> float:
    """Algorithmic HBM bytes of vca_group: V (bf16) read and labels written once
    per round, then labels read and the permutation written by the sort."""
    return w.iters * w.BH * w.N * (w.d * 2 + 4) + w.BH * w.N * 8


def prep_bytes(w) -> float:
    """Algorithmic HBM bytes of vca_prep_quant: Q, K, V (bf16) and the
    permutation read once; q8, k8 and the V residual (E4M3: 1 byte a value;
    NVFP4: half a byte plus one E4M3 scale per 16) written once; block means
    (bf16), Q/K block scales and V scales."""
    nb = w.N // 128
    v_res = w.d if w.vmode == "e4m3" else w.d // 2 + w.d // 16
    v_scale = w.d * 4 if w.vmode == "e4m3" else 4
    return w.BH * (w.N * (3 * w.d * 2 + 4 + 2 * w.d + v_res) + nb * (w.d * 2 + 8) + v_scale)


def table_line(w, peaks, reps: int = 3):
    import torch
    from bit_attention_video_smooth_gb300 import inputs as I
    from bit_attention_video_smooth_gb300 import vca

    vmode = vca.VCA_V_NVFP4 if w.vmode == "nvfp4" else vca.VCA_V_E4M3
    Q, K, V = I.make_qkv(w, seed=77, device="cuda")
    g = vca.alloc_group(w.B, w.H, w.N, w.k)
    p = vca.alloc_prep(w.B, w.H, w.N, vmode)
    O = torch.empty((w.B, w.H, w.N, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stages = {
        "group": lambda: vca.vca_group(V, w.k, w.iters, g.labels, g.perm, g.counts, g.centroids, g.ws, status),
        "prep": lambda: vca.vca_prep_quant(Q, K, V, g.perm, vmode, p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf,
                                           p.v_scale, p.v_mean, p.ws),
        "attention": lambda: vca.attention(p, w.B, w.H, w.N, expcast=w.expcast, out=O, dev_status=status),
    }
    ms = {}
    for name, fn in stages.items():
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / reps
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    # error against exact softmax attention (fp64 on the device) on sampled rows
    # of the first and last head
    errs = []
    rows = I.sample_rows(w.N, 32, seed=5).to("cuda").long()
    Qf, Kf, Vf = (t.view(w.BH, w.N, 128) for t in (Q, K, V))
    for h in (0, w.BH - 1):
        s = (Qf[h, rows].double() @ Kf[h].double().T) / (128 ** 0.5)
        ref = torch.softmax(s, dim=-1) @ Vf[h].double()
        got = O.view(w.BH, w.N, 128)[h, rows].double()
        errs.append(float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref)))
    # V-Smooth diagnostic: the share of V's energy that the 128-token block
    # means take out, blocks in cluster (permuted) order vs sequence order
    removed = {"sorted": [], "sequence": []}
    for h in (0, w.BH - 1):
        v = Vf[h].double()
        total = float((v * v).sum())
        for key, order in (("sorted", g.perm[h].long()), ("sequence", None)):
            vb = (v if order is None else v[order]).view(w.N // 128, 128, 128)
            res = vb - vb.mean(dim=1, keepdim=True)
            removed[key].append(1.0 - float((res * res).sum()) / total)
    # the QK Hadamard prep option: its prep time, and the error of attention over
    # the rotated operands on the same sampled rows
    p_h = vca.alloc_prep(w.B, w.H, w.N, vmode)
    prep_h = lambda: vca.prep_quant(Q, K, V, g.perm, vmode, out=p_h, qk_hadamard=True)
    for _ in range(2):
        prep_h()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        prep_h()
    e1.record()
    torch.cuda.synchronize()
    prep_h_ms = e0.elapsed_time(e1) / reps
    O_h = vca.attention(p_h, w.B, w.H, w.N, expcast=w.expcast)
    torch.cuda.synchronize()
    errs_h = []
    for h in (0, w.BH - 1):
        s = (Qf[h, rows].double() @ Kf[h].double().T) / (128 ** 0.5)
        ref = torch.softmax(s, dim=-1) @ Vf[h].double()
        got = O_h.view(w.BH, w.N, 128)[h, rows].double()
        errs_h.append(float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref)))
    del p_h, O_h
    # permutation reuse (the pages group on a quarter of the steps and reuse
    # the permutation over 4 adjacent ones): one group call and four prep +
    # attention steps against the four steps alone, each schedule timed once
    reuse = {}
    for key, sched in (("four_steps_ms", ["prep", "attention"] * 4),
                       ("group_and_four_steps_ms", ["group"] + ["prep", "attention"] * 4)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for name in sched:
            stages[name]()
        e1.record()
        torch.cuda.synchronize()
        reuse[key] = e0.elapsed_time(e1)
    reuse["group_overhead"] = reuse["group_and_four_steps_ms"] / reuse["four_steps_ms"] - 1.0
    # ExpCast against exact softmax on sampled score rows of the first head:
    # codes from the kernels' ExpCast arithmetic (the library's code entry, the
    # reference max = the row max), decoded E4M3, renormalised; total
    # variation per row
    tv = None
    if w.vmode == "e4m3":
        s2 = (Qf[0, rows].double() @ Kf[0].double().T) * (1.4426950408889634 / 128 ** 0.5)
        m2 = s2.max(dim=1, keepdim=True).values
        s32 = s2.float().contiguous()
        codes = torch.empty(s32.shape, dtype=torch.uint8, device="cuda")
        vca.vca_expcast_codes(s32, torch.ones_like(s32), m2.float().expand_as(s32).contiguous(), codes)
        ph = codes.view(torch.float8_e4m3fn).double()
        ph = ph / ph.sum(dim=1, keepdim=True)
        pe = torch.softmax(s2 * 0.6931471805599453, dim=1)
        per_row = 0.5 * (ph - pe).abs().sum(dim=1)
        tv = {"mean": float(per_row.mean()), "max": float(per_row.max()), "rows": int(per_row.numel())}
    peak, _ = attention_peak(w.vmode, peaks)
    hbm = (peaks or {}).get("hbm_gbs", 6800.0)
    gb, pb = group_bytes(w), prep_bytes(w)
    return {
        "config": w.name, "B": w.B, "H": w.H, "N": w.N, "vmode": w.vmode, "expcast": w.expcast, "k": w.k,
        "iters": w.iters,
        "attention_ms": ms["attention"], "attention_tflops": w.flops / ms["attention"] / 1e9,
        "attention_frac": w.flops / ms["attention"] / 1e9 / peak, "attention_peak_tflops": peak,
        "attention_frac_of_nominal": w.flops / ms["attention"] / 1e9 / attention_nominal(w.vmode),
        "group_ms": ms["group"], "group_gbs": gb / ms["group"] / 1e6, "group_frac": gb / ms["group"] / 1e6 / hbm,
        "prep_ms": ms["prep"], "prep_gbs": pb / ms["prep"] / 1e6, "prep_frac": pb / ms["prep"] / 1e6 / hbm,
        "hbm_peak_gbs": hbm, "rel_l2_vs_exact_attention": max(errs), "error_rows": "32 sampled rows x 2 heads",
        "energy_removed_by_block_means": {k: statistics.mean(v) for k, v in removed.items()},
        "perm_reuse_4_steps": reuse, "expcast_tv_vs_softmax": tv,
        "qk_hadamard": {"prep_ms": prep_h_ms, "rel_l2_vs_exact_attention": max(errs_h)},
    }


def run_table(args):
    import torch
    from bit_attention_video_smooth_gb300 import inputs as I
    torch.cuda.set_device(0)
    peaks = load_peaks()
    cfgs = [I.WORKLOADS["tiny"], I.WORKLOADS["wan"], I.WORKLOADS["wan_exp"], I.WORKLOADS["nvfp4"]]
    cfgs += [I.with_n(I.WORKLOADS["sweep"], n) for n in (4096, 16384, 32768, 70656, 131072)]
    for w in cfgs:
        print(json.dumps(table_line(w, peaks)), flush=True)
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.table:
        run_table(args)
        return
    from bit_attention_video_smooth_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    if args.N:
        w = I.with_n(w, args.N)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
    else:
        run_ours(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
