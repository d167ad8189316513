#!/usr/bin/env python3
"""Benchmark of the nanochat attention block on one B300 per rank.  Prints one JSON line (rank 0).

A step is one pass of the prefill forward over the long-context workload, the largest of the prefill workloads:
two nc_attn_fwd calls (windows 1024 and 8192 = full causal) on B=2, T=8192, Hq=12, Hkv=4, D=128, each call with its
own seeded q, k, v (seed = call index), all resident in HBM.  L2 is flushed (512 MiB write) before every timed step,
outside the timed events.  Each call runs the RoPE + QK-norm prologue kernel and the tcgen05 attention kernel.

value      in-band TFLOP/s of the whole job: 4 * D * N_vis(T, W) * B * Hq FLOPs per call, summed over the calls of
           all ranks, divided by the device time of the slowest rank (CUDA events, max over ranks).
roofline   the attention kernel (tensor-core bound) on the same workload: in-band FLOPs of its launches / their
           CUDA-event durations, against the measured bf16 dense peak.
prefill    one section per prefill workload (tiny, depth-12 SSSL, GQA, long-context): the step's in-band TFLOP/s, the
           attention kernel's own TFLOP/s and time per launch for each window, and the prologue's time and GB/s.
decode     the KV-cache decode step (64 sequences, cache lengths U[1, 4096], Hq=12, Hkv=4, W=2048), GB/s of the
           algorithmic bytes (K/V rows in the window, q, out, lengths, new rows) against the measured HBM peak;
           four cache copies are rotated so that every call reads HBM.
e2e        the same prefill metric through the public API with the inputs in pinned host memory: host-to-device
           copies of q, k, v and the device-to-host copy of every output inside the timed region.
cpu_baseline  the fp64 oracle on this machine's host cores on a bounded sample of the same workload.

--impl reference times the oracle instead (the reference arm): each step is a bounded sample of the workload.
With torchrun (WORLD_SIZE > 1) every rank runs an independent replica on its own GPU (weak scaling, no data-path
collective); rank 0 prints.
"""

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from seeded_inputs import (CHUNK, DECODE, DEPTH12, GQA, LONG, TINY, bwd_inputs, chunk_inputs,  # noqa: E402
                           decode_inputs, fwd_inputs)

METRIC = "attention fwd TFLOP/s (in-band) & % bf16 peak; decode GB/s & % HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# An earlier measurement of the same B300s (copy bandwidth, cuBLAS bf16 burst / sustained), kept for runs where the
# per-box MEASURED_PEAKS.json is absent.
RECORDED_PEAKS = {"hbm_gbs": 6514.2, "bf16_tflops": 1786.4, "bf16_tflops_sustained": 1387.5}


# ---------------------------------------------------------------------------------------------------------- counts
def n_vis(T, W):
    """Visible (query, key) pairs of one (batch, head): sum over i of min(i, W) + 1 (all i + 1 when unbounded)."""
    if W < 0 or W >= T - 1:
        return T * (T + 1) // 2
    return (W + 1) * (W + 2) // 2 + (T - 1 - W) * (W + 1)


def fwd_flops(B, T, Hq, D, W):
    """In-band FLOPs of one forward call: QK^T and PV, 2 * D each, over the visible pairs."""
    return 4 * D * n_vis(T, W) * B * Hq


def chunk_flops(B, Tq, p0, Hq, D, W):
    """In-band FLOPs of a chunk of Tq queries at positions p0 .. p0+Tq-1: 4 D per visible (query, key) pair."""
    a = np.arange(p0, p0 + Tq, dtype=np.int64)
    vis = a + 1 if W < 0 else np.minimum(a, W) + 1
    return 4 * D * int(vis.sum()) * B * Hq


def decode_bytes(lens, window, B, Hq, Hkv, D, with_new):
    """Algorithmic HBM bytes of one decode call: the K and V rows in each window, q, out, the lengths, and (with a new
    key) the new rows read and written into the cache."""
    rows = 0
    for p in lens:
        L = p + (1 if with_new else 0)
        lo = 0 if window < 0 else max(0, p - window)
        rows += max(0, min(L, p) - lo)          # rows read from the cache (the new row comes from k_new / v_new)
    b = rows * Hkv * D * 2 * 2
    b += 2 * B * Hq * D * 2 + 4 * B
    if with_new:
        b += 2 * (B * Hkv * D * 2) * 2          # read k_new, v_new; write both into the cache
    return b


# --------------------------------------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(RECORDED_PEAKS), "measured earlier on this GPU model (no per-box file)"


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class ClockSampler:
    """Samples SM clock, power and clock-event reasons of the GPU with `nvidia-smi -lms` while the timed region runs.

    Only samples whose nvidia-smi timestamp falls inside [t_begin, t_end] of the timed region are kept (host clock).
    """

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    FLAGS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index, interval_ms=20):
        self.proc = None
        self.lines = []
        self.interval_ms = interval_ms
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.target = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        except Exception:
            self.target = str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._read, daemon=True)
            self._thread.start()
            time.sleep(0.3)  # let the first samples arrive before the timed region starts
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, t_begin, t_end):
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": "nvidia-smi unavailable"}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._thread.join(timeout=5)
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), f[3], f[5:]))
            except ValueError:
                continue
        inside = [r for r in rows if t_begin - 0.03 <= r[0] <= t_end + 0.03]
        if not inside and rows:  # timed region shorter than the sampling interval: nearest sample
            inside = [min(rows, key=lambda r: abs(r[0] - 0.5 * (t_begin + t_end)))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": "no samples"}
        reasons = sorted({name for r in inside for name, v in zip(self.FLAGS, r[4]) if v.lower() == "active"})
        power = [float(r[3]) for r in inside if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": float(statistics.median(r[1] for r in inside)), "sm_max_mhz": inside[0][2],
                "reasons": reasons, "samples": len(inside), "power_w_max": max(power) if power else None,
                "timed_region_s": round(t_end - t_begin, 4), "source": f"nvidia-smi -lms {self.interval_ms}"}


def kernel_traffic(kernel, src_files):
    """DRAM bytes per launch from a committed ncu summary, when it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)[kernel]
    except Exception:
        return None
    if d.get("source_sha256") != source_digest(src_files):
        return None
    return d.get("bytes_per_launch")


def source_digest(src_files):
    """sha256 of the sources with comments and blank lines removed: edits to comments keep a capture valid, any
    change to the code invalidates it."""
    h = hashlib.sha256()
    for f in src_files:
        with open(os.path.join(ROOT, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


# -------------------------------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=ws)
    return ws, rank, local


def dist_max(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------------------- CPU (oracle)
def prologue_bytes(B, T, Hq, Hkv, D, out_bytes=2):
    """Algorithmic HBM bytes of the RoPE + QK-norm prologue: read q and k (bf16), write qn and kn (bf16, or e4m3 with
    out_bytes=1)."""
    return (2 + out_bytes) * B * T * (Hq + Hkv) * D


def oracle_fwd_sample(wl, W, batches, groups=None):
    """Times the fp64 oracle on the first `batches` batch rows (and the first `groups` kv-head groups, all when
    None) of one call of workload `wl` with window W.  Returns (in-band FLOPs, seconds)."""
    from oracle import ref
    G = wl.Hq // wl.Hkv
    ng = wl.Hkv if groups is None else groups
    q, k, v = fwd_inputs(wl.B, wl.T, wl.Hq, wl.Hkv, wl.D, seed=0)
    q, k, v = (x[:batches].double().numpy() for x in (q[:, :, :ng * G], k[:, :, :ng], v[:, :, :ng]))
    t0 = time.perf_counter()
    ref.attn_fwd(q, k, v, W)
    dt = time.perf_counter() - t0
    return fwd_flops(batches, wl.T, ng * G, wl.D, W), dt


def cpu_baseline():
    """The oracle on one whole long-context step: the W=1024 and the W=8192 call on both batch rows (about 509
    in-band GFLOP, some 10 s of host time)."""
    f1, t1 = oracle_fwd_sample(LONG, 1024, LONG.B)
    f2, t2 = oracle_fwd_sample(LONG, 8192, LONG.B)
    flops, dt = f1 + f2, t1 + t2
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"one long-context step (B=2, T=8192, Hq=12, Hkv=4): the W=1024 and W=8192 calls on both batch "
                      f"rows, numpy fp64, {flops / 1e9:.1f} in-band GFLOP in {dt:.1f} s on {cpu_model()} "
                      f"({os.cpu_count()} logical cores)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    flops_w, secs = [], []
    for it in range(args.warmup + args.steps):
        f, dt = oracle_fwd_sample(LONG, 1024, 1, groups=1)
        if it >= args.warmup:
            flops_w.append(f)
            secs.append(dt)
    value = sum(flops_w) / sum(secs) / 1e12
    cores = cpu_threads()
    sample = ("per step: batch row 0, kv-head group 0 (3 query heads) of the W=1024 call of the long-context "
              f"workload, numpy fp64, {cpu_model()}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": LONG_WORKLOAD, "reference_step": sample + " (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


ALL_SECTIONS = "e2e,prefill,fp8,decode,chunk,backward,cpu"

LONG_WORKLOAD = (f"{LONG.name}: B={LONG.B} T={LONG.T} Hq={LONG.Hq} Hkv={LONG.Hkv} D={LONG.D}, one step = calls with "
                 f"windows {list(LONG.windows)} (sliding window and full causal), distinct seeded q,k,v per call")


# ---------------------------------------------------------------------------------------------------- GPU arm
def prefill_section(nc, wl, dev, flush, n_steps, n_warmup=3, seeds=None, fp8=False):
    """Times one prefill workload: a step is one call per window of `wl` (call i on inputs of seed i, or seeds[i]).

    Returns (section dict, per-step event times in ms, layer tensors, workspace).  The step time comes from CUDA-graph
    replays of the whole step (the programmatic launch of each attention kernel overlaps its prologue's tail), each
    after an L2 flush outside the events.  Kernel times come from eager steps with CUDA events recorded around each
    kernel; a GPU sleep before each eager step lets the host queue the whole step first, so that no launch waits for
    the host inside the events.
    """
    stream = torch.cuda.current_stream()
    layers = []
    for li, W in enumerate(wl.windows):
        q, k, v = (t.to(dev) for t in fwd_inputs(wl.B, wl.T, wl.Hq, wl.Hkv, wl.D, seed=li if seeds is None else seeds[li]))
        layers.append((q, k, v, torch.empty_like(q), W))
    flops_layer = [fwd_flops(wl.B, wl.T, wl.Hq, wl.D, W) for W in wl.windows]
    flops_step = sum(flops_layer)
    ws_bytes = (nc.nc_attn_fwd_fp8_workspace_bytes if fp8 else nc.nc_attn_fwd_workspace_bytes)(
        wl.B, wl.T, wl.Hq, wl.Hkv, wl.D)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fwd = nc.nc_attn_fwd_fp8 if fp8 else nc.nc_attn_fwd

    def step(evs=None):
        for li, (q, k, v, o, W) in enumerate(layers):
            fwd(q, k, v, o, window=W, workspace=wsp, events=evs[li] if evs else None)

    for _ in range(max(3, n_warmup)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    for _ in range(max(3, n_warmup)):
        flush.fill_(1)
        g_step.replay()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(mk(), mk()) for _ in range(n_steps)]
    for s_ in range(n_steps):
        flush.fill_(s_ & 0xFF)
        step_ev[s_][0].record(stream)
        g_step.replay()
        step_ev[s_][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]

    # kernel times: events around each kernel in eager steps
    n_k = max(3, min(n_steps, 30))
    k_ev = [[(mk(), mk(), mk()) for _ in layers] for _ in range(n_k)]
    for s_ in range(n_k):
        flush.fill_(s_ & 0xFF)
        torch.cuda._sleep(2_000_000)            # ~1 ms at 2 GHz: the host queues the step meanwhile
        step(k_ev[s_])
    torch.cuda.synchronize()
    per_w = {}
    k2_tot_ms = 0.0
    k1_tot_ms = 0.0
    for li, (q, k, v, o, W) in enumerate(layers):
        k2 = [row[li][1].elapsed_time(row[li][2]) for row in k_ev]
        k1 = [row[li][0].elapsed_time(row[li][1]) for row in k_ev]
        k2_tot_ms += sum(k2)
        k1_tot_ms += sum(k1)
        us = 1e3 * statistics.mean(k2)
        key = str(W) if str(W) not in per_w else f"{W}#{li}"
        per_w[key] = {"attn_us_per_launch": us, "attn_tflops": flops_layer[li] / (us * 1e-6) / 1e12,
                      "prologue_us_per_launch": 1e3 * statistics.mean(k1)}
    pro_bytes = prologue_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.D, out_bytes=1 if fp8 else 2)
    pro_us = 1e3 * k1_tot_ms / (n_k * len(layers))
    attn_achieved = n_k * flops_step / (k2_tot_ms * 1e-3) / 1e12
    sec = {
        "workload": f"{wl.name}: B={wl.B} T={wl.T} Hq={wl.Hq} Hkv={wl.Hkv} D={wl.D}, windows {list(wl.windows)}",
        "flops_per_step": flops_step,
        "us_per_step": 1e3 * statistics.mean(step_ms),
        "tflops": n_steps * flops_step / (sum(step_ms) * 1e-3) / 1e12,
        "attn_tflops": attn_achieved,
        "attn_us_per_launch": 1e3 * k2_tot_ms / (n_k * len(layers)),
        "prologue_us_per_launch": pro_us,
        "prologue_gbs": pro_bytes / (pro_us * 1e-6) / 1e9,
        "prologue_bytes_per_launch": pro_bytes,
        "windows": per_w,
        "steps_timed": n_steps, "kernel_steps_timed": n_k,
    }
    return sec, step_ms, layers, wsp


def run_ours(args, ws, rank, local):
    from transformer_attention_06_b300 import nc_attn as nc

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def add_fracs(sec):
        sec["frac"] = sec["tflops"] / peaks["bf16_tflops"]
        sec["attn_frac"] = sec["attn_tflops"] / peaks["bf16_tflops"]
        sec["attn_frac_of_sustained"] = sec["attn_tflops"] / peaks["bf16_tflops_sustained"]
        sec["prologue_frac_of_hbm"] = sec["prologue_gbs"] / peaks["hbm_gbs"]
        for d in sec["windows"].values():
            d["attn_frac"] = d["attn_tflops"] / peaks["bf16_tflops"]
        return sec

    sections = set(args.sections.split(","))

    # ---- headline: the long-context step (another workload or the fp8 path only for profiling runs), with clocks
    # sampled during its timed region
    w = {"long": LONG, "depth12": DEPTH12, "gqa": GQA, "tiny": TINY}[args.workload]
    clocks = ClockSampler(local)
    clocks.start()
    dist_barrier(ws)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    head, step_ms, layers, wsp = prefill_section(nc, w, dev, flush, args.steps, args.warmup, fp8=args.fp8)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    clk = clocks.stop(t_wall0, t_wall1)
    dist_barrier(ws)
    add_fracs(head)
    flops_step = head["flops_per_step"]
    total_ms_max = dist_max(sum(step_ms), ws)
    value = ws * args.steps * flops_step / (total_ms_max * 1e-3) / 1e12
    traffic = kernel_traffic("attn_fwd_kernel", ["transformer_attention_06_b300/csrc/attn_fwd.cuh",
                                                 "transformer_attention_06_b300/csrc/common.cuh"])

    # ---- end to end through the public API with host buffers.  Every step copies its q, k, v from pinned host memory
    # and its outputs back, as a caller streaming batches would: copies in, compute and copies out run on three
    # streams, with two sets of device buffers so that a step's inputs arrive while the previous step computes and its
    # outputs leave while the next one starts (the link carries both directions at once).
    e2e = None
    if "e2e" in sections:
        host = [(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(), torch.empty_like(o, device="cpu").pin_memory())
                for (q, k, v, o, W) in layers]
        h2d = sum(x.numel() * x.element_size() for (q, k, v, _) in host for x in (q, k, v))
        d2h = sum(o.numel() * o.element_size() for (_, _, _, o) in host)
        dev_sets = [[(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o), W)
                     for (q, k, v, o, W) in layers] for _ in range(2)]
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        # enough steps that the pipeline's fill (the first inputs) and drain (the last outputs) are a small share
        n_e2e = min(max(20, args.steps), 40)
        n_warm = 2
        ev = lambda: torch.cuda.Event()  # noqa: E731
        h2d_done = [[ev() for _ in layers] for _ in range(2)]
        cmp_done = [[ev() for _ in layers] for _ in range(2)]
        d2h_done = [[ev() for _ in layers] for _ in range(2)]
        used = [[False] * len(layers) for _ in range(2)]
        torch.cuda.synchronize()
        t_begin, t_end = mk(), mk()
        for it in range(n_warm + n_e2e):
            if it == n_warm:
                torch.cuda.synchronize()
                t_begin.record(s_in)
            st = it % 2
            for li, ((hq, hk, hv, ho), (q, k, v, o, W)) in enumerate(zip(host, dev_sets[st])):
                with torch.cuda.stream(s_in):
                    if used[st][li]:
                        s_in.wait_event(cmp_done[st][li])      # the step before last has read these inputs
                    q.copy_(hq, non_blocking=True)
                    k.copy_(hk, non_blocking=True)
                    v.copy_(hv, non_blocking=True)
                    h2d_done[st][li].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(h2d_done[st][li])
                    if used[st][li]:
                        s_cmp.wait_event(d2h_done[st][li])     # its outputs have left
                    nc.nc_attn_fwd(q, k, v, o, window=W, workspace=wsp, stream=s_cmp)
                    cmp_done[st][li].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(cmp_done[st][li])
                    ho.copy_(o, non_blocking=True)
                    d2h_done[st][li].record(s_out)
                used[st][li] = True
        t_end.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = dist_max(t_begin.elapsed_time(t_end), ws)
        e2e = {"value": ws * n_e2e * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": e2e_ms / n_e2e,
               "timing": "copies in, compute and copies out on three streams, two device buffer sets; events from the "
                         "first timed copy-in to the last copy-out"}
        del host, dev_sets
    del layers, wsp
    torch.cuda.empty_cache()

    # ---- the other prefill workloads, one section each (the long-context section is the headline's)
    prefill = {LONG.name: head}
    if "prefill" in sections:
        for wl in (TINY, DEPTH12, GQA):
            sec, _, lay, wsp_ = prefill_section(nc, wl, dev, flush, 20)
            prefill[wl.name] = add_fracs(sec)
            del lay, wsp_
            torch.cuda.empty_cache()

    # ---- the prefill with e4m3 score operands: half of the in-band FLOPs (Q K^T) on the 8-bit tensor path at twice the
    # bf16 rate, the other half (P V) in bf16, so its peak is 4/3 of the bf16 peak
    prefill_fp8 = None
    if "fp8" in sections:
        prefill_fp8 = {}
        peak8 = peaks["bf16_tflops"] * 4.0 / 3.0
        for wl in (LONG, GQA, DEPTH12):
            sec, _, lay, wsp_ = prefill_section(nc, wl, dev, flush, 20, fp8=True)
            for d in [sec] + list(sec["windows"].values()):
                d["attn_frac"] = d["attn_tflops"] / peak8
            sec["frac"] = sec["tflops"] / peak8
            sec["prologue_frac_of_hbm"] = sec["prologue_gbs"] / peaks["hbm_gbs"]
            prefill_fp8[wl.name] = sec
            del lay, wsp_
            torch.cuda.empty_cache()
        prefill_fp8["peak_tflops"] = peak8
        prefill_fp8["peak_def"] = ("QK^T (half the in-band FLOPs) on e4m3 at 2x the bf16 rate, P V in bf16: 4/3 of the "
                                   "measured bf16 dense peak (the nominal fp8 : bf16 ratio is 2)")

    # ---- decode
    dec = None
    if "decode" in sections:
        dec = {}
        dw = DECODE
        for with_new in (False, True):
            d = decode_inputs(dw.B, dw.Hq, dw.Hkv, dw.D, dw.Tcap, dw.len_lo, dw.len_hi, seed=0, with_new=with_new)
            copies = [(d["kcache"].to(dev), d["vcache"].to(dev)) for _ in range(4)]
            qd, lens = d["q"].to(dev), d["cache_lens"].to(dev)
            kn = d["k_new"].to(dev) if with_new else None
            vn = d["v_new"].to(dev) if with_new else None
            out = torch.empty_like(qd)
            dws = torch.zeros(nc.nc_attn_decode_workspace_bytes(dw.B, dw.Hq, dw.Hkv, dw.D, dw.Tcap, dw.window),
                              dtype=torch.uint8, device=dev)
            nbytes = decode_bytes(d["cache_lens"].tolist(), dw.window, dw.B, dw.Hq, dw.Hkv, dw.D, with_new)
            n_dec = 40
            for i in range(max(3, args.warmup)):
                kc, vc = copies[i % 4]
                nc.nc_attn_decode(qd, kc, vc, lens, out, kn, vn, window=dw.window, workspace=dws)
            torch.cuda.synchronize()
            # 40 calls over the 4 rotated cache copies, captured once and replayed: device time per call without
            # host launch gaps (one call is far shorter than the host side of a launch).
            g_dec = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_dec):
                for i in range(n_dec):
                    kc, vc = copies[i % 4]
                    nc.nc_attn_decode(qd, kc, vc, lens, out, kn, vn, window=dw.window, workspace=dws)
            g_dec.replay()
            torch.cuda.synchronize()
            a, b = mk(), mk()
            reps = 3
            a.record(stream)
            for _ in range(reps):
                g_dec.replay()
            b.record(stream)
            torch.cuda.synchronize()
            n_dec *= reps
            us = dist_max(a.elapsed_time(b) * 1e3 / n_dec, ws)
            gbs = nbytes / (us * 1e-6) / 1e9
            dec["with_new" if with_new else "cache_only"] = {
                "value": gbs, "unit": "GB/s", "us_per_call": us, "bytes_per_call": nbytes,
                "frac": gbs / peaks["hbm_gbs"], "calls": n_dec}
            del copies
            torch.cuda.empty_cache()
        dec["config"] = (f"{dw.name}: B={dw.B} Hq={dw.Hq} Hkv={dw.Hkv} D={dw.D} Tcap={dw.Tcap} window={dw.window}, "
                         f"cache lengths U[{dw.len_lo},{dw.len_hi}] seed 0; 4 rotated cache copies (> L2); "
                         f"calls replayed from a CUDA graph")
        dec["peak_gbs"] = peaks["hbm_gbs"]

    # ---- chunked prefill against a KV cache
    chk = None
    if "chunk" in sections:
        cw = CHUNK
        d = chunk_inputs(cw.B, cw.Tq, cw.Hq, cw.Hkv, cw.D, cw.Tcap, seed=0)
        kc, vc = d["kcache"].to(dev), d["vcache"].to(dev)
        qd, kd, vd = d["q"].to(dev), d["k_new"].to(dev), d["v_new"].to(dev)
        lens = torch.full((cw.B,), cw.p0, dtype=torch.int32, device=dev)
        out = torch.empty_like(qd)
        cws = torch.empty(nc.nc_attn_prefill_chunk_workspace_bytes(cw.B, cw.Tq, cw.Hq, cw.Hkv, cw.D),
                          dtype=torch.uint8, device=dev)
        per_w = {}
        tot_flops = tot_us = 0.0
        for W in cw.windows:
            call = lambda: nc.nc_attn_prefill_chunk(qd, kd, vd, kc, vc, lens, out, window=W,  # noqa: E731
                                                    workspace=cws)
            for _ in range(max(3, args.warmup)):
                call()
            torch.cuda.synchronize()
            g_chk = torch.cuda.CUDAGraph()      # one call (two kernels); each call rewrites the same cache rows
            with torch.cuda.graph(g_chk):
                call()
            n_chk = 20
            evs = [(mk(), mk()) for _ in range(n_chk)]
            for i in range(n_chk):
                flush.fill_(i & 0xFF)
                evs[i][0].record(stream)
                g_chk.replay()
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            us = dist_max(sum(a.elapsed_time(b) for a, b in evs) * 1e3 / n_chk, ws)
            fl = chunk_flops(cw.B, cw.Tq, cw.p0, cw.Hq, cw.D, W)
            per_w[str(W)] = {"us_per_call": us, "tflops": fl / (us * 1e-6) / 1e12, "flops_per_call": fl}
            tot_flops += fl
            tot_us += us
        val = tot_flops / (tot_us * 1e-6) / 1e12
        chk = {"value": val, "unit": "TFLOP/s", "frac": val / peaks["bf16_tflops"], "windows": per_w,
               "config": (f"{cw.name}: B={cw.B} Tq={cw.Tq} appended at cache length {cw.p0}, Tcap={cw.Tcap}, "
                          f"Hq={cw.Hq} Hkv={cw.Hkv} D={cw.D}, windows {list(cw.windows)}; in-band FLOPs; each call "
                          f"replayed from a CUDA graph after a 512 MiB L2 flush outside the events")}
        del kc, vc

    # ---- backward pass (tcgen05 kernels) on the depth-12 layer shapes
    bwd = None
    if "backward" in sections:
        w = DEPTH12
        bq, bk, bv, bdo = (t.to(dev) for t in bwd_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, seed=0))
        bws = torch.empty(int(nc.lib.nc_attn_bwd_workspace_bytes(w.B, w.T, w.Hq, w.Hkv, w.D)), dtype=torch.uint8,
                          device=dev)
        per_w, tot_f, tot_us = {}, 0.0, 0.0
        for W in sorted(set(w.windows)):
            nc.nc_attn_bwd(bq, bk, bv, bdo, window=W, workspace=bws)
            torch.cuda.synchronize()
            n_b = 10
            evs = [(mk(), mk()) for _ in range(n_b)]
            for i in range(n_b):
                flush.fill_(i)
                evs[i][0].record(stream)
                nc.nc_attn_bwd(bq, bk, bv, bdo, window=W, workspace=bws)
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            us = dist_max(sum(a.elapsed_time(b) for a, b in evs) * 1e3 / n_b, ws)
            fl = 3.5 * fwd_flops(w.B, w.T, w.Hq, w.D, W)
            per_w[str(W)] = {"us_per_call": us, "tflops": fl / (us * 1e-6) / 1e12}
            tot_f += fl
            tot_us += us
        val = tot_f / (tot_us * 1e-6) / 1e12
        # the training path: the forward keeps its output and row statistics, the backward reuses them
        saved, s_f, s_us = {}, 0.0, 0.0
        for W in sorted(set(w.windows)):
            bo, blse = nc.nc_attn_fwd_lse(bq, bk, bv, window=W)
            nc.nc_attn_bwd_saved(bq, bk, bv, bo, bdo, blse, window=W, workspace=bws)
            torch.cuda.synchronize()
            n_b = 10
            evs = [(mk(), mk()) for _ in range(n_b)]
            for i in range(n_b):
                flush.fill_(i)
                evs[i][0].record(stream)
                nc.nc_attn_bwd_saved(bq, bk, bv, bo, bdo, blse, window=W, workspace=bws)
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            us = dist_max(sum(a.elapsed_time(b) for a, b in evs) * 1e3 / n_b, ws)
            fl = 2.5 * fwd_flops(w.B, w.T, w.Hq, w.D, W)
            saved[str(W)] = {"us_per_call": us, "tflops": fl / (us * 1e-6) / 1e12}
            s_f += fl
            s_us += us
            del bo, blse
        bwd = {"value": val, "unit": "TFLOP/s", "frac": val / peaks["bf16_tflops"], "windows": per_w,
               "config": (f"{w.name} layer shapes, windows {sorted(set(w.windows))}; one nc_attn_bwd_ws call: the forward "
                          f"recomputed for its row statistics, then dK/dV and dQ on tcgen05 and the norm/RoPE backward; "
                          f"dq, dk, dv in fp32; FLOPs counted as 3.5x the forward's in-band FLOPs (2 products of the "
                          f"forward, 5 of the backward); L2 flushed before each call"),
               "saved_statistics": {
                   "value": s_f / (s_us * 1e-6) / 1e12, "unit": "TFLOP/s",
                   "frac": s_f / (s_us * 1e-6) / 1e12 / peaks["bf16_tflops"], "windows": saved,
                   "config": ("one nc_attn_bwd_saved_ws call on the output and log-sum-exp kept by nc_attn_fwd_lse "
                              "(no forward recomputation; rowsum(dO O) from the kept output); FLOPs counted as 2.5x "
                              "the forward's in-band FLOPs (the backward's 5 products); L2 flushed before each call")}}
        del bq, bk, bv, bdo, bws

    st = nc.nc_attn_get_device_status(clear=True)
    cpu = None
    if rank == 0 and "cpu" in sections:
        cpu = cpu_baseline()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": LONG_WORKLOAD if w is LONG and not args.fp8 else
                       head["workload"] + (" (e4m3 scores)" if args.fp8 else "") + " [profiling run, not the headline]",
                       "l2": "512 MiB write before every timed step, outside the timed events",
                       "timing": "each step replayed from a CUDA graph of its four kernels; kernel times for the "
                                 "roofline from CUDA events around each kernel in eager steps",
                       "flops_per_step": flops_step, "parallelism": f"replicas x{ws}"},
            "frac_of_bf16_peak": value / ws / peaks["bf16_tflops"],
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel", "achieved": head["attn_tflops"],
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": head["attn_frac"],
                         "frac_of_sustained": head["attn_frac_of_sustained"],
                         "traffic": traffic, "peak_source": f"{peak_src} bf16 dense (burst)",
                         "achieved_def": "sum of in-band FLOPs of the attention-kernel launches / sum of their "
                                         "CUDA-event durations, on the long-context step",
                         "us_per_launch": head["attn_us_per_launch"],
                         "launches_timed": head["kernel_steps_timed"] * len(LONG.windows),
                         "prologue": {"bound": "hbm", "us_per_launch": head["prologue_us_per_launch"],
                                      "achieved_gbs": head["prologue_gbs"], "peak_gbs": peaks["hbm_gbs"],
                                      "frac": head["prologue_frac_of_hbm"]}},
            "prefill": prefill,
            "prefill_fp8": prefill_fp8,
            "decode": dec,
            "prefill_chunk": chk,
            "backward": bwd,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": args.steps * len(LONG.windows) * 2,
            "clocks": clk,
            "device_status": nc.status_string(st),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["long", "depth12", "gqa", "tiny"], default="long",
                    help="workload of the headline step (long-context unless a profiling run asks for another)")
    ap.add_argument("--fp8", action="store_true", help="headline step on the e4m3 path (profiling runs)")
    ap.add_argument("--sections", default=ALL_SECTIONS,
                    help="comma-separated sections timed after the headline step (default: all of " + ALL_SECTIONS + ")")
    args = ap.parse_args()
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
