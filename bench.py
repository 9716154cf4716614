"""Benchmark: sliding-window (+ sinks) attention on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl swa|reference]

One step is one bf16 prefill of the Mistral-like layer (B=1, H=32, Hkv=8,
d=128, n=16384, w=4096, g=0) -- the headline workload, reported as useful
TFLOP/s (4 * connections * d * B * H floating-point operations; masked or
padded tile work is not counted).  The decode half of the metric is measured
in the same run on the streaming-decode workload (B=32, H=32, Hkv=8, d=128,
w=4096, g=4, pos=100000): one cache append plus one decode per step, reported
as HBM GB/s over the algorithmic bytes (each cached K/V row read once).  The
other three configurations of the method are timed in the same run and
reported under "configs", each with its own roofline, clocks and CPU-oracle
baseline: the Gemma-3-like local layer (B=2, H=32, Hkv=16, n=32768, w=1024),
the long-context layer with sinks (B=1, H=32, Hkv=8, n=131072, w=4096, g=4)
and the tiny fp32 case (n=512, w=64, d=64, the CUDA-core fp32 kernel).

Timing: W warm-up steps, then K timed steps; L2 is flushed (a 256 MiB write,
then a 256 MiB read, so the flush's dirty lines are written back before the
timed region) before every timed launch and each launch is bracketed by CUDA events on the
launching stream.  Under torchrun every rank runs its own replica (weak
scaling); rank 0 prints one JSON line with the max time over ranks.

--impl reference times the CPU oracle (the only other implementation of this
method here) on a bounded sample of query rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

PREFILL_WORKLOADS = {
    "mistral_like_prefill": dict(B=1, H=32, Hkv=8, n=16384, d=128, w=4096, g=0, sink_scale=1.0),
    "gemma3_local_prefill": dict(B=2, H=32, Hkv=16, n=32768, d=128, w=1024, g=0, sink_scale=1.0),
    "long_sink_prefill": dict(B=1, H=32, Hkv=8, n=131072, d=128, w=4096, g=4, sink_scale=4.0),
    # the full-causal global layer of the Gemma-3 hybrid (w >= n)
    "gemma3_global_prefill": dict(B=2, H=32, Hkv=16, n=32768, d=128, w=32768, g=0,
                                  sink_scale=1.0),
    # plain multi-head attention (odd group: q-tile pairs in the pair kernel)
    "mha_prefill": dict(B=1, H=32, Hkv=32, n=16384, d=128, w=4096, g=0, sink_scale=1.0),
    # other fixed patterns (swa_prefill_pattern)
    "dilated_prefill": dict(B=1, H=32, Hkv=8, n=16384, d=128, w=1024, g=0, sink_scale=1.0,
                            pattern="dilated", r=4),
    "strided_prefill": dict(B=1, H=32, Hkv=8, n=65536, d=128, w=0, g=0, sink_scale=1.0,
                            pattern="strided", r=256),
    "landmark_prefill": dict(B=1, H=32, Hkv=8, n=16384, d=128, w=4096, g=4, sink_scale=4.0,
                             pattern="landmark", r=64),
}
PREFILL = PREFILL_WORKLOADS["mistral_like_prefill"]
# a prompt chunk of T tokens at position pos0 against a full rolling cache
CHUNK = dict(B=4, H=32, Hkv=8, d=128, w=4096, g=4, T=4096, pos0=100000, sink_scale=4.0)
DECODE = dict(B=32, H=32, Hkv=8, d=128, w=4096, g=4, pos=100000, sink_scale=4.0)
METRIC = "SWA prefill useful TFLOP/s (% bf16 peak); decode HBM GB/s (% peak)"
PREFILL_KERNEL_SRC = os.path.join(ROOT, "sink_sparse_attention_swa_b300", "csrc", "swa_prefill_tc.cu")
DECODE_KERNEL_SRC = os.path.join(ROOT, "sink_sparse_attention_swa_b300", "csrc", "swa_decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def pairs(n, w, g):
    """Connections of one head (window w including the current position, plus g sinks)."""
    total = n * (n + 1) // 2 if n <= w else w * (w + 1) // 2 + (n - w) * w
    m = n - w
    if m > 0:
        total += m * (m + 1) // 2 if m <= g else g * (g + 1) // 2 + (m - g) * g
    return total


def row_keys(i, c):
    """Keys query position i reads under workload c's pattern (i: int or array).
    window: the band and the sinks; dilated: i, i-r, ..., i-(w-1)r; strided:
    every (i-j) mod r == 0; landmark: the band, the sinks and the positions
    j mod r == 0 before the band that are not sinks."""
    i = np.asarray(i, dtype=np.int64)
    w, g = c["w"], c["g"]
    pat, r = c.get("pattern", "window"), c.get("r", 1)
    if pat == "dilated":
        return np.minimum(w, i // r + 1)
    if pat == "strided":
        return i // r + 1
    keys = np.minimum(i + 1, w) + np.minimum(g, np.maximum(0, i - w + 1))
    if pat == "landmark":
        lm = np.where(i >= w, (i - w) // r - (g + r - 1) // r + 1, 0)
        keys = keys + np.maximum(0, lm)
    return keys


def prefill_flops(c):
    if c.get("pattern", "window") == "window":
        return 4 * pairs(c["n"], c["w"], c["g"]) * c["d"] * c["B"] * c["H"]
    return 4 * int(row_keys(np.arange(c["n"]), c).sum()) * c["d"] * c["B"] * c["H"]


def chunk_flops(c):
    """Useful FLOPs of a chunk: query position P reads min(P+1, w) window keys
    plus min(g, P+1-w) sinks once the window has moved past them."""
    keys = 0
    for P in range(c["pos0"], c["pos0"] + c["T"]):
        keys += min(P + 1, c["w"]) + (min(c["g"], P + 1 - c["w"]) if P + 1 > c["w"] else 0)
    return 4 * keys * c["d"] * c["B"] * c["H"]


def prefill_bytes(c, elem=2):
    """Algorithmic HBM bytes of one prefill launch: Q, K, V read once, O written once."""
    q = c["B"] * c["H"] * c["n"] * c["d"] * elem
    kv = c["B"] * c["Hkv"] * c["n"] * c["d"] * elem
    return 2 * q + 2 * kv


def prefill_roofline(c, flops, launch_ms, pk, traffic, kernel):
    """The roofline of one prefill launch: the tensor-core bound (useful FLOPs at
    the measured bf16 peak) or, where the pattern reads few keys per query (the
    strided head at s = sqrt(n)), the HBM bound (Q, K, V, O once at the measured
    copy bandwidth), whichever takes longer."""
    nbytes = prefill_bytes(c)
    tflops = flops / (launch_ms * 1e-3) / 1e12
    gbs = nbytes / (launch_ms * 1e-3) / 1e9
    t_tensor = flops / (pk["bf16"] * 1e12)
    t_hbm = nbytes / (pk["hbm"] * 1e9)
    common = {"traffic": traffic, "kernel": kernel, "useful_flops_per_launch": flops,
              "algorithmic_bytes": nbytes,
              "tensor_bound_ms": t_tensor * 1e3, "hbm_bound_ms": t_hbm * 1e3}
    if t_hbm > t_tensor:
        return {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
                "frac": gbs / pk["hbm"], "peak_source": pk["src"] + " copy",
                "tensor_tflops": tflops, "tensor_frac": tflops / pk["bf16"], **common}
    return {"bound": "tensor", "achieved": tflops, "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": tflops / pk["bf16"], "peak_source": pk["src"] + " burst",
            "frac_of_sustained": tflops / pk["bf16_sustained"], **common}


def decode_bytes(c, elem=2):
    kv = c["B"] * c["Hkv"] * (c["w"] + c["g"]) * c["d"] * elem * 2
    qo = c["B"] * c["H"] * c["d"] * elem * 2
    return kv + qo


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    src="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, src="fallback")


def src_hash(path):
    """First 16 hex digits of the SHA-256 of a source file's code, with comments
    and blank lines removed: editing a comment keeps a capture valid, any change
    to the code does not."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def recorded_traffic(kernel, workload, src):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel source
    is unchanged since (the line carries the source hash); else None."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    h = src_hash(src)
    for line in text.splitlines():
        m = re.match(r"\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*([0-9a-f]{16})\s*\|\s*([0-9.e+]+)\s*\|", line)
        if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == h:
            return float(m.group(4))
    return None


class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# --------------------------------------------------------------------------- CPU oracle
_CPU_INPUTS = {}


def cpu_oracle_sample(min_seconds=10.0, max_seconds=30.0, seed=0, c=None):
    """Times the fp64 oracle on sampled query rows of a prefill workload until
    at least `min_seconds` have passed.  Returns (TFLOP/s of useful work,
    rows, seconds, threads)."""
    import oracle
    from sink_sparse_attention_swa_b300 import synthetic

    oracle.set_num_threads(os.cpu_count() or 1)
    c = PREFILL if c is None else c
    key = (tuple(sorted(c.items())), seed)
    if key not in _CPU_INPUTS:
        x = synthetic.prefill_inputs(c["B"], c["H"], c["Hkv"], c["n"], c["d"], c["w"], c["g"],
                                     dtype=c.get("dtype", "bf16"), seed=seed,
                                     sink_scale=c["sink_scale"], device="cpu")
        _CPU_INPUTS[key] = (x, x.K.double().numpy(), x.V.double().numpy())
    x, K, V = _CPU_INPUTS[key]
    rows_all = synthetic.sample_rows(c["B"], c["H"], c["n"], min(1 << 20, c["B"] * c["H"] * c["n"]),
                                     seed=1).numpy()
    done, t_total, flops = 0, 0.0, 0
    batch = 64
    while t_total < min_seconds and done < rows_all.shape[0]:
        rows = rows_all[done:done + batch]
        qr = np.stack([x.Q[b, h, i].double().numpy() for b, h, i in rows])
        t0 = time.perf_counter()
        if c.get("pattern", "window") == "window":
            oracle.prefill_rows(qr, K, V, c["H"], c["w"], c["g"], x.scale, rows)
        else:
            oracle.prefill_pattern_rows(qr, K, V, c["H"], c["w"], c["g"], c["r"], c["pattern"],
                                        x.scale, rows)
        t_total += time.perf_counter() - t0
        flops += 4 * c["d"] * int(row_keys(rows[:, 2], c).sum())
        done += rows.shape[0]
        if t_total < min_seconds / 4:
            batch *= 2
        if t_total > max_seconds:
            break
    return flops / t_total / 1e12, done, t_total, oracle.num_threads()


# --------------------------------------------------------------------------- GPU legs
class L2Flush:
    """Evicts L2 before a timed launch and leaves it clean: a 256 MiB write
    (larger than the 126 MB L2), then a 256 MiB read of a second buffer, so the
    dirty lines of the write are written back before the timed region starts
    instead of during it."""

    def __init__(self, device):
        n = 64 * 1024 * 1024  # 256 MiB of fp32
        self.w = torch.zeros(n, dtype=torch.float32, device=device)
        self.r = torch.ones(n, dtype=torch.float32, device=device)
        self.out = torch.zeros((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.add_(1)
        torch.sum(self.r, dim=0, out=self.out)


def time_launches(fn, steps, warmup, flush, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        flush()  # evict L2 (clean) before each timed launch
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def pipelined_e2e(host_in, host_out_like, compute, steps, warmup, stream, dev):
    """End-to-end steps through the public API from pinned host buffers, two
    steps in flight: step k's inputs go host->device on one stream while step
    k-1 computes on `stream`, and each step's output comes back device->host on
    a third stream.  Every step copies all of its inputs in and its output back
    inside the timed region.  compute(dev_inputs, dev_out) launches one step on
    `stream`.  Returns ms per step (device clock over the whole run)."""
    nb = 2
    dev_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in]
              for _ in range(nb)]
    dev_out = [torch.empty(host_out_like.shape, dtype=host_out_like.dtype, device=dev)
               for _ in range(nb)]
    host_out = [torch.empty_like(host_out_like).pin_memory() for _ in range(nb)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_done = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]

    def run(n, after=None):
        for k in range(n):
            b = k % nb
            with torch.cuda.stream(s_in):
                if after is not None and k == 0:
                    s_in.wait_event(after)
                if k >= nb:
                    s_in.wait_event(ev_done[b])  # step k-2 has finished reading buffer b
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if k >= nb:
                stream.wait_event(ev_out[b])  # step k-2's output has been read back
            compute(dev_in[b], dev_out[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                host_out[b].copy_(dev_out[b], non_blocking=True)
                ev_out[b].record(s_out)
        return (n - 1) % nb

    run(warmup)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    last = run(steps, after=start)
    stream.wait_event(ev_out[last])
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


# the configurations reported under "configs" in the default line, besides
# the headline prefill (value) and the decode leg
CONFIG_LEGS = ["gemma3_local_prefill", "long_sink_prefill", "tiny_fp32_prefill"]
TINY = dict(B=1, H=1, Hkv=1, n=512, d=64, w=64, g=0, sink_scale=1.0, dtype="f32")


def config_leg(name, args, swa, synthetic, world, rank, local, dev, stream, flush, pk):
    """One more configuration of the default run: K timed launches (L2 flushed
    before each), its clocks, roofline and a CPU-oracle baseline on sampled
    rows (rank 0, single process)."""
    c = TINY if name == "tiny_fp32_prefill" else PREFILL_WORKLOADS[name]
    dtype = c.get("dtype", "bf16")
    x = synthetic.prefill_inputs(c["B"], c["H"], c["Hkv"], c["n"], c["d"], c["w"], c["g"],
                                 dtype=dtype, seed=rank, sink_scale=c["sink_scale"], device=dev)
    out = torch.empty_like(x.Q)
    fn = lambda: swa.prefill(x.Q, x.K, x.V, c["w"], c["g"], x.scale, out=out, stream=stream)
    flops = prefill_flops(c)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        times = time_launches(fn, args.steps, args.warmup, flush, stream)
    barrier(world)
    assert swa.device_status(stream) == 0, "device status reported an error"
    launch_ms = float(np.mean(times))
    ms = max_over_ranks(launch_ms, world, dev)
    del x, out
    torch.cuda.empty_cache()
    leg = {"workload": name, **{k: v for k, v in c.items() if k != "sink_scale"},
           "sink_scale": c["sink_scale"], "dtype": dtype, "steps": args.steps,
           "ms_per_launch": ms, "unit": "TFLOP/s",
           "value": flops * world / (ms * 1e-3) / 1e12, "useful_flops_per_launch": flops,
           "clocks": clk.summary(), "gpu_launches": args.steps}
    if dtype == "bf16":
        kernel = ("swa_prefill_bf16_pair_sm103" if (c["H"] // c["Hkv"]) % 2 == 0
                  else "swa_prefill_bf16_sm103")
        leg["roofline"] = prefill_roofline(c, flops, launch_ms, pk,
                                           recorded_traffic(kernel, name, PREFILL_KERNEL_SRC),
                                           kernel)
    else:
        leg["roofline"] = None
        leg["note"] = ("the fp32 CUDA-core path, kept for exactness (max-abs 1e-5 against the "
                       "oracle); a latency-bound correctness case, not measured against a roofline")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs = min(args.cpu_seconds, 4.0)
        tfl, rows, s, thr = cpu_oracle_sample(secs, 3 * secs, c=c)
        _CPU_INPUTS.clear()  # host copies of this configuration's inputs
        leg["cpu_baseline"] = {
            "value": tfl, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"{rows} query rows of {name} (uniformly sampled over heads and "
                      f"positions), fp64, {s:.1f} s; a whole launch would take "
                      f"{flops / (tfl * 1e12):.1f} s (extrapolated from the rows)"}
    return leg


def run_swa(args):
    import sink_sparse_attention_swa_b300 as swa
    from sink_sparse_attention_swa_b300 import synthetic

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    c = PREFILL_WORKLOADS[args.workload]
    flush = L2Flush(dev)
    flops = prefill_flops(c)
    ms = value = traffic = kernel = launch_ms = None
    clk_summary = None
    e2e = None
    if args.only in ("all", "prefill"):
        x = synthetic.prefill_inputs(c["B"], c["H"], c["Hkv"], c["n"], c["d"], c["w"], c["g"],
                                     dtype="bf16", seed=rank, sink_scale=c["sink_scale"],
                                     device=dev)
        out = torch.empty_like(x.Q)
        if c.get("pattern", "window") == "window":
            swa_call = lambda Q, K, V, O: swa.prefill(Q, K, V, c["w"], c["g"], x.scale, out=O,
                                                      stream=stream)
        else:
            swa_call = lambda Q, K, V, O: swa.prefill_pattern(Q, K, V, c["pattern"], c["w"],
                                                              c["g"], c["r"], x.scale, out=O,
                                                              stream=stream)
        call = lambda Q, K, V: swa_call(Q, K, V, out)
        fn = lambda: call(x.Q, x.K, x.V)
        barrier(world)
        torch.cuda.synchronize()
        with Clocks(local) as clk:
            times = time_launches(fn, args.steps, args.warmup, flush, stream)
        barrier(world)
        clk_summary = clk.summary()
        ms = max_over_ranks(float(np.mean(times)), world, dev)
        value = flops * world / (ms * 1e-3) / 1e12
        launch_ms = float(np.mean(times))
        kernel = ("swa_prefill_bf16_pair_sm103" if (c["H"] // c["Hkv"]) % 2 == 0
                  else "swa_prefill_bf16_sm103")
        traffic = recorded_traffic(kernel, args.workload, PREFILL_KERNEL_SRC)

        if not args.no_e2e:
            # ---- end to end through the public API with host buffers
            Qh = x.Q.cpu().pin_memory()
            Kh = x.K.cpu().pin_memory()
            Vh = x.V.cpu().pin_memory()
            Oh = torch.empty_like(Qh).pin_memory()
            Qd, Kd, Vd = torch.empty_like(x.Q), torch.empty_like(x.K), torch.empty_like(x.V)

            def e2e_step():
                Qd.copy_(Qh, non_blocking=True)
                Kd.copy_(Kh, non_blocking=True)
                Vd.copy_(Vh, non_blocking=True)
                call(Qd, Kd, Vd)
                Oh.copy_(out, non_blocking=True)

            e2e_times = time_launches(e2e_step, max(2, args.steps // 2), 2, flush, stream)
            serial_ms = max_over_ranks(float(np.mean(e2e_times)), world, dev)
            del Qd, Kd, Vd
            torch.cuda.empty_cache()
            pipe_ms = pipelined_e2e(
                [Qh, Kh, Vh], Oh,
                lambda d, o: swa_call(d[0], d[1], d[2], o), max(4, args.steps), 2, stream, dev)
            e2e_ms = max_over_ranks(pipe_ms, world, dev)
            e2e = {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": (Qh.numel() + Kh.numel() + Vh.numel()) * 2,
                   "d2h_bytes_per_step": Oh.numel() * 2, "ms_per_step": e2e_ms,
                   "mode": "two steps in flight: H2D, compute and D2H on three streams",
                   "serial": {"value": flops * world / (serial_ms * 1e-3) / 1e12,
                              "ms_per_step": serial_ms}}
            del Qh, Kh, Vh, Oh
        del x, out
        torch.cuda.empty_cache()

    # ---- decode leg: append one token + decode, streaming-decode workload
    decode_line = None
    if args.only in ("all", "decode"):
        decode_line = decode_leg(args, swa, synthetic, world, rank, local, dev, stream, flush, pk)

    configs = None
    if args.only == "all" and not args.no_configs and args.workload == "mistral_like_prefill":
        configs = {nm: config_leg(nm, args, swa, synthetic, world, rank, local, dev, stream,
                                  flush, pk) for nm in CONFIG_LEGS}

    cpu = None
    if (rank == 0 and world == 1 and not args.no_cpu_baseline
            and args.only in ("all", "prefill")):
        tfl, rows, secs, thr = cpu_oracle_sample(args.cpu_seconds, 3 * args.cpu_seconds, c=c)
        cpu = {"value": tfl, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"{rows} query rows of {args.workload} (uniformly sampled over "
                         f"heads and positions), fp64, {secs:.1f} s"}

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, **c, "scale": "1/sqrt(d)",
                   "l2": "flushed before each timed launch: 256 MiB write, then 256 MiB read (L2 left clean)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "clocks": clk_summary,
        "e2e": e2e,
        "gpu_launches": ((args.steps if value is not None else 0)
                         + (decode_line["gpu_launches"] if decode_line else 0)
                         + sum(v["gpu_launches"] for v in (configs or {}).values())),
        "roofline": None if value is None else prefill_roofline(c, flops, launch_ms, pk,
                                                                traffic, kernel),
        "cpu_baseline": cpu,
        "decode": decode_line,
        "configs": configs,
    }
    print(json.dumps(line), flush=True)


def run_chunk(args):
    """Chunked prefill into the rolling cache, the serving call: one
    swa_prefill_chunk with append (gather the key lists, append the chunk to
    the cache, tensor-core attention) per step."""
    import sink_sparse_attention_swa_b300 as swa
    from sink_sparse_attention_swa_b300 import synthetic

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    c = CHUNK
    flush = L2Flush(dev)
    flops = chunk_flops(c)
    x = synthetic.chunk_inputs(c["B"], c["H"], c["Hkv"], c["d"], c["w"], c["g"], c["T"],
                               c["pos0"], seed=rank, sink_scale=c["sink_scale"], device=dev)
    out = torch.empty_like(x.q)
    nbytes = swa.prefill_chunk_workspace_bytes(c["B"], c["Hkv"], c["T"], c["d"], c["w"], c["g"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    fn = lambda: swa.prefill_chunk(x.q, x.k_new, x.v_new, x.Kc, x.Vc, x.pos0, c["w"], c["g"],
                                   x.scale, out=out, append=True, workspace=ws, stream=stream)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        times = time_launches(fn, args.steps, args.warmup, flush, stream)
    barrier(world)
    ms = max_over_ranks(float(np.mean(times)), world, dev)
    launch_ms = float(np.mean(times))
    e2e = None
    if not args.no_e2e:
        qh = x.q.cpu().pin_memory()
        kh = x.k_new.cpu().pin_memory()
        vh = x.v_new.cpu().pin_memory()
        oh = torch.empty_like(qh).pin_memory()
        qd, kd, vd = torch.empty_like(x.q), torch.empty_like(x.k_new), torch.empty_like(x.v_new)

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            swa.prefill_chunk(qd, kd, vd, x.Kc, x.Vc, x.pos0, c["w"], c["g"], x.scale, out=out,
                              append=True, workspace=ws, stream=stream)
            oh.copy_(out, non_blocking=True)

        e2e_times = time_launches(e2e_step, max(2, args.steps // 2), 2, flush, stream)
        serial_ms = max_over_ranks(float(np.mean(e2e_times)), world, dev)
        def chunk_step(d, o):
            # compute runs in order on one stream, so one workspace serves every step
            swa.prefill_chunk(d[0], d[1], d[2], x.Kc, x.Vc, x.pos0, c["w"], c["g"], x.scale,
                              out=o, append=True, workspace=ws, stream=stream)

        pipe_ms = pipelined_e2e([qh, kh, vh], oh, chunk_step, max(4, args.steps), 2, stream, dev)
        e2e_ms = max_over_ranks(pipe_ms, world, dev)
        e2e = {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": (qh.numel() + kh.numel() + vh.numel()) * 2,
               "d2h_bytes_per_step": oh.numel() * 2, "ms_per_step": e2e_ms,
               "mode": "two steps in flight: H2D, compute and D2H on three streams",
               "serial": {"value": flops * world / (serial_ms * 1e-3) / 1e12,
                          "ms_per_step": serial_ms},
               "note": "chunk q/k/v from pinned host memory, O back; the cache stays on the GPU"}
    assert swa.device_status(stream) == 0, "device status reported an error"
    if rank != 0:
        return
    achieved = flops / (launch_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": flops * world / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "chunked_prefill_stream", **c, "scale": "1/sqrt(d)",
                   "step": "swa_prefill_chunk with append (gather + cache append + attention)",
                   "l2": "flushed before each timed launch: 256 MiB write, then 256 MiB read (L2 left clean)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "clocks": clk.summary(),
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": achieved / pk["bf16"], "traffic": None,
                     "kernel": "whole call: swa_chunk_gather_k + swa_cache_append_k + "
                               "swa_prefill_bf16_pair_sm103",
                     "peak_source": pk["src"] + " burst",
                     "useful_flops_per_launch": flops},
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def decode_leg(args, swa, synthetic, world, rank, local, dev, stream, flush, pk):
    dc = DECODE
    dx = synthetic.decode_cache_inputs(dc["B"], dc["H"], dc["Hkv"], dc["d"], dc["w"], dc["g"],
                                       dc["pos"], dtype="bf16", seed=rank,
                                       sink_scale=dc["sink_scale"], device=dev)
    kn, vn = synthetic.token_stream(dc["B"], dc["Hkv"], dc["d"], 1, seed=rank + 1, device=dev)
    dout = torch.empty_like(dx.q)
    splits = args.splits  # 0: the library's automatic, balanced split
    ws_bytes = swa.decode_workspace_bytes(dc["B"], dc["H"], dc["Hkv"], dc["d"], dc["w"], dc["g"],
                                          splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    dfn_dec = lambda: swa.decode(dx.q, dx.Kc, dx.Vc, dx.pos, dc["w"], dc["g"], dx.scale, out=dout,
                                 workspace=ws, num_splits=splits, stream=stream)

    def dfn():
        swa.cache_append(dx.Kc, dx.Vc, kn, vn, dx.pos, dc["w"], dc["g"], stream=stream)
        dfn_dec()

    dsteps = max(args.steps, 10)
    with Clocks(local) as dclk:
        dtimes = time_launches(dfn, dsteps, args.warmup, flush, stream)
        dec_only = time_launches(dfn_dec, dsteps, args.warmup, flush, stream)
    dms = max_over_ranks(float(np.mean(dtimes)), world, dev)
    dbytes = decode_bytes(dc)
    dgbs = dbytes * world / (dms * 1e-3) / 1e9
    dec_ms = float(np.mean(dec_only))
    dec_traffic = recorded_traffic("swa_decode_split", "streaming_decode_sinks", DECODE_KERNEL_SRC)
    assert swa.device_status(stream) == 0, "device status reported an error"
    return {"workload": "streaming_decode_sinks", **{k: dc[k] for k in dc},
            "value": dgbs, "unit": "GB/s", "ms_per_step": dms,
            "step": "cache append (1 token) + decode", "num_splits": splits or "auto",
            "roofline": {"bound": "hbm", "achieved": dbytes / (dec_ms * 1e-3) / 1e9,
                         "peak": pk["hbm"], "unit": "GB/s",
                         "frac": dbytes / (dec_ms * 1e-3) / 1e9 / pk["hbm"],
                         "traffic": dec_traffic, "kernel": "swa_decode_split + merge",
                         "decode_only_ms": dec_ms, "algorithmic_bytes": dbytes,
                         "frac_of_8TBs": dbytes / (dec_ms * 1e-3) / 1e9 / 8000.0},
            "clocks": dclk.summary(), "gpu_launches": dsteps * 3}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(min(args.warmup, 1)):
        cpu_oracle_sample(min(per, 2.0), min(per, 2.0) * 3)
    vals, secs, rows_total, thr = [], 0.0, 0, 1
    for _ in range(args.steps):
        tfl, rows, s, thr = cpu_oracle_sample(per, 3 * per)
        vals.append(tfl)
        secs += s
        rows_total += rows
    value = float(np.mean(vals))
    flops = prefill_flops(PREFILL)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": flops / (value * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "mistral_like_prefill", **PREFILL, "scale": "1/sqrt(d)",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{rows_total} sampled query rows over {args.steps} steps, "
                                   f"{secs:.1f} s of fp64 CPU work; ms_per_step extrapolates "
                                   f"to the whole layer"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="swa", choices=["swa", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (Gemma-3-like, long-context, tiny fp32)")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "chunk"])
    ap.add_argument("--splits", type=int, default=0,
                    help="decode split count for tuning sweeps (0: automatic)")
    ap.add_argument("--workload", default="mistral_like_prefill", choices=sorted(PREFILL_WORKLOADS))
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only == "chunk":
        run_chunk(args)
    else:
        run_swa(args)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
