#!/usr/bin/env python3
"""Benchmark of the retention core on one B300 (or N replicas, one per GPU).

Headline workload (the one `value` reports): chunkwise recurrent retention,
long sequence -- b1 H16 N32768 dk256 dv512 chunk 256, bf16 Q/K/V ~ N(0,1)/16,
fp32 state, fp32 output.  A step is one full chunkwise forward over that
batch (intra-chunk products, cross-chunk read, state update; decay masks made
in registers).  The same JSON line also reports the decode workload (512
recurrent steps at b128 H16 dk256 dv512, fp32 state) and the parallel form
with all three normalisations and the GroupNorm/swish epilogue (b8 H8 N2048),
each with its own roofline.

Timing: W warm-up steps, then K steps between CUDA events on the launching
stream, bracketed by a barrier and synchronisation; inputs are larger than L2
(126 MB) so no flush is needed.  Multi-GPU (torchrun): independent replicas,
one per GPU, weak scaling; the elapsed time is the max over ranks.

`--impl reference` times the fp64 CPU oracle (the only reference this project
has) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_recurrence_sequence_chunkwise_b300 import inputs  # noqa: E402

METRIC = ("retention fwd tokens/s & % tensor peak (chunkwise); decode tokens/s & HBM GB/s")
E2E_SEGMENT = 2048          # tokens per streamed segment of the end-to-end leg (1024: 30.8 ms,
                            # 2048: 30.2, 4096: 30.4, 8192: 31.4 on chunkwise_long)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------------------- dist
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str | None = None, timeout_s: float | None = None):
        if self.world > 1:
            import datetime

            import torch.distributed as dist
            backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            kw = {"timeout": datetime.timedelta(seconds=timeout_s)} if timeout_s else {}
            dist.init_process_group(backend, **kw)
            self.pg = dist
        return self

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        """Max of a scalar over ranks (timing only; no data-path collective)."""
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() and self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(dist: Dist, elapsed_ms: float, units_per_rank: float) -> tuple[float, float]:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    worst = dist.max(elapsed_ms)
    return units_per_rank * dist.world / (worst / 1e3), worst


# ----------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ret_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if re.match(r"^[\d.]+$", r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        # samples taken while the GPU drew load (power above the idle floor)
        busy = [float(r[1]) for r in rows if re.match(r"^[\d.]+$", r[3]) and r[1].replace(".", "").isdigit()
                and power and float(r[3]) > min(power) + 0.25 * (max(power) - min(power))]
        loaded = busy or [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "samples_under_load": len(busy), "reasons": reasons}


def profile_traffic(summary_name: str, *source_files: str):
    """DRAM bytes per launch from a committed ncu summary, or None when a kernel source
    changed since the counters were taken (the summary records the hash of each source)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    hashes = set(re.findall(r"source_sha256:\s*([0-9a-f]{64})", text))
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (hashes and m_bytes):
        return None
    for f in source_files:
        src = os.path.join(ROOT, "linear_recurrence_sequence_chunkwise_b300", "csrc", f)
        if hashlib.sha256(open(src, "rb").read()).hexdigest() not in hashes:
            return None
    return float(m_bytes.group(1))


def timed(fn, steps: int, warmup: int, dist: Dist, stream=None, counter=None):
    """W untimed steps, then K steps between CUDA events on the launching stream.
    Returns (elapsed ms of this rank, counter delta over the timed steps)."""
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0 = counter() if counter else 0
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    c1 = counter() if counter else 0
    torch.cuda.synchronize()
    dist.barrier()
    return e0.elapsed_time(e1), c1 - c0


# ----------------------------------------------------------------------------- oracle arm
def oracle_chunkwise_sample(w, tokens: int, threads: int):
    """Oracle chunkwise on `threads` heads x `tokens` tokens of workload w, one head
    per host thread.  Returns (tokens/s, seconds, description)."""
    import oracle
    heads = threads
    q, k, v = inputs.qkv(inputs.Workload("sample", 1, heads, tokens, w.dk, w.dv, w.dtype,
                                         w.scale, chunk=w.chunk, seed=w.seed + 77))
    gam = inputs.gammas(w.H)[:heads] if heads <= w.H else (inputs.gammas(w.H) * 8)[:heads]

    def unit(h):
        return oracle.chunkwise(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], [gam[h]], w.chunk)

    oracle.default()
    t0 = time.perf_counter()
    oracle.map_units(unit, range(heads), threads)
    dt = time.perf_counter() - t0
    desc = (f"{heads} heads x {tokens} tokens of {w.name} (dk{w.dk} dv{w.dv} chunk {w.chunk}), "
            f"fp64 oracle, one head per host thread")
    return heads * tokens / dt, dt, desc


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return 0
    w = inputs.CHUNKWISE_LONG
    threads = max(1, min(os.cpu_count() or 1, w.H))
    tokens = 2048
    for _ in range(args.warmup):
        oracle_chunkwise_sample(w, tokens, threads)
    total, tps = 0.0, []
    for _ in range(args.steps):
        r, dt, desc = oracle_chunkwise_sample(w, tokens, threads)
        total += dt
        tps.append(r)
    value = args.steps * threads * tokens / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, "f32"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm
def workload_config(w, out_dtype: str):
    return {"workload": f"{w.name}: chunkwise retention b{w.b} H{w.H} N{w.N} dk{w.dk} dv{w.dv} "
                        f"chunk {w.chunk}, {w.dtype} q/k/v N(0,1)/sqrt(dk), fp32 state, "
                        f"{out_dtype} out, gamma_h = 1-2^(-5-h)",
            "b": w.b, "H": w.H, "N": w.N, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
            "out_dtype": out_dtype,
            "l2": "inputs (1.07 GB) larger than L2 (126 MB); no flush between steps"}


def bench_chunkwise(args, dist, rb, pk, out_dtype):
    w = inputs.CHUNKWISE_LONG
    q, k, v = inputs.qkv(w, "cuda")
    od = torch.float32 if out_dtype == "f32" else torch.bfloat16
    o = torch.empty(w.b, w.H, w.N, w.dv, dtype=od, device="cuda")
    fn = lambda: rb.retention_chunkwise(q, k, v, w.gamma, w.chunk, out=o)  # noqa: E731
    with Clocks(torch.cuda.current_device()) as clk:
        ms, launches = timed(fn, args.steps, args.warmup, dist, counter=rb.kernel_launches)
    rb.check_device_error()
    tokens = w.b * w.N
    value, worst = aggregate(dist, ms, tokens * args.steps)
    flops = inputs.algorithmic_flops("chunkwise", w)
    ms_step = worst / args.steps
    achieved = flops / (ms_step * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    in_bytes = 2 * (2 * w.b * w.H * w.N * w.dk + w.b * w.H * w.N * w.dv)
    out_bytes = w.b * w.H * w.N * w.dv * (4 if out_dtype == "f32" else 2)
    traffic = profile_traffic(f"chunkwise_tc_pair_{w.name}.md", "tc_chunkwise_pair.cu")
    res = {"value": value, "ms_per_step": ms_step, "launches": launches,
           "clocks": clk.summary(),
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "traffic": traffic,
                        "algorithmic_flops_per_launch": flops,
                        "algorithmic_bytes_per_launch": in_bytes + out_bytes,
                        "achieved_gbs": (in_bytes + out_bytes) / (ms_step * 1e-3) / 1e9}}
    # end to end through the C ABI with host buffers (retention_chunkwise_host): every step
    # copies q, k, v from pinned host memory and the output back; the sequence streams
    # through in segments whose state is carried exactly (eq.7), so the copies of one
    # segment overlap the compute of the next on separate streams.
    hq, hk, hv = (t.to("cpu").pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    seg = E2E_SEGMENT
    ws = torch.empty(rb.chunkwise_host_workspace_bytes(q.dtype, o.dtype, w.b, w.H, w.dk, w.dv, seg),
                     dtype=torch.uint8, device="cuda")

    def e2e_step():
        rb.retention_chunkwise_host(hq, hk, hv, w.gamma, w.chunk, ho, seg, workspace=ws)

    e2e_steps = max(1, min(args.steps, 5))
    ms_e2e, _ = timed(e2e_step, e2e_steps, 1, dist)
    e2e_val, _ = aggregate(dist, ms_e2e, tokens * e2e_steps)
    rb.check_device_error()
    link = host_link(((hq, q), (hk, k), (hv, v)), ((o, ho),))
    e2e_ms = ms_e2e / e2e_steps
    res["e2e"] = {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": in_bytes,
                  "d2h_bytes_per_step": out_bytes, "ms_per_step": e2e_ms,
                  "mode": f"retention_chunkwise_host: pinned host q/k/v/out, {w.N // seg} segments "
                          f"of {seg} tokens, H2D / compute / D2H on three streams, state carried "
                          f"on the device",
                  "link": link,
                  "link_frac": link["both_ms"] / e2e_ms}
    del q, k, v, o, hq, hk, hv, ho
    torch.cuda.empty_cache()
    return res


def host_link(h2d_pairs, d2h_pairs, reps: int = 3) -> dict:
    """The host link measured with the step's own pinned buffers: the H2D copies alone,
    the D2H copies alone and both at once on two streams (copy engines only, no kernel).
    both_ms is the floor of an end-to-end step that moves these bytes."""
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()

    def run(h2d: bool, d2h: bool) -> float:
        cur = torch.cuda.current_stream()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ev[0].record(cur)
        jobs = [(s_, pairs) for s_, on, pairs in ((sh, h2d, h2d_pairs), (sd, d2h, d2h_pairs)) if on]
        for s_, _ in jobs:          # both copy streams start from the same point
            s_.wait_stream(cur)
        for s_, pairs in jobs:
            with torch.cuda.stream(s_):
                for _ in range(reps):
                    for src, dst in pairs:
                        dst.copy_(src, non_blocking=True)
        for s_, _ in jobs:
            cur.wait_stream(s_)
        ev[1].record(cur)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / reps

    run(True, True)    # warm-up
    nb_h = sum(src.numel() * src.element_size() for src, _ in h2d_pairs)
    nb_d = sum(src.numel() * src.element_size() for src, _ in d2h_pairs)
    t_h, t_d, t_b = run(True, False), run(False, True), run(True, True)
    return {"h2d_gbs": nb_h / (t_h * 1e-3) / 1e9, "d2h_gbs": nb_d / (t_d * 1e-3) / 1e9,
            "h2d_ms": t_h, "d2h_ms": t_d, "both_ms": t_b}


def bench_decode(args, dist, rb, pk):
    w = inputs.DECODE
    state = inputs.decode_state(w, "cuda")
    qs, ks, vs = inputs.decode_all_inputs(w, "cuda")
    o = torch.empty(w.b, w.H, w.dv, dtype=torch.float32, device="cuda")

    def run_all():
        for t in range(w.steps):
            rb.retention_recurrent_step(qs[t], ks[t], vs[t], state, w.gamma, out=o)

    ms, _ = timed(run_all, 1, 1, dist)
    rb.check_device_error()
    ms_step = ms / w.steps
    tokens = w.b * w.steps
    value, _ = aggregate(dist, ms, tokens)
    state_bytes = 2 * 4 * w.b * w.H * w.dk * w.dv
    io_bytes = 2 * w.b * w.H * (2 * w.dk + w.dv) + 4 * w.b * w.H * w.dv
    gbs = (state_bytes + io_bytes) / (ms_step * 1e-3) / 1e9
    del state, qs, ks, vs, o
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: b{w.b} H{w.H} dk{w.dk} dv{w.dv}, {w.steps} steps, fp32 state "
                        f"N(0,0.1^2), bf16 q/k/v N(0,1)/16, fp32 out",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": profile_traffic("decode_decode.md", "decode.cu"),
                         "algorithmic_bytes_per_launch": state_bytes + io_bytes}}


def bench_parallel(args, dist, rb, pk):
    w = inputs.PARALLEL_NORM
    q, k, v = inputs.qkv(w, "cuda")
    g = inputs.gate(w, "cuda")
    out = torch.empty(w.b, w.N, w.H * w.dv, dtype=torch.float32, device="cuda")

    def step():
        # one kernel: parallel form, normalisations, GroupNorm and swish gate
        rb.retention_parallel_gated(q, k, v, g, w.gamma, w.flags, w.eps, out=out)

    steps = max(3, args.steps // 2)
    with Clocks(torch.cuda.current_device()) as clk:
        ms, _ = timed(step, steps, max(1, args.warmup // 2), dist)
    rb.check_device_error()
    ms_step = ms / steps
    tokens = w.b * w.N
    value, _ = aggregate(dist, ms, tokens * steps)
    flops = inputs.algorithmic_flops("parallel", w)
    achieved = flops / (ms_step * 1e-3) / 1e12
    del q, k, v, g, out
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: b{w.b} H{w.H} N{w.N} dk{w.dk} dv{w.dv}, bf16 in, all three "
                        "normalisations, GroupNorm(eps 1e-5)+swish gate epilogue fused "
                        "(retention_parallel_gated), fp32 out",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "traffic": profile_traffic(f"parallel_pair_{w.name}.md", "tc_parallel_pair.cu",
                                                    "tc_parallel.cu"),
                         "algorithmic_flops_per_launch": flops, **sustained_frac(achieved, pk)},
            "clocks": clk.summary()}


def bench_backward(args, dist, rb, pk):
    w = inputs.BACKWARD
    q, k, v = inputs.qkv(w, "cuda")
    do = inputs.dout(w, "cuda")
    grads = tuple(torch.empty(w.b, w.H, w.N, d, dtype=torch.float32, device="cuda")
                  for d in (w.dk, w.dk, w.dv))
    nbytes = rb.backward_workspace_bytes(torch.float32, w.b, w.H, w.N, w.dk, w.dv)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")

    def step():
        # five tensor-core passes: dv in reversed time on the caller's stream, the two dq
        # halves and the two dk halves (reversed time) as chains on two side streams
        rb.retention_chunkwise_backward(q, k, v, do, w.gamma, w.chunk, grads=grads, workspace=ws)

    def step_cuda_cores():
        rb.retention_chunkwise_backward(q, k, v, do, w.gamma, w.chunk, grads=grads,
                                        cuda_cores=True)

    steps = max(3, args.steps // 4)
    with Clocks(torch.cuda.current_device()) as clk:
        ms, _ = timed(step, steps, 3, dist)
    rb.check_device_error()
    ms_step = ms / steps
    ms_cc, _ = timed(step_cuda_cores, 3, 1, dist)
    rb.check_device_error()
    value, _ = aggregate(dist, ms, w.b * w.N * steps)
    flops = inputs.algorithmic_flops("backward", w)
    achieved = flops / (ms_step * 1e-3) / 1e12
    del q, k, v, do, grads, ws
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: gradient of chunkwise retention b{w.b} H{w.H} N{w.N} "
                        f"dk{w.dk} dv{w.dv} chunk {w.chunk}, bf16 q/k/v/dout N(0,1)/16, fp32 "
                        "dq/dk/dv (retention_chunkwise_backward_ws: tensor-core passes)",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "traffic": profile_traffic("chunkwise_backward_tc_backward.md",
                                                    "backward_tc.cu", "tc_chunkwise_pair.cu"),
                         "algorithmic_flops_per_launch": flops, **sustained_frac(achieved, pk)},
            "clocks": clk.summary(),
            "cuda_core_kernel_ms_per_step": ms_cc / 3}


def bench_rglru(args, dist, rb, pk):
    w = inputs.RGLRU
    x, ga, gx, lam = inputs.rglru_inputs(w, "cuda")
    y = torch.empty(w.b, w.N, w.dv, dtype=torch.float32, device="cuda")

    def step():
        rb.rglru_scan(x, ga, gx, lam, None, 8.0, out=y)

    steps = max(3, args.steps // 4)
    ms, _ = timed(step, steps, 3, dist)
    rb.check_device_error()
    ms_step = ms / steps
    value, _ = aggregate(dist, ms, w.b * w.N * steps)
    nbytes = w.b * w.N * w.dv * (3 * inputs.esize(w.dtype) + 4) + 4 * w.dv
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    del x, ga, gx, lam, y
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: RG-LRU scan (Griffin page) b{w.b} T{w.N} D{w.dv}, bf16 x and "
                        "gate pre-activations N(0,1), Lambda with a^8 ~ U(0.9,0.999), c 8, zero "
                        "initial state, fp32 y (rglru_scan)",
            "value": value, "unit": "steps/s (b*T per step)", "ms_per_step": ms_step,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": profile_traffic("rglru_scan_rglru.md", "rglru.cu"),
                         "algorithmic_bytes_per_launch": nbytes}}


def bench_xpos(args, dist, rb, pk):
    w = inputs.CHUNKWISE_LONG
    q, k, _ = inputs.qkv(w, "cuda")
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    theta = [10000.0 ** (-j / (w.dk // 2)) for j in range(w.dk // 2)]

    def step():
        rb.retention_xpos_rotate(q, k, theta, 0, q_out=qo, k_out=ko)

    steps = max(3, args.steps // 4)
    ms, _ = timed(step, steps, 3, dist)
    rb.check_device_error()
    ms_step = ms / steps
    value, _ = aggregate(dist, ms, w.b * w.N * steps)
    nbytes = 4 * q.numel() * q.element_size()      # q and k, each read and written once
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    del q, k, qo, ko
    torch.cuda.empty_cache()
    return {"workload": f"xpos: rotation of chunkwise_long's Q and K (b{w.b} H{w.H} N{w.N} "
                        f"dk{w.dk}, bf16 in and out, theta_j = 10000^(-2j/dk), positions 0..N-1)",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": profile_traffic("xpos_kernel_xpos.md", "xpos.cu"),
                         "algorithmic_bytes_per_launch": nbytes}}


def bench_chunkwise_bf16(args, dist, rb, pk):
    """The headline workload with a bf16 output (the state stays fp32)."""
    w = inputs.CHUNKWISE_LONG
    q, k, v = inputs.qkv(w, "cuda")
    o = torch.empty(w.b, w.H, w.N, w.dv, dtype=torch.bfloat16, device="cuda")
    fn = lambda: rb.retention_chunkwise(q, k, v, w.gamma, w.chunk, out=o)  # noqa: E731
    steps = max(3, args.steps // 2)
    ms, _ = timed(fn, steps, 3, dist)
    rb.check_device_error()
    kern = rb.last_kernel()
    ms_step = ms / steps
    value, _ = aggregate(dist, ms, w.b * w.N * steps)
    flops = inputs.algorithmic_flops("chunkwise", w)
    achieved = flops / (ms_step * 1e-3) / 1e12
    nbytes = 2 * (2 * w.b * w.H * w.N * w.dk + w.b * w.H * w.N * w.dv) + 2 * w.b * w.H * w.N * w.dv
    del q, k, v, o
    torch.cuda.empty_cache()
    return {"workload": f"{w.name} with bf16 output: b{w.b} H{w.H} N{w.N} dk{w.dk} dv{w.dv} chunk "
                        f"{w.chunk}, bf16 q/k/v, fp32 state, bf16 out ({kern})",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": None,
                         "algorithmic_flops_per_launch": flops,
                         "algorithmic_bytes_per_launch": nbytes,
                         "achieved_gbs": nbytes / (ms_step * 1e-3) / 1e9}}


def bench_sweep(args, dist, rb, pk):
    """The chunkwise training-shape sweep: b4 H16 dk256 dv512, N x chunk grid, fp32 out."""
    points = []
    for w in inputs.SWEEP:
        q, k, v = inputs.qkv(w, "cuda")
        o = torch.empty(w.b, w.H, w.N, w.dv, dtype=torch.float32, device="cuda")
        fn = lambda: rb.retention_chunkwise(q, k, v, w.gamma, w.chunk, out=o)  # noqa: E731
        steps = max(3, args.steps // 5)
        ms, _ = timed(fn, steps, 3, dist)
        rb.check_device_error()
        kern = rb.last_kernel()
        ms_step = ms / steps
        value, _ = aggregate(dist, ms, w.b * w.N * steps)
        flops = inputs.algorithmic_flops("chunkwise", w)
        achieved = flops / (ms_step * 1e-3) / 1e12
        points.append({"N": w.N, "chunk": w.chunk, "kernel": kern, "value": value,
                       "unit": "tokens/s", "ms_per_step": ms_step,
                       "roofline": {"bound": "tensor", "achieved": achieved,
                                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                    "frac": achieved / pk["bf16_tflops"], "traffic": None,
                                    "algorithmic_flops_per_launch": flops}})
        del q, k, v, o
        torch.cuda.empty_cache()
    return {"workload": "sweep: chunkwise retention b4 H16 dk256 dv512, N in {2048, 8192, 16384} "
                        "x chunk in {64, 128, 256}, bf16 q/k/v N(0,1)/16, fp32 state and out",
            "points": points}


MSR = dict(b=8, N=2048, D=4096, H=16, dk=256, dv=512, Dout=4096)


def bench_msr_layer(args, dist, rb, pk):
    """The gated multi-scale retention layer: four projections, the parallel form with all
    three normalisations and the gated GroupNorm fused, the output projection."""
    c = MSR
    b, N, D, H, dk, dv, Do = c["b"], c["N"], c["D"], c["H"], c["dk"], c["dv"], c["Dout"]
    x = inputs.randn((b, N, D), 8000, 1.0, "bf16", "cuda")
    shapes = [(D, H * dk), (D, H * dk), (D, H * dv), (D, H * dv), (H * dv, Do)]
    ws = [inputs.randn(sh, 8001 + i, sh[0] ** -0.5, "bf16", "cuda") for i, sh in enumerate(shapes)]
    gam = inputs.gammas(H)
    theta = [10000.0 ** (-j / (dk // 2)) for j in range(dk // 2)]
    out = torch.empty(b, N, Do, dtype=torch.bfloat16, device="cuda")
    wsb = torch.empty(rb.msr_layer_workspace_bytes(b, N, H, dk, dv, 0), dtype=torch.uint8,
                      device="cuda")

    def step():
        rb.retention_msr_layer(x, *ws, gam, theta, flags=7, out=out, workspace=wsb)

    steps = max(3, args.steps // 5)
    with Clocks(torch.cuda.current_device()) as clk:
        ms, _ = timed(step, steps, 3, dist)
    rb.check_device_error()
    ms_step = ms / steps
    value, _ = aggregate(dist, ms, b * N * steps)
    proj = 2.0 * b * N * D * (2 * H * dk + 2 * H * dv) + 2.0 * b * N * H * dv * Do
    core = float(b * H) * (dk + dv) * N * (N + 1)
    flops = proj + core
    achieved = flops / (ms_step * 1e-3) / 1e12
    del x, ws, out, wsb
    torch.cuda.empty_cache()
    return {"workload": f"msr_layer: gated multi-scale retention layer b{b} N{N} d_model{D} H{H} "
                        f"dk{dk} dv{dv} d_out{Do}, bf16 x and weights N(0, 1/fan_in), xPos on Q/K "
                        "fused into their projection, parallel form with all three "
                        "normalisations + GroupNorm/swish gate fused, bf16 out "
                        "(retention_msr_layer: six kernels)",
            "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": None,
                         "algorithmic_flops_per_launch": flops,
                         "flops_split": {"projections": proj, "retention_core": core},
                         **sustained_frac(achieved, pk)},
            "clocks": clk.summary()}


def sustained_frac(achieved: float, pk: dict) -> dict:
    """A dense tensor-core loop that runs long enough meets the board's power cap: the
    fraction of the sustained peak (a seconds-long cuBLAS loop) beside the burst one."""
    s = pk.get("bf16_tflops_sustained")
    return {"peak_sustained": s, "frac_of_sustained": achieved / s} if s else {}


def bench_gemm(args, dist, rb, pk):
    """The layer's projection GEMM alone (C = A W, the V/G projection shape)."""
    M, Nc, K = 16384, 8192, 4096
    a = inputs.randn((M, K), 8100, 1.0, "bf16", "cuda")
    w = inputs.randn((K, Nc), 8101, K ** -0.5, "bf16", "cuda")
    c = torch.empty(M, Nc, dtype=torch.bfloat16, device="cuda")
    steps = max(3, args.steps // 2)
    with Clocks(torch.cuda.current_device()) as clk:
        ms, _ = timed(lambda: rb.retention_gemm(a, w, out=c), steps, 3, dist)
    rb.check_device_error()
    ms_step = ms / steps
    flops = 2.0 * M * Nc * K
    achieved = flops / (ms_step * 1e-3) / 1e12
    value, _ = aggregate(dist, ms, M * steps)
    del a, w, c
    torch.cuda.empty_cache()
    return {"workload": f"gemm: projection GEMM C = A W, M{M} N{Nc} K{K}, bf16 in, fp32 "
                        "accumulate, bf16 out (retention_gemm)",
            "value": value, "unit": "rows/s", "ms_per_step": ms_step,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "traffic": profile_traffic("gemm_kernel_gemm.md", "tc_gemm.cu"),
                         "algorithmic_flops_per_launch": flops, **sustained_frac(achieved, pk)},
            "clocks": clk.summary()}


def cpu_baseline_leg():
    w = inputs.CHUNKWISE_LONG
    threads = max(1, min(os.cpu_count() or 1, w.H))
    tps, dt, desc = oracle_chunkwise_sample(w, 8192, threads)
    return {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": desc + f" ({dt:.1f} s wall)"}


# the legs reported beside the headline, in this order
EXTRA_LEGS = {"decode": bench_decode, "parallel": bench_parallel, "backward": bench_backward,
              "rglru": bench_rglru, "xpos": bench_xpos, "chunkwise_bf16": bench_chunkwise_bf16,
              "sweep": bench_sweep, "msr_layer": bench_msr_layer, "gemm": bench_gemm}


def run_ours(args, dist: Dist):
    from linear_recurrence_sequence_chunkwise_b300 import binding as rb
    rb.lib()
    pk, pk_src = peaks()
    out_dtype = args.out_dtype
    main = bench_chunkwise(args, dist, rb, pk, out_dtype)
    extra = {}
    if not args.only_headline:
        for name in args.legs.split(","):
            if name:
                extra[name] = EXTRA_LEGS[name](args, dist, rb, pk)
    cpu = cpu_baseline_leg() if (dist.rank == 0 and dist.world == 1 and not args.no_cpu) else None
    if dist.rank != 0:
        return 0
    w = inputs.CHUNKWISE_LONG
    line = {"metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(w, out_dtype),
            "roofline": main["roofline"], "peak_source": f"{pk_src} (MEASURED_PEAKS.json burst)"
            if pk_src == "measured" else "fallback",
            "cpu_baseline": cpu, "e2e": main["e2e"], "gpu_launches": main["launches"],
            "clocks": main["clocks"]}
    line.update(extra)
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- profiling
PROFILE_CASES = {
    # reduced sizes of the benched workloads, inputs still larger than L2
    "chunkwise": "chunkwise_long at N=8192: b1 H16 dk256 dv512 chunk 256, bf16 in, fp32 out",
    "decode": "decode at b32: H16 dk256 dv512, fp32 state (268 MB), bf16 q/k/v, fp32 out",
    "parallel": "parallel_norm (b8 H8 N2048 dk256 dv512, all normalisations) + epilogue",
    "backward": "backward (b4 H16 N2048 dk256 dv512 chunk 64), bf16 in, fp32 gradients (1.1 GB)",
    "rglru": "rglru (b8 T4096 D4096), bf16 x and gates, fp32 y (1.3 GB)",
    "xpos": "xpos rotation of chunkwise_long's Q and K (b1 H16 N32768 dk256, bf16, 1.1 GB)",
    "gemm": "projection GEMM M8192 N8192 K4096, bf16 in and out (0.2 GB)",
}


def run_profile(case: str) -> int:
    """Two untimed calls of one workload at a reduced size (the first is a warm-up
    that an ncu capture skips with -s).  For ncu captures only; prints no timing."""
    from linear_recurrence_sequence_chunkwise_b300 import binding as rb
    rb.lib()
    if case == "chunkwise":
        w = inputs.CHUNKWISE_LONG
        q, k, v = inputs.qkv(w, "cuda", N=8192)
        o = torch.empty(w.b, w.H, 8192, w.dv, dtype=torch.float32, device="cuda")
        calls = [lambda: rb.retention_chunkwise(q, k, v, w.gamma, w.chunk, out=o)]
    elif case == "decode":
        w = inputs.DECODE
        state = inputs.randn((32, w.H, w.dk, w.dv), w.seed + 5, w.state_std, "f32", "cuda")
        qs, ks, vs = (inputs.randn((32, w.H, d), w.seed + 101 + i, w.scale, "bf16", "cuda")
                      for i, d in enumerate((w.dk, w.dk, w.dv)))
        o = torch.empty(32, w.H, w.dv, dtype=torch.float32, device="cuda")
        calls = [lambda: rb.retention_recurrent_step(qs, ks, vs, state, w.gamma, out=o)]
    elif case == "backward":
        w = inputs.BACKWARD
        q, k, v = inputs.qkv(w, "cuda")
        do = inputs.dout(w, "cuda")
        grads = tuple(torch.empty(w.b, w.H, w.N, d, dtype=torch.float32, device="cuda")
                      for d in (w.dk, w.dk, w.dv))
        nbytes = rb.backward_workspace_bytes(torch.float32, w.b, w.H, w.N, w.dk, w.dv)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
        calls = [lambda: rb.retention_chunkwise_backward(q, k, v, do, w.gamma, w.chunk,
                                                         grads=grads, workspace=ws)]
    elif case == "xpos":
        w = inputs.CHUNKWISE_LONG
        q, k, _ = inputs.qkv(w, "cuda")
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        theta = [10000.0 ** (-j / (w.dk // 2)) for j in range(w.dk // 2)]
        calls = [lambda: rb.retention_xpos_rotate(q, k, theta, 0, q_out=qo, k_out=ko)]
    elif case == "gemm":
        a = inputs.randn((8192, 4096), 8100, 1.0, "bf16", "cuda")
        w = inputs.randn((4096, 8192), 8101, 4096 ** -0.5, "bf16", "cuda")
        cg = torch.empty(8192, 8192, dtype=torch.bfloat16, device="cuda")
        calls = [lambda: rb.retention_gemm(a, w, out=cg)]
    elif case == "rglru":
        w = inputs.RGLRU
        x, ga, gx, lam = inputs.rglru_inputs(w, "cuda")
        y = torch.empty(w.b, w.N, w.dv, dtype=torch.float32, device="cuda")
        calls = [lambda: rb.rglru_scan(x, ga, gx, lam, None, 8.0, out=y)]
    else:
        w = inputs.PARALLEL_NORM
        q, k, v = inputs.qkv(w, "cuda")
        g = inputs.gate(w, "cuda")
        out = torch.empty(w.b, w.N, w.H * w.dv, dtype=torch.float32, device="cuda")
        calls = [lambda: rb.retention_parallel_gated(q, k, v, g, w.gamma, w.flags, w.eps, out=out)]
    for _ in range(2):
        for c in calls:
            c()
    rb.check_device_error()
    torch.cuda.synchronize()
    print(f"profile case {case}: {PROFILE_CASES[case]}; launches {rb.kernel_launches()}")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--out-dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--only-headline", action="store_true")
    ap.add_argument("--legs", default=",".join(EXTRA_LEGS),
                    help="comma-separated legs reported beside the headline "
                         f"(default all: {','.join(EXTRA_LEGS)})")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES), default=None,
                    help="run two untimed calls of one reduced workload (for ncu) and exit")
    args = ap.parse_args(argv)
    unknown = [x for x in args.legs.split(",") if x and x not in EXTRA_LEGS]
    if unknown:
        ap.error(f"unknown legs {unknown}; choose from {sorted(EXTRA_LEGS)}")
    if args.profile:
        return run_profile(args.profile)
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)
    dist.init()
    try:
        return run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
