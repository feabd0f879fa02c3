"""Benchmark of the routed MXFP4 / e4m3 MoE layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--windows R] [--config all|NAME]
                    [--impl reference] [--weights mxfp4|fp8] [--act-scale e8m0|f32] [--peak-only]

One step = one forward of the whole layer (router, top-k, dispatch with
activation quantisation, gate/up grouped GEMM with SwiGLU and
re-quantisation, down grouped GEMM, combine) over one batch of T synthetic
tokens already resident in HBM.  Each workload is timed in R windows of K
steps (CUDA events on the forward's stream, barrier + synchronize around
each window); the median window gives ``ms_per_step``.  Prints one JSON
line.  Default (``--config all``): the line is the largest single-GPU
workload, the Pro-shaped prefill with skewed routing (T=16384, H=6144,
E=384 top-8, I=2048); the other four workloads ride in its ``per_config``
key, each with its own timing, roofline, stage times, routing statistics,
end-to-end rate, CPU baseline and clocks, and so do the Flash decode batch in
the fp32-scale activation mode and with the fp8 expert format.  The block-scaled tensor-core
rate the prefill rooflines divide by is measured in the same run
(``block_scaled_peak``).

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU: a barrier and a max over ranks bracket the timed region, and
``value`` is the tokens of all ranks divided by that time.

``--impl reference`` times the CPU oracle (fp64 restatement of the layer) on
the host cores on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s and % of roofline (HBM GB/s decode, tensor TFLOP/s prefill) on 1 B300"
HEADLINE = "pro-prefill-skew"      # the largest single-GPU workload
ORDER = ["toy", "flash-decode", "pro-decode", "flash-prefill", "pro-prefill-skew"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


ACT_SCALES = {"e8m0": 0, "f32": 1}


def workload_desc(cfg):
    return {"workload": cfg.name, "desc": cfg.desc, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I, "top_k": cfg.k,
            "seed": cfg.seed, "routing_bias": cfg.bias, "score": "sigmoid" if cfg.score_func == 0 else "softmax"}


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ["mx_gemm.cu", "ptx.cuh", "moe_internal.cuh"]:
        with open(os.path.join(ROOT, "fp8_mxfp4_expert_bf16_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock and throttle reasons while the timed region runs: NVML polled
    every 5 ms, or (if the NVML bindings do not load) an ``nvidia-smi -lms``
    sampler whose rows inside the marked window are kept."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    SMI_FIELDS = ["clocks_event_reasons.sw_power_cap", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.hw_thermal_slowdown"]

    def __init__(self, index):
        self.index = index
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._mark = False
        self.nv = None
        self.proc = None
        self.windows = []
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
        except Exception as e:   # noqa: BLE001
            self.nvml_error = str(e)

    def _run(self):
        get_reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        while not self._stop.is_set():
            if self._mark:
                try:
                    self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                    r = get_reasons(self.h) if get_reasons else 0
                    for bit, name in self.REASONS.items():
                        if r & bit:
                            self.reasons.add(name)
                except Exception:   # noqa: BLE001
                    pass
            time.sleep(0.005)

    def __enter__(self):
        if self.nv is not None:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        else:
            import subprocess
            q = "timestamp,clocks.sm,clocks.max.sm," + ",".join(self.SMI_FIELDS)
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "20"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:   # noqa: BLE001
                self.proc = None
            time.sleep(0.3)
        return self

    def mark(self, on):
        self._mark = on
        if self.nv is None:
            if on:
                self.windows.append([time.time(), None])
            elif self.windows:
                self.windows[-1][1] = time.time()

    def __exit__(self, *a):
        self._stop.set()
        if self.nv is not None:
            self.t.join()
        elif self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            import datetime
            rows = []
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 7:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(f[1]), float(f[2]), f[3:7]))
                except ValueError:
                    continue
            inside = [r for r in rows if any(w0 - 0.02 <= r[0] <= (w1 or w0) + 0.02 for w0, w1 in self.windows)]
            use = inside or rows[-3:]
            self.samples = [r[1] for r in use]
            self.max_mhz = use[0][2] if use else None
            names = ["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown"]
            for r in use:
                for n, v in zip(names, r[3]):
                    if v.lower() == "active":
                        self.reasons.add(n)
            self.source = "nvidia-smi" + ("" if inside else " (no sample inside the timed window; nearest kept)")

    def summary(self):
        if self.nv is None and not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"]}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples),
                "source": "nvml" if self.nv is not None else getattr(self, "source", "nvidia-smi")}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device: str) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself when torch.distributed is not initialised."""
    import torch
    import torch.distributed as tdist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if tdist.is_available() and tdist.is_initialized():
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, seconds_max: float, world: int) -> float:
    """Tokens per second of all ranks together: every replica processes its
    own batch, the job ends with its slowest rank."""
    return world * tokens_per_rank / seconds_max


def oracle_sample(inp, budget_s=12.0, act_scale_mode=0):
    """Time the CPU oracle, as it stands, on a bounded sample of the workload:
    oracle.forward routes every token of the batch and runs the expert FFNs
    of the sampled tokens.  A first call on one token sizes a second call
    whose sample fills the rest of the budget.  Returns (tokens, seconds,
    description)."""
    import oracle
    c = inp.cfg
    order = np.random.default_rng(12345).permutation(c.T)

    def call(toks):
        t0 = time.perf_counter()
        oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, c.k, c.score_func,
                       inp.logit_bias, inp.sel_bias, tokens=np.sort(toks), act_scale_mode=act_scale_mode,
                       weight_format=inp.weight_format)
        return time.perf_counter() - t0

    el = call(order[:1])
    done, calls = 1, 1
    n = int(max(0.0, budget_s - el) / max(el, 1e-3))
    if n >= 1:
        n = min(n, c.T - 1)
        el += call(order[1:1 + n])
        done += n
        calls += 1
    desc = (f"{done} tokens of the {c.name} batch in {calls} oracle calls (each routes all {c.T} tokens in fp64, "
            f"then runs the sampled tokens' {c.k} expert FFNs in fp64)")
    return done, el, desc


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        n = 1
    return max(n, os.cpu_count() or 1)


def config_dict(cfg, args):
    """The workload a line measures (identical in both arms)."""
    return dict(workload_desc(cfg), act_scale=args.act_scale, weights=args.weights)



def headline_config(args):
    import dataclasses
    name = HEADLINE if args.config == "all" else args.config
    cfg = synth.CONFIGS[name]
    if args.experts:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}-e{args.experts}", E=args.experts,
                                  desc=cfg.desc + f" (reduced to {args.experts} experts)")
    if args.tokens:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}-t{args.tokens}", T=args.tokens,
                                  desc=cfg.desc + f" (T overridden to {args.tokens})")
    return cfg


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    cfg = headline_config(args)
    inp = synth.make_inputs(cfg, weights=args.weights)
    mode = ACT_SCALES[args.act_scale]
    per_step = args.ref_budget / max(args.steps, 1)
    for _ in range(args.warmup):
        oracle_sample(inp, budget_s=0.0, act_scale_mode=mode)
    tokens, elapsed, desc = 0, 0.0, ""
    for _ in range(args.steps):
        n, el, desc = oracle_sample(inp, budget_s=per_step, act_scale_mode=mode)
        tokens += n
        elapsed += el
    value = tokens / elapsed
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"per step: {desc}; {tokens} tokens over {args.steps} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


PEAK_STEPS = 8192   # 4 x 8192 MMAs per SM per probe launch (~2 ms)


def burst_block_scaled_peak(device):
    """The tensor-core rate of the instruction the grouped GEMMs issue
    (moe_selftest_mma_peak: block-scaled e4m3 x E2M1, 128 x 256 x 32) as a
    burst: the best of five ~2 ms launches on a rested GPU."""
    import fp8_mxfp4_expert_bf16_b300 as moe
    moe.mma_peak(device, 1024, 3)
    bursts = [moe.mma_peak(device, PEAK_STEPS, 1) for _ in range(5)]
    b = max(bursts, key=lambda r: r["tflops"])
    return {"burst_tflops": b["tflops"], "burst_sm_mhz": b["sm_mhz"], "cycles_per_mma": b["cycles_per_mma"],
            "burst_ms": b["ms"]}


def sustained_block_scaled_peak(device, burst, seconds=3.0):
    """The same instruction issued back to back for about ``seconds``: the
    rate the chip holds under its power cap (the denominator for a kernel
    timed inside a long run of steps)."""
    import fp8_mxfp4_expert_bf16_b300 as moe
    n = max(1, int(seconds * 1000.0 / max(burst["burst_ms"], 0.1)))
    sus = moe.mma_peak(device, PEAK_STEPS, n)
    return dict(burst, sustained_tflops=sus["tflops"], sustained_sm_mhz=sus["sm_mhz"], sustained_ms=sus["ms"],
                how="moe_selftest_mma_peak: one CTA per SM issuing tcgen05.mma kind::mxf8f6f4.block_scale "
                    "128x256x32 (e4m3 x e2m1, E8M0 scales) from shared memory with the GEMMs' elected issue loop; "
                    f"burst = best of 5 launches of {4 * PEAK_STEPS} MMAs per SM before the workloads, sustained = "
                    f"{n} such launches back to back after them; SM clock from the SMs' cycle counters")


def expert_bytes(c, weights):
    """Algorithmic bytes of one expert's gate/up and down weights (with scales)."""
    if weights == "fp8":   # e4m3 bytes + a 4-byte scale per 128 x 128 block
        return (2 * c.I * c.H + 4 * (2 * c.I // 128) * (c.H // 128), c.H * c.I + 4 * (c.H // 128) * (c.I // 128))
    return (2 * c.I * c.H // 2 + 2 * c.I * c.H // 32, c.H * c.I // 2 + c.H * c.I // 32)


L2_BYTES = 126 * 1024 * 1024


def run_config(args, cfg, device, stream, P, peak, ws, rank, dist, cpu_budget):
    """Time one workload; returns its result entry (rank 0) or None."""
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    if dist:
        import torch.distributed as tdist
    c = cfg
    act_mode = ACT_SCALES[args.act_scale]
    inp = synth.make_inputs(cfg, weights=args.weights)
    layer = moe.MoELayer(c.H, c.I, c.E, c.k, c.T, c.score_func, device=device, act_scale_mode=act_mode)
    load = layer.load_weights_fp8 if args.weights == "fp8" else layer.load_weights
    load(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).to(f"cuda:{device}")
    y = torch.empty_like(x)
    eb13, eb2 = expert_bytes(c, args.weights)
    # weights that fit in L2 would be re-read from it: flush L2 between steps then
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=f"cuda:{device}") \
        if c.E * (eb13 + eb2) < 2 * L2_BYTES else None

    def barrier():
        torch.cuda.synchronize(device)
        if dist:
            tdist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            layer.forward(x, y, stream)
    layer.check_device_error()
    counts, _ = layer.expert_counts()
    active = int((counts > 0).sum())
    rows = int(counts.sum())
    g1_bytes, g2_bytes = active * eb13, active * eb2
    g1_flops = 2.0 * rows * (2 * c.I) * c.H
    g2_flops = 2.0 * rows * c.H * c.I
    decode = rows <= 64 * max(active, 1)   # a few rows per expert: streaming the weights binds

    def timed_window(k):
        """k forwards; device milliseconds (per-step events around each
        forward when L2 is flushed between steps, else one pair)."""
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(k):
                    layer.forward(x, y, stream)
                e1.record(stream)
            barrier()
            return e0.elapsed_time(e1)
        evs = []
        with torch.cuda.stream(stream):
            for _ in range(k):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                layer.forward(x, y, stream)
                e1.record(stream)
                evs.append((e0, e1))
        barrier()
        return sum(a.elapsed_time(b) for a, b in evs)

    windows = []
    with ClockSampler(device) as clk:
        for _ in range(args.windows):
            barrier()
            clk.mark(True)
            windows.append(timed_window(args.steps))
            clk.mark(False)
    layer.check_device_error()
    ms_med = statistics.median(windows)
    ms_max = max_over_ranks(ms_med, f"cuda:{device}")
    value = whole_job_rate(c.T * args.steps, ms_max / 1000.0, ws)
    launches = layer.launch_count() * args.steps

    # Kernel durations: K more forwards with the library's CUDA events between
    # the kernels on the forward's stream.  Those events stop consecutive
    # kernels from overlapping (programmatic dependent launch), so this
    # window is timed apart from the ones above.
    layer.set_profiling(True)
    ms_profiled = timed_window(args.steps) / args.steps
    stage = layer.stage_times()       # averages over the last <= 64 forwards of that window
    layer.set_profiling(False)
    layer.check_device_error()

    # end to end through the host-buffer entry point (pinned host memory):
    # every step copies its batch in and its output out inside the timed
    # region; consecutive steps overlap their copies with each other's
    # forwards (moe_forward_host_async), the region ends once the last
    # output has arrived in host memory
    # (R windows of K steps back to back, as the device-buffer windows; the
    # median window counts)
    xh = torch.from_numpy(inp.x.view(np.int16)).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        layer.forward_host(xh, yh, stream)
    barrier()
    e2e_windows = []
    for _ in range(args.windows):
        t0 = time.perf_counter()
        for _ in range(args.steps):
            layer.forward_host_async(xh, yh, stream)
        layer.host_sync()
        e2e_windows.append(time.perf_counter() - t0)
    el = statistics.median(e2e_windows)
    e2e_value = whole_job_rate(c.T * args.steps, max_over_ranks(el, f"cuda:{device}"), ws)

    g1_ms, g2_ms = stage["gemm1_gate_up"], stage["gemm2_down"]
    step_s = ms_max / args.steps / 1e3
    clocks = clk.summary()
    if flush is not None:
        roof = {"bound": "none", "note": f"the {c.E} experts' weights ({c.E * (eb13 + eb2) / 1e6:.1f} MB) fit in L2: "
                                        "a parity workload; L2 flushed between timed steps"}
    elif decode:
        ach = g1_bytes / (g1_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "k_mx_gemm<0> (gate/up grouped GEMM)", "achieved": ach,
                "peak": P["hbm_gbs"], "unit": "GB/s", "frac": ach / P["hbm_gbs"],
                "peak_source": f"{P['source']} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": g1_bytes, "traffic": ncu_traffic(cfg.name, "gemm1"),
                "down_gemm": {"achieved": g2_bytes / (g2_ms / 1e3) / 1e9, "bytes_per_launch": g2_bytes,
                              "frac": g2_bytes / (g2_ms / 1e3) / 1e9 / P["hbm_gbs"]},
                "layer_weight_gbs": (g1_bytes + g2_bytes) / step_s / 1e9,
                "layer_frac": (g1_bytes + g2_bytes) / step_s / 1e9 / P["hbm_gbs"]}
    else:
        # the tensor rate is filled in once the sustained peak is measured
        roof = {"bound": "tensor", "kernel": "k_mx_gemm<0> (gate/up grouped GEMM)",
                "achieved": g1_flops / (g1_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "algorithmic_flops_per_launch": g1_flops, "traffic": ncu_traffic(cfg.name, "gemm1"),
                "down_gemm": {"achieved": g2_flops / (g2_ms / 1e3) / 1e12},
                "layer_tflops": (g1_flops + g2_flops) / step_s / 1e12, "kernel_sm_mhz": clocks.get("sm_mhz")}

    cpu = None
    if rank == 0 and cpu_budget > 0:
        n, el, desc = oracle_sample(inp, budget_s=cpu_budget, act_scale_mode=act_mode)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc}
    entry = {
        "value": value, "unit": "tokens/s", "ms_per_step": ms_max / args.steps,
        "windows_ms_per_step": [w / args.steps for w in windows],
        "config": config_dict(cfg, args),
        "l2": ("weights fit in L2: L2 flushed (256 MB write) between timed steps" if flush is not None else
               "inputs larger than L2: every step streams the active experts' weights from HBM"),
        "roofline": roof, "stage_ms": stage,
        "stage_window": {"ms_per_step": ms_profiled,
                         "how": "a further window of K forwards with CUDA events between the kernels on the "
                                "forward's stream (stage_ms and the roofline's kernel time come from it)"},
        "routing": {"active_experts": active, "rows": rows, "max_count": int(counts.max()),
                    "min_count": int(counts.min()), "cv": float(counts.std() / max(counts.mean(), 1e-9))},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": c.T * c.H * 2,
                "d2h_bytes_per_step": c.T * c.H * 2, "windows_ms_per_step": [1e3 * w / args.steps for w in e2e_windows],
                "how": "moe_forward_host_async from pinned host buffers: every step's input copy, forward and output "
                       "copy inside the window, copies overlapping the neighbouring steps' forwards; host clock "
                       "from before the first call to after the last output arrived; median of the windows"},
        "gpu_launches": launches * args.windows,
        "clocks": clocks,
    }
    layer.close()
    del x, y, flush, inp
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    return entry if rank == 0 else None


def run_tp(args):
    """Tensor-parallel layer: rank r of the torchrun group holds shard r of
    the expert middle dimension; one step = its fp32 partial forward, a sum
    all-reduce over NCCL and one bf16 rounding (strong scaling: every rank
    works on the same batch).  With --tp 1 the same path runs on one GPU."""
    import torch
    from fp8_mxfp4_expert_bf16_b300.tp import TensorParallelMoE, make_shard
    ws, rank, local = dist_env()
    if ws != args.tp:
        raise SystemExit(f"--tp {args.tp} needs {args.tp} ranks (torchrun --nproc-per-node {args.tp}), got {ws}")
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
    cfg = headline_config(args)
    c = cfg
    inp = synth.make_inputs(cfg, weights=args.weights)
    layer = make_shard(c.H, c.I, c.E, c.k, c.T, args.tp, rank, c.score_func, local, ACT_SCALES[args.act_scale])
    load = layer.load_weights_fp8 if args.weights == "fp8" else layer.load_weights
    load(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    tp = TensorParallelMoE(layer)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty_like(x)

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            tdist.barrier()

    for _ in range(max(args.warmup, 3)):
        tp.forward(x, y)
    layer.check_device_error()
    windows = []
    with ClockSampler(local) as clk:
        for _ in range(args.windows):
            barrier()
            clk.mark(True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                tp.forward(x, y)
            e1.record()
            barrier()
            clk.mark(False)
            windows.append(e0.elapsed_time(e1))
    layer.check_device_error()
    ms = max_over_ranks(statistics.median(windows), f"cuda:{local}")
    if rank == 0:
        line = {"metric": METRIC, "value": c.T * args.steps / (ms / 1000.0), "unit": "tokens/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
                "dtype": "e4m3 x e2m1 (fp32 accumulate)", "data": "synthetic",
                "config": dict(config_dict(cfg, args), tp=args.tp), "parallelism": f"tp{args.tp}",
                "windows_ms_per_step": [w / args.steps for w in windows],
                "gpu_launches": (layer.launch_count() + 1) * args.steps * args.windows,
                "clocks": clk.summary(),
                "note": "tensor-parallel split of the expert middle dimension, one NCCL sum all-reduce per step"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    layer.close()
    return 0


def tensor_roofline(roof, peak, P):
    """Fractions of a tensor-bound entry: against the sustained block-scaled
    rate (the kernel is timed inside long runs of back-to-back steps), the
    burst rate, the instruction's rate at the SM clock sampled while the
    kernel ran (cycles per MMA x that clock), and twice the bf16 burst."""
    ach, pk = roof["achieved"], peak["sustained_tflops"]
    kclk = roof.pop("kernel_sm_mhz", None) or peak["sustained_sm_mhz"]
    pk_clk = peak["burst_tflops"] * kclk / peak["burst_sm_mhz"]
    roof.update(peak=pk, frac=ach / pk,
                peak_source=(f"block-scaled e4m3 x e2m1 MMA rate measured in this run, sustained "
                             f"({peak['sustained_sm_mhz']:.0f} MHz under the power cap; "
                             f"{peak['cycles_per_mma']:.1f} cycles per 128x256x32 MMA)"),
                frac_vs_burst_peak=ach / peak["burst_tflops"], burst_peak=peak["burst_tflops"],
                frac_at_kernel_clock=ach / pk_clk, peak_at_kernel_clock=pk_clk, kernel_sm_mhz=kclk,
                frac_vs_2x_bf16_burst=ach / (2.0 * P["bf16_tflops"]))
    roof["down_gemm"]["frac"] = roof["down_gemm"]["achieved"] / pk
    roof["layer_frac"] = roof["layer_tflops"] / pk
    return roof


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    dist = ws > 1
    if dist:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    device = local
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    P = peaks()
    burst = burst_block_scaled_peak(device)
    if args.peak_only:
        peak = sustained_block_scaled_peak(device, burst, args.peak_seconds)
        if rank == 0:
            print(json.dumps({"block_scaled_peak": peak, "measured_peaks": P}), flush=True)
        return 0
    head = headline_config(args)
    others = [n for n in ORDER if n != head.name] if args.config == "all" and not (args.experts or args.tokens) else []
    # the headline workload first (the GPU as the burst probe left it), then the others
    e = run_config(args, head, device, stream, P, None, ws, rank, dist,
                   0 if args.no_cpu_baseline else args.ref_budget)
    entries = {}
    for name in others:
        entries[name] = run_config(args, synth.CONFIGS[name], device, stream, P, None, ws, rank, dist,
                                   0 if args.no_cpu_baseline else args.ref_budget / 4)
    # the layer's two other formats on the Flash decode batch: fp32 activation
    # block scales, and the fp8 (V2.5) expert format
    if others and args.act_scale == "e8m0" and args.weights == "mxfp4":
        import copy
        for key, val in [("act_scale", "f32"), ("weights", "fp8")]:
            a2 = copy.copy(args)
            setattr(a2, key, val)
            entries[f"flash-decode/{key}={val}"] = run_config(a2, synth.CONFIGS["flash-decode"], device, stream, P,
                                                               None, ws, rank, dist, 0)
    peak = sustained_block_scaled_peak(device, burst, args.peak_seconds)
    if rank == 0:
        for ent in [e] + list(entries.values()):
            if ent["roofline"].get("bound") == "tensor":
                tensor_roofline(ent["roofline"], peak, P)
        line = {
            "metric": METRIC, "value": e["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": e["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e2m1 (fp32 accumulate)",
            "data": "synthetic", "config": e["config"], "parallelism": f"replicas{ws}",
            "windows": args.windows, "windows_ms_per_step": e["windows_ms_per_step"], "l2": e["l2"],
            "roofline": e["roofline"], "stage_ms": e["stage_ms"], "stage_window": e["stage_window"],
            "routing": e["routing"], "cpu_baseline": e["cpu_baseline"], "e2e": e["e2e"],
            "gpu_launches": e["gpu_launches"], "clocks": e["clocks"], "block_scaled_peak": peak,
            "per_config": entries,
        }
        print(json.dumps(line), flush=True)
    if dist:
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="forwards per timed window")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--windows", type=int, default=5, help="timed windows per workload (the median is reported)")
    ap.add_argument("--config", default="all", choices=["all"] + sorted(synth.CONFIGS),
                    help="all: the headline workload plus the other four in per_config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="mxfp4", choices=["mxfp4", "fp8"],
                    help="expert format: MXFP4 (default) or e4m3 with an fp32 scale per 128 x 128 block")
    ap.add_argument("--act-scale", default="e8m0", choices=sorted(ACT_SCALES),
                    help="activation block scales: power-of-two E8M0 (default) or fp32 amax/448")
    ap.add_argument("--peak-only", action="store_true", help="only measure the block-scaled tensor-core rate")
    ap.add_argument("--peak-seconds", type=float, default=3.0, help="length of the sustained peak measurement")
    ap.add_argument("--tp", type=int, default=0,
                    help="tensor-parallel layer over the torchrun group (N ranks = N shards, NCCL all-reduce)")
    ap.add_argument("--experts", type=int, default=None,
                    help="shrink the workload to this many experts (small profiling captures only)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the batch size T (small profiling captures only)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.tp:
        return run_tp(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
