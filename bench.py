"""Benchmark of the routed MXFP4 / e4m3 MoE layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step = one forward of the whole layer (router, top-k, dispatch with
activation quantisation, gate/up grouped GEMM with SwiGLU and
re-quantisation, down grouped GEMM, combine) over one batch of T synthetic
tokens already resident in HBM.  Prints one JSON line.  Default workload:
the Flash-shaped decode layer (T=64, H=4096, E=256 top-8, I=2048).

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU (the layer does not shard on one box): a barrier and a max over
ranks bracket the timed region, and ``value`` is the tokens of all ranks
divided by that time.

``--impl reference`` times the CPU oracle (fp64 restatement of the layer) on
the host cores on a bounded sample of the same workload.
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
DEFAULT_CONFIG = "flash-decode"


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


def oracle_sample(inp, budget_s=12.0, max_tokens=None, act_scale_mode=0):
    """Time the CPU oracle token by token on the workload (routing of the
    whole batch included in every call) until the time budget is spent."""
    import oracle
    c = inp.cfg
    rng = np.random.default_rng(12345)
    order = rng.permutation(c.T)
    t0 = time.perf_counter()
    done = 0
    for t in order:
        oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, c.k, c.score_func,
                       inp.logit_bias, inp.sel_bias, tokens=[int(t)], act_scale_mode=act_scale_mode,
                       weight_format=inp.weight_format)
        done += 1
        if time.perf_counter() - t0 >= budget_s or (max_tokens and done >= max_tokens):
            break
    el = time.perf_counter() - t0
    return done, el


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        n = 1
    return max(n, os.cpu_count() or 1)


def run_reference(args, cfg):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    inp = synth.make_inputs(cfg, weights=args.weights)
    tokens = 0
    elapsed = 0.0
    for _ in range(args.warmup):
        oracle_sample(inp, budget_s=args.ref_budget / max(args.steps, 1), max_tokens=1,
                      act_scale_mode=ACT_SCALES[args.act_scale])
    per = []
    for _ in range(args.steps):
        n, el = oracle_sample(inp, budget_s=args.ref_budget / max(args.steps, 1),
                              act_scale_mode=ACT_SCALES[args.act_scale])
        tokens += n
        elapsed += el
        per.append(el)
    value = tokens / elapsed
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_desc(cfg), act_scale=args.act_scale, weights=args.weights),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{tokens} tokens of the {cfg.name} batch, one oracle call per token "
                                   f"(routing of all {cfg.T} tokens + that token's {cfg.k} expert FFNs, fp64)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, cfg):
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe

    ws, rank, local = dist_env()
    dist = ws > 1
    if dist:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    device = local
    torch.cuda.set_device(device)
    inp = synth.make_inputs(cfg, weights=args.weights)
    c = cfg
    act_mode = ACT_SCALES[args.act_scale]
    layer = moe.MoELayer(c.H, c.I, c.E, c.k, c.T, c.score_func, device=device, act_scale_mode=act_mode)
    load = layer.load_weights_fp8 if args.weights == "fp8" else layer.load_weights
    load(inp.router_w, inp.logit_bias, inp.sel_bias, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).to(f"cuda:{device}")
    y = torch.empty_like(x)
    stream = torch.cuda.Stream(device)
    P = peaks()

    def barrier():
        torch.cuda.synchronize(device)
        if dist:
            tdist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            layer.forward(x, y, stream)
    layer.check_device_error()

    # routing statistics of this batch (for the algorithmic byte / flop counts)
    counts, _ = layer.expert_counts()
    active = int((counts > 0).sum())
    rows = int(counts.sum())
    if args.weights == "fp8":   # e4m3 bytes + a 4-byte scale per 128 x 128 block
        ebytes13 = 2 * c.I * c.H + 4 * (2 * c.I // 128) * (c.H // 128)
        ebytes2 = c.H * c.I + 4 * (c.H // 128) * (c.I // 128)
    else:                       # E2M1 nibbles + one E8M0 byte per 32
        ebytes13 = 2 * c.I * c.H // 2 + 2 * c.I * c.H // 32
        ebytes2 = c.H * c.I // 2 + c.H * c.I // 32
    g1_bytes = active * ebytes13
    g2_bytes = active * ebytes2
    g1_flops = 2.0 * rows * (2 * c.I) * c.H
    g2_flops = 2.0 * rows * c.H * c.I
    decode = rows <= 64 * max(active, 1)   # a few rows per expert: streaming the weights binds

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device) as clk:
        barrier()
        clk.mark(True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                layer.forward(x, y, stream)
            ev1.record(stream)
        barrier()
        clk.mark(False)
    ms_total = ev0.elapsed_time(ev1)
    launches = layer.launch_count() * args.steps
    layer.check_device_error()

    # Kernel durations: the same K forwards once more, with the library's CUDA
    # events recorded between the kernels on the forward's stream.  The events
    # stop consecutive kernels from overlapping (programmatic dependent
    # launch), so this window is timed separately from the one above.
    ev2 = torch.cuda.Event(enable_timing=True)
    ev3 = torch.cuda.Event(enable_timing=True)
    layer.set_profiling(True)
    barrier()
    with torch.cuda.stream(stream):
        ev2.record(stream)
        for _ in range(args.steps):
            layer.forward(x, y, stream)
        ev3.record(stream)
    barrier()
    ms_profiled = ev2.elapsed_time(ev3) / args.steps
    stage = layer.stage_times()       # averages over the last <= 64 forwards of that window
    layer.set_profiling(False)
    layer.check_device_error()

    ms_max = max_over_ranks(ms_total, f"cuda:{device}")
    value = whole_job_rate(c.T * args.steps, ms_max / 1000.0, ws)

    # end to end through the host-buffer entry point (pinned host memory)
    xh = torch.from_numpy(inp.x.view(np.int16)).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        layer.forward_host(xh, yh, stream)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        layer.forward_host(xh, yh, stream)
    el = time.perf_counter() - t0
    e2e_value = whole_job_rate(c.T * args.steps, max_over_ranks(el, f"cuda:{device}"), ws)

    g1_ms = stage["gemm1_gate_up"]
    g2_ms = stage["gemm2_down"]
    if decode:
        ach = g1_bytes / (g1_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "k_mx_gemm<0> (gate/up grouped GEMM)", "achieved": ach,
                "peak": P["hbm_gbs"], "unit": "GB/s", "frac": ach / P["hbm_gbs"],
                "peak_source": f"{P['source']} HBM copy bandwidth",
                "algorithmic_bytes_per_launch": g1_bytes,
                "traffic": ncu_traffic(cfg.name, "gemm1"),
                "down_gemm": {"achieved": g2_bytes / (g2_ms / 1e3) / 1e9, "bytes_per_launch": g2_bytes},
                "layer_weight_gbs": (g1_bytes + g2_bytes) / (ms_max / args.steps / 1e3) / 1e9}
    else:
        pk = 2.0 * P["bf16_tflops"]
        ach = g1_flops / (g1_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "k_mx_gemm<0> (gate/up grouped GEMM)", "achieved": ach, "peak": pk,
                "unit": "TFLOP/s", "frac": ach / pk,
                "peak_source": f"{P['source']} bf16 burst x 2 (nominal fp8/bf16 ratio; block-scaled fp8 peak not measured)",
                "algorithmic_flops_per_launch": g1_flops, "traffic": ncu_traffic(cfg.name, "gemm1"),
                "down_gemm": {"achieved": g2_flops / (g2_ms / 1e3) / 1e12},
                "layer_tflops": (g1_flops + g2_flops) / (ms_max / args.steps / 1e3) / 1e12}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n, el = oracle_sample(inp, budget_s=args.ref_budget, act_scale_mode=act_mode)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n} tokens of the {cfg.name} batch, one oracle call per token "
                         f"(routing of all {cfg.T} tokens + that token's {cfg.k} expert FFNs, fp64)"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e2m1 (fp32 accumulate)",
            "data": "synthetic", "config": dict(workload_desc(cfg), act_scale=args.act_scale, weights=args.weights,
                                               parallelism=f"replicas{ws}",
                                               l2="inputs larger than L2: every step streams the active experts' "
                                                  "weights from HBM"),
            "roofline": roof,
            "stage_ms": stage,
            "stage_window": {"ms_per_step": ms_profiled,
                             "how": "a second window of the same K forwards with CUDA events between the kernels "
                                    "on the forward's stream (stage_ms and the roofline's kernel time come from it)"},
            "routing": {"active_experts": active, "rows": rows, "max_count": int(counts.max()),
                        "min_count": int(counts.min())},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": c.T * c.H * 2,
                    "d2h_bytes_per_step": c.T * c.H * 2},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist:
        tdist.barrier()
        tdist.destroy_process_group()
    layer.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="mxfp4", choices=["mxfp4", "fp8"],
                    help="expert format: MXFP4 (default) or e4m3 with an fp32 scale per 128 x 128 block")
    ap.add_argument("--act-scale", default="e8m0", choices=sorted(ACT_SCALES),
                    help="activation block scales: power-of-two E8M0 (default) or fp32 amax/448")
    ap.add_argument("--experts", type=int, default=None,
                    help="shrink the workload to this many experts (small profiling captures only)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the batch size T (small profiling captures only)")
    args = ap.parse_args()
    cfg = synth.CONFIGS[args.config]
    import dataclasses
    if args.experts:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}-e{args.experts}", E=args.experts,
                                  desc=cfg.desc + f" (reduced to {args.experts} experts)")
    if args.tokens:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}-t{args.tokens}", T=args.tokens,
                                  desc=cfg.desc + f" (T overridden to {args.tokens})")
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
