"""Seeded synthetic inputs for the routed MXFP4 MoE layer.

Shared, as data only, by the tests, the smoke check and the benchmark.  It
holds none of the layer's arithmetic: it draws random numbers and stores
them in the layer's input formats (bf16 activations and router weights,
MXFP4 expert weights), nothing more.  The heavy drawing is in ``gen.c``
(counter-based SplitMix64, OpenMP), built with gcc on first use.

The five workloads follow the MiMo-V2.6 shapes: hidden 4,096 / 6,144,
256 / 384 experts, top-8, 2,048-wide expert middle, no shared expert (web
page "MiMo V2.6 Pro and Flash architecture teardown", sections "How Is the
Backbone Built?" and "How Big Is Each Expert?").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libsynth.so")

# stream ids (per seed) of the independent random sequences
_S_X, _S_WR, _S_W13, _S_W2 = 1, 2, 1 << 20, 2 << 20


def build(force: bool = False) -> str:
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_tab = None


def _L():
    global _lib, _tab
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, f, sz, p, i = ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
        lib.syn_normal_bf16.argtypes = [u64, u64, f, sz, p, p, i]
        lib.syn_normal_f32.argtypes = [u64, u64, f, sz, p, p, i]
        lib.syn_mxfp4_experts.argtypes = [u64, u64, i, i, i, f, p, p, p, i]
        lib.syn_expert_f32.argtypes = [u64, u64, i, i, i, f, p, p, i]
        lib.syn_fp8_experts.argtypes = [u64, u64, i, i, i, f, p, p, p, i]
        from scipy.special import ndtri
        n = 4096
        pts = np.arange(n + 1, dtype=np.float64) / n
        pts[0], pts[-1] = 2.0 ** -20, 1.0 - 2.0 ** -20
        _tab = np.ascontiguousarray(ndtri(pts).astype(np.float32))
        _lib = lib
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def normal_bf16(seed: int, stream: int, sigma: float, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _L().syn_normal_bf16(seed, stream, sigma, out.size, _p(out), _p(_tab), _tab.size - 1)
    return out


def normal_f32(seed: int, stream: int, sigma: float, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().syn_normal_f32(seed, stream, sigma, out.size, _p(out), _p(_tab), _tab.size - 1)
    return out


def mxfp4_experts(seed: int, stream_base: int, E: int, rows: int, K: int, sigma: float):
    packed = np.empty((E, rows, K // 2), dtype=np.uint8)
    scale = np.empty((E, rows, K // 32), dtype=np.uint8)
    _L().syn_mxfp4_experts(seed, stream_base, E, rows, K, sigma, _p(packed), _p(scale), _p(_tab), _tab.size - 1)
    return packed, scale


def fp8_experts(seed: int, stream_base: int, E: int, rows: int, K: int, sigma: float):
    """The same draws as ``mxfp4_experts`` stored as e4m3 codes u8 [E, rows, K]
    with one fp32 scale (amax / 448) per 128 x 128 block, f32 [E, rows/128, K/128]."""
    q = np.empty((E, rows, K), dtype=np.uint8)
    s = np.empty((E, rows // 128, K // 128), dtype=np.float32)
    _L().syn_fp8_experts(seed, stream_base, E, rows, K, sigma, _p(q), _p(s), _p(_tab), _tab.size - 1)
    return q, s


def expert_f32(seed: int, stream_base: int, E: int, rows: int, K: int, sigma: float) -> np.ndarray:
    """The fp32 draws behind ``mxfp4_experts`` (small cases only)."""
    out = np.empty((E, rows, K), dtype=np.float32)
    _L().syn_expert_f32(seed, stream_base, E, rows, K, sigma, _p(out), _p(_tab), _tab.size - 1)
    return out


@dataclass(frozen=True)
class Config:
    name: str
    T: int
    H: int
    E: int
    I: int
    k: int
    seed: int
    bias: str            # "none" | "normal:<sigma>" | "zipf:<s>"
    score_func: int = 0  # 0 sigmoid, 1 softmax
    desc: str = ""


CONFIGS = {
    "toy": Config("toy", 64, 512, 16, 256, 8, 0, "none",
                  desc="toy MoE layer T=64 H=512 E=16 top-8 I=256"),
    "flash-decode": Config("flash-decode", 64, 4096, 256, 2048, 8, 1, "none",
                           desc="Flash-shaped MoE layer decode T=64 H=4096 E=256 top-8 I=2048, uniform routing"),
    "flash-prefill": Config("flash-prefill", 8192, 4096, 256, 2048, 8, 2, "normal:0.5",
                            desc="Flash-shaped MoE layer prefill T=8192 H=4096 E=256 top-8 I=2048, "
                                 "per-expert logit bias N(0,0.5)"),
    "pro-decode": Config("pro-decode", 256, 6144, 384, 2048, 8, 3, "none",
                         desc="Pro-shaped MoE layer decode T=256 H=6144 E=384 top-8 I=2048, uniform routing"),
    "pro-prefill-skew": Config("pro-prefill-skew", 16384, 6144, 384, 2048, 8, 4, "zipf:1.1",
                               desc="Pro-shaped MoE layer prefill T=16384 H=6144 E=384 top-8 I=2048, "
                                    "Zipf(1.1) expert popularity via logit bias"),
}


@dataclass
class Inputs:
    cfg: Config
    x: np.ndarray            # u16 bf16 [T, H]
    router_w: np.ndarray     # u16 bf16 [E, H]
    logit_bias: np.ndarray   # f32 [E]
    sel_bias: np.ndarray     # f32 [E] (zero: the correction bias of a freshly initialised router)
    w13_q: np.ndarray        # mxfp4: u8 [E, 2I, H/2] (gate rows [0, I), up rows [I, 2I)); fp8: u8 e4m3 [E, 2I, H]
    w13_s: np.ndarray        # mxfp4: u8 E8M0 [E, 2I, H/32]; fp8: f32 [E, 2I/128, H/128]
    w2_q: np.ndarray         # mxfp4: u8 [E, H, I/2]; fp8: u8 e4m3 [E, H, I]
    w2_s: np.ndarray         # mxfp4: u8 [E, H, I/32]; fp8: f32 [E, H/128, I/128]
    extra: dict = field(default_factory=dict)
    weight_format: str = "mxfp4"   # "mxfp4" or "fp8" (e4m3 + fp32 scale per 128 x 128 block)


def logit_bias(cfg: Config) -> np.ndarray:
    """Per-expert router logit bias that shapes the routing mix.

    "none": zero (uniform routing).  "normal:s": N(0, s^2) per expert, numpy
    default_rng(seed).  "zipf:s": -s * ln(rank_e) with ranks a seeded random
    permutation of 1..E, so expert popularity falls off as a power of its rank.
    """
    E = cfg.E
    kind, _, arg = cfg.bias.partition(":")
    rng = np.random.default_rng(cfg.seed)
    if kind == "none":
        return np.zeros(E, dtype=np.float32)
    if kind == "normal":
        return rng.normal(0.0, float(arg), E).astype(np.float32)
    if kind == "zipf":
        ranks = rng.permutation(E) + 1
        return (-float(arg) * np.log(ranks.astype(np.float64))).astype(np.float32)
    raise ValueError(cfg.bias)


def make_inputs(cfg: Config | str, T: int | None = None, x_only: bool = False, weights: str = "mxfp4") -> Inputs:
    """Draw one workload: x ~ bf16(N(0,1)), Wr ~ bf16(N(0, 0.02^2)),
    expert weights fp32 N(0, 0.02^2) stored as MXFP4 (or, with
    weights="fp8", as e4m3 with an fp32 scale per 128 x 128 block)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    T = cfg.T if T is None else T
    s = cfg.seed
    x = normal_bf16(s, _S_X, 1.0, (T, cfg.H))
    if x_only:
        return Inputs(cfg, x, None, None, None, None, None, None, None)
    wr = normal_bf16(s, _S_WR, 0.02, (cfg.E, cfg.H))
    store = fp8_experts if weights == "fp8" else mxfp4_experts
    w13_q, w13_s = store(s, _S_W13, cfg.E, 2 * cfg.I, cfg.H, 0.02)
    w2_q, w2_s = store(s, _S_W2, cfg.E, cfg.H, cfg.I, 0.02)
    return Inputs(cfg, x, wr, logit_bias(cfg), np.zeros(cfg.E, dtype=np.float32),
                  w13_q, w13_s, w2_q, w2_s, weight_format=weights)


def custom_inputs(T, H, E, I, k, seed, bias="none", score_func=0, weights="mxfp4") -> Inputs:
    """A workload of any shape (edge cases in the tests)."""
    return make_inputs(Config(f"custom-{T}-{H}-{E}-{I}-{k}", T, H, E, I, k, seed, bias, score_func),
                       weights=weights)


def expert_weight_bytes(H: int, I: int, weights: str = "mxfp4") -> int:
    """Bytes of one expert: MXFP4, 3*H*I weights at 4 bits plus one scale
    byte per 32 weights (4.25 bits per weight); fp8, one byte per weight plus
    a 4-byte scale per 128 x 128 block."""
    if weights == "fp8":
        return 3 * H * I + 4 * (3 * H * I // (128 * 128))
    return 3 * H * I // 2 + 3 * H * I // 32
