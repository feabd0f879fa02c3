"""Routed MoE feed-forward layer with MXFP4 experts and e4m3 activations on B300.

Thin Python binding over the C ABI of ``libmoe_mx.so`` (declared in
``include/moe_mx.h``): argument marshalling only, every step of the layer
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no CPU fallback: if the library is missing or cannot be
loaded, importing the layer class raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

from .build import LIB as _LIB_PATH, build as _build

__all__ = ["MoELayer", "MoEError", "lib", "declared_symbols", "STAGES", "route_noalloc", "route_noalloc_check_error",
           "mxfp4_quantize", "mma_peak", "sum_partials_bf16"]

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_mx.h")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_CUDA", 4: "MOE_ERR_OOM",
          5: "MOE_ERR_NOT_LOADED", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_UNSUPPORTED", 8: "MOE_ERR_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("num_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("max_tokens", ctypes.c_int), ("score_func", ctypes.c_int),
                ("device", ctypes.c_int), ("act_scale_mode", ctypes.c_int), ("tp_size", ctypes.c_int),
                ("tp_rank", ctypes.c_int)]


ACT_SCALE_E8M0 = 0
ACT_SCALE_F32 = 1


_lib = None


def declared_symbols() -> list[str]:
    """Every function the C header declares."""
    with open(_HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:moe_status|int|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoe_mx.so (building it first if asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build() if build_if_missing else _LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libmoe_mx.so not built ({path}); run python -m fp8_mxfp4_expert_bf16_b300.build")
    L = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = {
        "moe_init": (S, [ctypes.POINTER(_Config), ctypes.POINTER(P)]),
        "moe_destroy": (S, [P]),
        "moe_load_weights": (S, [P, P, P, P, P, P, P, P]),
        "moe_load_weights_fp8": (S, [P, P, P, P, P, P, P, P]),
        "moe_forward": (S, [P, P, I, P, P]),
        "moe_forward_host": (S, [P, P, I, P, P]),
        "moe_forward_host_async": (S, [P, P, I, P, P]),
        "moe_host_sync": (S, [P]),
        "moe_forward_partial": (S, [P, P, I, P, P]),
        "moe_sum_partials_bf16": (S, [ctypes.POINTER(P), I, ctypes.c_size_t, P, P]),
        "moe_get_logits": (S, [P, P]),
        "moe_get_routing": (S, [P, P, P]),
        "moe_get_expert_counts": (S, [P, P, P]),
        "moe_get_permutation": (S, [P, P]),
        "moe_get_act_quant": (S, [P, P, P]),
        "moe_get_inter_quant": (S, [P, P, P]),
        "moe_get_act_scales_f32": (S, [P, P]),
        "moe_get_inter_scales_f32": (S, [P, P]),
        "moe_get_expert_out": (S, [P, P]),
        "moe_set_profiling": (S, [P, I]),
        "moe_get_stage_times": (S, [P, P, I]),
        "moe_stage_count": (I, []),
        "moe_stage_name": (ctypes.c_char_p, [I]),
        "moe_check_device_error": (S, [P]),
        "moe_selftest_wait_timeout": (S, [P, ctypes.c_uint]),
        "moe_last_launch_count": (I, [P]),
        "moe_last_error": (ctypes.c_char_p, [P]),
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_route_noalloc": (S, [P, I, I, P, P, P, I, I, I, P, P, P]),
        "moe_route_noalloc_check_error": (S, [P]),
        "moe_selftest_mma_peak": (S, [I, I, I, P]),
        "moe_selftest_mma_shape": (S, [I, I, I, I, P]),
        "moe_debug_fill_workspace": (S, [P, I]),
        "moe_mxfp4_quantize": (S, [P, ctypes.c_size_t, I, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _stages():
    L = lib()
    return [L.moe_stage_name(i).decode() for i in range(L.moe_stage_count())]


STAGES = None


def _ptr(a) -> int | None:
    """Address of a numpy array or a torch tensor (host or device); None -> NULL."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"], "arrays must be C-contiguous"
        return a.ctypes.data
    assert a.is_contiguous(), "tensors must be contiguous"
    return a.data_ptr()


class MoELayer:
    """One routed MoE layer on one GPU.

    Shapes: H hidden, I expert middle width, E experts, k top-k.  Weights in
    the packed MXFP4 layout of ``moe_load_weights`` (see the C header).
    """

    def __init__(self, hidden: int, inter: int, num_experts: int, top_k: int, max_tokens: int,
                 score_func: int = 0, device: int = 0, act_scale_mode: int = ACT_SCALE_E8M0,
                 tp_size: int = 1, tp_rank: int = 0):
        import torch  # noqa: F401  (device memory and streams)
        self.L = lib()
        self.H, self.I, self.E, self.k, self.max_tokens = hidden, inter, num_experts, top_k, max_tokens
        self.tp_size, self.tp_rank = tp_size, tp_rank
        self.I_loc = inter // max(tp_size, 1)       # this shard's slice of the expert middle dimension
        self.device = device
        self.act_scale_mode = act_scale_mode
        cfg = _Config(hidden, inter, num_experts, top_k, max_tokens, score_func, device, act_scale_mode, tp_size,
                      tp_rank)
        h = ctypes.c_void_p()
        st = self.L.moe_init(ctypes.byref(cfg), ctypes.byref(h))
        if st != 0:
            raise MoEError(st, self.L.moe_last_error(None).decode())
        self.h = h
        self.last_T = None

    # ------------------------------------------------------------ plumbing
    def _check(self, st: int):
        if st != 0:
            raise MoEError(st, self.L.moe_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.L.moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream(stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))

    # ------------------------------------------------------------ API
    def load_weights(self, router_w, logit_bias, sel_bias, w13_q, w13_s, w2_q, w2_s):
        """Copy the weights (numpy arrays or torch tensors, host or device)."""
        H, I, E = self.H, self.I, self.E
        for a, shape in [(router_w, (E, H)), (w13_q, (E, 2 * I, H // 2)), (w13_s, (E, 2 * I, H // 32)),
                         (w2_q, (E, H, I // 2)), (w2_s, (E, H, I // 32))]:
            assert tuple(a.shape) == shape, (tuple(a.shape), shape)
        for b in (logit_bias, sel_bias):
            assert b is None or tuple(b.shape) == (E,)
        self._check(self.L.moe_load_weights(self.h, _ptr(router_w), _ptr(logit_bias), _ptr(sel_bias),
                                            _ptr(w13_q), _ptr(w13_s), _ptr(w2_q), _ptr(w2_s)))

    def load_weights_fp8(self, router_w, logit_bias, sel_bias, w13, w13_scale, w2, w2_scale):
        """Experts in the fp8 block format: e4m3 codes u8 [E, 2I, H] / [E, H, I]
        with fp32 scales per 128 x 128 block [E, 2I/128, H/128] / [E, H/128, I/128]."""
        H, I, E = self.H, self.I, self.E
        for a, shape in [(router_w, (E, H)), (w13, (E, 2 * I, H)), (w13_scale, (E, 2 * I // 128, H // 128)),
                         (w2, (E, H, I)), (w2_scale, (E, H // 128, I // 128))]:
            assert tuple(a.shape) == shape, (tuple(a.shape), shape)
        for b in (logit_bias, sel_bias):
            assert b is None or tuple(b.shape) == (E,)
        self._check(self.L.moe_load_weights_fp8(self.h, _ptr(router_w), _ptr(logit_bias), _ptr(sel_bias),
                                                _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale)))

    def forward(self, x, y=None, stream=None):
        """x: cuda bf16 [T, H] -> y: cuda bf16 [T, H] (enqueued on the stream, no sync)."""
        import torch
        assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.shape[1] == self.H
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        self._check(self.L.moe_forward(self.h, _ptr(x), T, _ptr(y), self._stream(stream)))
        self.last_T = T
        return y

    def forward_partial(self, x, y32=None, stream=None):
        """x: cuda bf16 [T, H] -> y32: cuda fp32 [T, H], the gate-weighted sum
        before the bf16 rounding (a tensor-parallel shard's partial output)."""
        import torch
        assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.shape[1] == self.H
        T = x.shape[0]
        if y32 is None:
            y32 = torch.empty((T, self.H), dtype=torch.float32, device=x.device)
        assert y32.dtype == torch.float32 and tuple(y32.shape) == (T, self.H) and y32.is_contiguous()
        self._check(self.L.moe_forward_partial(self.h, _ptr(x), T, _ptr(y32), self._stream(stream)))
        self.last_T = T
        return y32

    def forward_host(self, x_host, y_host=None, stream=None):
        """Host bf16 bits (numpy uint16 or a CPU tensor) in and out; copies and
        synchronisation happen inside the library call."""
        T = x_host.shape[0]
        if y_host is None:
            y_host = np.empty((T, self.H), dtype=np.uint16)
        self._check(self.L.moe_forward_host(self.h, _ptr(x_host), T, _ptr(y_host), self._stream(stream)))
        self.last_T = T
        return y_host

    def forward_host_async(self, x_host, y_host, stream=None):
        """Enqueue a host-buffer forward (pinned numpy arrays or CPU tensors,
        bf16 bits) and return; host_sync() waits for every call so far.
        Consecutive calls overlap their copies with each other's forwards."""
        T = x_host.shape[0]
        self._check(self.L.moe_forward_host_async(self.h, _ptr(x_host), T, _ptr(y_host), self._stream(stream)))
        self.last_T = T
        return y_host

    def host_sync(self):
        self._check(self.L.moe_host_sync(self.h))

    def set_profiling(self, on: bool = True):
        self._check(self.L.moe_set_profiling(self.h, int(on)))

    def stage_times(self) -> dict:
        n = self.L.moe_stage_count()
        ms = np.zeros(n, dtype=np.float32)
        self._check(self.L.moe_get_stage_times(self.h, _ptr(ms), n))
        return {self.L.moe_stage_name(i).decode(): float(ms[i]) for i in range(n)}

    def check_device_error(self):
        self._check(self.L.moe_check_device_error(self.h))

    def launch_count(self) -> int:
        return self.L.moe_last_launch_count(self.h)

    def debug_fill_workspace(self, byte: int):
        """Fill every workspace buffer with ``byte`` (a forward must not read
        anything it did not write)."""
        self._check(self.L.moe_debug_fill_workspace(self.h, int(byte)))
        self.last_T = None

    # ------------------------------------------------------------ getters
    def logits(self):
        out = np.empty((self.last_T, self.E), dtype=np.float32)
        self._check(self.L.moe_get_logits(self.h, _ptr(out)))
        return out

    def routing(self):
        ids = np.empty((self.last_T, self.k), dtype=np.int32)
        gates = np.empty((self.last_T, self.k), dtype=np.float32)
        self._check(self.L.moe_get_routing(self.h, _ptr(ids), _ptr(gates)))
        return ids, gates

    def expert_counts(self):
        counts = np.empty(self.E, dtype=np.int32)
        offsets = np.empty(self.E + 1, dtype=np.int32)
        self._check(self.L.moe_get_expert_counts(self.h, _ptr(counts), _ptr(offsets)))
        return counts, offsets

    def permutation(self):
        perm = np.empty(self.last_T * self.k, dtype=np.int32)
        self._check(self.L.moe_get_permutation(self.h, _ptr(perm)))
        return perm

    def act_quant(self):
        """Q1 codes and block scales of the last forward: E8M0 bytes (u8), or
        float32 scales for a handle in the fp32-scale mode."""
        q = np.empty((self.last_T, self.H), dtype=np.uint8)
        if self.act_scale_mode == ACT_SCALE_F32:
            s = np.empty((self.last_T, self.H // 128), dtype=np.float32)
            self._check(self.L.moe_get_act_quant(self.h, _ptr(q), None))
            self._check(self.L.moe_get_act_scales_f32(self.h, _ptr(s)))
        else:
            s = np.empty((self.last_T, self.H // 128), dtype=np.uint8)
            self._check(self.L.moe_get_act_quant(self.h, _ptr(q), _ptr(s)))
        return q, s

    def inter_quant(self):
        """Q2 codes and block scales (perm order), as act_quant."""
        n = self.last_T * self.k
        q = np.empty((n, self.I_loc), dtype=np.uint8)
        if self.act_scale_mode == ACT_SCALE_F32:
            s = np.empty((n, self.I_loc // 128), dtype=np.float32)
            self._check(self.L.moe_get_inter_quant(self.h, _ptr(q), None))
            self._check(self.L.moe_get_inter_scales_f32(self.h, _ptr(s)))
        else:
            s = np.empty((n, self.I_loc // 128), dtype=np.uint8)
            self._check(self.L.moe_get_inter_quant(self.h, _ptr(q), _ptr(s)))
        return q, s

    def block_scales_f32(self, which: str = "act"):
        """Every block scale of Q1 ('act') or Q2 ('inter') as a float32 value."""
        rows = self.last_T if which == "act" else self.last_T * self.k
        width = self.H if which == "act" else self.I_loc
        s = np.empty((rows, width // 128), dtype=np.float32)
        f = self.L.moe_get_act_scales_f32 if which == "act" else self.L.moe_get_inter_scales_f32
        self._check(f(self.h, _ptr(s)))
        return s

    def expert_out(self):
        out = np.empty((self.last_T * self.k, self.H), dtype=np.float32)
        self._check(self.L.moe_get_expert_out(self.h, _ptr(out)))
        return out


def route_noalloc(x, router_w, logit_bias, sel_bias, k, score_func=0, ids=None, gates=None, stream=None):
    """Router + top-k for callers that cannot allocate device memory on their
    call path: all buffers are the caller's (contiguous cuda tensors on one
    device: x, router_w bf16; biases fp32 or None; ids int32 [T, k], gates
    fp32 [T, k]), the logits scratch is a fixed array inside the library
    (T * E <= 2^20).  Calls that overlap on the GPU share that array and must
    be serialised.  A kernel timeout is reported by route_noalloc_check_error."""
    import torch
    L = lib()
    T, H = x.shape
    E = router_w.shape[0]
    dev = x.device
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if gates is None:
        gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    for name, t, dt in [("x", x, torch.bfloat16), ("router_w", router_w, torch.bfloat16),
                        ("logit_bias", logit_bias, torch.float32), ("sel_bias", sel_bias, torch.float32),
                        ("ids", ids, torch.int32), ("gates", gates, torch.float32)]:
        if t is None:
            continue
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be a cuda tensor on {dev}")
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if router_w.shape[1] != H or tuple(ids.shape) != (T, k) or tuple(gates.shape) != (T, k):
        raise ValueError("shapes: x [T, H], router_w [E, H], ids and gates [T, k]")
    for b in (logit_bias, sel_bias):
        if b is not None and tuple(b.shape) != (E,):
            raise ValueError("biases must be [E]")
    with torch.cuda.device(dev):
        st = L.moe_route_noalloc(_ptr(x), T, H, _ptr(router_w), _ptr(logit_bias), _ptr(sel_bias), E, k,
                                 score_func, _ptr(ids), _ptr(gates), MoELayer._stream(stream))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())
    return ids, gates


def route_noalloc_check_error(device=None, stream=None):
    """Wait for the stream and raise MoEError if a kernel wait of an earlier
    route_noalloc call on the device gave up (the record is then cleared)."""
    import torch
    L = lib()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = L.moe_route_noalloc_check_error(MoELayer._stream(stream))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())


def mma_peak(device=0, steps_per_cta=8192, launches=1):
    """Block-scaled tensor-core throughput probe (see moe_selftest_mma_peak):
    returns dict(tflops, sm_mhz, cycles_per_mma, ms)."""
    L = lib()
    out = np.zeros(4, dtype=np.float32)
    st = L.moe_selftest_mma_peak(int(device), int(steps_per_cta), int(launches), _ptr(out))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())
    return {"tflops": float(out[0]), "sm_mhz": float(out[1]), "cycles_per_mma": float(out[2]), "ms": float(out[3])}


def mma_shape(n, tokens_on_n=False, device=0, steps_per_cta=4096):
    """Cost of one block-scaled 128 x n x 32 MMA (see moe_selftest_mma_shape):
    returns dict(cycles_per_mma, sm_mhz, tflops)."""
    L = lib()
    out = np.zeros(3, dtype=np.float32)
    st = L.moe_selftest_mma_shape(int(device), int(n), 1 if tokens_on_n else 0, int(steps_per_cta), _ptr(out))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())
    return {"cycles_per_mma": float(out[0]), "sm_mhz": float(out[1]), "tflops": float(out[2])}


def sum_partials_bf16(parts, y=None, stream=None):
    """bf16(parts[0] + parts[1] + ...): fp32 cuda tensors of one shape, added
    in list order in fp32 and rounded once (the tensor-parallel shards'
    partial outputs, or one all-reduced sum)."""
    import torch
    L = lib()
    p0 = parts[0]
    for p in parts:
        if not (p.is_cuda and p.dtype == torch.float32 and p.is_contiguous() and p.shape == p0.shape
                and p.device == p0.device):
            raise ValueError("partials must be contiguous fp32 cuda tensors of one shape on one device")
    if y is None:
        y = torch.empty(p0.shape, dtype=torch.bfloat16, device=p0.device)
    arr = (ctypes.c_void_p * len(parts))(*[p.data_ptr() for p in parts])
    with torch.cuda.device(p0.device):
        st = L.moe_sum_partials_bf16(arr, len(parts), p0.numel(), _ptr(y), MoELayer._stream(stream))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())
    return y


def mxfp4_quantize(w, stream=None):
    """fp32 cuda tensor [rows, K] -> (packed uint8 [rows, K/2], scales uint8 [rows, K/32]) on the device."""
    import torch
    L = lib()
    rows, K = w.shape
    packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=w.device)
    st = L.moe_mxfp4_quantize(_ptr(w), rows, K, _ptr(packed), _ptr(scales), MoELayer._stream(stream))
    if st != 0:
        raise MoEError(st, L.moe_last_error(None).decode())
    return packed, scales
