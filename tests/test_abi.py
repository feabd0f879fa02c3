"""The C-ABI library builds, loads without a GPU and exports every function
the header declares; host-side argument checks answer before any CUDA call."""
import ctypes
import subprocess

import pytest

import fp8_mxfp4_expert_bf16_b300 as moe


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    names = moe.declared_symbols()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", moe.build.LIB if hasattr(moe.build, "LIB") else moe._LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_library_is_sm103a_only_and_not_linked_to_libcuda():
    out = subprocess.run(["ldd", moe._LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


@pytest.mark.parametrize("field,value,status", [
    ("hidden", 100, 2), ("hidden", 0, 2), ("inter", 130, 2), ("num_experts", 0, 2), ("num_experts", 513, 2),
    ("top_k", 9, 2), ("top_k", 0, 2), ("max_tokens", 0, 2), ("score_func", 5, 1),
    ("tp_size", 9, 1), ("tp_size", -1, 1), ("tp_rank", 1, 1), ("tp_size", 3, 2)])
def test_init_rejects_bad_config_on_host(field, value, status):
    L = moe.lib()
    c = dict(hidden=512, inter=256, num_experts=16, top_k=8, max_tokens=64, score_func=0, device=0)
    c[field] = value
    cfg = moe._Config(**c)
    h = ctypes.c_void_p()
    assert L.moe_init(ctypes.byref(cfg), ctypes.byref(h)) == status
    assert h.value is None
    assert L.moe_last_error(None)


def test_null_handle_calls_fail_cleanly():
    L = moe.lib()
    assert L.moe_forward(None, None, 1, None, None) == 1
    assert L.moe_load_weights(None, None, None, None, None, None, None, None) == 1
    assert L.moe_get_routing(None, None, None) == 1
    assert L.moe_destroy(None) == 0
    assert L.moe_status_string(6) == b"device wait timed out"
    assert L.moe_stage_count() == 6 and L.moe_stage_name(3) == b"gemm1_gate_up"
