"""The block-scaled tensor-core throughput probe (the prefill roofline's
denominator) runs through the C ABI and reports plausible figures: the
instruction's cycle count and a rate consistent with it."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_mma_peak_probe():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    moe.mma_peak(0, 1024, 1)                       # warm-up
    r = moe.mma_peak(0, 4096, 3)
    print(r)
    assert 100.0 <= r["cycles_per_mma"] <= 400.0
    assert 300.0 <= r["sm_mhz"] <= 2200.0
    # rate implied by the cycle count and the clock on every SM, within 15%
    implied = 2 * 128 * 256 * 32 / r["cycles_per_mma"] * r["sm_mhz"] * 1e6 * nsm / 1e12
    assert abs(r["tflops"] - implied) <= 0.15 * implied, (r, implied)
    with pytest.raises(moe.MoEError):
        moe.mma_peak(0, 0, 1)
