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


def test_mma_shape_probe():
    """The instruction's cost per shape: 128 x 256 at about the peak probe's
    cycle count, and the tokens-on-N form (weights as A) no dearer than the
    128 x 256 form for N <= 128, at most N / 256 of its work per instruction."""
    import fp8_mxfp4_expert_bf16_b300 as moe
    moe.mma_shape(256, False, 0, 512)              # warm-up
    full = moe.mma_shape(256, False, 0, 4096)
    print("128x256", full)
    assert 100.0 <= full["cycles_per_mma"] <= 400.0
    for n in (16, 64, 128):
        r = moe.mma_shape(n, True, 0, 4096)
        print(f"128x{n} weights as A", r)
        assert 0.0 < r["cycles_per_mma"] <= full["cycles_per_mma"] * 1.05
    r = moe.mma_shape(128, False, 0, 4096)
    assert 0.0 < r["cycles_per_mma"] <= full["cycles_per_mma"] * 1.05
    for bad in [(8, False), (144, True), (272, False), (24, False)]:
        with pytest.raises(moe.MoEError):
            moe.mma_shape(bad[0], bad[1], 0, 16)
