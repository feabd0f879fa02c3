"""GPU MXFP4 quantiser against the oracle's OCP-rule quantiser: bit-exact
codes and scale bytes, including ties, saturation, zero blocks and extreme
magnitudes; and the packed output round-trips through the layer."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cases():
    rng = np.random.default_rng(21)
    w = rng.normal(0, 0.02, (300, 512)).astype(np.float32)
    w[0, :32] = 0.0                                                      # all-zero block
    w[1, :32] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.9] * 4, np.float32) * 2.0 ** -6
    w[1, 0] = 4.0 * 2.0 ** -6                                            # block amax fixes X = -6
    w[2, :32] *= 1e30                                                    # huge
    w[3, :32] *= 1e-30                                                   # tiny (fp32 subnormal range nearby)
    w[4, 32:64] = -w[4, 32:64]
    w[5, :] = rng.uniform(-1, 1, 512).astype(np.float32) * np.exp2(rng.integers(-20, 20, 512)).astype(np.float32)
    return w


def test_quantize_matches_oracle_bit_exact():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    w = _cases()
    p_g, s_g = moe.mxfp4_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    p_o, s_o = oracle.mxfp4_quant(w.astype(np.float64))
    assert np.array_equal(s_g.cpu().numpy(), s_o)
    assert np.array_equal(p_g.cpu().numpy(), p_o)


def test_quantize_reproduces_generator_weights():
    """The generator's fp32 draws quantised on the GPU give exactly the
    MXFP4 bytes the generator stored."""
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    w = synth.expert_f32(3, 7, 2, 64, 1024, 0.02).reshape(-1, 1024)
    p_ref, s_ref = synth.mxfp4_experts(3, 7, 2, 64, 1024, 0.02)
    p_g, s_g = moe.mxfp4_quantize(torch.from_numpy(np.ascontiguousarray(w)).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(p_g.cpu().numpy(), p_ref.reshape(-1, 512))
    assert np.array_equal(s_g.cpu().numpy(), s_ref.reshape(-1, 32))


def test_quantize_rejects_bad_shapes():
    import torch
    import fp8_mxfp4_expert_bf16_b300 as moe
    with pytest.raises(moe.MoEError) as ei:
        moe.mxfp4_quantize(torch.zeros((4, 40), device="cuda"))
    assert ei.value.status == 2
