"""bf16 -> fp16 conversion of the layer matrices (dflash_convert_bf16_to_f16) against
numpy's correctly rounded float64 -> float16 conversion of the same bf16 values."""
import numpy as np
import pytest

import dflash_inputs as di

pytestmark = pytest.mark.gpu


def _convert(bits: np.ndarray) -> np.ndarray:
    import torch
    import block_draft_model_proj_gb300 as dflash
    src = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    dst = torch.full(bits.shape, float("nan"), dtype=torch.float16, device="cuda")
    dflash.dflash_convert_bf16_to_f16(src, dst)
    return dst.cpu().numpy()


@pytest.mark.parametrize("n", [1, 7, 8, 4099, 1_000_003])
def test_conversion_is_round_to_nearest_even(lib, n):
    import block_draft_model_proj_gb300 as dflash
    rng = np.random.default_rng(n)
    v = (rng.standard_normal(n) * 0.02).astype(np.float32)
    special = np.array([0.0, -0.0, 2.0 ** -14, -(2.0 ** -14), 2.0 ** -20, 3e-7, 1e-9, 65280.0,
                        -65280.0, 1.0, 0.1, 2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25],
                       np.float32)
    v[:min(n, special.size)] = special[:min(n, special.size)]
    bits = di.f32_to_bf16_bits(v)
    got = _convert(bits)
    want = di.bf16_bits_to_f64(bits).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    dflash.dflash_device_status()


def test_values_beyond_fp16_range_are_reported(lib):
    import block_draft_model_proj_gb300 as dflash
    bits = di.f32_to_bf16_bits(np.array([1.0, 65536.0, -2.0], np.float32))
    got = _convert(bits)
    assert got[0] == 1.0 and np.isinf(got[1]) and got[2] == -2.0
    with pytest.raises(RuntimeError, match="fp16 range"):
        dflash.dflash_device_status()
    dflash.dflash_device_status()   # the first query reset the word
