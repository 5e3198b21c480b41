"""The device RoPE table against the rotation angles computed in fp64 ("DFlash", Configuration:
rotary position embedding with base rope_theta; "DFlash Draft Body", How It Works step 3:
positions of the drafted slots).  The table reduces each angle (p0 + p) * theta^(-2i/dh) to
[-pi, pi] in float32 (Cody and Waite's method with 2*pi and the inverse frequencies as float
pairs) before sincosf; the bound below allows that reduction's ~4e-7 plus sincosf's own
error, far under what the body's fp16 operands resolve."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL = 1e-6


def table64(p0, P, head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / head_dim)
    ang = (p0 + np.arange(P, dtype=np.float64))[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


@pytest.mark.parametrize("p0,P,head_dim,theta", [
    (0, 40000, 128, 1e6),          # every position of a 32k context and its blocks
    (0, 300, 64, 1e4),             # another head size and base
    ((1 << 20) - 64, 256, 128, 1e6),  # positions around 2^20
    ((1 << 24) - 32, 32, 128, 1e6),   # the largest positions the table takes
])
def test_rope_table_matches_fp64(lib, p0, P, head_dim, theta):
    import torch
    import block_draft_model_proj_gb300 as dflash
    cos_t = torch.empty((P, head_dim // 2), dtype=torch.float32, device="cuda")
    sin_t = torch.empty_like(cos_t)
    dflash.dflash_testing_rope_table(cos_t, sin_t, p0, head_dim, theta)
    torch.cuda.synchronize()
    c64, s64 = table64(p0, P, head_dim, theta)
    err_c = float(np.abs(cos_t.cpu().numpy().astype(np.float64) - c64).max())
    err_s = float(np.abs(sin_t.cpu().numpy().astype(np.float64) - s64).max())
    print(f"rope table p0={p0} P={P} dh={head_dim}: max |cos err| {err_c:.2e}, |sin err| {err_s:.2e}")
    assert err_c <= TOL and err_s <= TOL, (err_c, err_s)


def test_rope_table_rejects_positions_past_float32(lib):
    import torch
    import block_draft_model_proj_gb300 as dflash
    cos_t = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="2\\^24"):
        dflash.dflash_testing_rope_table(cos_t, torch.empty_like(cos_t), (1 << 24) - 32, 128, 1e6)
