"""The projection GEMM kernels in isolation (test hook of the library) vs an fp64 product of
the same bf16/fp16/fp32 operands.  Tensor-core (tcgen05) and CUDA-core engines, ragged shapes,
K-splits."""
import numpy as np
import pytest

import dflash_inputs as di

pytestmark = pytest.mark.gpu


def run(engine, dtype, M, N, K, splits, seed=0, lda_pad=0):
    import torch
    import block_draft_model_proj_gb300 as dflash
    rng = np.random.default_rng(seed)
    a32 = rng.standard_normal((M, K + lda_pad), dtype=np.float32)
    b32 = rng.standard_normal((N, K), dtype=np.float32)
    if dtype == "bf16":
        A = di.Tensor(di.f32_to_bf16_bits(a32), "bf16")
        B = di.Tensor(di.f32_to_bf16_bits(b32), "bf16")
        dt = dflash.DFLASH_DTYPE_BF16
        ref_a, ref_b = A.f64(), B.f64()
    elif dtype == "f16":
        a16, b16 = a32.astype(np.float16), b32.astype(np.float16)
        dt = dflash.DFLASH_DTYPE_F16
        ref_a, ref_b = a16.astype(np.float64), b16.astype(np.float64)
    else:
        A, B = di.Tensor(a32, "f32"), di.Tensor(b32, "f32")
        dt = dflash.DFLASH_DTYPE_F32
        ref_a, ref_b = A.f64(), B.f64()
    from dflash_testlib import np_to_device, to_device
    if dtype == "f16":
        dA, dB = np_to_device(a16), np_to_device(b16)
    else:
        dA, dB = to_device(A), to_device(B)
    dA = dA[:, :K] if lda_pad else dA
    ref_a = ref_a[:, :K]
    C = torch.full((splits, M, N), float("nan"), dtype=torch.float32, device="cuda")
    dflash.dflash_testing_gemm(engine, dt, dA, dB, C, splits)
    dflash.dflash_device_status()
    got = C.cpu().numpy().astype(np.float64).sum(axis=0)
    ref = ref_a @ ref_b.T
    return got, ref, K


def assert_close(got, ref, K):
    err = np.abs(got - ref)
    # fp32 accumulation of K unit-variance products: |err| ~ K * 2^-24 * |partial sums|
    tol = 4e-6 * K + 1e-5
    assert np.all(np.isfinite(got))
    assert float(err.max()) <= tol, (float(err.max()), tol)


TC_SHAPES = [
    (128, 256, 64, 1),       # one tile, one K step
    (256, 512, 640, 1),      # several tiles
    (300, 520, 200, 1),      # ragged M, N and K (K not a multiple of 64)
    (1, 8, 16, 1),           # tiny
    (16, 6144, 4096, 4),     # decode-shaped, K split
    (512, 4096, 1024, 3),    # uneven split
    (1000, 300, 4104, 2),    # K a multiple of 8 but not of 64
]


@pytest.mark.parametrize("M,N,K,splits", TC_SHAPES)
def test_tcgen05_gemm(lib, M, N, K, splits):
    import block_draft_model_proj_gb300 as dflash
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_TC, "bf16", M, N, K, splits)
    assert_close(got, ref, K)


@pytest.mark.parametrize("M,N,K,splits", [(300, 520, 200, 1), (1000, 300, 4104, 2),
                                          (128 * 24 + 64, 256 * 16, 192, 1)])
def test_tcgen05_gemm_cta_pairs_match_one_cta(lib, M, N, K, splits):
    """The CTA-pair form (256 x 256 per pair, cta_group::2 MMAs with M = 256) against the
    one-CTA form of the same GEMM: an odd M tile count (the last pair's second tile empty),
    K-splits, more pair units than pairs."""
    import block_draft_model_proj_gb300 as dflash
    got_pair, ref, _ = run(dflash.DFLASH_TESTING_ENGINE_TC, "bf16", M, N, K, splits, seed=7)
    dflash.dflash_testing_gemm_pairs(1)
    try:
        got_one, _, _ = run(dflash.DFLASH_TESTING_ENGINE_TC, "bf16", M, N, K, splits, seed=7)
    finally:
        dflash.dflash_testing_gemm_pairs(0)
    assert_close(got_pair, ref, K)
    assert_close(got_one, ref, K)
    diff = float(np.abs(got_pair - got_one).max())
    assert diff == 0.0, diff


@pytest.mark.parametrize("M,N,K,splits", [(128, 256, 64, 1), (300, 520, 200, 1),
                                          (16, 6144, 4096, 4), (1000, 300, 4104, 2)])
def test_tcgen05_gemm_f16(lib, M, N, K, splits):
    import block_draft_model_proj_gb300 as dflash
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_TC, "f16", M, N, K, splits, seed=5)
    assert_close(got, ref, K)


def test_tcgen05_gemm_f16_strided(lib):
    import block_draft_model_proj_gb300 as dflash
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_TC, "f16", 200, 256, 320, 1, lda_pad=64)
    assert_close(got, ref, K)


def test_tcgen05_gemm_strided_a(lib):
    import block_draft_model_proj_gb300 as dflash
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_TC, "bf16", 200, 256, 320, 1, lda_pad=64)
    assert_close(got, ref, K)


def test_tcgen05_gemm_persistent_many_tiles(lib):
    import block_draft_model_proj_gb300 as dflash
    # more tiles than SMs: each CTA walks several tiles and reuses both TMEM accumulators
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_TC, "bf16", 128 * 24, 256 * 16, 192, 1, seed=3)
    assert_close(got, ref, K)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K,splits", [(70, 90, 33, 1), (256, 128, 512, 3)])
def test_simt_gemm(lib, dtype, M, N, K, splits):
    import block_draft_model_proj_gb300 as dflash
    got, ref, K = run(dflash.DFLASH_TESTING_ENGINE_SIMT, dtype, M, N, K, splits)
    assert_close(got, ref, K)


# ---- weight-streaming GEMM (weights as the M operand, bf16 -> fp16 in tensor memory) ----

def run_ws(M, N, K, max_splits, w_dtype="bf16", tiles=None, seed=0, ldx_pad=0):
    import torch
    import block_draft_model_proj_gb300 as dflash
    from dflash_testlib import np_to_device
    rng = np.random.default_rng(seed)
    x16 = rng.standard_normal((M, K + ldx_pad)).astype(np.float16)
    w32 = rng.standard_normal((N, K), dtype=np.float32)
    if w_dtype == "bf16":
        wbits = di.f32_to_bf16_bits(w32)
        dW = np_to_device(wbits.view(np.int16)).view(torch.bfloat16)
        w64 = di.bf16_bits_to_f64(wbits)
        dt = dflash.DFLASH_DTYPE_BF16
    else:
        w16 = w32.astype(np.float16)
        dW = np_to_device(w16)
        w64 = w16.astype(np.float64)
        dt = dflash.DFLASH_DTYPE_F16
    dX = np_to_device(x16)
    dX = dX[:, :K] if ldx_pad else dX
    C = torch.full((max_splits, M, N), float("nan"), dtype=torch.float32, device="cuda")
    so = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl = None
    if tiles is not None:
        tl = np_to_device(np.array([len(tiles)] + list(tiles), np.int32))
    dflash.dflash_testing_gemm_ws(dX, dW, dt, C, max_splits, so, tl)
    dflash.dflash_device_status()
    s = int(so.cpu()[0])
    assert 1 <= s <= max_splits
    got = C[:s].cpu().numpy().astype(np.float64).sum(axis=0)
    ref = x16[:, :K].astype(np.float64) @ w64.T
    rows = np.arange(M) if tiles is None else np.concatenate(
        [np.arange(t * 128, min((t + 1) * 128, M)) for t in tiles])
    return got[rows], ref[rows], K, s


WS_SHAPES = [
    (128, 128, 64, 1),        # one unit, one K step
    (300, 520, 200, 1),       # ragged tokens, weight rows and K
    (16, 6144, 4096, 8),      # decode-shaped: splits chosen on the device
    (384, 4096, 4096, 4),     # three token tiles, O-projection shape
    (1000, 300, 4104, 3),     # K a multiple of 8 but not of 64
    (2048, 2048, 512, 1),     # many units per CTA: both accumulators reused
]


@pytest.mark.parametrize("M,N,K,splits", WS_SHAPES)
def test_weight_streaming_gemm_bf16_weights(lib, M, N, K, splits):
    got, ref, K, _ = run_ws(M, N, K, splits)
    assert_close(got, ref, K)


@pytest.mark.parametrize("M,N,K,splits", [(300, 520, 200, 2), (16, 6144, 4096, 8)])
def test_weight_streaming_gemm_f16_weights(lib, M, N, K, splits):
    got, ref, K, _ = run_ws(M, N, K, splits, w_dtype="f16", seed=2)
    assert_close(got, ref, K)


def test_weight_streaming_gemm_tile_list_and_stride(lib):
    # tiles 0 and 2 of four: the device schedule covers only those rows
    got, ref, K, _ = run_ws(512, 768, 320, 4, tiles=[0, 2], seed=4, ldx_pad=64)
    assert_close(got, ref, K)
