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
