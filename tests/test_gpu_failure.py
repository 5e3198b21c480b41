"""Failure detection on the GPU without a GPU fault: a bounded device wait that runs out.

The tensor-core GEMM is launched with its TMA producer withholding every copy and arrival
(a testing hook) and a 1 ms wait limit.  Its MMA thread's first wait can never complete, so
every CTA gives up after the limit, reports DFLASH_ERR_TIMEOUT through the device status
word, drains, frees its tensor memory and exits; the host reads the status and the device
stays usable.  Nothing traps, faults or waits without a bound."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pairs", [0, 1], ids=["cta_pairs", "one_cta"])
def test_withheld_producer_runs_out_its_wait_and_reports_timeout(lib, pairs):
    """Both forms of the 128 x 256-tile GEMM: CTA pairs (256 rows = two M tiles) and one
    CTA per tile."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    dflash.dflash_testing_gemm_pairs(pairs)
    try:
        _withheld_case(torch, dflash)
    finally:
        dflash.dflash_testing_gemm_pairs(0)


def _withheld_case(torch, dflash):
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn((256, 128), generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn((512, 128), generator=g, device="cuda").to(torch.bfloat16)
    C = torch.full((1, 256, 512), float("nan"), dtype=torch.float32, device="cuda")
    dflash.dflash_device_status(reset=True)
    dflash.dflash_testing_gemm_withheld(A, B, C, 1_000_000)
    with pytest.raises(RuntimeError, match="timed out"):
        dflash.dflash_device_status(reset=True)
    assert torch.isnan(C).all(), "an aborted GEMM writes nothing"
    # the status word was reset and the context still runs the same GEMM normally
    dflash.dflash_device_status()
    dflash.dflash_testing_gemm(dflash.DFLASH_TESTING_ENGINE_TC, dflash.DFLASH_DTYPE_BF16, A, B, C)
    dflash.dflash_device_status()
    ref = A.double() @ B.double().T
    assert float((C[0].double() - ref).abs().max()) < 1e-2


def test_withheld_wait_limit_is_validated_on_the_host(lib):
    import block_draft_model_proj_gb300 as dflash
    st = lib.dflash_testing_gemm_withheld(None, 8, None, 8, None, 8, 1, 1, 1, 10, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
