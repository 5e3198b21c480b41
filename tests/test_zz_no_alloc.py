"""dflash_verify_greedy_static: greedy verification for callers that cannot allocate device
memory (a host framework that owns the device memory pool, or a loop that must never call
cudaMalloc/cudaFree).  Its outputs must equal the workspace variant's, call after call,
although every call reuses the same fixed scratch array inside the library."""
import numpy as np
import pytest

import dflash_inputs as di

pytestmark = pytest.mark.gpu


def _run(logits: di.Tensor, draft: np.ndarray, eos: int, static: bool):
    import torch
    import block_draft_model_proj_gb300 as dflash
    from dflash_testlib import to_device
    B, S, V = logits.shape
    dl = to_device(logits)
    dd = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).cuda()
    em = torch.full((B, S), -9, dtype=torch.int32, device="cuda")
    ne = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ac = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ch = torch.full((B, S), -9, dtype=torch.int32, device="cuda")
    dt = dflash.DFLASH_DTYPE_BF16 if logits.dtype == "bf16" else dflash.DFLASH_DTYPE_F32
    fn = dflash.dflash_verify_greedy_static if static else dflash.dflash_verify_greedy
    fn(dl, dt, dd, B, S - 1, V, eos, em, ne, ac, ch)
    dflash.dflash_device_status()
    return [t.cpu().numpy() for t in (ch, em, ne, ac)]


def _same(a, b):
    for x, y, name in zip(a, b, ("choices", "emitted", "num_emitted", "accepted")):
        assert np.array_equal(x, y), name


def _cases():
    w8 = di.WORKLOADS["decode_8b_b8_ctx4096"]
    yield di.gen_verify(w8)
    w1 = di.WORKLOADS["tiny_f32"]
    yield di.gen_verify(w1)


def test_static_matches_workspace_variant_twice_in_a_row(lib):
    # two different inputs back to back: the second call must not see the first one's
    # partials, and each must equal the workspace variant bit for bit
    for vi in _cases():
        first = _run(vi.logits, vi.draft, -1, static=True)
        _same(first, _run(vi.logits, vi.draft, -1, static=False))
    for vi in _cases():
        second = _run(vi.logits, vi.draft, -1, static=True)
        _same(second, _run(vi.logits, vi.draft, -1, static=False))
        assert np.array_equal(second[3], vi.planted_prefix)


def test_static_at_the_row_limit(lib):
    # B * (gamma + 1) = 16384 rows: one chunk per row, the whole static array in use
    rng = np.random.default_rng(77)
    B, S, V = 1024, 16, 96
    x = rng.integers(-3, 4, size=(B, S, V)).astype(np.float32)
    logits = di.Tensor(di.f32_to_bf16_bits(x), "bf16")
    draft = rng.integers(0, 3, size=(B, S - 1)).astype(np.int32)
    for _ in range(2):
        _same(_run(logits, draft, 1, static=True), _run(logits, draft, 1, static=False))


def test_static_rejects_more_rows_than_its_scratch(lib):
    import block_draft_model_proj_gb300 as dflash
    st = lib.dflash_verify_greedy_static(None, 1, None, 16385, 0, 10, -1, None, None, None, None,
                                         None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    assert b"static scratch limit" in lib.dflash_last_error()
