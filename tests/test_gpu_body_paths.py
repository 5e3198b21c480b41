"""Context projection + draft body vs the fp64 oracle on every dispatch path the library
takes, at sizes the oracle finishes in seconds ("DFlash Draft Body", How It Works steps 3
and 4; "DFlash", How it works: dual-source K/V).

The library picks its kernels from the sizes of a call, so each case below is chosen to
land on one side of a boundary:

* context rows B*L at most 512 or more (the context K/V projection reads fp16 copies of
  bf16 layer weights either way);
* attention with one key chunk (the unit normalises its own rows) or several chunks
  merged by the combine pass: L <= 256 vs above, and long contexts with many chunks;
* query tiles holding 1, 2, 4, 16 or 64 blocks (S * Hq/Hkv = 128, 64, 32, 8, 2 rows per
  block), with N not a multiple of the blocks per tile;
* draft slots T = B*N*S of 16, 24, 60, 128 (weight-streaming GEMM, K-split gate/up),
  136 and 512 (weight-streaming GEMM, SwiGLU epilogue), 520 (128 x 256-tile GEMM on fp16
  copies made in the call), and fp16 weights held by the caller;
* matrix widths that are not multiples of 64;
* explicit anchors at the edges: anchor 0 (no context key), the last candidate L - 2,
  a mask hole inside the 16-key group at the prefix boundary, fewer candidates than N.

Every case compares every block with the oracle element by element (max-abs 2e-2 and
relative RMS 5e-3 over valid slots, exact zeros elsewhere).
"""
import numpy as np
import pytest

import dflash_inputs as di
from dflash_testlib import Case

pytestmark = pytest.mark.gpu

BASE = dict(target_hidden=128, num_target_layers=2, hidden=256, num_layers=2, num_heads=4,
            num_kv_heads=2, head_dim=128, intermediate=384, block_size=4, dtype="bf16")


def workload(name, index=20, shape=None, **wk):
    s = dict(BASE)
    s.update(shape or {})
    kw = dict(batch=2, seq_len=160, num_anchors=3, padded_rows=((1, 90),))
    kw.update(wk)
    return di.Workload(name, index, di.DraftShape(**s), **kw)


def all_blocks(c):
    return [(b, k) for b in range(c.w.batch) for k in range(c.N)]


def check(w, gpu_plan=True, f16_layers=False, plan=None, mask=None):
    c = Case(w, plan=plan, mask=mask)
    got = c.run_gpu(gpu_plan=gpu_plan and plan is None and mask is None, f16_layers=f16_layers,
                    check_cache=True)
    stats = c.compare(got, all_blocks(c))
    assert stats["n"] > 0
    return c, got


def test_smoke_shape_with_device_plan(lib):
    """The exact shape of the package's smoke check, the device plan chained into the body
    (160 context rows per row: the context K/V projection of at most 512 rows)."""
    check(di.smoke_workload())


CONTEXT_LENGTHS = [128, 160, 256, 264, 304, 1000, 4104]


@pytest.mark.parametrize("L", CONTEXT_LENGTHS)
def test_context_lengths(lib, L):
    # <= 256: one key chunk; above: several chunks and the combine pass
    check(workload(f"ctx_{L}", seq_len=L, padded_rows=((1, L * 9 // 16),)))


def test_long_context_many_chunks(lib):
    check(workload("ctx_20000", index=21, batch=1, seq_len=20000, num_anchors=6,
                   padded_rows=()))


# (S, Hq, Hkv) -> rows per block S * Hq/Hkv and blocks per 128-row query tile
TILE_PACKINGS = [(16, 8, 1, 1), (16, 8, 2, 2), (8, 8, 2, 4), (4, 4, 2, 16), (2, 4, 4, 64)]


@pytest.mark.parametrize("S,Hq,Hkv,bpt", TILE_PACKINGS)
@pytest.mark.parametrize("L", [160, 304])
def test_blocks_per_query_tile(lib, S, Hq, Hkv, bpt, L):
    assert 128 // (S * Hq // Hkv) == bpt
    check(workload(f"pack_{S}_{Hq}_{Hkv}", index=22, shape=dict(block_size=S, num_heads=Hq,
                                                                 num_kv_heads=Hkv),
                   seq_len=L, num_anchors=bpt + 1 if bpt < 16 else 5))


# (B, N) with S = 4: T = B * N * 4 draft slots
TOKEN_COUNTS = [(1, 4), (2, 3), (3, 5), (4, 8), (2, 17), (4, 32), (2, 65)]


@pytest.mark.parametrize("B,N", TOKEN_COUNTS)
def test_token_counts(lib, B, N):
    check(workload(f"tok_{B * N * 4}", index=23, batch=B, num_anchors=N, seq_len=304,
                   padded_rows=((B - 1, 200),)))


@pytest.mark.parametrize("B,N", [(2, 17), (2, 65)])
def test_token_counts_with_fp16_layers_held(lib, B, N):
    check(workload(f"tok16_{B * N * 4}", index=23, batch=B, num_anchors=N, seq_len=304,
                   padded_rows=((B - 1, 200),)), f16_layers=True)


@pytest.mark.parametrize("shape", [dict(target_hidden=136), dict(intermediate=392),
                                   dict(hidden=320), dict(num_layers=3, intermediate=200)])
def test_ragged_widths(lib, shape):
    check(workload("ragged", index=24, shape=shape, seq_len=264))


def plan_from_anchors(mask, anchors, S):
    """Block validity and positions of explicitly chosen anchors, by the plan's own rule:
    slot j of the block anchored at a sits at position a + j and is valid when positions a
    and a + j are both valid ("DFlash Draft Body", How It Works steps 1 and 4)."""
    B, N = anchors.shape
    L = mask.shape[1]
    valid = np.zeros((B, N, S), np.uint8)
    pos = np.full((B, N, S), -1, np.int32)
    for b in range(B):
        for k in range(N):
            a = int(anchors[b, k])
            if a < 0:
                continue
            for j in range(S):
                pos[b, k, j] = a + j
                ok = a + j < L and mask[b, a] != 0 and mask[b, a + j] != 0
                valid[b, k, j] = 1 if ok else 0
    return {"anchors": anchors.astype(np.int32), "block_valid": valid, "position_ids": pos}


def test_edge_anchors(lib):
    """Anchor 0 reads no context key; anchor L - 2 is the last candidate (its tail slots
    past L are invalid); a mask hole straddles the prefix boundary inside one 16-key group;
    a row with fewer candidates than N has empty slots (-1) at the end."""
    w = workload("edges", index=25, batch=3, seq_len=264, num_anchors=4, padded_rows=())
    L = w.seq_len
    mask = np.ones((3, L), np.uint8)
    mask[1, 117:123] = 0           # anchor 123: keys 117..122 excluded, group 112..127
    mask[1, 130:131] = 0
    mask[2, 6:] = 0                # 5 candidates 0..4 ... take 3 of them, one slot empty
    anchors = np.array([[0, 1, 200, L - 2],
                        [16, 123, 127, 128],
                        [0, 2, 4, -1]], np.int32)
    plan = plan_from_anchors(mask, anchors, w.shape.block_size)
    c, got = check(w, plan=plan, mask=mask)
    assert np.all(got[2, 3] == 0.0)
    assert plan["block_valid"][0, 3, 2:].sum() == 0   # past L


def test_every_slot_invalid_in_a_row(lib):
    """A row whose mask has a single valid token has no window: all of its slots are
    exactly zero and the other rows are unaffected."""
    check(workload("nowin", index=26, batch=3, seq_len=160, num_anchors=4,
                   padded_rows=((0, 1),)))


@pytest.fixture
def fused_epilogues(lib):
    """Every projection on the 128 x 256-tile GEMM uses the fused epilogues (Q/K RoPE and the
    attention layouts from the QKV projection, the residual add from O and down); at these
    sizes the library would otherwise pick a K-split and the row passes."""
    import block_draft_model_proj_gb300 as dflash
    dflash.dflash_testing_fused_epilogues(1)
    yield
    dflash.dflash_testing_fused_epilogues(0)


# (B, N, S, Hq, Hkv, padded rows, fp16 layers held): slots T = B*N*S above 128 (fp16 held) or
# 512 (bf16 converted in the call) run on the 128 x 256-tile GEMM.  N*S not a multiple of 8
# leaves pad columns in V^T; a row with a single valid token makes whole 128-slot tiles
# invalid (skipped by the GEMM, zeroed once per call); T not a multiple of 128 is ragged.
FUSED_CASES = [
    (2, 65, 4, 4, 2, ((1, 200),), True),     # T = 520, N*S = 260 (pad 4)
    (2, 65, 4, 4, 2, ((1, 200),), False),    # the same with bf16 weights (converted)
    (3, 64, 4, 4, 2, ((0, 1),), False),      # row 0 invalid: tiles 0, 1 skipped
    (2, 17, 16, 8, 2, ((1, 150),), True),    # 4 blocks per query tile, T = 544
    (3, 33, 4, 8, 8, ((2, 100),), True),     # Hq = Hkv: 24 heads, N*S = 132 (pad 4)
]


@pytest.mark.parametrize("B,N,S,Hq,Hkv,pad,f16", FUSED_CASES)
def test_fused_epilogues(lib, fused_epilogues, B, N, S, Hq, Hkv, pad, f16):
    check(workload(f"fused_{B}_{N}_{S}_{Hq}_{Hkv}", index=27,
                   shape=dict(block_size=S, num_heads=Hq, num_kv_heads=Hkv),
                   batch=B, num_anchors=N, seq_len=304, padded_rows=pad), f16_layers=f16)
