"""GPU anchor plan vs the oracle: bit-exact anchors, block_valid, loss_mask, position_ids."""
import os

import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_plan(mask, sids, step, seed, N, S):
    import torch
    import block_draft_model_proj_gb300 as dflash
    B, L = mask.shape
    dm = torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).cuda()
    ds = torch.from_numpy(np.ascontiguousarray(sids, np.int64)).cuda()
    anchors = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    bv = torch.full((B, N, S), 9, dtype=torch.uint8, device="cuda")
    lm = torch.full((B, N, S), 9, dtype=torch.uint8, device="cuda")
    pid = torch.full((B, N, S), -7, dtype=torch.int32, device="cuda")
    cl = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    dflash.dflash_plan(dm, ds, step, seed, N, S, anchors, bv, lm, pid, ctx_len=cl)
    dflash.dflash_device_status()
    return {"anchors": anchors.cpu().numpy(), "block_valid": bv.cpu().numpy(),
            "loss_mask": lm.cpu().numpy(), "position_ids": pid.cpu().numpy(),
            "ctx_len": cl.cpu().numpy()}


def expected_ctx_len(ref):
    """Largest anchor of a block with a valid slot, per row (0 if none), from the oracle plan."""
    a, v = ref["anchors"], ref["block_valid"].astype(bool).any(axis=-1)
    return np.array([max([int(x) for x, ok in zip(a[b], v[b]) if ok] + [0])
                     for b in range(a.shape[0])], np.int32)


def assert_same_plan(got, ref):
    for k in ("anchors", "block_valid", "loss_mask", "position_ids"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["ctx_len"], expected_ctx_len(ref))


@pytest.mark.parametrize("name", ["plan_small.txt", "plan_shared_sid.txt"])
def test_golden_plans(lib, name):
    from test_oracle_plan import _read_plan_golden
    mask, sids, step, seed, N, S, anchors = _read_plan_golden(os.path.join(GOLDEN, name))
    got = gpu_plan(mask, sids, step, seed, N, S)
    assert np.array_equal(got["anchors"], anchors)
    assert_same_plan(got, orc.build_plan(mask, sids, step, seed, N, S))


@pytest.mark.parametrize("wname", ["tiny_f32", "train_8b_b4_l2048", "longctx_8b_l32768",
                                   "train_8b_b16_l4096"])
def test_workload_plans(lib, wname):
    w = di.WORKLOADS[wname]
    mask, sids = di.gen_mask(w), di.gen_sample_ids(w)
    for step in (w.plan_step, w.plan_step + 1):
        got = gpu_plan(mask, sids, step, w.plan_seed, w.num_anchors, w.shape.block_size)
        ref = orc.build_plan(mask, sids, step, w.plan_seed, w.num_anchors, w.shape.block_size)
        assert_same_plan(got, ref)
    if w.shared_sid_groups:
        for grp in w.shared_sid_groups:
            for b in grp:
                assert np.array_equal(got["anchors"][b], got["anchors"][grp[0]])
    if w.padded_rows:
        for row, _ in w.padded_rows:
            assert np.all(got["anchors"][row] == -1)
            assert np.all(got["loss_mask"][row] == 0)


@pytest.mark.parametrize("trial", range(6))
def test_random_masks_and_shared_ids(lib, trial):
    rng = np.random.default_rng(500 + trial)
    B = int(rng.integers(1, 9))
    L = int(rng.integers(1, 3000))
    N = int(rng.integers(1, 70))
    S = int(rng.integers(1, 20))
    mask = (rng.random((B, L)) < rng.uniform(0.3, 1.0)).astype(np.uint8)
    for b in range(B):
        mask[b, int(rng.integers(0, L + 1)):] = 0
    sids = rng.integers(0, max(1, B // 2), size=B).astype(np.int64)
    seed = int(rng.integers(0, 2 ** 63))
    step = int(rng.integers(-5, 10 ** 9))
    got = gpu_plan(mask, sids, step, seed, N, S)
    assert_same_plan(got, orc.build_plan(mask, sids, step, seed, N, S))


def test_many_anchors_take_every_candidate(lib):
    mask = np.ones((2, 50), np.uint8)
    mask[1, 10:] = 0
    got = gpu_plan(mask, np.array([1, 2]), 3, 4, 1024, 16)
    assert list(got["anchors"][0][:49]) == list(range(49))
    assert np.all(got["anchors"][0][49:] == -1)
    assert list(got["anchors"][1][:9]) == list(range(9))
    assert_same_plan(got, orc.build_plan(mask, np.array([1, 2]), 3, 4, 1024, 16))


def test_plan_is_deterministic_across_calls(lib):
    w = di.WORKLOADS["train_8b_b16_l4096"]
    mask, sids = di.gen_mask(w), di.gen_sample_ids(w)
    a = gpu_plan(mask, sids, 0, 1, 32, 16)
    b = gpu_plan(mask, sids, 0, 1, 32, 16)
    assert_same_plan(a, b)
