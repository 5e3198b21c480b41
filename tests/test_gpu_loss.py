"""The draft loss on the GPU (dflash_decayed_ce_loss) vs the fp64 oracle: the frozen
lm_head's cross-entropy against the ground-truth tokens over loss_mask with exponential
positional decay ("DFlash", How it works, Loss; "DFlash Draft Body", How It Works step 4).

The GPU rounds the hidden states to bf16 for the lm_head GEMM (the lm_head is the target's
own bf16 matrix); the per-slot cross-entropy is held to the body's bound (max-abs 2e-2,
relative RMS 5e-3) and the loss to 1e-3 relative."""
import numpy as np
import pytest

import dflash_inputs as di
from dflash_testlib import np_to_device, to_device
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu


def _hidden(w, seed):
    """Stand-in for the body's output: unit-RMS rows (the final norm's scale), fp32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((w.batch, w.num_anchors, w.shape.block_size, w.shape.hidden),
                               dtype=np.float32)


def _run(hidden, lm, targets, mask, S, V, decay):
    import torch
    import block_draft_model_proj_gb300 as dflash
    T = int(np.prod(mask.shape))
    D = hidden.shape[-1]
    ce = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    dflash.dflash_decayed_ce_loss(np_to_device(hidden.reshape(T, D)), to_device(lm),
                                  np_to_device(targets.reshape(T)), np_to_device(mask.reshape(T)),
                                  T, S, D, V, decay, ce, loss)
    dflash.dflash_device_status()
    return float(loss.cpu()[0]), ce.cpu().numpy().reshape(mask.shape)


def _check(w, V, decay, seed):
    s = w.shape
    mask_in = di.gen_mask(w)
    plan = orc.build_plan(mask_in, di.gen_sample_ids(w), 0, w.plan_seed, w.num_anchors,
                          s.block_size)
    lm_mask = plan["loss_mask"]
    hidden = _hidden(w, seed)
    lm = di.gen_lm_head(w, V)
    targets = di.gen_targets(w, V)
    loss, ce = _run(hidden, lm, targets, lm_mask, s.block_size, V, decay)
    ref_loss, ref_ce = orc.decayed_ce_loss(hidden.astype(np.float64), lm.f64(), targets, lm_mask,
                                           decay)
    m = lm_mask.astype(bool)
    assert np.all(ce[~m] == 0.0)
    err = ce[m] - ref_ce[m]
    assert np.all(np.isfinite(ce))
    assert float(np.max(np.abs(err))) <= 2e-2
    assert float(np.sqrt(np.sum(err ** 2) / np.sum(ref_ce[m] ** 2))) <= 5e-3
    assert abs(loss - ref_loss) <= 1e-3 * abs(ref_loss)
    return loss, ce, hidden, lm, targets, lm_mask


def test_small_ragged_vocab(lib):
    shape = di.DraftShape(target_hidden=128, num_target_layers=2, hidden=256, num_layers=1,
                          num_heads=4, num_kv_heads=2, head_dim=128, intermediate=256,
                          block_size=4, dtype="bf16")
    w = di.Workload("loss_small", 50, shape, batch=3, seq_len=300, num_anchors=7,
                    padded_rows=((2, 60),))
    _check(w, 1000, 2.0, 1)


def test_full_vocab_training_shape(lib):
    """B=4 L=2048, 8 blocks of 16 slots, D = 4096, the full 151936-entry vocab."""
    w = di.WORKLOADS["train_8b_b4_l2048"]
    loss, ce, hidden, lm, targets, mask = _check(w, 151936, 4.0, 2)
    # deterministic, and slots outside the loss mask do not matter
    h2 = hidden.copy()
    h2[~mask.astype(bool)] = 50.0
    t2 = targets.copy()
    t2[~mask.astype(bool)] = -7
    loss2, ce2 = _run(h2, lm, t2, mask, w.shape.block_size, 151936, 4.0)
    assert loss2 == loss and np.array_equal(ce2, ce)


def test_target_outside_the_vocab_reports_device_check(lib):
    import block_draft_model_proj_gb300 as dflash
    shape = di.DraftShape(target_hidden=128, num_target_layers=2, hidden=128, num_layers=1,
                          num_heads=4, num_kv_heads=2, head_dim=128, intermediate=256,
                          block_size=4, dtype="bf16")
    w = di.Workload("loss_bad", 51, shape, batch=1, seq_len=64, num_anchors=2)
    mask = np.ones((1, 2, 4), np.uint8)
    mask[:, :, 0] = 0
    targets = np.zeros((1, 2, 4), np.int32)
    targets[0, 1, 2] = 500
    try:
        with pytest.raises(RuntimeError, match="index check"):
            _run(_hidden(w, 3), di.gen_lm_head(w, 300), targets, mask, 4, 300, 1.0)
    finally:
        dflash.dflash_device_status(reset=True)
