"""GPU context projection + draft body vs the fp64 oracle, plus the body's structural
guarantees on the GPU (block isolation, strict prefix, no writes to the context K/V, exact
zeros at invalid slots, identical rows for shared sample ids)."""
import numpy as np
import pytest

import dflash_inputs as di
from dflash_testlib import Case, small_bf16_workload
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu


def test_small_bf16_full_parity_with_gains(lib):
    w = small_bf16_workload()
    mask = di.gen_mask(w)
    mask[2, 50:60] = 0              # a hole inside the context
    c = Case(w, gain_std=0.1, mask=mask)
    got = c.run_gpu(check_cache=True)
    blocks = [(b, k) for b in range(w.batch) for k in range(c.N)]
    c.compare(got, blocks)


def test_tiny_f32_config_full_parity(lib):
    w = di.WORKLOADS["tiny_f32"]
    c = Case(w)
    got = c.run_gpu()
    stats = c.compare(got, [(0, k) for k in range(c.N)])
    assert stats["n"] > 0


def test_train_8b_b4_parity(lib):
    w = di.WORKLOADS["train_8b_b4_l2048"]
    c = Case(w)
    got = c.run_gpu(check_cache=True)
    # row 3 is padded to one valid token: no window, every slot exactly zero
    assert np.all(got[3] == 0.0)
    c.compare(got, [(0, k) for k in range(c.N)] + [(2, 0), (2, 1)])


def test_train_8b_b4_parity_with_prepared_f16_layers(lib):
    """The same workload with fp16 copies of the layer matrices prepared once: more than 128
    tokens with fp16 weights take the 128 x 256-tile GEMM instead of the weight-streaming
    one; both meet the bound, and their outputs differ only by accumulation order."""
    w = di.WORKLOADS["train_8b_b4_l2048"]
    c = Case(w)
    got = c.run_gpu(f16_layers=True)
    assert np.all(got[3] == 0.0)
    c.compare(got, [(0, k) for k in range(c.N)] + [(1, 3)])


@pytest.mark.parametrize("batch", [1, 8, 32, 64])
def test_decode_8b_parity(lib, batch):
    w = di.WORKLOADS[f"decode_8b_b{batch}_ctx4096"]
    c = Case(w)
    got = c.run_gpu()
    c.compare(got, [(0, 0)] + ([(batch - 1, 0)] if batch > 1 else []))


def test_longctx_8b_sampled_parity(lib):
    w = di.WORKLOADS["longctx_8b_l32768"]
    c = Case(w)
    got = c.run_gpu()
    anchors = c.plan["anchors"][0]
    # the three shortest prefixes and the longest one (several 4096-key chunks merged by
    # the combine pass)
    ks = [int(k) for k in np.argsort(anchors)[:3]] + [int(np.argmax(anchors))]
    assert int(anchors[ks[-1]]) >= 16384
    c.compare(got, [(0, k) for k in ks])
    assert np.all(np.isfinite(got))


def test_train_8b_b16_sampled_parity_and_shared_rows(lib):
    w = di.WORKLOADS["train_8b_b16_l4096"]
    c = Case(w)
    got = c.run_gpu()
    for grp in w.shared_sid_groups:
        for b in grp[1:]:
            assert np.array_equal(got[b], got[grp[0]]), "rows sharing a sample id must match"
    ks = [int(k) for k in np.argsort(c.plan["anchors"][8])[:2]]
    c.compare(got, [(8, k) for k in ks] + [(0, 0)])


def test_block_isolation_and_strict_prefix_on_gpu(lib):
    """Perturbing other blocks' embeddings, or the target context at/after a block's anchor,
    leaves that block's output bit-identical; perturbing its strict prefix changes it."""
    w = small_bf16_workload()
    c = Case(w)
    base = c.run_gpu()
    b = 0
    k = int(np.argmax(c.plan["anchors"][b]))
    a = int(c.plan["anchors"][b, k])
    assert a > 10
    emb2 = di.Tensor(c.emb.data.copy(), c.emb.dtype)
    rng = np.random.default_rng(0)
    for kk in range(c.N):
        if kk != k:
            emb2.data[b, kk] = di.f32_to_bf16_bits(rng.standard_normal(emb2.data[b, kk].shape)
                                                   .astype(np.float32))
    H = di.gen_target_hidden(w)
    H2 = di.Tensor(H.data.copy(), H.dtype)
    H2.data[b, a:] = di.f32_to_bf16_bits(
        5 * rng.standard_normal(H2.data[b, a:].shape).astype(np.float32))
    got = c.run_gpu(emb=emb2, hidden=H2)
    assert np.array_equal(got[b, k], base[b, k])
    H3 = di.Tensor(H.data.copy(), H.dtype)
    H3.data[b, a - 1] = di.f32_to_bf16_bits(
        5 * rng.standard_normal(H3.data[b, a - 1].shape).astype(np.float32))
    got3 = c.run_gpu(hidden=H3)
    assert not np.array_equal(got3[b, k], base[b, k])


def _ctx_len_of(plan):
    a, v = plan["anchors"], plan["block_valid"].astype(bool).any(axis=-1)
    return [max([int(x) for x, ok in zip(a[b], v[b]) if ok] + [0]) for b in range(a.shape[0])]


@pytest.mark.parametrize("wname", ["small", "train_8b_b4_l2048"])
def test_skipping_unread_context_and_empty_slot_tiles_changes_nothing(lib, wname):
    """Context rows no block reads (c >= ctx_len) and 128-slot tiles without a valid slot are
    skipped by the projections; the body's outputs must be bit-identical to the full run."""
    w = small_bf16_workload() if wname == "small" else di.WORKLOADS[wname]
    c = Case(w)
    full = c.run_gpu()
    cl = _ctx_len_of(c.plan)
    assert min(cl) < w.seq_len
    skipped = c.run_gpu(ctx_len=cl)
    assert np.array_equal(full, skipped)


def test_out_of_range_position_reports_device_check(lib):
    import block_draft_model_proj_gb300 as dflash
    w = small_bf16_workload()
    c = Case(w)
    c.plan = {k: v.copy() for k, v in c.plan.items()}
    b, k = 0, 0
    assert c.plan["block_valid"][b, k, 0]
    c.plan["position_ids"][b, k, 0] = w.seq_len + 10_000   # beyond L + S
    with pytest.raises(RuntimeError, match="index check"):
        c.run_gpu()
    dflash.dflash_device_status(reset=True)


def test_prepared_f16_layer_weights_match_in_call_conversion(lib):
    """Layer matrices converted once (DFLASH_FLAG_F16_LAYERS) and converted inside each call
    feed the same GEMMs: the outputs are bit-identical."""
    c = Case(small_bf16_workload())
    assert np.array_equal(c.run_gpu(), c.run_gpu(f16_layers=True))


def test_activation_outside_fp16_range_is_reported(lib):
    """A gain of 1e5 on the first input norm pushes the normalised activations past the fp16
    range: the device status reports DFLASH_ERR_RANGE."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    c = Case(small_bf16_workload())
    g = c.model.dev_layers[0]["g_in"]
    c.model.dev_layers[0]["g_in"] = torch.full_like(g, 1e5)
    try:
        with pytest.raises(RuntimeError, match="fp16 range"):
            c.run_gpu()
    finally:
        c.model.dev_layers[0]["g_in"] = g
        dflash.dflash_device_status(reset=True)
