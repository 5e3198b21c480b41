"""GPU context projection + draft body vs the fp64 oracle, plus the body's structural
guarantees on the GPU (block isolation, strict prefix, no writes to the context K/V, exact
zeros at invalid slots, identical rows for shared sample ids)."""
import numpy as np
import pytest

import dflash_inputs as di
from dflash_testlib import SynthModel, compare_hidden, np_to_device, to_device, tol_for
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu


class Case:
    """One workload's inputs, the GPU outputs, and oracle access to selected blocks."""

    def __init__(self, w: di.Workload, gain_std=0.0, plan=None, mask=None):
        self.w = w
        s = w.shape
        self.model = SynthModel(w, gain_std)
        self.mask = di.gen_mask(w) if mask is None else mask
        self.sids = di.gen_sample_ids(w)
        if plan is None:
            if w.inference:
                a, v, p = di.inference_block_layout(w)
                plan = {"anchors": a, "block_valid": v, "position_ids": p}
            else:
                plan = orc.build_plan(self.mask, self.sids, w.plan_step, w.plan_seed,
                                      w.num_anchors, s.block_size)
        self.plan = plan
        self.emb = di.gen_block_emb(w)
        self.N = plan["anchors"].shape[1]

    def run_gpu(self, emb=None, hidden=None, mask=None, check_cache=False, ctx_len=None,
                f16_layers=False):
        """f16_layers: hand the library fp16 copies of the layer matrices (prepared once,
        DFLASH_FLAG_F16_LAYERS) instead of the bf16 ones it converts inside each call."""
        import torch
        import block_draft_model_proj_gb300 as dflash
        w, s = self.w, self.w.shape
        B, L, N, S = w.batch, w.seq_len, self.N, s.block_size
        cfg = dflash.make_config(s, f16_layers=f16_layers)
        wts = self.model.lib_weights()
        if f16_layers:
            wts = dflash.prepare_f16_layers(wts)
        H = to_device(di.gen_target_hidden(w) if hidden is None else hidden)
        kv = torch.empty((s.num_layers, B, 2, s.num_kv_heads, L, s.head_dim),
                         dtype=dflash.kv_cache_dtype(cfg),
                         device="cuda")
        cl = None if ctx_len is None else np_to_device(np.asarray(ctx_len, np.int32))
        dflash.dflash_project_context(cfg, wts, H, B, L, 0, L, kv, ctx_len=cl)
        del H
        out = torch.full((B, N, S, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
        m = np_to_device(self.mask if mask is None else mask)
        before = kv.clone() if check_cache else None
        dflash.dflash_body_forward(cfg, wts, to_device(self.emb if emb is None else emb),
                                   np_to_device(self.plan["anchors"]),
                                   np_to_device(self.plan["block_valid"]),
                                   np_to_device(self.plan["position_ids"]), m, kv, B, L, N, out)
        dflash.dflash_device_status()
        if check_cache:
            assert torch.equal(before, kv), "the body must not write the context K/V"
        return out.cpu().numpy()

    def oracle_blocks(self, blocks, emb=None, hidden_fn=None, mask=None):
        """blocks: list of (b, k).  Returns {(b, k): [S, D] fp64}."""
        w, s = self.w, self.w.shape
        mask = self.mask if mask is None else mask
        emb = (self.emb if emb is None else emb).f64()
        out = {}
        by_row = {}
        for b, k in blocks:
            by_row.setdefault(b, []).append(k)
        for b, ks in by_row.items():
            need = max(min(int(self.plan["anchors"][b, k]), w.seq_len) for k in ks)
            need = max(need, 1)
            rows = (di.gen_target_hidden_rows(w, b, 0, need) if hidden_fn is None
                    else hidden_fn(b, need))
            kv = orc.project_context_row(s, self.model.top64(), self.model.layer64, rows.f64())
            for k in ks:
                out[(b, k)] = orc.block_forward(
                    s, self.model.top64(), self.model.layer64, emb[b, k],
                    int(self.plan["anchors"][b, k]), self.plan["block_valid"][b, k], mask[b], kv,
                    self.plan["position_ids"][b, k])
        return out

    def compare(self, got, blocks, ref=None):
        ref = self.oracle_blocks(blocks) if ref is None else ref
        g = np.stack([got[b, k] for b, k in blocks])
        r = np.stack([ref[(b, k)] for b, k in blocks])
        v = np.stack([self.plan["block_valid"][b, k] for b, k in blocks])
        return compare_hidden(g, r, v, tol_for(self.w.shape))


def small_bf16_workload():
    """Several tiles in every GEMM dimension plus ragged tails; masks with holes."""
    shape = di.DraftShape(target_hidden=192, num_target_layers=2, hidden=256, num_layers=2,
                          num_heads=4, num_kv_heads=2, head_dim=128, intermediate=392,
                          block_size=4, dtype="bf16")
    return di.Workload("small_bf16", 7, shape, batch=3, seq_len=304, num_anchors=5,
                       padded_rows=((1, 170),), verify_batch=0, vocab=0)


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


@pytest.mark.parametrize("batch", [1, 8])
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
    ks = [int(k) for k in np.argsort(anchors)[:3]]        # shortest prefixes
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
