"""The inference cache on the GPU: a body reading a cache longer than its context, and the
cache update of a generation cycle ("DFlash: drafting, verification, and speed", One
DFlash generation cycle: only the anchor and the accepted proposals stay in a cache; the
draft and target caches stay aligned), checked against the oracle's commit rule and
context projection."""
import numpy as np
import pytest

import dflash_inputs as di
from dflash_testlib import SynthModel, compare_hidden, np_to_device, to_device, tol_for
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu

BF16 = di.DraftShape(target_hidden=128, num_target_layers=2, hidden=256, num_layers=2,
                     num_heads=4, num_kv_heads=2, head_dim=128, intermediate=384, block_size=4,
                     dtype="bf16")
F32 = di.DraftShape(target_hidden=64, num_target_layers=2, hidden=128, num_layers=2,
                    num_heads=4, num_kv_heads=2, head_dim=64, intermediate=256, block_size=4,
                    dtype="f32")


def _hidden(w, b, P, tag, shape):
    """Synthetic target hidden states of P positions for row b (stream `tag`)."""
    rng = np.random.default_rng([w.data_seed, 77, tag, b])
    x = rng.standard_normal((P, shape.concat_width), dtype=np.float32)
    return di.Tensor(di.f32_to_bf16_bits(x) if shape.dtype == "bf16" else x, shape.dtype)


def _stack(ts):
    return di.Tensor(np.stack([t.data for t in ts]), ts[0].dtype)


class Cycle:
    """A context of L0 positions per request, then appends of verified blocks."""

    def __init__(self, shape, B=3, L0=100, L_cache=264, index=40):
        import torch
        import block_draft_model_proj_gb300 as dflash
        self.dflash, self.torch = dflash, torch
        self.shape, self.B, self.L0, self.L_cache = shape, B, L0, L_cache
        self.w = di.Workload("cycle", index, shape, batch=B, seq_len=L_cache, num_anchors=1)
        self.model = SynthModel(self.w)
        self.cfg = dflash.make_config(shape)
        self.ctx = [_hidden(self.w, b, L0, 0, shape) for b in range(B)]

    def run(self, blocks, accepted_lists, emb):
        """blocks: list over cycles of [B] lists of Tensors [S, W]; accepted_lists: list
        over cycles of int arrays [B] or None.  Returns (out, cache_len, kv)."""
        torch, dflash, s = self.torch, self.dflash, self.shape
        B, L_cache, S = self.B, self.L_cache, s.block_size
        wts = self.model.lib_weights()
        kv = torch.zeros((s.num_layers, B, 2, s.num_kv_heads, L_cache, s.head_dim),
                         dtype=dflash.kv_cache_dtype(self.cfg), device="cuda")
        dflash.dflash_project_context(self.cfg, wts, to_device(_stack(self.ctx)), B, self.L0, 0,
                                      L_cache, kv)
        cache_len = torch.full((B,), self.L0, dtype=torch.int32, device="cuda")
        for blk, acc in zip(blocks, accepted_lists):
            a = None if acc is None else np_to_device(np.asarray(acc, np.int32))
            dflash.dflash_append_context(self.cfg, wts, to_device(_stack(blk)), B, S, a,
                                         cache_len, L_cache, kv)
        lens = cache_len.cpu().numpy()
        anchors = lens.reshape(B, 1).astype(np.int32)
        pos = (anchors[:, :, None] + np.arange(S, dtype=np.int32)).astype(np.int32)
        valid = np.ones((B, 1, S), np.uint8)
        mask = np.ones((B, L_cache), np.uint8)
        out = torch.full((B, 1, S, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
        dflash.dflash_body_forward(self.cfg, wts, to_device(emb), np_to_device(anchors),
                                   np_to_device(valid), np_to_device(pos), np_to_device(mask),
                                   kv, B, L_cache, 1, out)
        dflash.dflash_device_status()
        return out.cpu().numpy(), lens, kv

    def oracle(self, blocks, accepted_lists, emb):
        s, S = self.shape, self.shape.block_size
        outs = []
        for b in range(self.B):
            hid = self.ctx[b].f64()
            for blk, acc in zip(blocks, accepted_lists):
                hid = orc.commit_verified(hid, blk[b].f64(), S - 1 if acc is None else int(acc[b]))
            kvr = orc.project_context_row(s, self.model.top64(), self.model.layer64, hid)
            n = hid.shape[0]
            outs.append(orc.block_forward(s, self.model.top64(), self.model.layer64,
                                          emb.f64()[b, 0], n, np.ones(S, np.uint8),
                                          np.ones(self.L_cache, np.uint8), kvr,
                                          n + np.arange(S)))
        return np.stack(outs)[:, None], [h for h in outs]


def _blocks(cyc, tags):
    return [[_hidden(cyc.w, b, cyc.shape.block_size, t, cyc.shape) for b in range(cyc.B)]
            for t in tags]


def _emb(cyc):
    rng = np.random.default_rng(cyc.w.data_seed + 5)
    x = rng.standard_normal((cyc.B, 1, cyc.shape.block_size, cyc.shape.hidden), dtype=np.float32)
    return di.Tensor(di.f32_to_bf16_bits(x) if cyc.shape.dtype == "bf16" else x,
                     cyc.shape.dtype)


@pytest.mark.parametrize("shape", [BF16, F32], ids=["bf16", "f32"])
def test_two_cycles_of_append_then_draft_match_the_oracle(lib, shape):
    cyc = Cycle(shape)
    blocks = _blocks(cyc, [1, 2])
    accepted = [np.array([0, 3, 1]), np.array([2, 0, 3])]
    emb = _emb(cyc)
    got, lens, _ = cyc.run(blocks, accepted, emb)
    assert list(lens) == [100 + 1 + 3, 100 + 4 + 1, 100 + 2 + 4]
    ref, _ = cyc.oracle(blocks, accepted, emb)
    compare_hidden(got, ref, np.ones(got.shape[:-1], bool), tol_for(shape))


def test_rejected_positions_never_reach_the_next_block(lib):
    """Rollback: the hidden states of rejected proposals (and their suffix) may be anything;
    the cache below the committed length and the next block's output are bit-identical."""
    cyc = Cycle(BF16, index=41)
    blocks = _blocks(cyc, [1, 2])
    accepted = [np.array([0, 3, 1]), np.array([2, 0, 2])]
    emb = _emb(cyc)
    got, lens, kv = cyc.run(blocks, accepted, emb)
    rng = np.random.default_rng(9)
    noisy = []
    for blk, acc in zip(blocks, accepted):
        nb = []
        for b, t in enumerate(blk):
            d = t.data.copy()
            tail = d[int(acc[b]) + 1:]
            tail[...] = di.f32_to_bf16_bits(
                30 * rng.standard_normal(tail.shape).astype(np.float32))
            nb.append(di.Tensor(d, t.dtype))
        noisy.append(nb)
    got2, lens2, kv2 = cyc.run(noisy, accepted, emb)
    assert np.array_equal(lens, lens2)
    assert np.array_equal(got, got2)
    k1, k2 = kv.cpu(), kv2.cpu()
    for b in range(cyc.B):
        n = int(lens[b])
        assert np.array_equal(k1[:, b, 0, :, :n].numpy(), k2[:, b, 0, :, :n].numpy())
        assert np.array_equal(k1[:, b, 1].reshape(-1, 128, cyc.L_cache)[:, :, :n].numpy(),
                              k2[:, b, 1].reshape(-1, 128, cyc.L_cache)[:, :, :n].numpy())
    # committing the whole block instead (accepted = NULL) changes the next block
    got3, lens3, _ = cyc.run(noisy, [None, None], emb)
    assert list(lens3) == [100 + 8] * cyc.B
    assert not np.array_equal(got3, got)


def test_cycle_chained_through_device_verification(lib):
    """accepted comes straight from dflash_verify_greedy on the device (no host round trip)
    and drives the append; the cache lengths advance by accepted + 1."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    cyc = Cycle(BF16, index=42)
    S = cyc.shape.block_size
    vw = di.scaled(cyc.w, verify_batch=cyc.B, vocab=3000)
    vi = di.gen_verify(vw)
    em = torch.empty((cyc.B, S), dtype=torch.int32, device="cuda")
    ne = torch.empty((cyc.B,), dtype=torch.int32, device="cuda")
    ac = torch.empty_like(ne)
    dflash.dflash_verify_greedy(to_device(vi.logits), dflash.DFLASH_DTYPE_BF16,
                                np_to_device(vi.draft), cyc.B, S - 1, vi.logits.shape[2], -1, em,
                                ne, ac)
    wts = cyc.model.lib_weights()
    kv = torch.zeros((cyc.shape.num_layers, cyc.B, 2, cyc.shape.num_kv_heads, cyc.L_cache, 128),
                     dtype=torch.float16, device="cuda")
    cache_len = torch.full((cyc.B,), cyc.L0, dtype=torch.int32, device="cuda")
    blk = _blocks(cyc, [3])[0]
    dflash.dflash_append_context(cyc.cfg, wts, to_device(_stack(blk)), cyc.B, S, ac, cache_len,
                                 cyc.L_cache, kv)
    dflash.dflash_device_status()
    assert np.array_equal(cache_len.cpu().numpy(), cyc.L0 + vi.planted_prefix + 1)


def test_append_past_the_cache_end_is_rejected_on_the_device(lib):
    import torch
    import block_draft_model_proj_gb300 as dflash
    cyc = Cycle(BF16, B=2, index=43)
    S = cyc.shape.block_size
    wts = cyc.model.lib_weights()
    kv = torch.zeros((cyc.shape.num_layers, 2, 2, cyc.shape.num_kv_heads, cyc.L_cache, 128),
                     dtype=torch.float16, device="cuda")
    cache_len = torch.tensor([cyc.L_cache - 2, 10], dtype=torch.int32, device="cuda")
    blk = _blocks(cyc, [4])[0]
    try:
        with pytest.raises(RuntimeError, match="index check"):
            dflash.dflash_append_context(cyc.cfg, wts, to_device(_stack(blk)), 2, S, None,
                                         cache_len, cyc.L_cache, kv)
            dflash.dflash_device_status()
    finally:
        dflash.dflash_device_status(reset=True)
    # the overflowing row keeps its length; the other one commits its 4 positions
    assert list(cache_len.cpu().numpy()) == [cyc.L_cache - 2, 14]


def test_body_reads_a_cache_longer_than_its_context(lib):
    """A context of 200 positions in planes of 264: the body runs with L = 264 (the planes'
    stride) and blocks anchored anywhere up to right after the context."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    s, B, L0, Lc = BF16, 2, 200, 264
    w = di.Workload("longcache", 44, s, batch=B, seq_len=Lc, num_anchors=3)
    model = SynthModel(w)
    cfg = dflash.make_config(s)
    H = di.Tensor(di.gen_target_hidden(w).data[:, :L0].copy(), "bf16")
    kv = torch.zeros((s.num_layers, B, 2, s.num_kv_heads, Lc, 128), dtype=torch.float16,
                     device="cuda")
    dflash.dflash_project_context(cfg, model.lib_weights(), to_device(H), B, L0, 0, Lc, kv)
    anchors = np.array([[3, 120, 200], [57, 199, 200]], np.int32)
    S = s.block_size
    pos = (anchors[:, :, None] + np.arange(S)).astype(np.int32)
    valid = np.ones((B, 3, S), np.uint8)
    mask = np.zeros((B, Lc), np.uint8)
    mask[:, :L0] = 1
    emb = di.gen_block_emb(w)
    out = torch.full((B, 3, S, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    dflash.dflash_body_forward(cfg, model.lib_weights(), to_device(emb), np_to_device(anchors),
                               np_to_device(valid), np_to_device(pos), np_to_device(mask), kv, B,
                               Lc, 3, out)
    dflash.dflash_device_status()
    got = out.cpu().numpy()
    ref = np.zeros_like(got, dtype=np.float64)
    for b in range(B):
        kvr = orc.project_context_row(s, model.top64(), model.layer64, H.f64()[b])
        for k in range(3):
            ref[b, k] = orc.block_forward(s, model.top64(), model.layer64, emb.f64()[b, k],
                                          int(anchors[b, k]), valid[b, k], mask[b], kvr, pos[b, k])
    compare_hidden(got, ref, valid.astype(bool), tol_for(s))
