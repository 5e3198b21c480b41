"""Shared test plumbing: seeded inputs on the device, fp64 views for the oracle, comparisons.

Both sides get the same seeded inputs from dflash_inputs; nothing here computes any part of
the method.
"""
from __future__ import annotations

import numpy as np

import dflash_inputs as di
from oracle import dflash_oracle as orc

# bf16 body tolerance (the stated bound) and the fp32 configuration's bound
TOL_BF16 = {"max_abs": 2e-2, "rel_rms": 5e-3}
TOL_F32 = {"max_abs": 1e-4, "rel_rms": 1e-4}


def tol_for(shape) -> dict:
    return TOL_BF16 if shape.dtype == "bf16" else TOL_F32


def to_device(t: di.Tensor, device="cuda"):
    import torch
    if t.dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).to(device).view(
            torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(t.data)).to(device)


def np_to_device(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class SynthModel:
    """Synthetic draft weights of one workload: device tensors + lazy fp64 copies."""

    def __init__(self, w: di.Workload, gain_std: float = 0.0, device="cuda", need_device=True):
        self.w = w
        self.shape = w.shape
        self.gain_std = gain_std
        self._top = di.gen_top_weights(w, gain_std)
        self._layers = [di.gen_layer_weights(w, l, gain_std) for l in range(w.shape.num_layers)]
        self._f64_layers = {}
        self._f64_top = None
        self.dev_top = self.dev_layers = None
        if need_device:
            self.dev_top = {k: to_device(v, device) for k, v in self._top.items()}
            self.dev_layers = [{k: to_device(v, device) for k, v in lw.items()} for lw in self._layers]

    def top64(self) -> dict:
        if self._f64_top is None:
            self._f64_top = {k: v.f64() for k, v in self._top.items()}
        return self._f64_top

    def layer64(self, l: int) -> dict:
        if l not in self._f64_layers:
            self._f64_layers[l] = {k: v.f64() for k, v in self._layers[l].items()}
        return self._f64_layers[l]

    def lib_weights(self):
        import block_draft_model_proj_gb300 as dflash
        return dflash.Weights(self.dev_top, self.dev_layers)


def compare_hidden(got: np.ndarray, ref: np.ndarray, valid: np.ndarray, tol: dict) -> dict:
    """got/ref [..., D] over block slots; valid [...] bool.  Invalid slots must be exactly 0."""
    valid = valid.astype(bool)
    assert np.all(got[~valid] == 0.0), "invalid slots must be exactly zero"
    g, r = got[valid].astype(np.float64), ref[valid]
    if g.size == 0:
        return {"max_abs": 0.0, "rel_rms": 0.0, "n": 0}
    err = g - r
    stats = {"max_abs": float(np.max(np.abs(err))),
             "rel_rms": float(np.sqrt(np.sum(err * err) / max(np.sum(r * r), 1e-300))),
             "n": int(valid.sum())}
    print(f"parity: max_abs={stats['max_abs']:.3e} rel_rms={stats['rel_rms']:.3e} "
          f"over {stats['n']} slots")
    assert np.all(np.isfinite(g))
    assert stats["max_abs"] <= tol["max_abs"], stats
    assert stats["rel_rms"] <= tol["rel_rms"], stats
    return stats


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
                f16_layers=False, gpu_plan=False):
        """f16_layers: hand the library fp16 copies of the layer matrices (prepared once,
        DFLASH_FLAG_F16_LAYERS) instead of the bf16 ones it converts inside each call.
        gpu_plan: the body reads the plan dflash_plan writes on the device (as a caller
        chains them), checked bit for bit against the oracle plan first."""
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
        if gpu_plan:
            assert mask is None, "the device plan is drawn from the case's own mask"
            plan = {"anchors": torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    "block_valid": torch.empty((B, N, S), dtype=torch.uint8, device="cuda"),
                    "loss_mask": torch.empty((B, N, S), dtype=torch.uint8, device="cuda"),
                    "position_ids": torch.empty((B, N, S), dtype=torch.int32, device="cuda")}
            dflash.dflash_plan(m, np_to_device(self.sids), w.plan_step, w.plan_seed, N, S,
                               plan["anchors"], plan["block_valid"], plan["loss_mask"],
                               plan["position_ids"])
            for k, v in plan.items():
                assert np.array_equal(v.cpu().numpy(), self.plan[k]), k
        else:
            plan = {k: np_to_device(self.plan[k])
                    for k in ("anchors", "block_valid", "position_ids")}
        before = kv.clone() if check_cache else None
        dflash.dflash_body_forward(cfg, wts, to_device(self.emb if emb is None else emb),
                                   plan["anchors"], plan["block_valid"], plan["position_ids"], m,
                                   kv, B, L, N, out)
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
