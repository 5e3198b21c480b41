"""Shared test plumbing: seeded inputs on the device, fp64 views for the oracle, comparisons.

Both sides get the same seeded inputs from dflash_inputs; nothing here computes any part of
the method.
"""
from __future__ import annotations

import numpy as np

import dflash_inputs as di

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
