"""Pins for the oracle's decayed cross-entropy over the drafted blocks (CPU only)."""
import math

import numpy as np
import pytest
from scipy.special import log_softmax

from oracle import dflash_oracle as orc


def test_position_weights():
    w = orc.position_weights(6, 2.0)
    assert w[0] == 0.0 and w[1] == 1.0
    assert np.allclose(w[2:] / w[1:-1], math.exp(-0.5))
    assert np.all(np.diff(w[1:]) < 0)            # earlier positions weigh more
    with pytest.raises(ValueError):
        orc.position_weights(4, 0.0)


def _case(seed, B=2, N=3, S=5, D=16, V=11):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((B, N, S, D))
    wl = rng.standard_normal((V, D)) * 0.3
    t = rng.integers(0, V, size=(B, N, S))
    m = (rng.random((B, N, S)) < 0.7).astype(np.uint8)
    m[:, :, 0] = 0
    return h, wl, t, m


def test_matches_scipy_log_softmax():
    h, wl, t, m = _case(1)
    loss, ce = orc.decayed_ce_loss(h, wl, t, m, 3.0)
    ref = -np.take_along_axis(log_softmax(h @ wl.T, axis=-1), t[..., None], -1)[..., 0]
    assert np.allclose(ce[m.astype(bool)], ref[m.astype(bool)], atol=1e-12)
    assert np.all(ce[~m.astype(bool)] == 0)
    w = orc.position_weights(h.shape[2], 3.0)[None, None, :] * m
    assert loss == pytest.approx(float((w * ref).sum() / w.sum()), abs=1e-12)


def test_uniform_logits_give_log_vocab():
    h, wl, t, m = _case(2)
    loss, ce = orc.decayed_ce_loss(h, np.zeros_like(wl), t, m, 1.0)
    assert loss == pytest.approx(math.log(wl.shape[0]), abs=1e-12)
    assert np.allclose(ce[m.astype(bool)], math.log(wl.shape[0]))


def test_decay_limits():
    h, wl, t, m = _case(3)
    # a very slow decay: the plain mean over masked slots
    loss, ce = orc.decayed_ce_loss(h, wl, t, m, 1e12)
    assert loss == pytest.approx(float(ce[m.astype(bool)].mean()), rel=1e-9)
    # a very fast decay: only the first predicted slot counts
    loss, ce = orc.decayed_ce_loss(h, wl, t, m, 1e-3)
    assert loss == pytest.approx(float(ce[:, :, 1][m[:, :, 1].astype(bool)].mean()), rel=1e-9)


def test_masked_slots_do_not_matter():
    h, wl, t, m = _case(4)
    base, _ = orc.decayed_ce_loss(h, wl, t, m, 2.0)
    h2, t2 = h.copy(), t.copy()
    off = ~m.astype(bool)
    h2[off] = 100.0
    t2[off] = 0
    again, _ = orc.decayed_ce_loss(h2, wl, t2, m, 2.0)
    assert again == base
    assert orc.decayed_ce_loss(h, wl, t, np.zeros_like(m), 2.0)[0] == 0.0
