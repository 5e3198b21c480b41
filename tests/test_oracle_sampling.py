"""Pins for the oracle's speculative-sampling verification (CPU only): the counter-based
uniform draws, the exponential-race sampler, and the acceptance / residual rule of page
"DFlash: drafting, verification, and speed", Sampling with temperature is not argmax
matching -- checked against what the mathematics fixes (the output distribution equals the
target's whatever the proposal, the acceptance rate 1 - TV(p, q), the greedy limit)."""
import math

import numpy as np
import pytest
from scipy import stats

from oracle import dflash_oracle as orc


def test_counter_uniform_grid_and_spread():
    u = np.array([orc.counter_uniform(7, b, i) for b in range(40) for i in range(100)])
    assert np.all((u > 0) & (u < 1))
    # every value is (k + 1/2) * 2^-23 for an integer k, and survives a round trip to fp32
    k = u * 2 ** 23 - 0.5
    assert np.array_equal(k, np.round(k))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert orc.counter_uniform(0) == ((orc.splitmix64_mix(0) >> 41) + 0.5) * 2.0 ** -23
    assert len(set(u.tolist())) == len(u)
    # uniform over 16 bins (chi-square at 1e-3)
    counts = np.histogram(u, bins=16, range=(0, 1))[0]
    assert stats.chisquare(counts).pvalue > 1e-3
    assert orc.counter_uniform(7, 3, 4) == orc.counter_uniform(7, 3, 4)
    assert orc.counter_uniform(7, 3, 4) != orc.counter_uniform(8, 3, 4)


def test_race_sample_single_weight_and_scale_invariance():
    w = np.array([0.0, 0.0, 3.5, 0.0])
    assert all(orc.race_sample(w, s, 1) == 2 for s in range(20))
    w = np.array([0.1, 0.7, 0.2, 0.4, 0.0])
    for s in range(50):
        assert orc.race_sample(w, s, 2) == orc.race_sample(4.0 * w, s, 2)
        assert orc.race_sample(w, s, 2) != 4


def test_race_sample_distribution():
    w = np.array([0.05, 0.5, 0.0, 0.25, 0.2])
    n = 4000
    draws = [orc.race_sample(w, 11, t) for t in range(n)]
    counts = np.bincount(draws, minlength=len(w))
    assert counts[2] == 0
    nz = w > 0
    assert stats.chisquare(counts[nz], n * w[nz] / w.sum()).pvalue > 1e-3


def _dist(rng, V, alpha=1.0):
    x = rng.gamma(alpha, size=V)
    return x / x.sum()


@pytest.mark.parametrize("gamma", [1, 2])
def test_first_emitted_token_follows_the_target(gamma):
    """Whatever the proposal q, the first emitted token is distributed as p_0 (the proposal
    is drawn from q, then accepted with min(1, p/q) or replaced by a residual sample)."""
    rng = np.random.default_rng(5 + gamma)
    V = 5
    p = np.stack([_dist(rng, V) for _ in range(gamma + 1)])
    q = np.stack([_dist(rng, V, 0.5) for _ in range(gamma)])
    n = 4000
    first = np.zeros(V, np.int64)
    accepted0 = 0
    for t in range(n):
        draft = [int(rng.choice(V, p=q[i])) for i in range(gamma)]
        out, acc = orc.verify_sampling_block(p, q, draft, seed=99, b=t)
        first[out[0]] += 1
        accepted0 += acc > 0
    assert stats.chisquare(first, n * p[0]).pvalue > 1e-3
    # acceptance probability of the first proposal: sum_y min(p(y), q(y)) = 1 - TV(p, q)
    a = np.minimum(p[0], q[0]).sum()
    se = math.sqrt(a * (1 - a) / n)
    assert abs(accepted0 / n - a) < 4 * se


def test_greedy_limit():
    """One-hot target and proposal distributions: accept exactly when the proposal is the
    target's choice, the residual is the target's choice, the bonus is the last choice --
    greedy verification of the same block."""
    rng = np.random.default_rng(3)
    V, gamma = 7, 4
    for t in range(200):
        choices = rng.integers(0, V, size=gamma + 1)
        draft = [int(c) if rng.random() < 0.7 else int(rng.integers(0, V)) for c in choices[:-1]]
        p = np.eye(V)[choices]
        q = np.eye(V)[draft]
        got = orc.verify_sampling_block(p, q, draft, seed=t, b=0)
        assert got == orc.verify_greedy_block(draft, [int(c) for c in choices])


def test_equal_distributions_accept_everything_and_eos_stops():
    rng = np.random.default_rng(4)
    V, gamma = 6, 3
    p = np.stack([_dist(rng, V) for _ in range(gamma + 1)])
    draft = [1, 2, 3]
    out, acc = orc.verify_sampling_block(p, p[:gamma], draft, seed=1, b=0)
    assert acc == gamma and out[:gamma] == draft and len(out) == gamma + 1
    out, acc = orc.verify_sampling_block(p, p[:gamma], draft, seed=1, b=0, eos_token=2)
    assert out == [1, 2] and acc == 2
    # a proposal the draft could not have drawn (q(y) = 0) is accepted whenever p(y) > 0
    q = np.stack([_dist(rng, V) for _ in range(gamma)])
    q[0, 5] = 0.0
    out, acc = orc.verify_sampling_block(p, q, [5, 1, 1], seed=2, b=0)
    assert acc >= 1 and out[0] == 5
    with pytest.raises(ValueError):
        orc.verify_sampling_block(p, q, [1, 2], seed=1, b=0)


def test_batched_form_uses_temperature_softmax():
    rng = np.random.default_rng(8)
    B, S, V = 3, 4, 9
    logits = rng.standard_normal((B, S, V))
    q = np.stack([np.stack([_dist(rng, V) for _ in range(S - 1)]) for _ in range(B)])
    draft = rng.integers(0, V, size=(B, S - 1)).astype(np.int32)
    em, num, acc = orc.verify_sampling(logits, 0.7, q, draft, seed=5)
    for b in range(B):
        p = np.exp(logits[b] / 0.7)
        p /= p.sum(axis=1, keepdims=True)
        out, a = orc.verify_sampling_block(p, q[b], draft[b], 5, b)
        assert list(em[b, :num[b]]) == out and acc[b] == a
        assert np.all(em[b, num[b]:] == -1)
