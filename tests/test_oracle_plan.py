"""Pins for the oracle's batch plan (anchor sampling, validity, loss mask); CPU only."""
import os

import numpy as np
import pytest

from oracle import dflash_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_reference_outputs():
    # Reference outputs of the SplitMix64 generator (Steele, Lea & Flood 2014; the public
    # splitmix64.c by S. Vigna): seed 1234567 and seed 0.
    assert orc.splitmix64_stream(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert orc.splitmix64_stream(0, 1) == [0xE220A8397B1DCDAF]


def test_anchor_key_takes_twos_complement_of_negatives():
    assert orc.anchor_key(1, -1, 5, 2) == orc.anchor_key(1, (1 << 64) - 1, 5, 2)
    assert orc.anchor_key(1, 2, -7, 2) == orc.anchor_key(1, 2, (1 << 64) - 7, 2)


def test_candidates_rule_small_case():
    # valid(a) and valid(a + 1); position L is out of range
    assert orc.anchor_candidates([1, 1, 0, 1, 1, 1, 0, 1]) == [0, 3, 4]
    assert orc.anchor_candidates([1]) == []
    assert orc.anchor_candidates([0, 0, 0]) == []
    assert orc.anchor_candidates([1, 1]) == [0]


def _brute_force_anchors(mask_row, sid, step, seed, n):
    """Selection by rank counting: a candidate is chosen iff fewer than n candidates have a
    smaller (key, position) pair."""
    L = len(mask_row)
    cands = [a for a in range(L) if mask_row[a] and a + 1 < L and mask_row[a + 1]]
    keys = {a: orc.anchor_key(seed, step, sid, a) for a in cands}
    chosen = []
    for a in cands:
        rank = sum(1 for c in cands if (keys[c], c) < (keys[a], a))
        if rank < n:
            chosen.append(a)
    chosen.sort()
    return chosen + [-1] * (n - len(chosen))


@pytest.mark.parametrize("trial", range(20))
def test_anchor_choice_brute_force(trial):
    rng = np.random.default_rng(100 + trial)
    L = int(rng.integers(1, 40))
    mask = (rng.random(L) < 0.8).astype(np.uint8)
    sid = int(rng.integers(-2 ** 63, 2 ** 63 - 1))
    step, seed = int(rng.integers(0, 1000)), int(rng.integers(0, 2 ** 64 - 1, dtype=np.uint64))
    n = int(rng.integers(1, 12))
    assert orc.choose_anchors(list(mask), sid, step, seed, n) == \
        _brute_force_anchors(list(mask), sid, step, seed, n)


def _random_case(rng, B=6, L=50, N=5, S=4):
    mask = np.ones((B, L), np.uint8)
    for b in range(B):
        vl = int(rng.integers(0, L + 1))
        mask[b, vl:] = 0
        holes = rng.random(L) < 0.1
        mask[b, holes] = 0
    sids = rng.integers(0, 4, size=B).astype(np.int64)
    return mask, sids, N, S


def test_plan_invariants():
    rng = np.random.default_rng(7)
    for trial in range(10):
        mask, sids, N, S = _random_case(rng)
        p = orc.build_plan(mask, sids, step=trial, seed=99, num_anchors=N, block_size=S)
        B, L = mask.shape
        for b in range(B):
            a = p["anchors"][b]
            real = [int(x) for x in a if x >= 0]
            assert real == sorted(set(real))                       # sorted, unique
            assert all(x == -1 for x in a[len(real):])               # empty slots last
            for k in range(N):
                for j in range(S):
                    if a[k] < 0:
                        assert p["block_valid"][b, k, j] == 0 and p["position_ids"][b, k, j] == -1
                        continue
                    pos = a[k] + j
                    assert p["position_ids"][b, k, j] == pos
                    want = (a[k] < L and mask[b, a[k]] == 1 and pos < L and mask[b, pos] == 1)
                    assert p["block_valid"][b, k, j] == int(want)
        assert np.all(p["loss_mask"][:, :, 0] == 0)
        assert np.all(p["loss_mask"] <= p["block_valid"])
        assert np.array_equal(p["loss_mask"][:, :, 1:], p["block_valid"][:, :, 1:])


def test_leader_anchors_are_candidates_and_count():
    rng = np.random.default_rng(8)
    mask, _, N, S = _random_case(rng)
    sids = np.arange(mask.shape[0], dtype=np.int64)    # all distinct: every row leads
    p = orc.build_plan(mask, sids, 0, 1, N, S)
    for b in range(mask.shape[0]):
        cands = orc.anchor_candidates(list(mask[b]))
        real = [int(x) for x in p["anchors"][b] if x >= 0]
        assert set(real) <= set(cands)
        assert len(real) == min(N, len(cands))


def test_rows_without_window_have_no_valid_slot():
    mask = np.zeros((3, 10), np.uint8)
    mask[1, 0] = 1            # one valid token: no window
    mask[2, :] = 1
    mask[2, 1::2] = 0          # alternating: no two consecutive valid tokens
    p = orc.build_plan(mask, np.array([1, 2, 3]), 0, 0, 3, 4)
    assert np.all(p["anchors"] == -1)
    assert np.all(p["block_valid"] == 0) and np.all(p["loss_mask"] == 0)


def test_determinism_and_sensitivity():
    rng = np.random.default_rng(9)
    mask = np.ones((4, 300), np.uint8)
    sids = np.array([11, 12, 13, 14], np.int64)
    p1 = orc.build_plan(mask, sids, 5, 77, 8, 4)
    p2 = orc.build_plan(mask.copy(), sids.copy(), 5, 77, 8, 4)
    for k in p1:
        assert np.array_equal(p1[k], p2[k])
    assert not np.array_equal(orc.build_plan(mask, sids, 6, 77, 8, 4)["anchors"], p1["anchors"])
    assert not np.array_equal(orc.build_plan(mask, sids, 5, 78, 8, 4)["anchors"], p1["anchors"])
    # rows with distinct sample ids and identical masks draw different anchors
    assert not np.array_equal(p1["anchors"][0], p1["anchors"][1])
    del rng


def test_shared_sample_id_rows_get_leader_anchors():
    mask = np.ones((4, 64), np.uint8)
    mask[3, 40:] = 0                       # follower with a shorter valid span
    sids = np.array([7, 9, 7, 7], np.int64)
    p = orc.build_plan(mask, sids, 0, 3, 10, 4)
    assert np.array_equal(p["anchors"][0], p["anchors"][2])
    assert np.array_equal(p["anchors"][0], p["anchors"][3])
    assert not np.array_equal(p["anchors"][0], p["anchors"][1])
    # the follower's validity comes from its own mask
    for k in range(10):
        a = p["anchors"][3, k]
        for j in range(4):
            assert p["block_valid"][3, k, j] == int(a >= 0 and a < 40 and a + j < 40)


def test_anchor_uniformity_chi_square():
    # statistical sanity: over many seeds every candidate position is picked about N/|C| often
    L, N, trials = 24, 4, 3000
    counts = np.zeros(L)
    mask = [1] * L
    for t in range(trials):
        for a in orc.choose_anchors(mask, 5, 0, t, N):
            counts[a] += 1
    cands = L - 1
    exp = trials * N / cands
    chi2 = float(np.sum((counts[:cands] - exp) ** 2 / exp))
    assert counts[L - 1] == 0
    # 22 degrees of freedom: P(chi2 > 50) < 1e-3
    assert chi2 < 50.0


def _read_plan_golden(path):
    with open(path) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    hdr = dict(kv.split("=") for kv in lines[0].split())
    B, L, N, S = (int(hdr[k]) for k in ("B", "L", "N", "S"))
    step, seed = int(hdr["step"]), int(hdr["seed"])
    rows = lines[1:]
    mask = np.array([[int(c) for c in rows[b].split(":")[1].strip()] for b in range(B)], np.uint8)
    sids = np.array([int(r.split(":")[1]) for r in rows[B:2 * B]], np.int64)
    anchors = np.array([[int(t) for t in r.split(":")[1].split()] for r in rows[2 * B:3 * B]],
                       np.int32)
    return mask, sids, step, seed, N, S, anchors


@pytest.mark.parametrize("name", ["plan_small.txt", "plan_shared_sid.txt"])
def test_plan_golden_vectors(name):
    mask, sids, step, seed, N, S, anchors = _read_plan_golden(os.path.join(GOLDEN, name))
    p = orc.build_plan(mask, sids, step, seed, N, S)
    assert np.array_equal(p["anchors"], anchors)
