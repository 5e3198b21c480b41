"""Pins for the oracle's greedy verification (CPU only)."""
import os

import numpy as np
import pytest

from oracle import dflash_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = [int(t) for t in rest.split()]
    return vals


def test_worked_example_from_pages():
    g = _read_golden("verify_worked_example.txt")
    emitted, accepted = orc.verify_greedy_block(g["draft"], g["target_choices"])
    assert emitted == g["emitted"]
    assert accepted == g["accepted"][0]


def test_all_match_emits_bonus():
    emitted, accepted = orc.verify_greedy_block([1, 2, 3], [1, 2, 3, 7])
    assert emitted == [1, 2, 3, 7] and accepted == 3


def test_first_mismatch():
    emitted, accepted = orc.verify_greedy_block([5, 2, 3], [1, 2, 3, 7])
    assert emitted == [1] and accepted == 0


def test_later_matches_after_mismatch_do_not_count():
    # only the continuous prefix survives; position 3 matching is irrelevant
    emitted, accepted = orc.verify_greedy_block([1, 9, 3, 4], [1, 2, 3, 4, 5])
    assert emitted == [1, 2] and accepted == 1


def test_eos_stops_without_bonus():
    emitted, accepted = orc.verify_greedy_block([1, 0, 3], [1, 0, 3, 7], eos_token=0)
    assert emitted == [1, 0] and accepted == 2


def test_eos_as_correction_is_emitted():
    # a mismatching proposal: the target's choice (which may be EOS) is emitted and the block ends
    emitted, accepted = orc.verify_greedy_block([1, 4, 3], [1, 0, 3, 7], eos_token=0)
    assert emitted == [1, 0] and accepted == 1


def test_empty_draft_emits_bonus_only():
    emitted, accepted = orc.verify_greedy_block([], [42])
    assert emitted == [42] and accepted == 0


@pytest.mark.parametrize("n_choices", [3, 5])
def test_length_mismatch_raises(n_choices):
    with pytest.raises(ValueError):
        orc.verify_greedy_block([1, 2, 3], list(range(n_choices)))


def test_argmax_fast_agrees_with_loop_on_ties():
    rng = np.random.default_rng(3)
    # small integer values make ties common
    rows = rng.integers(-3, 4, size=(200, 37)).astype(np.float64)
    fast = orc.argmax_lowest_fast(rows)
    for r in range(rows.shape[0]):
        assert fast[r] == orc.argmax_lowest(rows[r])
        # lowest index among the maxima
        assert fast[r] == min(np.nonzero(rows[r] == rows[r].max())[0])


def test_argmax_signed_zero_and_negatives():
    row = np.array([-1.0, -0.0, 0.0, -0.5])
    assert orc.argmax_lowest(row) == 1       # -0.0 == +0.0: the first wins
    assert orc.argmax_lowest(np.array([-3.0, -2.0, -2.0])) == 1


def test_batched_verify_brute_force():
    rng = np.random.default_rng(11)
    B, S, V = 64, 6, 13
    logits = rng.integers(-2, 3, size=(B, S, V)).astype(np.float64)
    choices_ref = np.array([[orc.argmax_lowest(logits[b, i]) for i in range(S)] for b in range(B)])
    # drafts that follow the choices for a random number of steps
    draft = rng.integers(0, V, size=(B, S - 1)).astype(np.int32)
    for b in range(B):
        k = rng.integers(0, S)
        draft[b, :k] = choices_ref[b, :k]
    ch, em, num, acc = orc.verify_greedy(logits, draft)
    assert np.array_equal(ch, choices_ref)
    for b in range(B):
        # brute force: the accepted count is the length of the longest agreeing prefix
        k = 0
        while k < S - 1 and draft[b, k] == choices_ref[b, k]:
            k += 1
        assert acc[b] == k
        assert num[b] == k + 1
        assert list(em[b, :k]) == list(draft[b, :k])
        assert em[b, k] == choices_ref[b, k]
        assert np.all(em[b, k + 1:] == -1)


def test_batched_verify_rejects_bad_shapes():
    with pytest.raises(ValueError):
        orc.verify_greedy(np.zeros((2, 4, 8)), np.zeros((2, 4), np.int32))


def test_commit_keeps_anchor_and_accepted_proposals_only():
    """The pages' worked example: proposals [10, 20, 99, 40] against target choices
    [10, 20, 30, 40, 50] accept 2; the anchor and the two accepted proposals stay, the
    rejected 99 and its suffix 40 go, although 40 matched its target choice."""
    g = _read_golden("verify_worked_example.txt")
    _, accepted = orc.verify_greedy_block(g["draft"], g["target_choices"])
    prev = np.arange(6, dtype=np.float64).reshape(3, 2)          # 3 committed positions
    # the verified block's states: anchor, then the four proposals (tagged by token id)
    block = np.array([[-1, -1]] + [[t, t] for t in g["draft"]], np.float64)
    out = orc.commit_verified(prev, block, accepted)
    assert out.shape == (3 + accepted + 1, 2)
    assert np.array_equal(out[:3], prev)
    assert [int(x) for x in out[3:, 0]] == [-1, 10, 20]
    assert 99 not in out and 40 not in out


@pytest.mark.parametrize("gamma", [0, 1, 4, 15])
def test_commit_length_follows_verification(gamma):
    rng = np.random.default_rng(gamma)
    for _ in range(20):
        choices = list(rng.integers(0, 3, size=gamma + 1))
        draft = list(rng.integers(0, 3, size=gamma))
        emitted, acc = orc.verify_greedy_block(draft, choices)
        block = rng.standard_normal((gamma + 1, 3))
        out = orc.commit_verified(np.zeros((5, 3)), block, acc)
        # the retained block positions are exactly the anchor plus the accepted proposals;
        # without an EOS stop that is also the number of emitted tokens
        assert out.shape[0] == 5 + acc + 1 == 5 + len(emitted)
        assert np.array_equal(out[5:], block[:acc + 1])
    with pytest.raises(ValueError):
        orc.commit_verified(np.zeros((1, 3)), np.zeros((4, 3)), 4)
