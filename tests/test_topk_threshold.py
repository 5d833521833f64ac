"""The warp top-k's selection rule, checked on the host.

One warp holds a token's keys, lane l the keys of positions l, l + 32, ...
The kernel takes t0 = the k-th largest of the 32 lanes' maxima, gathers every
key >= t0 with its position, and when there are at most 64 of them sorts them
by (key descending, position ascending) and keeps the first k; otherwise it
falls back to the bitwise search. The rule is exact because the k lanes with
the largest maxima hold k distinct keys >= t0, so t0 is at most the k-th
largest key and every key ranked above a selected one is gathered too. This
restates the rule and checks it against a plain sort on random, tied and
degenerate key sets (keys past the expert count are 0, below every real key).
"""
import numpy as np
import pytest


def select_by_threshold(keys, k):
    """keys: [32 * NK] in position order. Returns the k positions, or None
    when the kernel takes the bitwise search instead: k > 16, or more than 64
    keys reach the threshold."""
    if k > 16:
        return None
    lanes = keys.reshape(-1, 32).T            # lane l: positions l + 32 i
    t0 = np.sort(lanes.max(axis=1))[::-1][k - 1]
    cand = [(int(keys[p]), p) for p in range(len(keys)) if keys[p] >= t0]
    assert len(cand) >= k
    if len(cand) > 64:
        return None
    cand.sort(key=lambda kp: (-kp[0], kp[1]))
    return [p for _, p in cand[:k]]


def reference(keys, k):
    order = sorted(range(len(keys)), key=lambda p: (-int(keys[p]), p))
    return order[:k]


@pytest.mark.parametrize("E,k", [(896, 16), (1024, 32), (256, 8), (32, 4), (7, 3), (100, 9),
                                 (32, 32), (1024, 1)])
def test_threshold_select_matches_a_full_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    fallbacks = 0
    for trial in range(60):
        keys = np.zeros(1024, np.uint32)
        if trial % 3 == 0:      # distinct keys
            keys[:E] = rng.permutation(np.arange(1, E + 1, dtype=np.uint32) * 7919)
        elif trial % 3 == 1:    # a coarse grid: many ties
            keys[:E] = rng.integers(1, 6, E).astype(np.uint32)
        else:                   # a fine grid: some ties around the k-th key
            keys[:E] = rng.integers(1, 4 * E, E).astype(np.uint32)
        got = select_by_threshold(keys, k)
        if got is None:
            fallbacks += 1
            continue
        assert got == reference(keys, k)
    if k <= 16:   # (k > 16: the bitwise search decides)
        assert fallbacks < 60


def test_all_equal_keys_take_the_fallback():
    keys = np.zeros(1024, np.uint32)
    keys[:896] = 5
    assert select_by_threshold(keys, 16) is None
