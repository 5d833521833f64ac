"""The cache replacement rule's reference, pinned by a hand-worked sequence."""
import pytest

from stream_lru import LruModel


def test_hand_worked_sequence():
    m = LruModel(n_experts=8, n_slots=3)
    # call 1: both miss, empty slots (stamp 0) in slot order
    assert m.call([0, 1]) == [(0, 0), (1, 1)]
    # call 2: 1 hits (slot 1 stamp 2); 2 takes the oldest free slot: slot 2 (stamp 0)
    assert m.call([1, 2]) == [(2, 2)]
    # call 3: 3 takes slot 0 (stamp 1 < stamp 2 of slots 1 and 2), evicting 0
    assert m.call([3]) == [(3, 0)]
    assert m.slot_of[0] == -1 and m.expert_of == [3, 1, 2]
    # call 4: 2 hits; 0 misses and takes slot 1 (stamp 2) over slot 0 (stamp 3), evicting 1
    assert m.call([0, 2]) == [(0, 1)]
    assert m.expert_of == [3, 0, 2] and m.slot_of[1] == -1
    assert m.stamp == [3, 4, 4] and m.clock == 4
    assert (m.hits, m.misses) == (2, 5)


def test_missing_experts_take_slots_in_expert_order():
    m = LruModel(n_experts=10, n_slots=4)
    m.call([9, 3, 5, 1])            # unordered input: handled in expert order
    assert m.expert_of == [1, 3, 5, 9]
    m.call([2, 8])                  # ties in stamp (all 1): lower slot first
    assert m.expert_of == [2, 8, 5, 9]


def test_no_slot_for_every_active_expert_raises():
    m = LruModel(n_experts=10, n_slots=2)
    with pytest.raises(ValueError):
        m.call([0, 1, 2])


def test_all_hits_keep_the_state_but_advance_stamps():
    m = LruModel(n_experts=6, n_slots=3)
    m.call([0, 1, 2])
    before = list(m.expert_of)
    assert m.call([2, 0, 1]) == []
    assert m.expert_of == before and m.stamp == [2, 2, 2]
