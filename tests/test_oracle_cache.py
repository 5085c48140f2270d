"""Pins of the oracle's expert-cache plan (no GPU).

The plan is the exact-miss expert cache of AFN-019 "Hide SSD misses before
the router knows they exist", section "Two storage workloads, not one"
(whole records; score(record) = P(use before eviction) x expected exposed
latency avoided / resident bytes; LRU as the comparison baseline).  With one expert
routed per call it is textbook demand paging, so the classic worked examples
of page replacement fix FIFO and LRU; LRU's inclusion property (a stack
algorithm never faults more with more frames) must hold on any trace; the
score policy is pinned by hand-worked small cases that separate it from LRU.
"""
import numpy as np
import pytest

import oracle

# Silberschatz, Galvin and Gagne, "Operating System Concepts", chapter on
# page replacement: this reference string with three frames takes 15 faults
# under FIFO and 12 under LRU.
TEXTBOOK = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]
# Belady's anomaly (Belady, Nelson and Shedler 1969): FIFO takes 9 faults with
# three frames and 10 with four; LRU takes 10 and 8.
BELADY = [1, 2, 3, 4, 1, 2, 5, 1, 2, 3, 4, 5]


def one_hot(e, E):
    c = np.zeros(E, np.int32)
    c[e] = 1
    return c


def faults(seq, S, policy, E=16, decay=0.9):
    cp = oracle.CachePlan(E, S, policy, decay)
    for e in seq:
        full, ml, ms = cp.step(one_hot(e, E))
        assert not full
    return int(cp.stats[3])


@pytest.mark.parametrize("policy,S,want", [("fifo", 3, 15), ("lru", 3, 12)])
def test_textbook_reference_string(policy, S, want):
    assert faults(TEXTBOOK, S, policy) == want


@pytest.mark.parametrize("policy,S,want", [("fifo", 3, 9), ("fifo", 4, 10), ("lru", 3, 10), ("lru", 4, 8)])
def test_belady_anomaly(policy, S, want):
    assert faults(BELADY, S, policy) == want


def test_lru_inclusion_property():
    """LRU is a stack algorithm: with one more slot the resident set after
    every call contains the smaller cache's, and faults never increase."""
    rng = np.random.default_rng(5)
    E = 12
    seq = rng.zipf(1.3, size=400) % E
    prev = None
    for S in range(1, 9):
        cp = oracle.CachePlan(E, S, "lru")
        sets = []
        for e in seq:
            cp.step(one_hot(int(e), E))
            sets.append(set(int(x) for x in cp.expert_of if x >= 0))
        if prev is not None:
            assert cp.stats[3] <= prev[0]
            assert all(a <= b for a, b in zip(prev[1], sets))
        prev = (int(cp.stats[3]), sets)


def test_score_keeps_the_frequent_expert_where_lru_drops_it():
    """Two slots; calls route A, A, A, B, C.  LRU evicts A (used last in call
    3, B in call 4).  With decay 0.9 the use rates before call 5 are
    A: 0.9^2 * (1 + 0.9 + 0.81) = 2.1951, B: 0.9: SCORE evicts B.  With decay
    0.5 they are A: 0.25 * 1.75 = 0.4375, B: 0.5: SCORE evicts A."""
    A, B, Cx, E = 0, 1, 2, 4

    def resident(policy, decay):
        cp = oracle.CachePlan(E, 2, policy, decay)
        for e in (A, A, A, B, Cx):
            cp.step(one_hot(e, E))
        return sorted(int(x) for x in cp.expert_of), cp

    assert resident("lru", 0.9)[0] == [B, Cx]
    got, cp = resident("score", 0.9)
    assert got == [A, Cx]
    np.testing.assert_allclose(cp.score[:3], [2.1951, 0.9, 1.0], rtol=1e-6)
    assert resident("score", 0.5)[0] == [B, Cx]


def test_score_with_zero_decay_takes_the_lowest_slot():
    """decay 0: every candidate's use rate is 0, so the lowest unpinned slot
    is always the victim."""
    cp = oracle.CachePlan(8, 3, "score", 0.0)
    for e in range(6):
        cp.step(one_hot(e, 8))
    assert cp.expert_of.tolist() == [5, 1, 2]


def test_pinned_slots_are_never_victims():
    """Slots of experts routed in the same call stay; FIFO skips them in
    rotation order."""
    E = 8
    cp = oracle.CachePlan(E, 3, "fifo")
    c = np.zeros(E, np.int32)
    c[[0, 1, 2]] = 1
    cp.step(c)
    assert cp.expert_of.tolist() == [0, 1, 2] and cp.hand[0] == 0
    c = np.zeros(E, np.int32)
    c[[0, 3]] = [2, 1]
    full, ml, ms = cp.step(c)
    assert not full and ml.tolist() == [3] and ms.tolist() == [1]
    assert cp.expert_of.tolist() == [0, 3, 2] and cp.hand[0] == 2
    assert cp.stats.tolist() == [1, 1, 1, 4]


def test_cache_full_changes_no_slot():
    E = 8
    for policy in ("fifo", "lru", "score"):
        cp = oracle.CachePlan(E, 2, policy)
        cp.step(one_hot(5, E))
        before = (cp.slot_of.copy(), cp.expert_of.copy(), cp.hand[0], cp.last_use.copy())
        c = np.zeros(E, np.int32)
        c[[1, 2, 3]] = 1
        full, ml, ms = cp.step(c)
        assert full and len(ml) == 0
        assert np.array_equal(cp.slot_of, before[0]) and np.array_equal(cp.expert_of, before[1])
        assert cp.hand[0] == before[2] and np.array_equal(cp.last_use, before[3])
        assert cp.hand[1] == 2 and cp.stats.tolist() == [0, 0, 0, 1]


@pytest.mark.parametrize("policy", ["fifo", "lru", "score"])
def test_plan_invariants_on_multi_route_calls(policy):
    """Calls routing several experts: after a call that fits, every routed
    expert is resident; the misses are exactly the routed experts that were
    not; slots and experts stay a bijection."""
    rng = np.random.default_rng(11)
    E, S = 64, 20
    cp = oracle.CachePlan(E, S, policy, 0.8)
    for _ in range(200):
        c = np.zeros(E, np.int32)
        c[rng.choice(E, size=int(rng.integers(1, 24)), replace=False)] = 1
        resident = set(int(x) for x in cp.expert_of if x >= 0)
        full, ml, ms = cp.step(c)
        routed = set(int(e) for e in np.nonzero(c)[0])
        if full:
            assert len(routed - resident) > S - len(routed & resident)
            continue
        assert ml.tolist() == sorted(routed - resident)
        assert len(set(ms.tolist())) == len(ms)
        assert routed <= set(int(x) for x in cp.expert_of if x >= 0)
        for e in range(E):
            if cp.slot_of[e] >= 0:
                assert cp.expert_of[cp.slot_of[e]] == e
        for s in range(S):
            if cp.expert_of[s] >= 0:
                assert cp.slot_of[cp.expert_of[s]] == s
