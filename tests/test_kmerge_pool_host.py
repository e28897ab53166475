"""The K-Merge pool's policy on the host (no GPU): storage never exceeds the
budget B, an adapter that fits is stored as its own entry, one that does not
is merged into the most similar entry (ties: lowest index) once the caller
reports the merge's outcome, and an adapter larger than B is never stored.

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"K-Merge: online LoRA adapter management for the edge" (steps 1-4 and the
budget-B paragraph); the readings are in include/bitdelta_kmerge.h.
"""
import random

import pytest

import bit_weight_delta_gb300 as bd

MB = 1 << 20


@pytest.fixture
def pool():
    p = bd.KMergePool(3 * MB)
    yield p
    p.close()


def test_store_until_the_budget_then_hit(pool):
    assert pool.request(7, MB) == ("store", 0)
    assert pool.request(3, MB) == ("store", 1)
    assert pool.request(7, MB) == ("hit", 0)
    assert pool.request(9, MB) == ("store", 2)
    st = pool.stats()
    assert st["used_bytes"] == 3 * MB and st["entries"] == 3 and st["hits"] == 1


def test_overflow_asks_for_similarity_then_merges_into_the_argmax(pool):
    for a in (0, 1, 2):
        pool.request(a, MB)
    assert pool.request(5, MB) == ("need_similarity", -1)
    assert pool.stats()["used_bytes"] == 3 * MB        # nothing changed
    assert pool.request(5, MB, [0.1, 0.7, 0.3]) == ("merge", 1)
    assert pool.entry_of(5) == -1                      # pending until commit
    pool.commit(5, 1, True, MB)
    assert pool.entry_of(5) == 1
    assert pool.entry_info(1) == (MB, 2)
    assert pool.request(5, MB) == ("hit", 1)
    assert pool.stats()["used_bytes"] == 3 * MB


def test_ties_go_to_the_lowest_entry(pool):
    for a in (0, 1, 2):
        pool.request(a, MB)
    assert pool.request(8, MB, [0.4, 0.9, 0.9]) == ("merge", 1)
    pool.commit(8, 1, False, MB)
    assert pool.request(8, MB, [0.2, 0.2, 0.2]) == ("merge", 0)


def test_rejected_merge_changes_nothing(pool):
    for a in (0, 1, 2):
        pool.request(a, MB)
    before = pool.stats()
    assert pool.request(4, MB, [0.5, 0.1, 0.2]) == ("merge", 0)
    pool.commit(4, 0, False, MB)
    after = pool.stats()
    assert pool.entry_of(4) == -1 and pool.entry_info(0) == (MB, 1)
    assert after["used_bytes"] == before["used_bytes"] and after["merges_rejected"] == 1


def test_larger_than_budget_is_rejected(pool):
    assert pool.request(1, 3 * MB + 1) == ("reject", -1)
    assert pool.stats()["entries"] == 0 and pool.stats()["rejects"] == 1


def test_merge_that_would_exceed_the_budget_is_refused(pool):
    pool.request(0, 2 * MB)
    pool.request(1, MB)
    assert pool.request(2, MB, [0.3, 0.6]) == ("merge", 1)
    with pytest.raises(bd.BitDeltaError):
        pool.commit(2, 1, True, 1 * MB + 1)     # 2 MB + 1 MB + 1 > B
    pool.commit(2, 1, True, MB)                 # the merge is still pending: retry
    assert pool.entry_of(2) == 1 and pool.stats()["used_bytes"] == 3 * MB


def test_bad_arguments(pool):
    pool.request(0, 2 * MB)
    pool.request(1, MB)
    with pytest.raises(bd.BitDeltaError):
        pool.request(2, MB, [0.5])                  # one value per entry
    with pytest.raises(bd.BitDeltaError):
        pool.request(2, MB, [0.5, float("nan")])
    with pytest.raises(bd.BitDeltaError):
        pool.request(2, MB, [0.5, 1.5])             # not a cosine
    with pytest.raises(bd.BitDeltaError):
        pool.commit(2, 0, True, MB)                 # nothing pending
    assert pool.request(2, MB, [0.5, 0.2]) == ("merge", 0)
    with pytest.raises(bd.BitDeltaError):
        pool.request(3, MB, [0.5, 0.2])             # another merge is pending
    with pytest.raises(bd.BitDeltaError):
        pool.commit(2, 1, True, MB)                 # not the proposed entry
    with pytest.raises(bd.BitDeltaError):
        pool.request(-1, MB)
    with pytest.raises(bd.BitDeltaError):
        pool.request(4, 0)
    with pytest.raises(bd.BitDeltaError):
        bd.KMergePool(0)


def test_random_requests_never_exceed_the_budget():
    """Random request streams (sizes 1-4 MB, budget 10 MB, random
    similarities, random merge outcomes and merged sizes): the pool never
    holds more than B, every covered adapter maps to exactly one entry, the
    entries' adapter counts add up, and a merge always targets the argmax."""
    rng = random.Random(5)
    for trial in range(20):
        budget = 10 * MB
        pool = bd.KMergePool(budget)
        sizes = {a: rng.randint(1, 4) * MB for a in range(40)}
        covered = {}
        for _ in range(300):
            a = rng.randrange(40)
            act, e = pool.request(a, sizes[a])
            if act == "need_similarity":
                n = pool.stats()["entries"]
                cos = [rng.choice([-0.5, 0.0, 0.25, 0.5, 1.0]) for _ in range(n)]
                act, e = pool.request(a, sizes[a], cos)
                assert act == "merge" and e == cos.index(max(cos))
                accept = rng.random() < 0.7
                merged = rng.randint(1, 4) * MB
                used = pool.stats()["used_bytes"]
                fits = used - pool.entry_info(e)[0] + merged <= budget
                if accept and not fits:
                    with pytest.raises(bd.BitDeltaError):
                        pool.commit(a, e, True, merged)
                    pool.commit(a, e, False, merged)
                else:
                    pool.commit(a, e, accept, merged)
                    if accept:
                        covered[a] = e
            elif act == "store":
                covered[a] = e
            elif act == "hit":
                assert covered[a] == e
            st = pool.stats()
            assert st["used_bytes"] <= budget
            assert sum(pool.entry_info(i)[0] for i in range(st["entries"])) == st["used_bytes"]
            assert sum(pool.entry_info(i)[1] for i in range(st["entries"])) == len(covered)
            for b, eb in covered.items():
                assert pool.entry_of(b) == eb
        pool.close()
