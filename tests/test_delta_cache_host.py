"""The delta cache's policy on a host arena (no GPU): cold load on first
request, hits afterwards, LRU eviction among variants nobody holds, the
highest-traffic variants pinned, requests refused (BD_ERR_CACHE_FULL) rather
than evicting a held or pinned delta, and thread safety.

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"Infrastructure details" (cold start, LRU weighted by request rate with the
top variants pinned, one load per variant however many requests queue)."""
import random
import threading

import pytest
import torch

import bit_weight_delta_gb300 as bd

SLOT = 4096


def blob(variant: int, n: int = 3000) -> torch.Tensor:
    g = torch.Generator().manual_seed(variant)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


def make(n_slots: int, pin: int, variants=range(4)):
    arena = torch.zeros(n_slots * SLOT + 256, dtype=torch.uint8)
    off = (-arena.data_ptr()) % 256      # 256-byte aligned start
    cache = bd.DeltaCache(arena[off:off + n_slots * SLOT], SLOT, pin_top_k=pin)
    blobs = {v: blob(v) for v in variants}
    for v, b in blobs.items():
        cache.register(v, b)
    return cache, blobs


def use(cache, v):
    view = cache.acquire(v)
    data = view.clone()
    cache.release(v)
    return data


def test_cold_load_then_hit():
    cache, blobs = make(2, 0)
    assert torch.equal(use(cache, 1), blobs[1])
    assert cache.stats()["loads"] == 1
    assert torch.equal(use(cache, 1), blobs[1])
    st = cache.stats()
    assert st == {**st, "acquires": 2, "hits": 1, "loads": 1, "evictions": 0,
                  "bytes_loaded": blobs[1].numel()}


def test_lru_evicts_the_least_recently_used_free_slot():
    cache, blobs = make(2, 0)
    use(cache, 0)           # t1
    use(cache, 1)           # t2
    use(cache, 2)           # t3: evicts 0 (least recent)
    assert cache.slot_of(0) == -1 and cache.slot_of(1) >= 0 and cache.slot_of(2) >= 0
    use(cache, 1)           # t4: hit
    assert torch.equal(use(cache, 0), blobs[0])   # t5: evicts 2 (t3 < t4)
    assert cache.slot_of(2) == -1 and cache.slot_of(1) >= 0
    assert cache.stats()["evictions"] == 2


def test_top_traffic_variants_stay_resident():
    cache, _ = make(2, 1, variants=range(5))
    for _ in range(5):
        use(cache, 0)       # variant 0: the most traffic -> pinned
    for v in (1, 2, 3, 4, 1, 3):
        use(cache, v)
        assert cache.slot_of(0) >= 0, f"pinned variant evicted by {v}"
    assert cache.stats()["evictions"] == 5


def test_pinning_follows_traffic():
    cache, _ = make(2, 1, variants=range(4))
    use(cache, 0)
    for _ in range(3):
        use(cache, 1)       # 1 overtakes 0 in traffic
    use(cache, 2)           # the only evictable slot holds 0
    assert cache.slot_of(0) == -1 and cache.slot_of(1) >= 0


def test_held_variants_are_never_evicted_and_full_is_reported():
    cache, blobs = make(2, 0)
    a = cache.acquire(0)
    b = cache.acquire(1)
    assert cache.try_acquire(2) is None            # both slots held: refused
    with pytest.raises(bd.BitDeltaError) as e:
        cache.acquire(2)
    assert e.value.code == 8                        # BD_ERR_CACHE_FULL
    assert torch.equal(a.clone(), blobs[0]) and torch.equal(b.clone(), blobs[1])
    cache.release(1)
    assert torch.equal(use(cache, 2), blobs[2])     # 1 was free: evicted
    assert cache.slot_of(0) >= 0
    cache.release(0)


def test_pinned_and_held_slots_make_the_cache_full():
    cache, _ = make(2, 1)
    for _ in range(3):
        use(cache, 0)                               # pinned
    held = cache.acquire(1)
    assert cache.try_acquire(2) is None
    cache.release(1)
    assert held is not None and cache.try_acquire(2) is not None
    cache.release(2)


def test_two_holders_share_one_slot():
    cache, blobs = make(2, 0)
    a = cache.acquire(3)
    b = cache.acquire(3)
    assert a.data_ptr() == b.data_ptr()
    assert cache.stats()["loads"] == 1 and cache.stats()["hits"] == 1
    cache.release(3)
    cache.release(3)
    with pytest.raises(bd.BitDeltaError):
        cache.release(3)                            # nothing held any more


def test_reregister_invalidates_a_free_slot():
    cache, _ = make(2, 0)
    use(cache, 1)
    new = blob(99)
    cache.register(1, new)
    assert cache.slot_of(1) == -1
    assert torch.equal(use(cache, 1), new)
    held = cache.acquire(1)
    with pytest.raises(bd.BitDeltaError):
        cache.register(1, blob(7))                  # held: refused
    assert held is not None
    cache.release(1)


def test_bad_arguments():
    cache, _ = make(2, 0)
    with pytest.raises(bd.BitDeltaError):
        cache.acquire(42)                           # not registered
    with pytest.raises(bd.BitDeltaError):
        cache.register(5, torch.zeros(SLOT + 1, dtype=torch.uint8))   # larger than a slot
    arena = torch.zeros(3 * SLOT, dtype=torch.uint8)
    with pytest.raises(bd.BitDeltaError):
        bd.DeltaCache(arena, 1000)                  # slot size not a multiple of 256


def test_threads_acquire_and_release_concurrently():
    cache, blobs = make(3, 1, variants=range(6))
    errors = []

    def worker(seed):
        rng = random.Random(seed)
        for _ in range(300):
            v = rng.randrange(6)
            view = cache.try_acquire(v)
            if view is None:
                continue
            if not torch.equal(view.clone(), blobs[v]):
                errors.append(v)
            cache.release(v)

    threads = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    st = cache.stats()
    assert not errors
    assert st["acquires"] == st["hits"] + st["queued_behind_load"] + st["loads"]
    assert st["loads"] == st["evictions"] + sum(cache.slot_of(v) >= 0 for v in range(6))
