"""The host tier (lora_host_register / lora_acquire / lora_prefetch / lora_release):
more adapters than the pool's slots, swapped in asynchronously with LRU eviction.

Parity: every layer call of a request stream, enqueued without any host
synchronisation between swap-ins and calls, matches the fp64 oracle for the adapters
the request named. Policy: hits, misses and evictions equal those of a plain LRU model
of the same request stream (held adapters are not evictable).
"""
from collections import OrderedDict

import numpy as np
import pytest

import lora_inputs as L
import oracle
from _helpers import assert_parity, to_dev, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
al = pytest.importorskip("adapter_linear_gb300")

D_IN, D_OUT, SLOTS, KEYS = 256, 384, 4, 12


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    al.load_library()
    torch.cuda.set_device(0)


def adapters(seed=51):
    return {100 + k: L.make_adapter(seed, k, D_IN, D_OUT, 8 if k % 3 else 16,
                                    2.0 * (8 if k % 3 else 16) + k, std=0.1)
            for k in range(KEYS)}


def tier_pool(ads, slots=SLOTS):
    pool = al.LoraPool(slots, 16, D_IN, D_OUT)
    for key, a in ads.items():
        pool.host_register(key, to_dev(a.A), to_dev(a.B), a.rank, a.alpha)
    return pool


class LruModel:
    """Capacity-limited LRU over keys; held keys are skipped when choosing a victim."""

    def __init__(self, cap):
        self.cap, self.lru = cap, OrderedDict()
        self.hits = self.misses = self.evictions = 0

    def acquire(self, key, held):
        if key in self.lru:
            self.hits += 1
        else:
            self.misses += 1
            if len(self.lru) == self.cap:
                victim = next(k for k in self.lru if k not in held)
                del self.lru[victim]
                self.evictions += 1
            self.lru[key] = True
        self.lru.move_to_end(key)


def test_request_stream_parity_and_lru_policy():
    ads = adapters()
    pool = tier_pool(ads)
    W = L.normal_bf16(52, L.ROLE_W, 0, (D_OUT, D_IN), 1.0 / 16)
    Wd = to_dev(W)
    g = L.rng_for(53, L.ROLE_IDS)
    keys = np.array(sorted(ads))
    p = 1.0 / np.arange(1, KEYS + 1)
    p /= p.sum()
    model = LruModel(SLOTS)
    stream = torch.cuda.Stream()
    pending = []
    with torch.cuda.stream(stream):
        for r in range(40):
            req = list(dict.fromkeys(int(k) for k in g.choice(keys, size=3, p=p)))
            held = set()
            slot_of = {}
            for k in req:
                model.acquire(k, held)
                held.add(k)
                slot_of[k] = pool.acquire(k, stream)
            T = 48
            pick = g.integers(-1, len(req), size=T)
            key_ids = [req[i] if i >= 0 else -1 for i in pick]
            ids = np.array([slot_of[k] if k >= 0 else -1 for k in key_ids], np.int32)
            X = L.normal_bf16(54, L.ROLE_X, r, (T, D_IN), 1.0)
            Y = pool.linear(to_dev(X), Wd, to_dev(ids), stream=stream)
            for k in req:
                pool.release(slot_of[k])
            pending.append((X, key_ids, Y))
    stream.synchronize()
    assert pool.check_errors() == al.LORA_OK
    st = pool.cache_stats()
    assert (st["hits"], st["misses"], st["evictions"]) == \
        (model.hits, model.misses, model.evictions), st
    assert st["misses"] > SLOTS and st["evictions"] > 0  # the stream did churn
    assert st["registered"] == KEYS and st["resident"] == SLOTS
    # parity: key k's adapter in oracle slot k - 100
    tup = {k - 100: (a.A, a.B, a.rank, a.alpha) for k, a in ads.items()}
    for X, key_ids, Y in pending:
        ids = np.array([k - 100 if k >= 0 else -1 for k in key_ids], np.int32)
        ref = oracle.lora_linear(X, W, ids, tup, KEYS)
        assert_parity(to_host_f64(Y), ref, "host-tier request")
    pool.close()


def test_held_adapters_are_not_evicted():
    ads = adapters()
    pool = tier_pool(ads)
    slots = [pool.acquire(100 + k) for k in range(SLOTS)]
    assert len(set(slots)) == SLOTS
    with pytest.raises(al.LoraError) as e:
        pool.acquire(100 + SLOTS)            # every slot is held
    assert e.value.status == al.LORA_ERR_OOM
    pool.release(slots[1])                   # key 101 may go now
    s = pool.acquire(100 + SLOTS)
    assert s == slots[1]
    assert pool.cache_stats()["evictions"] == 1
    pool.close()


def test_prefetch_then_hit_and_manual_slots_stay():
    ads = adapters()
    pool = tier_pool(ads, slots=SLOTS + 1)
    manual = L.make_adapter(55, 0, D_IN, D_OUT, 16, 8.0, std=0.1)
    pool.load_adapter(0, to_dev(manual.A), to_dev(manual.B), 16, 8.0)
    pool.prefetch(105)
    assert pool.cache_stats()["resident"] == 1
    s = pool.acquire(105)
    st = pool.cache_stats()
    assert (st["hits"], st["misses"]) == (1, 0)
    pool.release(s)
    for k in range(KEYS):                    # churn through every key
        pool.release(pool.acquire(100 + k))
    assert pool.cache_stats()["resident"] == SLOTS
    # the manual slot 0 still holds its adapter
    W = L.normal_bf16(56, L.ROLE_W, 0, (D_OUT, D_IN), 1.0 / 16)
    X = L.normal_bf16(56, L.ROLE_X, 0, (8, D_IN), 1.0)
    ids = np.array([0, -1, 0, 0, -1, 0, 0, 0], np.int32)
    Y = pool.linear(to_dev(X), to_dev(W), to_dev(ids))
    torch.cuda.synchronize()
    ref = oracle.lora_linear(X, W, ids, {0: (manual.A, manual.B, 16, 8.0)}, 1)
    assert_parity(to_host_f64(Y), ref, "manual slot after churn")
    pool.close()


def test_host_tier_errors_and_unload_interplay():
    ads = adapters()
    pool = tier_pool(ads)
    E = al.LoraError
    a = ads[100]
    with pytest.raises(E) as e:
        pool.host_register(100, to_dev(a.A), to_dev(a.B), a.rank, a.alpha)
    assert e.value.status == al.LORA_ERR_SLOT_OCCUPIED
    with pytest.raises(E) as e:
        pool.acquire(999)
    assert e.value.status == al.LORA_ERR_ARG
    s = pool.acquire(100)
    with pytest.raises(E) as e:
        pool.host_unregister(100)            # held
    assert e.value.status == al.LORA_ERR_IN_USE
    with pytest.raises(E) as e:
        pool.unload_adapter(s)               # held through the tier
    assert e.value.status == al.LORA_ERR_IN_USE
    pool.release(s)
    with pytest.raises(E) as e:
        pool.release(s)                      # not held any more
    assert e.value.status == al.LORA_ERR_ARG
    pool.unload_adapter(s)                   # drops it from the cache; the key stays
    assert pool.cache_stats()["resident"] == 0
    s2 = pool.acquire(100)
    assert pool.cache_stats()["misses"] == 2
    pool.release(s2)
    pool.host_unregister(100)
    assert pool.cache_stats()["registered"] == KEYS - 1
    with pytest.raises(E) as e:
        pool.acquire(100)
    assert e.value.status == al.LORA_ERR_ARG
    pool.close()
