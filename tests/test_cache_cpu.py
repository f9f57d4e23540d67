"""The expert cache's policy on the host (no GPU): ds_moe_cache with no device
tables only plans, so every decision it makes can be checked here.

The policy ("Page the experts off the SSD": routed experts are paged in
through a cache that never becomes a correctness structure): after a call of
layer l, each expert the call used that already has a slot is a hit and
refreshes its slot; each expert it missed takes the first free slot, else
the least recently used slot that this call did not use (ties: the lower
slot), else stays in host memory.  Checked against a small model of that
rule written out here, on scripted cases and on a long random trace over
several layers with Zipf-skewed use.
"""
import ctypes

import numpy as np
import pytest

import bit_quantized_routed_router_gb300 as ds
from bit_quantized_routed_router_gb300 import MoEShape


def shape(E=16):
    return MoEShape(n_embd=1024, n_expert=E, n_ff=1024, n_ff_shared=512, top_k=4)


def cache(n_layers, n_slots, E=16):
    host = [np.zeros(16, np.uint8) for _ in range(n_layers)]  # never read: planning only
    return ds.ExpertCache(shape(E), host, None, n_slots, None)


def used(E, *experts):
    c = np.zeros(E, np.int32)
    c[list(experts)] = 1
    return c


class ModelLRU:
    """The policy restated: slots hold (layer, expert) with a last-use tick."""

    def __init__(self, n_layers, E, n_slots):
        self.where = {}  # (layer, e) -> slot
        self.owner = [None] * n_slots
        self.last = [0] * n_slots
        self.tick = 0
        self.hits = self.misses = 0

    def record(self, layer, counts):
        self.tick += 1
        fills, want = [], []
        for e in np.flatnonzero(counts > 0):
            s = self.where.get((layer, int(e)))
            if s is None:
                self.misses += 1
                want.append(int(e))
            else:
                self.hits += 1
                self.last[s] = self.tick
        for e in want:
            free = [s for s, o in enumerate(self.owner) if o is None]
            if free:
                s = free[0]
            else:
                old = [s for s in range(len(self.owner)) if self.last[s] < self.tick]
                if not old:
                    break
                s = min(old, key=lambda j: (self.last[j], j))
                del self.where[self.owner[s]]
            self.owner[s] = (layer, e)
            self.where[(layer, e)] = s
            self.last[s] = self.tick
            fills.append((s, e))
        return fills


def test_free_slots_first_then_hits():
    c = cache(1, 4)
    assert c.record(0, used(16, 3, 7)) == [(0, 3), (1, 7)]
    assert c.slot(0, 3) == 0 and c.slot(0, 7) == 1 and c.slot(0, 5) == -1
    assert c.record(0, used(16, 3, 7)) == []
    assert c.stats() == {"hits": 2, "misses": 2, "resident": 2}


def test_least_recently_used_slot_is_evicted():
    c = cache(1, 3)
    c.record(0, used(16, 0, 1, 2))   # slots 0,1,2 at tick 1
    c.record(0, used(16, 1))         # slot 1 refreshed
    c.record(0, used(16, 2))         # slot 2 refreshed
    assert c.record(0, used(16, 9)) == [(0, 9)]  # slot 0 (expert 0) is the oldest
    assert c.slot(0, 0) == -1 and c.slot(0, 9) == 0
    assert c.record(0, used(16, 10)) == [(1, 10)]


def test_experts_of_the_same_call_are_never_evicted():
    c = cache(1, 2)
    assert c.record(0, used(16, 0, 1, 2, 3)) == [(0, 0), (1, 1)]
    assert c.slot(0, 2) == -1 and c.slot(0, 3) == -1
    # both slots used by this call: the miss stays in host memory
    assert c.record(0, used(16, 0, 1, 5)) == []
    assert c.slot(0, 5) == -1
    assert c.stats() == {"hits": 2, "misses": 5, "resident": 2}


def test_budget_zero_keeps_everything_in_host_memory():
    c = cache(2, 0)
    for layer in (0, 1, 0):
        assert c.record(layer, used(16, 1, 2, 3)) == []
    assert all(c.slot(l, e) == -1 for l in range(2) for e in range(16))
    assert c.stats() == {"hits": 0, "misses": 9, "resident": 0}


def test_eviction_across_layers_clears_the_other_table():
    c = cache(2, 2)
    c.record(0, used(16, 4, 5))
    assert c.record(1, used(16, 4)) == [(0, 4)]
    assert c.slot(0, 4) == -1 and c.slot(1, 4) == 0 and c.slot(0, 5) == 1


def test_counts_zero_or_negative_are_unused():
    c = cache(1, 4)
    counts = np.array([0, -1, 2] + [0] * 13, np.int32)
    assert c.record(0, counts) == [(0, 2)]


@pytest.mark.parametrize("n_slots", [1, 5, 24, 64])
def test_random_trace_matches_the_model(n_slots):
    n_layers, E, k = 3, 32, 4
    rng = np.random.default_rng(n_slots)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    c, m = cache(n_layers, n_slots, E), ModelLRU(n_layers, E, n_slots)
    for step in range(400):
        layer = step % n_layers
        counts = np.zeros(E, np.int32)
        for _ in range(int(rng.integers(1, 5))):  # 1..4 tokens, k distinct experts each
            counts[rng.choice(E, size=k, replace=False, p=p)] += 1
        assert c.record(layer, counts) == m.record(layer, counts), step
    for l in range(n_layers):
        for e in range(E):
            assert c.slot(l, e) == m.where.get((l, e), -1)
    st = c.stats()
    assert (st["hits"], st["misses"]) == (m.hits, m.misses)
    assert st["resident"] == sum(o is not None for o in m.owner)


def test_host_argument_checks():
    L = ds.lib()
    sh = shape()
    out = ctypes.c_void_p()
    err = ctypes.create_string_buffer(256)
    host = (ctypes.c_void_p * 1)(None)
    assert L.ds_moe_cache_create(ctypes.byref(sh.c()), 1, host, None, 2, None, ctypes.byref(out), err, 256) \
        == ds.DS_ERR_INVALID_ARG
    buf = np.zeros(16, np.uint8)
    host = (ctypes.c_void_p * 1)(buf.ctypes.data)
    assert L.ds_moe_cache_create(ctypes.byref(sh.c()), 0, host, None, 2, None, ctypes.byref(out), err, 256) \
        == ds.DS_ERR_INVALID_ARG
    # device tables need slots when the cache holds experts
    fake = ctypes.c_void_p(256)
    assert L.ds_moe_cache_create(ctypes.byref(sh.c()), 1, host, None, 2, fake, ctypes.byref(out), err, 256) \
        == ds.DS_ERR_INVALID_ARG
    c = cache(2, 2)
    with pytest.raises(ds.DsMoeError):
        c.slot(2, 0)
    with pytest.raises(ds.DsMoeError):
        c.slot(0, 16)
    with pytest.raises(ds.DsMoeError):
        c.record(5, used(16, 1))
    # a planning-only cache cannot run a layer
    assert L.ds_moe_cache_layer(c.handle, 0, None, None, 1, None, None, 0, None, err, 256) == ds.DS_ERR_INVALID_ARG
    assert b"device tables" in err.value
