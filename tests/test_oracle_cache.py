"""Pins for the expert-cache oracle (oracle.cache_oracle) and the library's
host-side policy (moe_expert_cache_plan), which must take the same decisions.

| property                          | pinned by                                               |
|-----------------------------------|---------------------------------------------------------|
| the stated policy, step by step   | tests/golden/expert_cache_lru.json, worked by hand      |
| least recently used is optimal    | never fewer misses than Belady's optimum (exhaustive     |
|   in no case, and never worse     | search on tiny traces); equal to it when C = E          |
|   than loading everything         |                                                         |
| LRU stack property                | one-expert steps: misses never grow with more slots     |
| needed experts stay resident      | invariant after every step                              |
| counters                          | hits + misses = total expert lookups                    |
| library == oracle                 | identical loads and maps on random traces (C ABI, CPU)  |

Planted policy mistakes at the end (FIFO, MRU, highest-slot ties) each fail."""
from __future__ import annotations

import ctypes
import itertools
import json
import pathlib
import random

import pytest

from oracle.cache_oracle import CacheTooSmall, LRUCache, simulate

GOLDEN = pathlib.Path(__file__).parent / "golden" / "expert_cache_lru.json"


def test_golden_trace():
    g = json.loads(GOLDEN.read_text())
    c, loads = simulate(g["trace"], g["E"], g["C"])
    assert [[list(x) for x in step] for step in loads] == g["loads"]
    assert (c.hits, c.misses) == (g["hits"], g["misses"])
    assert c.slot_of == g["final_slot_of"]


def _random_trace(rng, E, C, steps, max_need=None):
    max_need = max_need or C
    return [rng.sample(range(E), rng.randint(1, max_need)) for _ in range(steps)]


def _belady_min_misses(trace, E, C):
    """Exhaustive search: the fewest misses any replacement choice achieves."""
    best = [None]

    def rec(i, resident, misses):
        if best[0] is not None and misses >= best[0]:
            return
        if i == len(trace):
            best[0] = misses
            return
        need = set(trace[i])
        miss = sorted(need - resident)
        keep_pool = sorted(resident - need)
        free = C - len(resident)
        n_evict = max(0, len(miss) - free)
        for ev in itertools.combinations(keep_pool, n_evict):
            rec(i + 1, (resident - set(ev)) | need, misses + len(miss))

    rec(0, frozenset(), 0)
    return best[0]


def test_never_better_than_optimal_and_optimal_when_everything_fits():
    rng = random.Random(5)
    for _ in range(60):
        E, C = rng.randint(2, 5), None
        C = rng.randint(1, E)
        trace = _random_trace(rng, E, C, rng.randint(1, 7))
        c, _ = simulate(trace, E, C)
        opt = _belady_min_misses(trace, E, C)
        assert c.misses >= opt
        if C == E:
            assert c.misses == len(set(e for s in trace for e in s)) == opt


def test_lru_stack_property_on_single_expert_steps():
    rng = random.Random(7)
    for _ in range(40):
        E = rng.randint(2, 8)
        trace = [[rng.randrange(E)] for _ in range(30)]
        misses = [simulate(trace, E, C)[0].misses for C in range(1, E + 1)]
        assert all(a >= b for a, b in zip(misses, misses[1:])), misses


def test_invariants_and_counters():
    rng = random.Random(9)
    for _ in range(30):
        E = rng.randint(2, 10)
        C = rng.randint(2, E)
        c = LRUCache(E, C)
        lookups = 0
        for need in _random_trace(rng, E, C, 25):
            c.plan(need)
            lookups += len(set(need))
            for e in need:
                assert c.expert_in[c.slot_of[e]] == e
            assert len([s for s in c.expert_in if s >= 0]) <= C
        assert c.hits + c.misses == lookups


def test_too_many_needed_is_an_error():
    c = LRUCache(4, 2)
    with pytest.raises(CacheTooSmall):
        c.plan([0, 1, 2])


# ------------------------------------------------------------------ library
@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_55_b300 import _lib, build
    build.build()
    return _lib


def _lib_plan(L, st, E, need):
    arr = (ctypes.c_int * E)(*[1 if e in need else 0 for e in range(E)])
    le, ls, n = (ctypes.c_int * E)(), (ctypes.c_int * E)(), ctypes.c_int()
    rc = L.load().moe_expert_cache_plan(ctypes.byref(st), arr, le, ls, ctypes.byref(n))
    return rc, [(le[i], ls[i]) for i in range(n.value)]


def test_library_policy_matches_oracle(lib):
    rng = random.Random(11)
    for _ in range(50):
        E = rng.randint(1, 32)
        C = rng.randint(1, E)
        st = lib.ExpertCacheState()
        assert lib.load().moe_expert_cache_init(ctypes.byref(st), E, C) == 0
        ref = LRUCache(E, C)
        for need in _random_trace(rng, E, C, 40):
            rc, loads = _lib_plan(lib, st, E, set(need))
            assert rc == 0
            assert loads == ref.plan(need)
            assert list(st.slot_of)[:E] == ref.slot_of
            assert list(st.expert_in)[:C] == ref.expert_in
        assert (st.hits, st.misses, st.step) == (ref.hits, ref.misses, ref.step)


def test_library_rejects_bad_states_and_oversized_steps(lib):
    L = lib.load()
    st = lib.ExpertCacheState()
    assert L.moe_expert_cache_init(ctypes.byref(st), 8, 9) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_expert_cache_init(ctypes.byref(st), 33, 2) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_expert_cache_init(ctypes.byref(st), 8, 2) == 0
    rc, _ = _lib_plan(lib, st, 8, {0, 1, 2})
    assert rc == lib.MOE_ERR_UNSUPPORTED and st.step == 0 and st.misses == 0
    st.slot_of[0] = 1  # maps that disagree
    rc, _ = _lib_plan(lib, st, 8, {0})
    assert rc == lib.MOE_ERR_INVALID_ARG


# ------------------------------------------------------------------ planted mistakes
class _FIFO(LRUCache):
    """First in, first out: the use mark is set on loading only."""

    def touch(self, slot, loaded_now):
        if loaded_now:
            self.last_use[slot] = self.step


class _MRU(LRUCache):
    def victim(self, candidates):
        return max(candidates, key=lambda s: (self.last_use[s], -s))


class _HighTie(LRUCache):
    def victim(self, candidates):
        return min(candidates, key=lambda s: (self.last_use[s], -s))


@pytest.mark.parametrize("cls", [_FIFO, _MRU, _HighTie])
def test_planted_policy_mistakes_fail_the_golden_trace(cls):
    g = json.loads(GOLDEN.read_text())
    c = cls(g["E"], g["C"])
    loads = [[list(x) for x in c.plan(step)] for step in g["trace"]]
    assert loads != g["loads"] or c.slot_of != g["final_slot_of"]
