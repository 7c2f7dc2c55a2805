"""The slot residency policy (host logic in the library, no GPU): LRU assignment of adapter ids to
slots with pinning, checked against a small independent model of the rule and on hand cases."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def mlora():
    from rank_adapter_gemm_token_gb300 import build, mlora
    build.build()
    mlora.load()
    return mlora


class LruModel:
    """The rule written out plainly: resident ids keep their slot; a new id takes the lowest free
    slot, else the unpinned slot not used by this step whose last use is oldest (lowest index on
    ties); failing steps change nothing."""

    def __init__(self, S):
        self.S, self.id_of, self.last, self.tick, self.pinned = S, [-1] * S, [0] * S, 0, set()

    def assign(self, ids):
        distinct = list(dict.fromkeys(i for i in ids if i >= 0))
        if len(distinct) > self.S:
            return None
        id_of, last, now = list(self.id_of), list(self.last), self.tick + 1
        for i in distinct:
            if i in id_of:
                last[id_of.index(i)] = now
        loads = []
        for i in distinct:
            if i in id_of:
                continue
            free = [s for s in range(self.S) if id_of[s] == -1]
            if free:
                best = free[0]
            else:
                cand = [s for s in range(self.S) if last[s] < now and id_of[s] not in self.pinned]
                if not cand:
                    return None
                best = min(cand, key=lambda s: (last[s], s))
            id_of[best], last[best] = i, now
            loads.append((i, best))
        self.id_of, self.last, self.tick = id_of, last, now
        return [-1 if i < 0 else id_of.index(i) for i in ids], loads


def test_hits_keep_their_slot_and_misses_evict_the_least_recent(mlora):
    c = mlora.mlora_slot_cache_create(3)
    slots, loads = mlora.mlora_slot_cache_assign(c, [10, 11, -1, 10])
    assert slots.tolist() == [0, 1, -1, 0] and loads == [(10, 0), (11, 1)]
    slots, loads = mlora.mlora_slot_cache_assign(c, [12])
    assert slots.tolist() == [2] and loads == [(12, 2)]
    slots, loads = mlora.mlora_slot_cache_assign(c, [11, 13])          # 10 is the least recent
    assert slots.tolist() == [1, 0] and loads == [(13, 0)]
    assert mlora.mlora_slot_cache_lookup(c, 10) == -1 and mlora.mlora_slot_cache_lookup(c, 13) == 0
    mlora.mlora_slot_cache_destroy(c)


def test_pinned_ids_stay_and_failures_change_nothing(mlora):
    c = mlora.mlora_slot_cache_create(2)
    mlora.mlora_slot_cache_assign(c, [1, 2])
    mlora.mlora_slot_cache_pin(c, 1)
    slots, loads = mlora.mlora_slot_cache_assign(c, [3])                # 1 is pinned: 2 goes
    assert slots.tolist() == [1] and loads == [(3, 1)]
    with pytest.raises(mlora.MloraError) as e:                          # 3 ids, 2 slots
        mlora.mlora_slot_cache_assign(c, [4, 5, 6])
    assert e.value.status == mlora.MLORA_ERR_NO_FREE_SLOT
    mlora.mlora_slot_cache_pin(c, 3)
    with pytest.raises(mlora.MloraError) as e:                          # both slots pinned
        mlora.mlora_slot_cache_assign(c, [7])
    assert e.value.status == mlora.MLORA_ERR_NO_FREE_SLOT
    assert mlora.mlora_slot_cache_lookup(c, 1) == 0 and mlora.mlora_slot_cache_lookup(c, 3) == 1
    mlora.mlora_slot_cache_evict(c, 3)
    slots, loads = mlora.mlora_slot_cache_assign(c, [7])                # the freed slot
    assert slots.tolist() == [1] and loads == [(7, 1)]
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_slot_cache_assign(c, [-2])
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    mlora.mlora_slot_cache_destroy(c)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_steps_follow_the_rule(mlora, seed):
    rng = np.random.default_rng(seed)
    S = 6
    c = mlora.mlora_slot_cache_create(S)
    model = LruModel(S)
    for step in range(300):
        if rng.uniform() < 0.05:
            i, pin = int(rng.integers(0, 12)), bool(rng.integers(0, 2))
            mlora.mlora_slot_cache_pin(c, i, pin)
            if pin:
                model.pinned.add(i)
            else:
                model.pinned.discard(i)
        ids = rng.integers(-1, 12, size=int(rng.integers(1, 10))).tolist()
        want = model.assign(ids)
        if want is None:
            with pytest.raises(mlora.MloraError):
                mlora.mlora_slot_cache_assign(c, ids)
        else:
            slots, loads = mlora.mlora_slot_cache_assign(c, ids)
            assert slots.tolist() == want[0] and loads == want[1], step
    mlora.mlora_slot_cache_destroy(c)
