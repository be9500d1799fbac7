"""The FIFO of host-offloaded KV chunks ("SparseSpec-MLSys26", 动态 KV 管理:
on device-memory pressure requests' KV goes to the host chunk by chunk, first
in first out, and offloaded requests come back -- ahead of new ones -- as soon
as device memory is free).  Plain host code behind the C ABI; no GPU needed.
The checks are the properties the header states: a request's chunks tile its
positions, requests come back whole and in the order they left, the resident
count never passes the capacity, new requests wait while offloaded ones are
queued, and a refused call changes nothing."""
import ctypes

import numpy as np
import pytest

import sparse_self_speculative_pillar_gb300 as P


def state(f):
    return (f.capacity, f.resident, f.chunk, f.head, f.count, bytes(f.q[:f.count]) if f.count else b"")


def test_chunks_tile_each_request_and_requests_come_back_in_eviction_order():
    f = P.pillar_offload_init(capacity=10000, chunk=256)
    lens = {11: 1000, 5: 37, 42: 4096, 7: 256}
    for req, n in lens.items():
        assert P.pillar_offload_reserve(f, n, new_request=True)
    order = [42, 11, 7, 5]
    for req in order:
        nc = P.pillar_offload_evict(f, req, lens[req])
        assert nc == -(-lens[req] // 256)
    assert f.resident == 0
    chunks = P.pillar_offload_reload(f)
    assert [c[0] for c in chunks if c[3]] == order  # whole requests, in the order they left
    for req in order:
        mine = [c for c in chunks if c[0] == req]
        assert [c[1] for c in mine] == list(range(0, lens[req], 256))
        assert sum(c[2] for c in mine) == lens[req] and all(c[2] == 256 for c in mine[:-1])
        assert mine[-1][3] == 1 and all(c[3] == 0 for c in mine[:-1])
    assert f.count == 0 and f.resident == sum(lens.values())


def test_reload_takes_whole_requests_that_fit_and_keeps_strict_order():
    f = P.pillar_offload_init(capacity=1000, chunk=100)
    assert P.pillar_offload_reserve(f, 1000, new_request=True)
    P.pillar_offload_evict(f, 1, 600)  # resident 400
    P.pillar_offload_evict(f, 2, 150)  # resident 250
    assert f.resident == 250
    assert P.pillar_offload_reserve(f, 300, new_request=False)  # a running request grows: 550
    # 450 free: request 1 (600) does not fit, and request 2 (150) must not overtake it
    assert P.pillar_offload_reload(f) == []
    P.pillar_offload_release(f, 300)  # 750 free
    got = P.pillar_offload_reload(f)
    assert [c[0] for c in got] == [1] * 6 + [2, 2] and f.count == 0 and f.resident == 1000
    # a chunk budget that cannot hold the next request's chunks stops there
    P.pillar_offload_evict(f, 3, 350)
    assert P.pillar_offload_reload(f, max_out=3) == [] and f.count == 4
    assert [c[0] for c in P.pillar_offload_reload(f, max_out=4)] == [3] * 4


def test_new_requests_wait_while_offloaded_ones_are_queued():
    f = P.pillar_offload_init(capacity=100, chunk=16)
    assert P.pillar_offload_reserve(f, 60, new_request=True)
    P.pillar_offload_evict(f, 0, 60)
    assert not P.pillar_offload_reserve(f, 10, new_request=True)  # offloaded work comes back first
    assert P.pillar_offload_reserve(f, 10, new_request=False)     # a resident request may still grow
    assert P.pillar_offload_reload(f) != [] and f.count == 0
    assert P.pillar_offload_reserve(f, 30, new_request=True)
    assert not P.pillar_offload_reserve(f, 1, new_request=False)  # 100 of 100 in use


def test_random_traffic_keeps_the_counts_consistent():
    rng = np.random.default_rng(17)
    cap = 50000
    f = P.pillar_offload_init(capacity=cap, chunk=512)
    resident = {}     # req -> length
    queued = []       # requests in eviction order, with lengths
    nxt = 0
    for _ in range(3000):
        op = rng.integers(5)
        if op == 0:
            n = int(rng.integers(1, 6000))
            if P.pillar_offload_reserve(f, n, new_request=True):
                assert not queued
                resident[nxt] = n
                nxt += 1
        elif op == 1 and resident:
            req = int(rng.choice(list(resident)))
            n = int(rng.integers(1, 300))
            if P.pillar_offload_reserve(f, n, new_request=False):
                resident[req] += n
        elif op == 2 and resident:
            req = int(rng.choice(list(resident)))
            try:
                P.pillar_offload_evict(f, req, resident[req])
            except P.PillarError:  # the queue is full: nothing changed
                continue
            queued.append((req, resident.pop(req)))
        elif op == 3 and resident:
            req = int(rng.choice(list(resident)))
            P.pillar_offload_release(f, resident.pop(req))
        else:
            got = P.pillar_offload_reload(f)
            back = [c[0] for c in got if c[3]]
            assert back == [r for r, _ in queued[:len(back)]]
            for r, n in queued[:len(back)]:
                assert sum(c[2] for c in got if c[0] == r) == n
                resident[r] = n
            queued = queued[len(back):]
        assert f.resident == sum(resident.values()) <= cap
        assert f.count == sum(-(-n // 512) for _, n in queued)


def test_refused_calls_change_nothing():
    f = P.pillar_offload_init(capacity=100, chunk=1)
    assert P.pillar_offload_reserve(f, 100, new_request=True)
    before = state(f)
    for bad in (lambda: P.pillar_offload_evict(f, 0, 101), lambda: P.pillar_offload_evict(f, 0, 0),
                lambda: P.pillar_offload_release(f, 101), lambda: P.pillar_offload_release(f, -1),
                lambda: P.pillar_offload_reserve(f, -1, new_request=False)):
        with pytest.raises(P.PillarError):
            bad()
        assert state(f) == before
    # more chunks than the queue holds
    g = P.pillar_offload_init(capacity=P.OFFLOAD_QUEUE + 10, chunk=1)
    assert P.pillar_offload_reserve(g, P.OFFLOAD_QUEUE + 10, new_request=True)
    before = state(g)
    with pytest.raises(P.PillarError):
        P.pillar_offload_evict(g, 0, P.OFFLOAD_QUEUE + 1)
    assert state(g) == before
    for cap, chunk in ((-1, 4), (10, 0)):
        with pytest.raises(P.PillarError):
            P.pillar_offload_init(cap, chunk)


def test_struct_layout():
    assert ctypes.sizeof(P.PillarOffloadChunk) == 16
    assert ctypes.sizeof(P.PillarOffloadFifo) == 32 + 16 * P.OFFLOAD_QUEUE
