"""Host offload of KV on the GPU ("SparseSpec-MLSys26", 动态 KV 管理: a
request's KV goes to host memory chunk by chunk and comes back before the
request is scheduled again).  pillar_kv_offload packs slot blocks into
page-locked host rows (written by the kernel through their device mapping),
pillar_kv_reload puts them back in whatever slots the allocator hands out.
Checked against the oracle's gather and append, with out-of-range slots
flagged, pageable host memory refused, and an attention step over a request
whose KV travelled through the host, driven by the offload FIFO."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import sparse_self_speculative_pillar_gb300 as P  # noqa: E402
from tests._gpu_common import Gpu, compare_attn, run_oracle  # noqa: E402


def _shape(Hkv, D, num_slots):
    return P.make_shape(B=1, Hq=Hkv, Hkv=Hkv, D=D, k=1, max_sparse=0, max_len=1, num_slots=num_slots)


@pytest.mark.parametrize("D,Hkv,n,num_slots", [(128, 8, 2000, 8192), (64, 3, 37, 257), (128, 1, 1, 5)])
def test_offload_and_reload_round_trip(D, Hkv, n, num_slots):
    rng = np.random.default_rng(D + n)
    k_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    v_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    slots = rng.permutation(num_slots)[:n].astype(np.int32)
    want_k, want_v, skipped = oracle.kv_offload(k_pool, v_pool, slots)
    assert not skipped
    shape = _shape(Hkv, D, num_slots)
    dk, dv = torch.from_numpy(k_pool).cuda(), torch.from_numpy(v_pool).cuda()
    hk = torch.zeros((n, Hkv, D), dtype=torch.int16).pin_memory()
    hv = torch.zeros((n, Hkv, D), dtype=torch.int16).pin_memory()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ds = torch.from_numpy(slots).cuda()
    P.pillar_kv_offload(shape, dk, dv, ds, hk, hv, device_flags=flags)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hk.numpy(), want_k)
    np.testing.assert_array_equal(hv.numpy(), want_v)
    # back into other slots of cleared pools
    new = np.roll(slots, 1)
    dk.zero_()
    dv.zero_()
    P.pillar_kv_reload(shape, hk, hv, torch.from_numpy(new).cuda(), dk, dv, device_flags=flags)
    torch.cuda.synchronize()
    ek, ev, _ = oracle.kv_append(np.zeros_like(k_pool), np.zeros_like(v_pool), want_k, want_v, new)
    np.testing.assert_array_equal(dk.cpu().numpy(), ek)
    np.testing.assert_array_equal(dv.cpu().numpy(), ev)
    assert int(flags.item()) == 0


def test_out_of_range_slots_are_flagged_and_pageable_memory_refused():
    D, Hkv, num_slots = 64, 2, 16
    rng = np.random.default_rng(8)
    k_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    slots = np.array([3, num_slots, -4, 15], np.int32)
    want, _, skipped = oracle.kv_offload(k_pool, k_pool, slots)
    assert skipped
    shape = _shape(Hkv, D, num_slots)
    dk = torch.from_numpy(k_pool).cuda()
    hk = torch.zeros((4, Hkv, D), dtype=torch.int16).pin_memory()
    hv = torch.zeros((4, Hkv, D), dtype=torch.int16).pin_memory()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pillar_kv_offload(shape, dk, dk, torch.from_numpy(slots).cuda(), hk, hv, device_flags=flags)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hk.numpy(), want)  # skipped rows left as they were (zero)
    assert int(flags.item()) == P.FLAG_SLOT
    pageable = torch.zeros((4, Hkv, D), dtype=torch.int16)  # not page-locked: no device address
    with pytest.raises(P.PillarError):
        P.pillar_kv_offload(shape, dk, dk, torch.from_numpy(slots).cuda(), pageable, hv)
    with pytest.raises(P.PillarError):
        P.pillar_kv_reload(shape, pageable, hv, torch.from_numpy(slots).cuda(), dk, dk)


def test_attention_over_requests_that_went_through_the_host():
    """Two requests of a step are offloaded (the FIFO chunks their positions),
    their slots are given to other data, and they are reloaded into fresh
    slots in the order they left; with the slot table updated the step's
    outputs are bit for bit those of the step before the move, and match the
    oracle."""
    w = W.generate(W.scaled("qwen3_8b", B=10, length_scale=0.08, seed_offset=21))
    g = Gpu(w)
    g.attn()
    assert g.attn_flags() == 0
    before = g.host()
    shape = g.shape
    used = set(w.slot_table.tolist())
    spare = np.array([s for s in range(w.num_slots) if s not in used], np.int32)
    victims = [int(np.nonzero(w.req_mode == 1)[0][0]), int(np.nonzero(w.req_mode == 0)[0][0])]
    lens = {b: int(w.req_len[b]) for b in victims}
    assert spare.size >= sum(lens.values())
    f = P.pillar_offload_init(capacity=int(sum(w.req_len)), chunk=128)
    assert P.pillar_offload_reserve(f, int(sum(w.req_len)), new_request=True)
    host = {}
    for b in victims:  # offload chunk by chunk
        P.pillar_offload_evict(f, b, lens[b])
        off = int(w.kv_off[b])
        slots = torch.from_numpy(w.slot_table[off:off + lens[b]].copy()).cuda()
        hk = torch.empty((lens[b], w.Hkv, w.D), dtype=torch.int16).pin_memory()
        hv = torch.empty((lens[b], w.Hkv, w.D), dtype=torch.int16).pin_memory()
        for c0 in range(0, lens[b], 128):
            c1 = min(lens[b], c0 + 128)
            P.pillar_kv_offload(shape, g.k_pool, g.v_pool, slots[c0:c1], hk[c0:c1], hv[c0:c1])
        host[b] = (hk, hv)
        g.k_pool[slots.long()] = 7  # the freed slots are reused by other data
        g.v_pool[slots.long()] = -7
    torch.cuda.synchronize()
    chunks = P.pillar_offload_reload(f)
    assert [c[0] for c in chunks if c[3]] == victims
    table = w.slot_table.copy()
    free = list(spare)
    for req, first, n, _ in chunks:  # back, chunk by chunk, into fresh slots
        new = np.array(free[:n], np.int32)
        free = free[n:]
        hk, hv = host[req]
        P.pillar_kv_reload(shape, hk[first:first + n], hv[first:first + n], torch.from_numpy(new).cuda(),
                           g.k_pool, g.v_pool)
        off = int(w.kv_off[req])
        table[off + first:off + first + n] = new
    g.slot_table.copy_(torch.from_numpy(table).cuda())
    g.out.zero_()
    g.logits.zero_()
    g.attn()
    assert g.attn_flags() == 0
    after = g.host()
    np.testing.assert_array_equal(after["out"], before["out"])
    np.testing.assert_array_equal(after["logits"], before["logits"])
    compare_attn(w, after, run_oracle(w))
