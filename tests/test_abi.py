"""The C-ABI library builds for sm_103a, loads, and exports every entry point
declared in include/pillar.h; host-side argument checks return the
documented codes without touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import sparse_self_speculative_pillar_gb300 as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pillar.h")).read()
    return sorted(set(re.findall(r"PILLAR_API\s+[\w\s\*]*?\b(pillar_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    P.build()
    return P.load()


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(P.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_shape_struct_matches_header_layout():
    # 12 int32, then int64 (8-aligned at 48), float, 3 int32 -> 72 bytes
    assert ctypes.sizeof(P.PillarShape) == 72
    assert P.PillarShape.num_slots.offset == 48
    assert P.PillarShape.schedule.offset == 60
    assert P.PillarShape.wait_timeout_us.offset == 64
    # pillar_buckets_t: int32 nbuckets, then PILLAR_MAX_BUCKETS int32 counts
    src = open(os.path.join(ROOT, "include", "pillar.h")).read()
    assert int(re.search(r"#define PILLAR_MAX_BUCKETS (\d+)", src).group(1)) == P.MAX_BUCKETS
    assert ctypes.sizeof(P.PillarBuckets) == 4 * (1 + P.MAX_BUCKETS)


def _shape(**kw):
    base = dict(B=4, Hq=32, Hkv=8, D=128, k=8, max_sparse=64, max_len=8192, num_slots=1 << 20, max_topk=410)
    base.update(kw)
    return P.make_shape(**base)


def test_workspace_sizes_and_argument_checks(lib):
    n = P.pillar_attn_workspace_bytes(_shape())
    assert n > 0 and n % 256 == 0
    for sched in (P.SCHEDULE_DRAFT_ONLY, P.SCHEDULE_VERIFY_ONLY, P.SCHEDULE_UNIFORM_ROWS, P.SCHEDULE_NAIVE_JOINT):
        assert P.pillar_attn_workspace_bytes(_shape(schedule=sched)) == n  # the schedule needs no other room
    assert P.pillar_topk_workspace_bytes(_shape(), 3) >= 3 * 8 * 8192 * 4
    for bad in (dict(D=96), dict(Hq=30), dict(k=15, Hq=40, Hkv=8), dict(max_len=0), dict(row_lo=3, row_hi=2),
                dict(verify_chunk=100), dict(draft_chunk=8192), dict(Hq=72, Hkv=8), dict(schedule=5), dict(wait_timeout_us=-1),
                dict(schedule=-1)):
        with pytest.raises(P.PillarError) as e:
            P.pillar_attn_workspace_bytes(_shape(**bad))
        assert e.value.status == -1
    # shapes whose workspace size would not fit in 64 bits are refused, not wrapped
    huge = _shape(B=1 << 27, Hq=64, Hkv=8, k=7, max_len=(1 << 31) - 1, verify_chunk=64, max_sparse=0)
    with pytest.raises(P.PillarError) as e:
        P.pillar_attn_workspace_bytes(huge)
    assert e.value.status == -1
    with pytest.raises(P.PillarError) as e:
        P.pillar_topk_workspace_bytes(_shape(max_len=1 << 30), (1 << 31) - 1)
    assert e.value.status == -1
    big = _shape(B=512, k=12, Hq=32, Hkv=8, max_len=32768, max_sparse=4096)  # large but real
    assert P.pillar_attn_workspace_bytes(big) > 0
    s = _shape()
    # null workspace -> -2, with no device work enqueued
    st = lib.pillar_attn_unified(ctypes.byref(s), *([ctypes.c_void_p(16)] * 11), None, 0, None)
    assert st == -2
    # null tensor -> -1
    st = lib.pillar_attn_unified(ctypes.byref(s), None, *([ctypes.c_void_p(16)] * 10), ctypes.c_void_p(256), 1 << 40,
                                 None)
    assert st == -1
    # a logits pointer that is 4- but not 8-byte aligned -> -1 (pairs of logits are stored together)
    ptrs = [ctypes.c_void_p(256)] * 11
    ptrs[9] = ctypes.c_void_p(256 + 4)
    st = lib.pillar_attn_unified(ctypes.byref(s), *ptrs, ctypes.c_void_p(256), 1 << 40, None)
    assert st == -1
    # Top-K: a pointer that is not 4-byte aligned -> -1, before anything is enqueued
    tptr = [ctypes.c_void_p(256)] * 7
    tptr[5] = ctypes.c_void_p(256 + 2)
    assert lib.pillar_topk_select(ctypes.byref(s), 3, *tptr, ctypes.c_void_p(256), 1 << 40, None) == -1
    assert lib.pillar_topk_select_noalloc(ctypes.byref(s), 3, *tptr, None, None) == -1
    # B == 0 -> nothing to do
    s0 = _shape(B=0)
    assert lib.pillar_attn_unified(ctypes.byref(s0), *([None] * 12), 0, None) == 0
    assert lib.pillar_topk_select(ctypes.byref(s), 0, *([None] * 8), 0, None) == 0
    assert P.pillar_status_string(-4).startswith("device")
    # pillar_kv_append: host checks before anything is enqueued
    assert lib.pillar_kv_append(ctypes.byref(s), None, None, None, 0, None, None, None, None) == 0  # no tokens
    assert lib.pillar_kv_append(ctypes.byref(s), None, None, None, -1, None, None, None, None) == -1
    assert lib.pillar_kv_append(ctypes.byref(s), None, None, None, 3, None, None, None, None) == -1
    odd = ctypes.c_void_p(16 + 8)  # not 16-byte aligned
    assert lib.pillar_kv_append(ctypes.byref(s), odd, odd, odd, 3, odd, odd, None, None) == -1


def test_workspace_covers_the_most_items_the_planner_can_emit():
    """The planner splits a verify request of L keys into ceil(L / chunk)
    items (chunk = verify_chunk, or by default 1024 keys below 8192 positions
    and 2048 from there on) and a draft list of n keys into ceil(n /
    draft_chunk) items (2048 keys by default); every item of a split (request, KV head) writes
    (k+1)*G partial rows of D fp32 values plus an LSE.  The workspace must
    hold that many item records and partial rows for the worst batch of the
    shape."""
    rng = np.random.default_rng(21)
    for _ in range(200):
        Hkv = int(rng.integers(1, 9))
        G = int(rng.integers(1, 9))
        k = int(rng.integers(0, 64 // G))
        D = int(rng.choice([64, 128]))
        vc = int(rng.choice([0, 64, 128, 1024, 2048]))
        dc = int(rng.choice([0, 64, 512, 2048]))
        s = _shape(B=int(rng.integers(1, 300)), Hq=G * Hkv, Hkv=Hkv, D=D, k=k,
                   max_len=int(rng.integers(1, 40000)), max_sparse=int(rng.integers(0, 5000)),
                   verify_chunk=vc, draft_chunk=dc, row_lo=min(1, k), row_hi=k + 1)
        units = s.B * Hkv
        v_items = -(-s.max_len // (vc or 1024))          # the default's smaller chunk gives the most items
        d_items = -(-s.max_sparse // (dc or 2048)) if s.max_sparse else 1  # draft items: 2048 keys by default
        items = units * max(v_items, d_items, 1)
        rows = items * (k + 1) * G
        need = items * 16 + rows * (D + 1) * 4              # item records + partial rows (D values + LSE)
        assert P.pillar_attn_workspace_bytes(s) >= need
