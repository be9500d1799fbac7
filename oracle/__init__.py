"""fp64 CPU oracle for the PillarAttn unified step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It restates, in plain C compiled with
gcc, what the GPU path computes (see ``pillar_oracle.c`` for the page
citations and the readings of points the pages leave open).  It shares no
code with the CUDA library and never calls it.

Pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, invariants and brute force.  Nothing in it is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pillar_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libpillar_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no target-specific flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        lib.oracle_attn_unified.argtypes = [i32, i32, i32, i32, i32, i64, f64, i32,
                                            P, P, P, P, P, P, P, P, P, P, P, P, i32]
        lib.oracle_attn_unified.restype = i32
        lib.oracle_topk_select.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                           P, P, P, P, P, P, P, i32]
        lib.oracle_topk_select.restype = i32
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = f64
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def bf16_to_f64(bits: int) -> float:
    """Exact value of one bf16 bit pattern (the oracle's own widening)."""
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


@dataclass
class AttnResult:
    out: np.ndarray        # [T_q, Hq, D] fp64
    lse: np.ndarray        # [T_q, Hq] fp64 (draft rows included)
    logits: np.ndarray     # packed [sum_v Hq*(k+1)*L_v] fp64 (selected verify requests)
    status: int


def attn_unified(*, Hq, Hkv, D, k, scale, q, k_pool, v_pool, slot_table, req_mode, req_len,
                 sparse_idx, sparse_cnt, select=None, want_logits=True, nthreads=None):
    """Run the unified draft/verify step in fp64 (see ``oracle_attn_unified``).

    bf16 arrays are passed as their uint16 bit patterns.  ``select`` (bool [B])
    restricts the work to some requests; the logits buffer is then packed over
    the selected verify requests only.
    """
    req_mode = _c(req_mode, np.int32)
    req_len = _c(req_len, np.int32)
    B = int(req_mode.shape[0])
    q = _c(q, np.uint16)
    T_q = int(q.shape[0])
    sparse_idx = _c(sparse_idx, np.int32)
    max_sparse = int(sparse_idx.shape[-1]) if sparse_idx.size else 0
    sel = None if select is None else _c(np.asarray(select).astype(bool), np.uint8)
    out = np.zeros((T_q, Hq, D), np.float64)
    lse = np.full((T_q, Hq), np.nan, np.float64)
    ver = (req_mode == 1) if sel is None else ((req_mode == 1) & sel.astype(bool))
    n_logits = int(Hq * (k + 1) * req_len[ver].astype(np.int64).sum()) if want_logits else 0
    logits = np.empty(n_logits, np.float64) if want_logits else None
    st = _load().oracle_attn_unified(
        B, Hq, Hkv, D, k, int(k_pool.shape[0]), float(scale), max_sparse,
        _ptr(q), _ptr(_c(k_pool, np.uint16)), _ptr(_c(v_pool, np.uint16)),
        _ptr(_c(slot_table, np.int32)), _ptr(req_mode), _ptr(req_len),
        _ptr(sparse_idx), _ptr(_c(sparse_cnt, np.int32)), _ptr(sel),
        _ptr(out), _ptr(lse), _ptr(logits), int(nthreads or default_threads()))
    if st == -1:
        raise ValueError("oracle_attn_unified: bad dimensions")
    if st == -5:
        raise MemoryError("oracle_attn_unified")
    return AttnResult(out, lse, logits if logits is not None else np.empty(0), st)


@dataclass
class TopkResult:
    next_idx: np.ndarray   # [V, Hkv, max_topk] int32 (first next_cnt entries valid)
    next_cnt: np.ndarray   # [V, Hkv] int32
    scores: np.ndarray     # packed [sum_v Hkv*L_v] fp64
    status: int


def topk_select(*, Hq, Hkv, k, row_lo, row_hi, logits, lse, L, K, max_topk, nthreads=None):
    """Averaged exact scores and Top-K per (verify request, KV head), in fp64.

    ``logits`` is packed [V][Hq][k+1][L_v]; ``lse`` is [V, Hq, k+1].
    """
    L = _c(L, np.int32)
    K = _c(K, np.int32)
    V = int(L.shape[0])
    logits = _c(logits, np.float64)
    lse = _c(lse, np.float64)
    next_idx = np.full((V, Hkv, max(max_topk, 1)), -1, np.int32)
    next_cnt = np.zeros((V, Hkv), np.int32)
    scores = np.empty(int(Hkv * L.astype(np.int64).sum()), np.float64)
    st = _load().oracle_topk_select(V, Hq, Hkv, k, row_lo, row_hi, max_topk, _ptr(logits), _ptr(lse),
                                    _ptr(L), _ptr(K), _ptr(next_idx), _ptr(next_cnt), _ptr(scores),
                                    int(nthreads or default_threads()))
    if st == -5:
        raise MemoryError("oracle_topk_select")
    if st == -1 and V:
        raise ValueError("oracle_topk_select: bad arguments")
    return TopkResult(next_idx[:, :, :max_topk], next_cnt, scores, st)


def verify_lse_of(res: AttnResult, req_mode, k, Hq, select=None):
    """Gather the verify rows' LSE into the [V, Hq, k+1] layout of the GPU dump."""
    req_mode = np.asarray(req_mode)
    rows = []
    q_off = 0
    for b, m in enumerate(req_mode):
        n = k + 1 if m == 1 else 1
        if m == 1 and (select is None or select[b]):
            rows.append(res.lse[q_off:q_off + n, :].T)  # [Hq, k+1]
        q_off += n
    if not rows:
        return np.zeros((0, Hq, k + 1))
    return np.stack(rows, 0)


def kv_append(k_pool, v_pool, k_new, v_new, slots):
    """The pools after appending new tokens ("SparseSpec-MLSys26", Unified
    batch scheduler + fused attention kernel: page size 1, one slot per
    token): copies of k_pool / v_pool [num_slots, Hkv, D] in which row
    slots[i] holds token i's rows k_new[i] / v_new[i]; a slot outside
    [0, num_slots) is skipped.  Returns (k, v, any_skipped).  One token at a
    time, in order."""
    k = np.array(k_pool, copy=True)
    v = np.array(v_pool, copy=True)
    skipped = False
    for i, s in enumerate(np.asarray(slots).tolist()):
        if 0 <= s < k.shape[0]:
            k[s] = k_new[i]
            v[s] = v_new[i]
        else:
            skipped = True
    return k, v, skipped


def kv_offload(k_pool, v_pool, slots):
    """The packed rows an offload writes to host memory ("SparseSpec-MLSys26",
    动态 KV 管理: a request's KV goes to the host chunk by chunk): row i holds
    the slot block k_pool[slots[i]] / v_pool[slots[i]]; a slot outside
    [0, num_slots) leaves its row as it was (zeros here) and is reported.
    Returns (k_rows, v_rows, any_skipped).  One row at a time, in order."""
    slots = np.asarray(slots).tolist()
    k = np.zeros((len(slots),) + tuple(k_pool.shape[1:]), dtype=np.asarray(k_pool).dtype)
    v = np.zeros((len(slots),) + tuple(v_pool.shape[1:]), dtype=np.asarray(v_pool).dtype)
    skipped = False
    for i, s in enumerate(slots):
        if 0 <= s < k_pool.shape[0]:
            k[i] = k_pool[s]
            v[i] = v_pool[s]
        else:
            skipped = True
    return k, v, skipped


def draft_lists_after_topk(next_idx, next_cnt, verify_len, phase, slot_table=None, kv_off=None):
    """Critical lists of the draft steps that follow a verify step
    ("SparseSpec-MLSys26", PillarAttn: the Top-K of the verify step's exact
    scores is the critical set of the next k draft steps; the tokens appended
    since are attended as well).

    For verify request v and KV head h, at draft phase p (p tokens appended
    since the verify step, whose length was L_v = verify_len[v]), the list is
    the Top-K positions next_idx[v, h, :next_cnt[v, h]] (all below L_v),
    followed by the appended positions L_v, ..., L_v + p - 1, in ascending
    order.  ``phase`` is one p for all requests or one per request.  With
    ``slot_table`` and ``kv_off`` (request v's slots start at kv_off[v] and
    cover its L_v + p positions), each listed position's slot is returned as
    well.  Returns (lists [V, Hkv, n_max] int32, counts [V, Hkv] int32,
    slots like lists or None); entries past a count are 0."""
    next_idx = np.asarray(next_idx)
    next_cnt = np.asarray(next_cnt)
    V, Hkv = next_cnt.shape
    Lv = np.asarray(verify_len, np.int64)
    ph = np.broadcast_to(np.asarray(phase, np.int64), (V,))
    built = {}
    n_max = 1
    for v in range(V):
        for h in range(Hkv):
            crit = [int(x) for x in next_idx[v, h, :int(next_cnt[v, h])]]
            lst = sorted(crit) + [int(Lv[v]) + i for i in range(int(ph[v]))]
            built[(v, h)] = lst
            n_max = max(n_max, len(lst))
    lists = np.zeros((V, Hkv, n_max), np.int32)
    counts = np.zeros((V, Hkv), np.int32)
    slots = np.zeros((V, Hkv, n_max), np.int32) if slot_table is not None else None
    for (v, h), lst in built.items():
        counts[v, h] = len(lst)
        for i, pos in enumerate(lst):
            lists[v, h, i] = pos
            if slots is not None:
                slots[v, h, i] = int(slot_table[int(kv_off[v]) + pos])
    return lists, counts, slots
