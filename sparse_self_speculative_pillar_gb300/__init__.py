"""GB300 (sm_103a) PillarAttn unified step: thin Python binding over the C ABI.

Every step of the path runs in the CUDA library built from ``csrc/``; this
module only marshals arguments (torch tensors or raw device pointers) into
the ``extern "C"`` entry points declared in ``include/pillar.h`` and turns
non-zero status codes into exceptions.  There is no fallback: if the
library is missing or cannot be loaded, every call raises.

Entry points (same names as the C ABI):
  pillar_attn_workspace_bytes(shape)
  pillar_attn_unified(shape, q, k_pool, v_pool, slot_table, req_mode, req_len,
                      sparse_idx, sparse_cnt, out, verify_logits, verify_lse,
                      workspace, stream=None)
  pillar_topk_workspace_bytes(shape, V)
  pillar_topk_select(shape, V, verify_logits, verify_lse, req_len, group_map, K,
                     next_idx, next_cnt, workspace, stream=None)
  pillar_get_error(workspace, stream=None)
  pillar_status_string(status)
  pillar_attn_unified_slotted(shape, ..., sparse_slot, out, ...)   (draft lists with their slots)
  pillar_attn_plan(shape, req_mode, req_len, sparse_cnt, workspace, stream=None)
  pillar_attn_run(shape, q, k_pool, v_pool, slot_table, sparse_idx, out, verify_logits, verify_lse,
                  workspace, sparse_slot=None, stream=None)  (one plan, several runs)
  pillar_draft_lists(shape, V, next_idx, next_cnt, group_map, verify_len, req_len, slot_table,
                     sparse_idx, sparse_cnt, sparse_slot=None, device_flags=None, stream=None)
  pillar_topk_select_noalloc(shape, V, ..., device_flags=None, stream=None)
  pillar_kv_append(shape, k_new, v_new, slots, k_pool, v_pool, device_flags=None, stream=None)
  pillar_kv_offload(shape, k_pool, v_pool, slots, host_k, host_v, device_flags=None, stream=None)
  pillar_kv_reload(shape, host_k, host_v, slots, k_pool, v_pool, device_flags=None, stream=None)
  pillar_buckets_init(k), pillar_buckets_admit(pb), pillar_buckets_retire(pb, bucket),
  pillar_buckets_step(pb, buckets, step)    (host-side phase buckets)
  pillar_offload_init(capacity, chunk), pillar_offload_reserve(f, n, new_request),
  pillar_offload_release(f, n), pillar_offload_evict(f, req, len),
  pillar_offload_reload(f, max_out)         (host-side FIFO of offloaded KV chunks)
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "PillarShape", "make_shape", "PillarError", "load", "library_path", "build",
    "pillar_attn_workspace_bytes", "pillar_attn_unified", "pillar_attn_unified_slotted", "pillar_draft_lists",
    "pillar_attn_plan", "pillar_attn_run",
    "pillar_topk_workspace_bytes", "pillar_topk_select", "pillar_topk_select_noalloc", "pillar_get_error", "pillar_status_string",
    "FLAG_INDEX", "FLAG_SLOT", "FLAG_REQUEST", "FLAG_COUNT", "FLAG_TIMEOUT", "FLAG_TOPK",
    "SCHEDULE_UNIFIED", "SCHEDULE_DRAFT_ONLY", "SCHEDULE_VERIFY_ONLY", "SCHEDULE_UNIFORM_ROWS", "SCHEDULE_NAIVE_JOINT",
    "pillar_kv_append", "PillarBuckets", "pillar_buckets_init", "pillar_buckets_admit", "pillar_buckets_retire", "pillar_buckets_step",
    "pillar_kv_offload", "pillar_kv_reload", "PillarOffloadFifo", "pillar_offload_init", "pillar_offload_reserve",
    "pillar_offload_release", "pillar_offload_evict", "pillar_offload_reload",
]

FLAG_INDEX, FLAG_SLOT, FLAG_REQUEST, FLAG_COUNT, FLAG_TIMEOUT, FLAG_TOPK = 1, 2, 4, 8, 16, 32
# values of PillarShape.schedule (PILLAR_SCHEDULE_* in the header)
SCHEDULE_UNIFIED, SCHEDULE_DRAFT_ONLY, SCHEDULE_VERIFY_ONLY, SCHEDULE_UNIFORM_ROWS, SCHEDULE_NAIVE_JOINT = 0, 1, 2, 3, 4
EXPORTED = ("pillar_attn_workspace_bytes", "pillar_attn_unified", "pillar_attn_unified_slotted",
            "pillar_draft_lists", "pillar_topk_workspace_bytes",
            "pillar_topk_select", "pillar_topk_select_noalloc", "pillar_get_error", "pillar_status_string",
            "pillar_kv_append", "pillar_buckets_init", "pillar_buckets_admit", "pillar_buckets_retire",
            "pillar_buckets_step", "pillar_kv_offload", "pillar_kv_reload", "pillar_offload_init",
            "pillar_attn_plan", "pillar_attn_run",
            "pillar_offload_reserve", "pillar_offload_release", "pillar_offload_evict", "pillar_offload_reload")
MAX_BUCKETS = 64  # PILLAR_MAX_BUCKETS
OFFLOAD_QUEUE = 1024  # PILLAR_OFFLOAD_QUEUE
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024 + 256


class PillarShape(ctypes.Structure):
    """Mirror of ``pillar_shape_t``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32),
        ("k", ctypes.c_int32), ("max_sparse", ctypes.c_int32), ("max_len", ctypes.c_int32),
        ("row_lo", ctypes.c_int32), ("row_hi", ctypes.c_int32), ("max_topk", ctypes.c_int32),
        ("verify_chunk", ctypes.c_int32), ("draft_chunk", ctypes.c_int32), ("num_slots", ctypes.c_int64),
        ("sm_scale", ctypes.c_float), ("schedule", ctypes.c_int32),
        ("wait_timeout_us", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


def make_shape(*, B, Hq, Hkv, D, k, max_sparse, max_len, num_slots, max_topk=1, row_lo=1, row_hi=None,
               verify_chunk=0, draft_chunk=0, sm_scale=0.0, schedule=0, wait_timeout_us=0) -> PillarShape:
    return PillarShape(B=B, Hq=Hq, Hkv=Hkv, D=D, k=k, max_sparse=max_sparse, max_len=max_len,
                       row_lo=row_lo, row_hi=(k + 1) if row_hi is None else row_hi, max_topk=max(1, max_topk),
                       verify_chunk=verify_chunk, draft_chunk=draft_chunk, num_slots=num_slots,
                       sm_scale=sm_scale, schedule=schedule, wait_timeout_us=wait_timeout_us)


class PillarOffloadChunk(ctypes.Structure):
    """pillar_offload_chunk_t: one chunk of an offloaded request's positions."""
    _fields_ = [("req", ctypes.c_int32), ("first", ctypes.c_int32), ("n", ctypes.c_int32), ("last", ctypes.c_int32)]


class PillarOffloadFifo(ctypes.Structure):
    """pillar_offload_fifo_t: resident slot count and the queue of offloaded chunks."""
    _fields_ = [("capacity", ctypes.c_int64), ("resident", ctypes.c_int64), ("chunk", ctypes.c_int32),
                ("head", ctypes.c_int32), ("count", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("q", PillarOffloadChunk * OFFLOAD_QUEUE)]


class PillarBuckets(ctypes.Structure):
    """pillar_buckets_t: the request count of each of the k+1 phase buckets."""
    _fields_ = [("nbuckets", ctypes.c_int32), ("count", ctypes.c_int32 * MAX_BUCKETS)]


class PillarError(RuntimeError):
    def __init__(self, fn, status, flags=None):
        self.status = status
        self.flags = flags
        msg = f"{fn}: status {status} ({pillar_status_string(status)})"
        if flags is not None:
            msg += f", device flags 0x{flags:x}"
        super().__init__(msg)


_lib = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load():
    """Load the CUDA library (built in-tree by ``build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"the sm_103a library is not built ({path}); run __graft_entry__.build()")
    import torch  # noqa: F401  -- makes the CUDA runtime of the process available first
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    SP = ctypes.POINTER(PillarShape)
    lib.pillar_attn_workspace_bytes.argtypes = [SP, ctypes.POINTER(ctypes.c_size_t)]
    lib.pillar_attn_unified.argtypes = [SP] + [P] * 11 + [P, ctypes.c_size_t, P]
    lib.pillar_attn_unified_slotted.argtypes = [SP] + [P] * 12 + [P, ctypes.c_size_t, P]
    lib.pillar_draft_lists.argtypes = [SP, ctypes.c_int32] + [P] * 11
    lib.pillar_attn_plan.argtypes = [SP, P, P, P, P, ctypes.c_size_t, P]
    lib.pillar_attn_run.argtypes = [SP] + [P] * 10 + [ctypes.c_size_t, P]
    lib.pillar_topk_workspace_bytes.argtypes = [SP, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    lib.pillar_topk_select.argtypes = [SP, ctypes.c_int32] + [P] * 7 + [P, ctypes.c_size_t, P]
    lib.pillar_topk_select_noalloc.argtypes = [SP, ctypes.c_int32] + [P] * 8 + [P]
    lib.pillar_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.pillar_status_string.argtypes = [ctypes.c_int]
    lib.pillar_kv_append.argtypes = [SP, P, P, P, ctypes.c_int32, P, P, P, P]
    BP = ctypes.POINTER(PillarBuckets)
    I32P = ctypes.POINTER(ctypes.c_int32)
    lib.pillar_buckets_init.argtypes = [BP, ctypes.c_int32]
    lib.pillar_buckets_admit.argtypes = [BP, I32P]
    lib.pillar_buckets_retire.argtypes = [BP, ctypes.c_int32]
    lib.pillar_buckets_step.argtypes = [BP, I32P, ctypes.c_int32, ctypes.c_int64, I32P, I32P,
                                        ctypes.POINTER(ctypes.c_int64)]
    lib.pillar_kv_offload.argtypes = [SP, P, P, P, ctypes.c_int32, P, P, P, P]
    lib.pillar_kv_reload.argtypes = [SP, P, P, P, ctypes.c_int32, P, P, P, P]
    FP = ctypes.POINTER(PillarOffloadFifo)
    lib.pillar_offload_init.argtypes = [FP, ctypes.c_int64, ctypes.c_int32]
    lib.pillar_offload_reserve.argtypes = [FP, ctypes.c_int64, ctypes.c_int32, I32P]
    lib.pillar_offload_release.argtypes = [FP, ctypes.c_int64]
    lib.pillar_offload_evict.argtypes = [FP, ctypes.c_int32, ctypes.c_int32, I32P]
    lib.pillar_offload_reload.argtypes = [FP, ctypes.POINTER(PillarOffloadChunk), ctypes.c_int32, I32P]
    lib.pillar_status_string.restype = ctypes.c_char_p
    for n in EXPORTED:
        if n == "pillar_status_string":
            continue
        getattr(lib, n).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    """Device pointer of a CUDA tensor (or a raw int pointer, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("device tensors only")
    if not x.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return x.data_ptr()


def _nbytes(x):
    if isinstance(x, int):
        raise ValueError("a raw workspace pointer needs an explicit size")
    return x.numel() * x.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def pillar_status_string(status: int) -> str:
    if _lib is None:
        try:
            load()
        except Exception:  # pragma: no cover
            return "library not loaded"
    return _lib.pillar_status_string(int(status)).decode()


def pillar_attn_workspace_bytes(shape: PillarShape) -> int:
    out = ctypes.c_size_t(0)
    st = load().pillar_attn_workspace_bytes(ctypes.byref(shape), ctypes.byref(out))
    if st:
        raise PillarError("pillar_attn_workspace_bytes", st)
    return int(out.value)


def pillar_attn_unified(shape, q, k_pool, v_pool, slot_table, req_mode, req_len, sparse_idx, sparse_cnt, out,
                        verify_logits, verify_lse, workspace, stream=None, ws_bytes=None):
    st = load().pillar_attn_unified(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(slot_table), _ptr(req_mode), _ptr(req_len),
        _ptr(sparse_idx), _ptr(sparse_cnt), _ptr(out), _ptr(verify_logits), _ptr(verify_lse), _ptr(workspace),
        ws_bytes if ws_bytes is not None else _nbytes(workspace), _stream(stream))
    if st:
        raise PillarError("pillar_attn_unified", st)


def pillar_attn_unified_slotted(shape, q, k_pool, v_pool, slot_table, req_mode, req_len, sparse_idx, sparse_cnt,
                                sparse_slot, out, verify_logits, verify_lse, workspace, stream=None, ws_bytes=None):
    st = load().pillar_attn_unified_slotted(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(slot_table), _ptr(req_mode), _ptr(req_len),
        _ptr(sparse_idx), _ptr(sparse_cnt), _ptr(sparse_slot), _ptr(out), _ptr(verify_logits), _ptr(verify_lse),
        _ptr(workspace), ws_bytes if ws_bytes is not None else _nbytes(workspace), _stream(stream))
    if st:
        raise PillarError("pillar_attn_unified_slotted", st)


def pillar_attn_plan(shape, req_mode, req_len, sparse_cnt, workspace, stream=None, ws_bytes=None):
    """The device planner alone: offsets and work items of the batch, into the workspace."""
    st = load().pillar_attn_plan(ctypes.byref(shape), _ptr(req_mode), _ptr(req_len), _ptr(sparse_cnt), _ptr(workspace),
                                 ws_bytes if ws_bytes is not None else _nbytes(workspace), _stream(stream))
    if st:
        raise PillarError("pillar_attn_plan", st)


def pillar_attn_run(shape, q, k_pool, v_pool, slot_table, sparse_idx, out, verify_logits, verify_lse, workspace,
                    sparse_slot=None, stream=None, ws_bytes=None):
    """The attention kernel and the merge on the plan in the workspace (one layer of the batch the plan describes)."""
    st = load().pillar_attn_run(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(slot_table), _ptr(sparse_idx), _ptr(sparse_slot),
        _ptr(out), _ptr(verify_logits), _ptr(verify_lse), _ptr(workspace),
        ws_bytes if ws_bytes is not None else _nbytes(workspace), _stream(stream))
    if st:
        raise PillarError("pillar_attn_run", st)


def pillar_draft_lists(shape, V, next_idx, next_cnt, group_map, verify_len, req_len, slot_table, sparse_idx,
                       sparse_cnt, sparse_slot=None, device_flags=None, stream=None):
    """The draft step's lists (and, with sparse_slot, their slots) from a verify step's Top-K."""
    st = load().pillar_draft_lists(
        ctypes.byref(shape), int(V), _ptr(next_idx), _ptr(next_cnt), _ptr(group_map), _ptr(verify_len),
        _ptr(req_len), _ptr(slot_table), _ptr(sparse_idx), _ptr(sparse_cnt), _ptr(sparse_slot), _ptr(device_flags),
        _stream(stream))
    if st:
        raise PillarError("pillar_draft_lists", st)


def pillar_topk_workspace_bytes(shape: PillarShape, V: int) -> int:
    out = ctypes.c_size_t(0)
    st = load().pillar_topk_workspace_bytes(ctypes.byref(shape), int(V), ctypes.byref(out))
    if st:
        raise PillarError("pillar_topk_workspace_bytes", st)
    return int(out.value)


def pillar_topk_select(shape, V, verify_logits, verify_lse, req_len, group_map, K, next_idx, next_cnt, workspace,
                       stream=None, ws_bytes=None):
    st = load().pillar_topk_select(
        ctypes.byref(shape), int(V), _ptr(verify_logits), _ptr(verify_lse), _ptr(req_len), _ptr(group_map), _ptr(K),
        _ptr(next_idx), _ptr(next_cnt), _ptr(workspace), ws_bytes if ws_bytes is not None else _nbytes(workspace),
        _stream(stream))
    if st:
        raise PillarError("pillar_topk_select", st)


def pillar_topk_select_noalloc(shape, V, verify_logits, verify_lse, req_len, group_map, K, next_idx, next_cnt,
                               device_flags=None, stream=None):
    """pillar_topk_select for callers that cannot allocate device memory: the
    library's built-in scratch array replaces the workspace.  Calls sharing a
    device must not overlap on the GPU; the first call on a device should come
    before any stream capture."""
    st = load().pillar_topk_select_noalloc(
        ctypes.byref(shape), int(V), _ptr(verify_logits), _ptr(verify_lse), _ptr(req_len), _ptr(group_map), _ptr(K),
        _ptr(next_idx), _ptr(next_cnt), _ptr(device_flags), _stream(stream))
    if st:
        raise PillarError("pillar_topk_select_noalloc", st)


def pillar_get_error(workspace, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns the flags."""
    flags = ctypes.c_int32(0)
    st = load().pillar_get_error(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    if st not in (0, -4):
        raise PillarError("pillar_get_error", st)
    return int(flags.value)


def pillar_kv_append(shape, k_new, v_new, slots, k_pool, v_pool, device_flags=None, stream=None):
    """Scatter n new tokens' K/V rows ([n, Hkv, D] bf16) into the pools at
    slots[0..n); out-of-range slots are skipped and flagged in device_flags."""
    n = int(slots.numel()) if not isinstance(slots, int) else None
    if n is None:
        raise ValueError("slots must be a tensor (its length is the token count)")
    st = load().pillar_kv_append(ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(slots), n, _ptr(k_pool),
                                 _ptr(v_pool), _ptr(device_flags), _stream(stream))
    if st:
        raise PillarError("pillar_kv_append", st)


def _host_ptr(x):
    """Address of a host buffer for the offload copies (a CPU tensor, page-locked
    or not: the library refuses memory the device cannot address), a CUDA
    tensor, or a raw int pointer."""
    if x is None or isinstance(x, int):
        return x
    return x.data_ptr()


def pillar_kv_offload(shape, k_pool, v_pool, slots, host_k, host_v, device_flags=None, stream=None):
    """Pack the slot blocks k_pool[slots[i]], v_pool[slots[i]] into rows i of
    host_k, host_v ([n, Hkv, D] bf16, page-locked host memory, e.g. a tensor
    made with pin_memory=True); out-of-range slots are skipped and flagged."""
    n = int(slots.numel())
    st = load().pillar_kv_offload(ctypes.byref(shape), _ptr(k_pool), _ptr(v_pool), _ptr(slots), n,
                                  _host_ptr(host_k), _host_ptr(host_v), _ptr(device_flags), _stream(stream))
    if st:
        raise PillarError("pillar_kv_offload", st)


def pillar_kv_reload(shape, host_k, host_v, slots, k_pool, v_pool, device_flags=None, stream=None):
    """The way back: rows i of host_k, host_v go to the slot blocks slots[i]."""
    n = int(slots.numel())
    st = load().pillar_kv_reload(ctypes.byref(shape), _host_ptr(host_k), _host_ptr(host_v), _ptr(slots), n,
                                 _ptr(k_pool), _ptr(v_pool), _ptr(device_flags), _stream(stream))
    if st:
        raise PillarError("pillar_kv_reload", st)


# --------------------------------------------------------------- offload FIFO (host side)

def pillar_offload_init(capacity: int, chunk: int) -> PillarOffloadFifo:
    f = PillarOffloadFifo()
    st = load().pillar_offload_init(ctypes.byref(f), int(capacity), int(chunk))
    if st:
        raise PillarError("pillar_offload_init", st)
    return f


def pillar_offload_reserve(f: PillarOffloadFifo, n: int, new_request: bool) -> bool:
    """True if n more device slots were granted (see the header)."""
    g = ctypes.c_int32(0)
    st = load().pillar_offload_reserve(ctypes.byref(f), int(n), 1 if new_request else 0, ctypes.byref(g))
    if st:
        raise PillarError("pillar_offload_reserve", st)
    return bool(g.value)


def pillar_offload_release(f: PillarOffloadFifo, n: int) -> None:
    st = load().pillar_offload_release(ctypes.byref(f), int(n))
    if st:
        raise PillarError("pillar_offload_release", st)


def pillar_offload_evict(f: PillarOffloadFifo, req: int, length: int) -> int:
    """Queue request `req`'s positions [0, length) for the host; returns its chunk count."""
    nc = ctypes.c_int32(0)
    st = load().pillar_offload_evict(ctypes.byref(f), int(req), int(length), ctypes.byref(nc))
    if st:
        raise PillarError("pillar_offload_evict", st)
    return int(nc.value)


def pillar_offload_reload(f: PillarOffloadFifo, max_out: int = OFFLOAD_QUEUE):
    """Chunks to bring back now, as (req, first, n, last) tuples, oldest requests first."""
    out = (PillarOffloadChunk * max(1, max_out))()
    nout = ctypes.c_int32(0)
    st = load().pillar_offload_reload(ctypes.byref(f), out, int(max_out), ctypes.byref(nout))
    if st:
        raise PillarError("pillar_offload_reload", st)
    return [(c.req, c.first, c.n, c.last) for c in out[:nout.value]]


# --------------------------------------------------------------- phase buckets (host side)

def pillar_buckets_init(k: int) -> PillarBuckets:
    pb = PillarBuckets()
    st = load().pillar_buckets_init(ctypes.byref(pb), int(k))
    if st:
        raise PillarError("pillar_buckets_init", st)
    return pb


def pillar_buckets_admit(pb: PillarBuckets) -> int:
    """Bucket of a new request (the least loaded one, lowest index among equals)."""
    b = ctypes.c_int32(-1)
    st = load().pillar_buckets_admit(ctypes.byref(pb), ctypes.byref(b))
    if st:
        raise PillarError("pillar_buckets_admit", st)
    return int(b.value)


def pillar_buckets_retire(pb: PillarBuckets, bucket: int) -> None:
    st = load().pillar_buckets_retire(ctypes.byref(pb), int(bucket))
    if st:
        raise PillarError("pillar_buckets_retire", st)


def pillar_buckets_step(pb: PillarBuckets, buckets, step: int):
    """(req_mode, phase, q_rows) of the requests with these buckets at `step`
    (lists of ints and the step's query-row count)."""
    n = len(buckets)
    arr = (ctypes.c_int32 * max(1, n))(*buckets)
    mode = (ctypes.c_int32 * max(1, n))()
    phase = (ctypes.c_int32 * max(1, n))()
    rows = ctypes.c_int64(0)
    st = load().pillar_buckets_step(ctypes.byref(pb), arr, n, int(step), mode, phase, ctypes.byref(rows))
    if st:
        raise PillarError("pillar_buckets_step", st)
    return list(mode)[:n], list(phase)[:n], int(rows.value)
