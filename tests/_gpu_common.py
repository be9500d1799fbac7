"""Shared helpers of the GPU parity tests: upload a seeded workload, run the
CUDA path through the C ABI, run the fp64 oracle on the same inputs, and
compare with the stated tolerances.

Tolerances: attention outputs, LSE and logits agree with the oracle to
|gpu - oracle| <= 2e-2 + 1e-2 * |oracle| elementwise (bf16 inputs, fp32
accumulation); -inf logits agree exactly.  Top-K index sets agree exactly,
except for positions whose oracle score lies within 1e-5 (relative) of the
oracle's K-th score.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import sparse_self_speculative_pillar_gb300 as P
import workloads as W

ATOL, RTOL = 2e-2, 1e-2
TIE_REL = 1e-5


def _t(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


class Gpu:
    """Device copies of one workload (pool built on the device by scattering the
    logical K/V rows into their slots)."""

    def __init__(self, w: W.Workload, **shape_kw):
        self.w = w
        self.q = _t(w.q)
        st = _t(w.slot_table).long()
        self.k_pool = torch.zeros((w.num_slots, w.Hkv, w.D), dtype=torch.int16, device="cuda")
        self.v_pool = torch.zeros_like(self.k_pool)
        self.k_pool[st] = _t(w.k_logical)
        self.v_pool[st] = _t(w.v_logical)
        self.slot_table = _t(w.slot_table)
        self.req_mode = _t(w.req_mode)
        self.req_len = _t(w.req_len)
        self.sparse_idx = _t(w.sparse_idx)
        self.sparse_cnt = _t(w.sparse_cnt)
        self.group_map = _t(w.verify_batch_index)
        self.K = _t(w.topk_K)
        self.V = w.V
        kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, max_sparse=w.max_sparse,
                  max_len=int(max(1, w.req_len.max())), num_slots=w.num_slots,
                  max_topk=int(w.topk_K.max()) if w.V else 1)
        kw.update(shape_kw)
        self.shape = P.make_shape(**kw)
        T_q = w.q.shape[0]
        n_logits = int(w.Hq * (w.k + 1) * w.verify_len.astype(np.int64).sum())
        self.out = torch.empty((T_q, w.Hq, w.D), dtype=torch.int16, device="cuda")
        self.logits = torch.full((max(1, n_logits),), float("nan"), dtype=torch.float32, device="cuda")
        self.lse = torch.full((max(1, w.V), w.Hq, w.k + 1), float("nan"), dtype=torch.float32, device="cuda")
        self.ws = torch.empty(P.pillar_attn_workspace_bytes(self.shape), dtype=torch.uint8, device="cuda")
        self.tws = torch.empty(P.pillar_topk_workspace_bytes(self.shape, max(1, w.V)), dtype=torch.uint8,
                               device="cuda")
        self.next_idx = torch.full((max(1, w.V), w.Hkv, self.shape.max_topk), -1, dtype=torch.int32, device="cuda")
        self.next_cnt = torch.full((max(1, w.V), w.Hkv), -1, dtype=torch.int32, device="cuda")

    def attn(self, stream=None):
        P.pillar_attn_unified(self.shape, self.q, self.k_pool, self.v_pool, self.slot_table, self.req_mode,
                              self.req_len, self.sparse_idx, self.sparse_cnt, self.out, self.logits, self.lse,
                              self.ws, stream=stream)

    def topk(self, stream=None):
        P.pillar_topk_select(self.shape, self.V, self.logits, self.lse, self.req_len, self.group_map, self.K,
                             self.next_idx, self.next_cnt, self.tws, stream=stream)

    def attn_flags(self):
        return P.pillar_get_error(self.ws)

    def topk_flags(self):
        return P.pillar_get_error(self.tws)

    def host(self):
        torch.cuda.synchronize()
        out = W.bf16_bits_to_f32(self.out.cpu().numpy().view(np.uint16)).astype(np.float64)
        return dict(out=out, logits=self.logits.cpu().numpy().astype(np.float64),
                    lse=self.lse.cpu().numpy().astype(np.float64),
                    next_idx=self.next_idx.cpu().numpy(), next_cnt=self.next_cnt.cpu().numpy())


def run_oracle(w: W.Workload, select=None, sparse_idx=None, sparse_cnt=None, use_pool=None):
    """fp64 oracle on the same inputs.  Small pools are passed as they are (real
    slot table); large ones as the logical rows with an identity table, which
    is the same arithmetic on the same values."""
    if use_pool is None:
        use_pool = w.num_slots * w.Hkv * w.D <= (1 << 26)
    if use_pool:
        kp, vp, table = w.pool("k"), w.pool("v"), w.slot_table
    else:
        kp, vp, table = w.k_logical, w.v_logical, np.arange(len(w.slot_table), dtype=np.int32)
    return oracle.attn_unified(Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, scale=1 / math.sqrt(w.D), q=w.q, k_pool=kp,
                               v_pool=vp, slot_table=table, req_mode=w.req_mode, req_len=w.req_len,
                               sparse_idx=w.sparse_idx if sparse_idx is None else sparse_idx,
                               sparse_cnt=w.sparse_cnt if sparse_cnt is None else sparse_cnt, select=select)


def close(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    ninf_r, ninf_g = np.isneginf(ref), np.isneginf(gpu)
    assert np.array_equal(ninf_r, ninf_g), f"{what}: -inf pattern differs ({(ninf_r != ninf_g).sum()} entries)"
    m = ~ninf_r
    assert np.all(np.isfinite(gpu[m])), f"{what}: non-finite values"
    err = np.abs(gpu[m] - ref[m])
    bound = ATOL + RTOL * np.abs(ref[m])
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err {err.max():.3e} "
                           f"at ref {ref[m][np.argmax(err)]:.4f}")
    return float(err.max()) if err.size else 0.0


def compare_attn(w: W.Workload, g: dict, r: oracle.AttnResult, select=None):
    """Elementwise comparison of out (all rows of selected requests), verify
    logits and LSE."""
    q_off = w.q_off
    ver_idx = list(w.verify_batch_index)
    off_g = np.concatenate([[0], np.cumsum(w.verify_len.astype(np.int64) * w.Hq * (w.k + 1))])
    lse_orc = oracle.verify_lse_of(r, w.req_mode, w.k, w.Hq, select=select)
    o_off = 0
    vsel = 0
    worst = {"out": 0.0, "logits": 0.0, "lse": 0.0}
    for b in range(w.B):
        if select is not None and not select[b]:
            continue
        nq = w.k + 1 if w.req_mode[b] == 1 else 1
        worst["out"] = max(worst["out"], close(g["out"][q_off[b]:q_off[b] + nq], r.out[q_off[b]:q_off[b] + nq],
                                               f"out of request {b}"))
        if w.req_mode[b] == 1:
            v = ver_idx.index(b)
            n = int(w.Hq * (w.k + 1) * w.req_len[b])
            worst["logits"] = max(worst["logits"], close(g["logits"][off_g[v]:off_g[v] + n], r.logits[o_off:o_off + n],
                                                         f"logits of request {b}"))
            worst["lse"] = max(worst["lse"], close(g["lse"][v], lse_orc[vsel], f"lse of request {b}"))
            o_off += n
            vsel += 1
    return worst


def compare_topk(gpu_idx, gpu_cnt, ref: oracle.TopkResult, L, K, Hkv, what="topk"):
    """Sets equal outside the tie band of the oracle's K-th score; ascending
    output; counts equal."""
    s_off = np.concatenate([[0], np.cumsum(np.asarray(L, np.int64) * Hkv)])
    mism = 0
    for v in range(len(L)):
        for g in range(Hkv):
            n = int(ref.next_cnt[v, g])
            assert gpu_cnt[v, g] == n, f"{what}: count of ({v},{g}) {gpu_cnt[v, g]} != {n}"
            gi = gpu_idx[v, g, :n]
            assert np.all(np.diff(gi) > 0), f"{what}: ({v},{g}) not strictly ascending"
            ri = ref.next_idx[v, g, :n]
            if np.array_equal(gi, ri):
                continue
            sc = ref.scores[s_off[v] + g * L[v]: s_off[v] + (g + 1) * L[v]]
            kth = np.sort(sc)[::-1][n - 1] if n else 0.0
            diff = np.setxor1d(gi, ri)
            assert np.all(diff >= 0) and np.all(diff < L[v])
            near = np.abs(sc[diff] - kth) <= TIE_REL * abs(kth)
            assert near.all(), (f"{what}: ({v},{g}) differs outside the tie band at {diff[~near][:8]} "
                                f"(scores {sc[diff[~near][:4]]}, K-th {kth})")
            mism += len(diff)
    return mism
