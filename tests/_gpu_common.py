"""Shared helpers of the GPU parity tests: run the fp64 oracle on the same
inputs as the CUDA path (uploaded by workloads.device.Gpu) and compare with
the stated tolerances.

Tolerances (bf16 inputs, fp32 accumulation), checked as two quantities on
every compared block (a request's output rows, its logits, its LSEs):
  * max-abs: max_i |gpu_i - oracle_i| <= 2e-2;
  * rel:     ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2;
-inf logits agree exactly.  Top-K index sets agree exactly, except for
positions whose oracle score lies within 1e-5 (relative) of the oracle's K-th
score.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import workloads as W
# the device set of a workload lives beside the generator (no arithmetic, no oracle)
from workloads.device import Gpu, to_device  # noqa: F401

ATOL, RTOL = 2e-2, 1e-2
TIE_REL = 1e-5


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
    """Both tolerances on one block; returns (max-abs error, relative l2 error)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    ninf_r, ninf_g = np.isneginf(ref), np.isneginf(gpu)
    assert np.array_equal(ninf_r, ninf_g), f"{what}: -inf pattern differs ({(ninf_r != ninf_g).sum()} entries)"
    m = ~ninf_r
    assert np.all(np.isfinite(gpu[m])), f"{what}: non-finite values"
    if not m.any():
        return 0.0, 0.0
    d = gpu[m] - ref[m]
    err = np.abs(d)
    max_abs = float(err.max())
    nr = float(np.linalg.norm(ref[m]))
    rel = float(np.linalg.norm(d)) / nr if nr > 0 else float(np.linalg.norm(d))
    assert max_abs <= ATOL, (f"{what}: max-abs error {max_abs:.3e} > {ATOL} at ref {ref[m][np.argmax(err)]:.4f} "
                             f"({(err > ATOL).sum()} of {err.size} elements)")
    assert rel <= RTOL, f"{what}: relative l2 error {rel:.3e} > {RTOL}"
    return max_abs, rel


def compare_attn(w: W.Workload, g: dict, r: oracle.AttnResult, select=None):
    """Every element of out (all rows of the selected requests), verify logits
    and LSE; returns the worst max-abs and relative errors of each."""
    q_off = w.q_off
    ver_idx = list(w.verify_batch_index)
    off_g = np.concatenate([[0], np.cumsum(w.verify_len.astype(np.int64) * w.Hq * (w.k + 1))])
    lse_orc = oracle.verify_lse_of(r, w.req_mode, w.k, w.Hq, select=select)
    o_off = 0
    vsel = 0
    worst = {f"{q}_{e}": 0.0 for q in ("out", "logits", "lse") for e in ("abs", "rel")}

    def note(q, ar):
        worst[q + "_abs"] = max(worst[q + "_abs"], ar[0])
        worst[q + "_rel"] = max(worst[q + "_rel"], ar[1])

    for b in range(w.B):
        if select is not None and not select[b]:
            continue
        nq = w.k + 1 if w.req_mode[b] == 1 else 1
        note("out", close(g["out"][q_off[b]:q_off[b] + nq], r.out[q_off[b]:q_off[b] + nq], f"out of request {b}"))
        if w.req_mode[b] == 1:
            v = ver_idx.index(b)
            n = int(w.Hq * (w.k + 1) * w.req_len[b])
            note("logits", close(g["logits"][off_g[v]:off_g[v] + n], r.logits[o_off:o_off + n],
                                 f"logits of request {b}"))
            note("lse", close(g["lse"][v], lse_orc[vsel], f"lse of request {b}"))
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
