"""The next draft step's critical lists built on the device after Top-K
("SparseSpec-MLSys26", 核心方法 / PillarAttn: the Top-K of a verify step is
the critical set of the next k draft steps; the tokens appended since are
attended as well), and the draft step that reads their pre-translated slots.

A stride is played out on one pool: the requests that verify do so over a
prefix of their context (L - p positions, p = 1..k), the Top-K runs on the
GPU's own dump, pillar_draft_lists turns it into the lists of the draft step
in which those requests have grown back to L positions, and that draft step
runs with and without the translated slots."""
import math

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import sparse_self_speculative_pillar_gb300 as P  # noqa: E402
from tests._gpu_common import Gpu, compare_attn, run_oracle, to_device  # noqa: E402

SENTINEL = -7


def play_stride(seed, recipe="qwen3_8b", B=10, length_scale=0.05):
    wd = W.generate(W.scaled(recipe, B=B, length_scale=length_scale, seed_offset=seed))
    gd = Gpu(wd)  # the pool; the draft step's own lists for the requests that were drafts already
    S = np.nonzero(wd.req_mode == 1)[0].astype(np.int32)  # the requests that verified
    k, G = wd.k, wd.G
    p = (1 + (S % k)).astype(np.int32)                     # tokens appended since, 1..k
    Lv = (wd.req_len[S] - p).astype(np.int32)
    kv_off_d = wd.kv_off
    # the verify step: requests S over their prefixes, fresh query rows, the prefixes of their slots
    table_v = np.concatenate([wd.slot_table[kv_off_d[b]:kv_off_d[b] + int(lv)] for b, lv in zip(S, Lv)])
    q_v = W.query_rows(wd, (k + 1) * len(S), 1000 + seed)
    K = np.clip(-(-Lv.astype(np.int64) * wd.recipe.s_num // wd.recipe.s_den), 1, Lv).astype(np.int32)
    kmax = int(K.max())
    shape_v = P.make_shape(B=len(S), Hq=wd.Hq, Hkv=wd.Hkv, D=wd.D, k=k, max_sparse=1, max_len=int(Lv.max()),
                           num_slots=wd.num_slots, max_topk=kmax)
    V = len(S)
    n_log = int(wd.Hq * (k + 1) * Lv.astype(np.int64).sum())
    logits = torch.empty(n_log, dtype=torch.float32, device="cuda")
    lse = torch.empty((V, wd.Hq, k + 1), dtype=torch.float32, device="cuda")
    out_v = torch.empty(((k + 1) * V, wd.Hq, wd.D), dtype=torch.int16, device="cuda")
    ws = torch.empty(P.pillar_attn_workspace_bytes(shape_v), dtype=torch.uint8, device="cuda")
    tws = torch.empty(P.pillar_topk_workspace_bytes(shape_v, V), dtype=torch.uint8, device="cuda")
    next_idx = torch.full((V, wd.Hkv, kmax), -1, dtype=torch.int32, device="cuda")
    next_cnt = torch.zeros((V, wd.Hkv), dtype=torch.int32, device="cuda")
    lv_d = to_device(Lv)
    P.pillar_attn_unified(shape_v, to_device(q_v), gd.k_pool, gd.v_pool, to_device(table_v.astype(np.int32)),
                          to_device(np.ones(V, np.int32)), lv_d, torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros((V, wd.Hkv), dtype=torch.int32, device="cuda"), out_v, logits, lse, ws)
    P.pillar_topk_select(shape_v, V, logits, lse, lv_d, to_device(np.arange(V, dtype=np.int32)), to_device(K),
                         next_idx, next_cnt, tws)
    assert P.pillar_get_error(ws) == 0 and P.pillar_get_error(tws) == 0
    # the draft step: every request a draft with one query row; S's lists come from the device
    max_sparse = max(wd.max_sparse, kmax + k)
    si = np.full((wd.B, wd.Hkv, max_sparse), SENTINEL, np.int32)
    sc = np.full((wd.B, wd.Hkv), SENTINEL, np.int32)
    for b in np.nonzero(wd.req_mode == 0)[0]:
        si[b, :, :wd.max_sparse] = wd.sparse_idx[b]
        sc[b] = wd.sparse_cnt[b]
    ss = np.where(si >= 0, 0, SENTINEL).astype(np.int32)  # slots of the lists the host already has
    for b in np.nonzero(wd.req_mode == 0)[0]:
        for h in range(wd.Hkv):
            n = int(sc[b, h])
            ss[b, h, :n] = wd.slot_table[kv_off_d[b] + si[b, h, :n]]
    si_d, sc_d, ss_d = to_device(si), to_device(sc), to_device(ss)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape_d = P.make_shape(B=wd.B, Hq=wd.Hq, Hkv=wd.Hkv, D=wd.D, k=k, max_sparse=max_sparse,
                           max_len=int(wd.req_len.max()), num_slots=wd.num_slots, max_topk=kmax)
    P.pillar_draft_lists(shape_d, V, next_idx, next_cnt, to_device(S), lv_d, gd.req_len, gd.slot_table, si_d, sc_d,
                         ss_d, flags)
    torch.cuda.synchronize()
    return dict(wd=wd, gd=gd, S=S, p=p, Lv=Lv, next_idx=next_idx.cpu().numpy(), next_cnt=next_cnt.cpu().numpy(),
                si=si_d.cpu().numpy(), sc=sc_d.cpu().numpy(), ss=ss_d.cpu().numpy(), si_host=si, sc_host=sc,
                shape_d=shape_d, flags=int(flags.item()), si_d=si_d, sc_d=sc_d, ss_d=ss_d)


def test_device_lists_and_slots_match_the_oracle():
    c = play_stride(61)
    wd, S = c["wd"], c["S"]
    assert c["flags"] == 0
    lists, counts, slots = oracle.draft_lists_after_topk(c["next_idx"], c["next_cnt"], c["Lv"], c["p"],
                                                         slot_table=wd.slot_table, kv_off=wd.kv_off[S])
    for v, b in enumerate(S):
        np.testing.assert_array_equal(c["sc"][b], counts[v])
        for h in range(wd.Hkv):
            n = int(counts[v, h])
            np.testing.assert_array_equal(c["si"][b, h, :n], lists[v, h, :n])
            np.testing.assert_array_equal(c["ss"][b, h, :n], slots[v, h, :n])
            assert np.all(c["si"][b, h, n:] == SENTINEL)  # nothing past the count
    others = np.setdiff1d(np.arange(wd.B), S)
    np.testing.assert_array_equal(c["si"][others], c["si_host"][others])  # other rows untouched
    np.testing.assert_array_equal(c["sc"][others], c["sc_host"][others])


@pytest.mark.parametrize("recipe,B,scale", [("qwen3_8b", 10, 0.05), ("stress", 14, 0.04), ("tiny", 4, 1.0)])
def test_draft_step_on_device_lists(recipe, B, scale):
    """The draft step over the device-built lists: with pre-translated slots it
    writes bit for bit what the position-only call writes, and both match the
    oracle."""
    c = play_stride(62, recipe, B, scale)
    wd, gd = c["wd"], c["gd"]
    assert c["flags"] == 0
    q1 = wd.q[wd.q_off]  # one query row per request
    mode = torch.zeros(wd.B, dtype=torch.int32, device="cuda")
    outs = []
    for slotted in (False, True):
        out = torch.empty((wd.B, wd.Hq, wd.D), dtype=torch.int16, device="cuda")
        lg = torch.empty(1, dtype=torch.float32, device="cuda")
        ls = torch.empty((1, wd.Hq, wd.k + 1), dtype=torch.float32, device="cuda")
        ws = torch.empty(P.pillar_attn_workspace_bytes(c["shape_d"]), dtype=torch.uint8, device="cuda")
        args = (c["shape_d"], to_device(q1), gd.k_pool, gd.v_pool, gd.slot_table, mode, gd.req_len, c["si_d"],
                c["sc_d"])
        if slotted:
            P.pillar_attn_unified_slotted(*args, c["ss_d"], out, lg, ls, ws)
        else:
            P.pillar_attn_unified(*args, out, lg, ls, ws)
        assert P.pillar_get_error(ws) == 0
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    # the oracle over the same lists
    w2 = W.generate(W.scaled(recipe, B=B, length_scale=scale, seed_offset=62))
    w2.req_mode = np.zeros(wd.B, np.int32)
    w2.q = q1
    w2.sparse_idx, w2.sparse_cnt = np.maximum(c["si"], 0), c["sc"]
    w2.topk_K = np.zeros(0, np.int32)
    ref = run_oracle(w2)
    res = dict(out=W.bf16_bits_to_f32(outs[1].view(np.uint16)).astype(np.float64),
               logits=np.zeros(0), lse=np.zeros((0, wd.Hq, wd.k + 1)))
    compare_attn(w2, res, ref)


def test_draft_lists_flags():
    """A group_map entry outside the batch, a length that went down since the
    verify step, and a list longer than max_sparse are flagged; nothing is
    written out of bounds, and the long list is cut to max_sparse."""
    Hkv, K, B = 2, 6, 3
    shape = P.make_shape(B=B, Hq=4, Hkv=Hkv, D=64, k=3, max_sparse=8, max_len=100, num_slots=1000, max_topk=K)
    nidx = to_device(np.tile(np.arange(K, dtype=np.int32) * 3, (3, Hkv, 1)))
    ncnt = to_device(np.full((3, Hkv), K, np.int32))
    req_len = to_device(np.array([50, 40, 60], np.int32))
    table = to_device(np.arange(150, dtype=np.int32))
    si = to_device(np.full((B, Hkv, 8), SENTINEL, np.int32))
    sc = to_device(np.full((B, Hkv), SENTINEL, np.int32))
    ss = to_device(np.full((B, Hkv, 8), SENTINEL, np.int32))
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    # v0 -> b=7 (outside the batch); v1 -> b=1 whose length shrank (45 > 40); v2 -> b=2, 6 + 5 > 8 entries
    P.pillar_draft_lists(shape, 3, nidx, ncnt, to_device(np.array([7, 1, 2], np.int32)),
                         to_device(np.array([30, 45, 55], np.int32)), req_len, table, si, sc, ss, flags)
    f = int(flags.item())
    assert f & P.FLAG_REQUEST and f & P.FLAG_COUNT
    si, sc, ss = si.cpu().numpy(), sc.cpu().numpy(), ss.cpu().numpy()
    assert np.all(si[0] == SENTINEL) and np.all(sc[0] == SENTINEL)  # b = 0: no verify request maps to it
    assert np.all(sc[1] == 0) and np.all(si[1] == SENTINEL)         # shrunk length: an empty list
    assert np.all(sc[2] == 8)
    for h in range(Hkv):
        np.testing.assert_array_equal(si[2, h], [0, 3, 6, 9, 12, 15, 55, 56])
        np.testing.assert_array_equal(ss[2, h], 90 + si[2, h])      # request 2's slots start at 50 + 40
