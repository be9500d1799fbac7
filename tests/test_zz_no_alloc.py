"""pillar_topk_select_noalloc: Top-K without a caller-provided workspace.

Callers whose device memory belongs to another allocator (a framework's
caching allocator, a serving process that reserves all of HBM up front), or
that cannot afford cudaMalloc's implicit synchronisation, use this entry
point; its scratch is an array built into the library.  These checks call
it through the C ABI twice in a row and require the same critical lists as
pillar_topk_select (which takes a workspace), and a clear refusal when a
shape needs more scratch than the array holds.  The file is collected last
so that a stop-at-first-failure run has already run everything else.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import sparse_self_speculative_pillar_gb300 as P  # noqa: E402
from tests._gpu_common import Gpu  # noqa: E402


def test_noalloc_topk_matches_the_workspace_entry_point_twice():
    w = W.generate(W.scaled("qwen3_8b", B=28, length_scale=0.2, seed_offset=31))
    g = Gpu(w)
    g.attn()
    g.topk()
    assert g.attn_flags() == 0 and g.topk_flags() == 0
    ref_idx = g.next_idx.cpu().numpy()
    ref_cnt = g.next_cnt.cpu().numpy()
    for _ in range(2):
        idx = torch.full_like(g.next_idx, -1)
        cnt = torch.full_like(g.next_cnt, -1)
        flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        P.pillar_topk_select_noalloc(g.shape, g.V, g.logits, g.lse, g.req_len, g.group_map, g.K, idx, cnt,
                                     device_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
        got = idx.cpu().numpy()
        for v in range(w.V):
            for h in range(w.Hkv):
                n = ref_cnt[v, h]
                np.testing.assert_array_equal(got[v, h, :n], ref_idx[v, h, :n])


def test_noalloc_topk_refuses_shapes_beyond_its_scratch():
    # 8 verify requests x 8 KV heads x 65600 positions: more scores than the built-in array holds
    shape = P.make_shape(B=8, Hq=32, Hkv=8, D=128, k=8, max_sparse=1, max_len=65600, num_slots=1, max_topk=16)
    assert P.pillar_topk_workspace_bytes(shape, 8) > P.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(P.PillarError) as e:
        P.pillar_topk_select_noalloc(shape, 8, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert e.value.status == -5
    # the largest shape that fits is accepted
    shape_ok = P.make_shape(B=8, Hq=32, Hkv=8, D=128, k=8, max_sparse=1, max_len=65535, num_slots=1, max_topk=16)
    assert P.pillar_topk_workspace_bytes(shape_ok, 8) <= P.NOALLOC_SCRATCH_BYTES


def test_noalloc_error_word_reports_each_call_alone():
    """The built-in scratch keeps the previous call's contents; its error word
    starts every call clean all the same: a flagged call followed by a clean
    one reports nothing, a clean one followed by a flagged one the flag."""
    Hq, Hkv, k, L, K = 4, 2, 2, 200, 9
    rng = np.random.default_rng(44)
    lg = rng.standard_normal((1, Hq, k + 1, L)).astype(np.float32)
    lse = np.log(np.exp(lg.astype(np.float64)).sum(-1)).astype(np.float32)
    shape = P.make_shape(B=2, Hq=Hq, Hkv=Hkv, D=64, k=k, max_sparse=1, max_len=L, num_slots=1, max_topk=K)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = [dev(lg.ravel()), dev(lse), dev(np.array([L, 50], np.int32))]
    good, bad = dev(np.array([0], np.int32)), dev(np.array([7], np.int32))  # batch index 7: no such request
    Kd = dev(np.array([K], np.int32))
    nidx = torch.full((1, Hkv, K), -1, dtype=torch.int32, device="cuda")
    ncnt = torch.full((1, Hkv), -1, dtype=torch.int32, device="cuda")
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    P.pillar_topk_select_noalloc(shape, 1, *args, bad, Kd, nidx, ncnt, device_flags=flags)
    P.pillar_topk_select_noalloc(shape, 1, *args, good, Kd, nidx, ncnt, device_flags=flags)
    assert int(flags.item()) == 0
    P.pillar_topk_select_noalloc(shape, 1, *args, bad, Kd, nidx, ncnt, device_flags=flags)
    assert int(flags.item()) == P.FLAG_REQUEST
