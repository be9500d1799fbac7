"""Full-size workloads in the launch configuration the benchmark times
(default chunking, one persistent CTA per SM).  The oracle recomputes a
sample of requests one by one -- the shortest and longest verify requests
and a spread of draft requests -- and every output of those requests is
compared; the remaining requests are checked for properties that hold at any
size (finite outputs, -inf exactly past each verify row's causal limit,
ascending Top-K lists of the right length)."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
from tests._gpu_common import Gpu, compare_attn, compare_topk, run_oracle  # noqa: E402

FULL = ["qwen3_1p7b", "qwen3_8b", "qwen3_14b", "stress", "stress_all_draft", "stress_all_verify"]


def _sample(w, n_draft=4, seed=0):
    sel = np.zeros(w.B, bool)
    ver = np.nonzero(w.req_mode == 1)[0]
    dra = np.nonzero(w.req_mode == 0)[0]
    if len(ver):
        sel[ver[np.argmin(w.req_len[ver])]] = True
        sel[ver[np.argmax(w.req_len[ver])]] = True
    if len(dra):
        rng = np.random.default_rng(seed)
        sel[rng.choice(dra, size=min(n_draft, len(dra)), replace=False)] = True
        sel[dra[np.argmax(w.req_len[dra])]] = True
    return sel


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    w = W.generate(name)
    g = Gpu(w)
    g.attn()
    g.topk()
    assert g.attn_flags() == 0 and g.topk_flags() == 0
    res = g.host()
    sel = np.ones(w.B, bool) if name == "qwen3_1p7b" else _sample(w)
    ref = run_oracle(w, select=sel)
    compare_attn(w, res, ref, select=sel)

    # properties of every request
    assert np.all(np.isfinite(res["out"]))
    off = 0
    for v, b in enumerate(w.verify_batch_index):
        L = int(w.req_len[b])
        lg = res["logits"][off:off + w.Hq * (w.k + 1) * L].reshape(w.Hq, w.k + 1, L)
        off += lg.size
        for j in range(w.k + 1):
            lim = L - (w.k + 1) + j
            assert np.all(np.isfinite(lg[:, j, :lim + 1])) and np.all(np.isneginf(lg[:, j, lim + 1:]))
        n = res["next_cnt"][v]
        assert np.all(n == w.topk_K[v])
        for h in range(w.Hkv):
            assert np.all(np.diff(res["next_idx"][v, h, :n[h]]) > 0)

    # Top-K of the sampled verify requests against the oracle's own dump
    if w.V:
        vsel = [v for v, b in enumerate(w.verify_batch_index) if sel[b]]
        Ls = w.verify_len[vsel]
        Ks = w.topk_K[vsel]
        t = oracle.topk_select(Hq=w.Hq, Hkv=w.Hkv, k=w.k, row_lo=1, row_hi=w.k + 1, logits=ref.logits,
                               lse=oracle.verify_lse_of(ref, w.req_mode, w.k, w.Hq, select=sel), L=Ls, K=Ks,
                               max_topk=g.shape.max_topk)
        compare_topk(res["next_idx"][vsel], res["next_cnt"][vsel], t, Ls, Ks, w.Hkv)
