"""Full-size workloads in the launch configuration the benchmark times
(default chunking, one persistent CTA per SM).  Every request of every
workload is compared element by element with the fp64 oracle -- its output
rows, and for a verify request its logits and LSEs -- and the Top-K of every
verify request is compared with the oracle's Top-K of the oracle's own dump.
The oracle runs over groups of consecutive requests so that the host holds a
bounded slice of the fp64 logits at a time; the worst errors of each workload
are printed (pytest -s shows them)."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
from tests._gpu_common import Gpu, compare_attn, compare_topk, run_oracle  # noqa: E402

FULL = ["qwen3_1p7b", "qwen3_8b", "qwen3_14b", "stress", "stress_all_draft", "stress_all_verify"]
GROUP_LOGITS = 1 << 27   # fp64 logits the oracle may hold per group (1 GiB)
GROUP_REQUESTS = 64


def request_groups(w):
    """Consecutive requests, each group's verify logits within GROUP_LOGITS."""
    groups, cur, n_log = [], [], 0
    for b in range(w.B):
        lb = int(w.Hq * (w.k + 1) * w.req_len[b]) if w.req_mode[b] == 1 else 0
        if cur and (n_log + lb > GROUP_LOGITS or len(cur) == GROUP_REQUESTS):
            groups.append(cur)
            cur, n_log = [], 0
        cur.append(b)
        n_log += lb
    if cur:
        groups.append(cur)
    return groups


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_request(name):
    w = W.generate(name)
    g = Gpu(w)
    g.attn()
    g.topk()
    assert g.attn_flags() == 0 and g.topk_flags() == 0
    res = g.host(logits_f64=False)
    worst, topk_diff, compared = {}, 0, 0
    for grp in request_groups(w):
        sel = np.zeros(w.B, bool)
        sel[grp] = True
        ref = run_oracle(w, select=sel)
        for key, v in compare_attn(w, res, ref, select=sel).items():
            worst[key] = max(worst.get(key, 0.0), v)
        compared += len(grp)
        vsel = [v for v, b in enumerate(w.verify_batch_index) if sel[b]]
        if vsel:
            Ls, Ks = w.verify_len[vsel], w.topk_K[vsel]
            t = oracle.topk_select(Hq=w.Hq, Hkv=w.Hkv, k=w.k, row_lo=1, row_hi=w.k + 1, logits=ref.logits,
                                   lse=oracle.verify_lse_of(ref, w.req_mode, w.k, w.Hq, select=sel), L=Ls, K=Ks,
                                   max_topk=g.shape.max_topk)
            topk_diff += compare_topk(res["next_idx"][vsel], res["next_cnt"][vsel], t, Ls, Ks, w.Hkv)
    assert compared == w.B
    print(f"\n{name}: {w.B} requests ({w.V} verify) compared element by element; worst max-abs / rel-l2 error: "
          + ", ".join(f"{q} {worst[q + '_abs']:.2e} / {worst[q + '_rel']:.2e}" for q in ("out", "logits", "lse"))
          + f"; Top-K positions differing inside the tie band: {topk_diff}")
