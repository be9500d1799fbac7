"""Pins for the fp64 oracle: closed forms, invariants and brute force.

Each test fixes something the pages or plain mathematics determine, chosen so
that a plausible mistake in the oracle (a dropped term, a wrong sign or index,
a transposed operand, a wrong mask bound, a wrong averaging set) fails one of
them.  Definitions come from "SparseSpec-MLSys26", section 核心方法 /
PillarAttn (draft attends its critical set; verify is full causal attention
that dumps logits and LSE; exact scores are rematerialised, averaged over the
k draft rows and the GQA group's heads, and Top-K'd), and from the same
page's unified-batch section (page size 1: every position reaches its K/V
through a per-request slot table).
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import workloads as W

F = W.f32_to_bf16_bits


def bf(x):
    return F(np.asarray(x, np.float32))


def widen(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def make_case(rng, *, Hq, Hkv, D, k, lens, modes, lists=None, pool_extra=7, permute=True, scale=None):
    """Random bf16 case with a permuted page-size-1 pool."""
    lens = np.asarray(lens, np.int32)
    modes = np.asarray(modes, np.int32)
    B = len(lens)
    total = int(lens.sum())
    pool = total + pool_extra
    perm = rng.permutation(pool) if permute else np.arange(pool)
    table = perm[:total].astype(np.int32)
    kp = bf(rng.standard_normal((pool, Hkv, D)))
    vp = bf(rng.standard_normal((pool, Hkv, D)))
    T_q = int(np.where(modes == 1, k + 1, 1).sum())
    q = bf(rng.standard_normal((T_q, Hq, D)))
    max_sparse = 1
    if lists:
        max_sparse = max(max_sparse, max(len(v) for v in lists.values()))
    si = np.zeros((B, Hkv, max_sparse), np.int32)
    sc = np.zeros((B, Hkv), np.int32)
    for (b, h), lst in (lists or {}).items():
        si[b, h, :len(lst)] = lst
        sc[b, h] = len(lst)
    return dict(Hq=Hq, Hkv=Hkv, D=D, k=k, scale=(1 / math.sqrt(D)) if scale is None else scale, q=q,
                k_pool=kp, v_pool=vp, slot_table=table, req_mode=modes, req_len=lens, sparse_idx=si,
                sparse_cnt=sc)


def run(case, **kw):
    return oracle.attn_unified(**case, **kw)


# --------------------------------------------------------------------------- widening / rounding

def test_bf16_widening_exact_values():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x3F00) == 0.5
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133  # smallest subnormal
    assert oracle.bf16_to_f64(0x7F80) == math.inf


def test_generator_rounds_to_nearest_even():
    one = np.float32(1.0)
    ulp = 2.0 ** -7                      # bf16 spacing at 1.0
    assert F(np.float32(1.0 + ulp / 2))[()] == 0x3F80          # tie -> even (1.0)
    assert F(np.float32(1.0 + 3 * ulp / 2))[()] == 0x3F82      # tie -> even (1+2ulp)
    assert F(np.float32(1.0 + ulp / 2 + 2 ** -20))[()] == 0x3F81  # above the tie -> up
    assert F(one)[()] == 0x3F80
    assert F(np.float32(-2.0))[()] == 0xC000


# --------------------------------------------------------------------------- closed forms

def _three_key_case(mode):
    """q = (1, 0); keys (0,0), (1,0), (2,0); scale 1 => logits 0, 1, 2.
    V rows (1,0), (0,1), (1,1)."""
    kp = bf([[[0, 0]], [[1, 0]], [[2, 0]]])
    vp = bf([[[1, 0]], [[0, 1]], [[1, 1]]])
    k = 0
    q = bf([[[1, 0]]])
    lists = np.array([[[0, 1, 2]]], np.int32)
    return dict(Hq=1, Hkv=1, D=2, k=k, scale=1.0, q=q, k_pool=kp, v_pool=vp,
                slot_table=np.arange(3, dtype=np.int32), req_mode=np.array([mode], np.int32),
                req_len=np.array([3], np.int32), sparse_idx=lists, sparse_cnt=np.array([[3]], np.int32))


@pytest.mark.parametrize("mode", [0, 1])
def test_closed_form_three_keys(mode):
    r = run(_three_key_case(mode))
    e = math.e
    Z = 1 + e + e * e
    assert r.status == 0
    assert abs(r.lse[0, 0] - math.log(Z)) < 1e-14
    assert abs(r.out[0, 0, 0] - (1 + e * e) / Z) < 1e-14
    assert abs(r.out[0, 0, 1] - (e + e * e) / Z) < 1e-14
    if mode == 1:
        np.testing.assert_array_equal(r.logits, [0.0, 1.0, 2.0])


def test_zero_query_gives_uniform_weights():
    rng = np.random.default_rng(1)
    L = 37
    c = make_case(rng, Hq=2, Hkv=1, D=16, k=2, lens=[L], modes=[1])
    c["q"][:] = 0
    r = run(c)
    vrows = widen(c["v_pool"][c["slot_table"], 0, :])
    for j in range(3):
        n = L - 3 + j + 1
        assert abs(r.lse[j, 0] - math.log(n)) < 1e-13
        np.testing.assert_allclose(r.out[j, 0], vrows[:n].mean(0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_value():
    rng = np.random.default_rng(2)
    D, L = 8, 20
    lst = [1, 4, 5, 9, 13, 19]
    c = make_case(rng, Hq=1, Hkv=1, D=D, k=1, lens=[L], modes=[0], lists={(0, 0): lst}, scale=0.25)
    kv = np.zeros(D, np.float32)
    kv[0] = 3.0
    c["k_pool"][:] = bf(kv)
    qv = np.zeros(D, np.float32)
    qv[0] = 2.0
    c["q"][:] = bf(qv)
    r = run(c)
    logit = 0.25 * 6.0
    assert abs(r.lse[0, 0] - (logit + math.log(len(lst)))) < 1e-13
    vrows = widen(c["v_pool"][c["slot_table"][lst], 0, :])
    np.testing.assert_allclose(r.out[0, 0], vrows.mean(0), rtol=0, atol=1e-14)


def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    c = make_case(rng, Hq=4, Hkv=2, D=32, k=3, lens=[10], modes=[0], lists={(0, 0): [7], (0, 1): [2]})
    r = run(c)
    for h in range(4):
        g = h // 2
        t = [7, 2][g]
        slot = c["slot_table"][t]
        np.testing.assert_array_equal(r.out[0, h], widen(c["v_pool"][slot, g]))
        logit = c["scale"] * float(widen(c["q"][0, h]) @ widen(c["k_pool"][slot, g]))
        assert abs(r.lse[0, h] - logit) < 1e-12


def test_empty_list_gives_zero_and_minus_inf():
    rng = np.random.default_rng(4)
    c = make_case(rng, Hq=2, Hkv=1, D=8, k=2, lens=[9], modes=[0], lists={(0, 0): []})
    r = run(c)
    assert np.all(r.out == 0) and np.all(r.lse == -np.inf)


# --------------------------------------------------------------------------- invariants

def _mixed_case(rng, D=32, Hq=4, Hkv=2, k=3):
    lens = [40, 53, 29, 64]
    modes = [1, 0, 1, 0]
    lists = {}
    for b in (1, 3):
        for h in range(Hkv):
            n = rng.integers(1, lens[b])
            lists[(b, h)] = np.sort(rng.choice(lens[b], n, replace=False))
    return make_case(rng, Hq=Hq, Hkv=Hkv, D=D, k=k, lens=lens, modes=modes, lists=lists)


def test_full_list_draft_equals_verify_last_row():
    """Sparse attention whose list is the whole context equals full attention
    (the two are separate loops in the oracle)."""
    rng = np.random.default_rng(5)
    k, L, Hq, Hkv, D = 4, 70, 4, 2, 32
    cv = make_case(rng, Hq=Hq, Hkv=Hkv, D=D, k=k, lens=[L], modes=[1])
    rv = run(cv)
    cd = dict(cv)
    cd["req_mode"] = np.array([0], np.int32)
    cd["q"] = cv["q"][k:k + 1].copy()     # the last verify row's query
    cd["sparse_idx"] = np.tile(np.arange(L, dtype=np.int32), (1, Hkv, 1))
    cd["sparse_cnt"] = np.full((1, Hkv), L, np.int32)
    rd = run(cd)
    np.testing.assert_allclose(rd.out[0], rv.out[k], rtol=0, atol=1e-13)
    np.testing.assert_allclose(rd.lse[0], rv.lse[k], rtol=0, atol=1e-13)


def test_verify_row_equals_draft_over_its_causal_prefix():
    rng = np.random.default_rng(6)
    k, L, Hq, Hkv, D = 5, 33, 6, 3, 16
    cv = make_case(rng, Hq=Hq, Hkv=Hkv, D=D, k=k, lens=[L], modes=[1])
    rv = run(cv)
    for j in range(k + 1):
        upto = L - (k + 1) + j + 1
        cd = dict(cv)
        cd["req_mode"] = np.array([0], np.int32)
        cd["q"] = cv["q"][j:j + 1].copy()
        si = np.zeros((1, Hkv, L), np.int32)
        si[:, :, :upto] = np.arange(upto)
        cd["sparse_idx"] = si
        cd["sparse_cnt"] = np.full((1, Hkv), upto, np.int32)
        rd = run(cd)
        np.testing.assert_allclose(rd.out[0], rv.out[j], rtol=0, atol=1e-13)
        np.testing.assert_allclose(rd.lse[0], rv.lse[j], rtol=0, atol=1e-13)


def test_softmax_rows_sum_to_one_and_mask_is_causal():
    rng = np.random.default_rng(7)
    c = _mixed_case(rng)
    r = run(c)
    k, Hq = c["k"], c["Hq"]
    off = 0
    for b in np.nonzero(c["req_mode"] == 1)[0]:
        L = int(c["req_len"][b])
        lg = r.logits[off:off + Hq * (k + 1) * L].reshape(Hq, k + 1, L)
        off += Hq * (k + 1) * L
        lse = oracle.verify_lse_of(r, c["req_mode"], k, Hq)[list(np.nonzero(c["req_mode"] == 1)[0]).index(b)]
        for h in range(Hq):
            for j in range(k + 1):
                lim = L - (k + 1) + j
                assert np.all(np.isfinite(lg[h, j, :lim + 1]))
                assert np.all(lg[h, j, lim + 1:] == -np.inf)
                s = np.exp(lg[h, j, :lim + 1] - lse[h, j]).sum()
                assert abs(s - 1.0) < 1e-13


def test_future_positions_do_not_change_a_verify_row():
    rng = np.random.default_rng(8)
    k, L = 3, 25
    c = make_case(rng, Hq=2, Hkv=1, D=16, k=k, lens=[L], modes=[1])
    r0 = run(c)
    # perturb K/V of the last position: only the last row can see it
    s_last = c["slot_table"][L - 1]
    c2 = {**c, "k_pool": c["k_pool"].copy(), "v_pool": c["v_pool"].copy()}
    c2["k_pool"][s_last] = bf(rng.standard_normal(c2["k_pool"][s_last].shape))
    c2["v_pool"][s_last] = bf(rng.standard_normal(c2["v_pool"][s_last].shape))
    r1 = run(c2)
    np.testing.assert_array_equal(r1.out[:k], r0.out[:k])
    np.testing.assert_array_equal(r1.lse[:k], r0.lse[:k])
    assert np.abs(r1.out[k] - r0.out[k]).max() > 1e-6


def test_slot_translation_is_a_relabelling():
    """Moving every row to another slot (and the table with it) changes nothing."""
    rng = np.random.default_rng(9)
    c = _mixed_case(rng)
    r0 = run(c)
    pool = c["k_pool"].shape[0]
    pi = rng.permutation(pool)
    c2 = dict(c)
    c2["k_pool"] = np.empty_like(c["k_pool"])
    c2["v_pool"] = np.empty_like(c["v_pool"])
    c2["k_pool"][pi] = c["k_pool"]
    c2["v_pool"][pi] = c["v_pool"]
    c2["slot_table"] = pi[c["slot_table"]].astype(np.int32)
    r1 = run(c2)
    np.testing.assert_array_equal(r1.out, r0.out)
    np.testing.assert_array_equal(r1.lse, r0.lse)
    np.testing.assert_array_equal(r1.logits, r0.logits)


def test_requests_are_independent_of_their_batch():
    rng = np.random.default_rng(10)
    c = _mixed_case(rng)
    r_all = run(c)
    k = c["k"]
    q_off = np.concatenate([[0], np.cumsum(np.where(c["req_mode"] == 1, k + 1, 1))[:-1]])
    kv_off = np.concatenate([[0], np.cumsum(c["req_len"])[:-1]])
    for b in range(len(c["req_len"])):
        nq = k + 1 if c["req_mode"][b] else 1
        L = int(c["req_len"][b])
        c1 = dict(c)
        c1["req_mode"] = c["req_mode"][b:b + 1]
        c1["req_len"] = c["req_len"][b:b + 1]
        c1["q"] = c["q"][q_off[b]:q_off[b] + nq]
        c1["slot_table"] = c["slot_table"][kv_off[b]:kv_off[b] + L]
        c1["sparse_idx"] = c["sparse_idx"][b:b + 1]
        c1["sparse_cnt"] = c["sparse_cnt"][b:b + 1]
        r1 = run(c1)
        np.testing.assert_array_equal(r1.out, r_all.out[q_off[b]:q_off[b] + nq])
    sel = np.array([False, True, True, False])
    r_sel = run(c, select=sel)
    np.testing.assert_array_equal(r_sel.out[q_off[1]:q_off[3]], r_all.out[q_off[1]:q_off[3]])


def test_query_head_uses_kv_head_h_over_G():
    """Swapping the two KV heads and the two query-head groups swaps the outputs."""
    rng = np.random.default_rng(11)
    k, L, Hq, Hkv = 2, 19, 4, 2
    c = make_case(rng, Hq=Hq, Hkv=Hkv, D=16, k=k, lens=[L, 12], modes=[1, 0],
                  lists={(1, 0): [0, 3, 11], (1, 1): [5, 6]})
    r0 = run(c)
    c2 = dict(c)
    c2["k_pool"] = c["k_pool"][:, ::-1].copy()
    c2["v_pool"] = c["v_pool"][:, ::-1].copy()
    c2["q"] = np.concatenate([c["q"][:, 2:], c["q"][:, :2]], axis=1).copy()
    c2["sparse_idx"] = c["sparse_idx"][:, ::-1].copy()
    c2["sparse_cnt"] = c["sparse_cnt"][:, ::-1].copy()
    r1 = run(c2)
    np.testing.assert_array_equal(r1.out[:, :2], r0.out[:, 2:])
    np.testing.assert_array_equal(r1.out[:, 2:], r0.out[:, :2])


def test_split_lists_merge_back_by_lse():
    """Attention over a list equals the LSE-weighted merge of attention over a
    partition of it: o = sum_i exp(lse_i - lse) o_i with lse = log sum exp(lse_i).
    A wrong LSE (e.g. a missing max shift) breaks this."""
    rng = np.random.default_rng(12)
    L = 90
    full = np.arange(L)
    parts = [full[:17], full[17:60], full[60:]]
    lists = {(0, 0): full}
    c = make_case(rng, Hq=2, Hkv=1, D=32, k=1, lens=[L], modes=[0], lists=lists)
    rf = run(c)
    outs, lses = [], []
    for p in parts:
        cp = dict(c)
        si = np.zeros((1, 1, L), np.int32)
        si[0, 0, :len(p)] = p
        cp["sparse_idx"] = si
        cp["sparse_cnt"] = np.array([[len(p)]], np.int32)
        rp = run(cp)
        outs.append(rp.out[0])
        lses.append(rp.lse[0])
    lses = np.array(lses)
    lse = np.logaddexp.reduce(lses, axis=0)
    o = sum(np.exp(lses[i] - lse)[:, None] * outs[i] for i in range(3))
    np.testing.assert_allclose(lse, rf.lse[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, rf.out[0], rtol=0, atol=1e-12)


def test_scale_multiplies_the_logits():
    """Doubling the scale equals doubling every query (exact in bf16)."""
    rng = np.random.default_rng(13)
    c = _mixed_case(rng)
    c1 = dict(c, scale=2 * c["scale"])
    c2 = dict(c, q=bf(2 * widen(c["q"]).astype(np.float32)))
    r1, r2 = run(c1), run(c2)
    np.testing.assert_array_equal(r1.out, r2.out)
    np.testing.assert_array_equal(r1.logits, r2.logits)


def test_out_of_range_entries_are_skipped_and_reported():
    rng = np.random.default_rng(14)
    c = make_case(rng, Hq=2, Hkv=1, D=16, k=1, lens=[30], modes=[0], lists={(0, 0): [1, 5, 30, 7]})
    r = run(c)
    assert r.status == -4
    c_ok = make_case(np.random.default_rng(14), Hq=2, Hkv=1, D=16, k=1, lens=[30], modes=[0],
                     lists={(0, 0): [1, 5, 7]})
    r_ok = run(c_ok)
    np.testing.assert_array_equal(r.out, r_ok.out)


# --------------------------------------------------------------------------- Top-K pins

def _topk_of(logits_rows, lse_rows, L, K, Hq=1, Hkv=1, k=0, row_lo=0, row_hi=1, max_topk=None):
    return oracle.topk_select(Hq=Hq, Hkv=Hkv, k=k, row_lo=row_lo, row_hi=row_hi,
                              logits=np.asarray(logits_rows, np.float64).ravel(),
                              lse=np.asarray(lse_rows, np.float64).reshape(-1, Hq, k + 1),
                              L=np.array(L, np.int32), K=np.array(K, np.int32),
                              max_topk=max_topk or max(K) if len(K) else 1)


@pytest.mark.parametrize("seed", range(12))
def test_topk_matches_brute_force_subset_enumeration(seed):
    """The chosen set is the max-sum K-subset of scores; among max-sum subsets
    the lexicographically smallest (ties go to lower positions)."""
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(2, 13))
    K = int(rng.integers(1, L + 1))
    Hq, Hkv, k = 2, 1, 2
    # coarse logits so that exact ties happen
    lg = rng.integers(-3, 3, size=(Hq, k + 1, L)).astype(np.float64)
    lse = np.log(np.exp(lg).sum(-1))
    res = _topk_of(lg, lse, [L], [K], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=3)
    score = res.scores[:L]
    best, best_set = -np.inf, None
    for sub in itertools.combinations(range(L), K):  # lexicographic order
        s = math.fsum(score[list(sub)])
        if s > best + 1e-12:
            best, best_set = s, sub
    got = tuple(res.next_idx[0, 0, :res.next_cnt[0, 0]])
    assert got == best_set


def test_topk_ties_take_lower_positions_and_output_is_ascending():
    L = 10
    lg = np.zeros((1, 1, L))
    lg[0, 0, [2, 5, 8]] = 1.0            # three equal maxima
    lse = np.log(np.exp(lg).sum(-1))
    res = _topk_of(lg, lse, [L], [2])
    assert list(res.next_idx[0, 0, :2]) == [2, 5]
    res = _topk_of(lg, lse, [L], [5])
    assert list(res.next_idx[0, 0, :5]) == [0, 1, 2, 5, 8]


def test_topk_scores_average_softmax_rows():
    """With full softmax rows the averaged scores sum to 1; with one row and
    one head they are that row's softmax."""
    rng = np.random.default_rng(20)
    Hq, Hkv, k, L = 6, 2, 3, 17
    lg = rng.standard_normal((Hq, k + 1, L))
    lse = np.log(np.exp(lg).sum(-1))
    res = _topk_of(lg, lse, [L], [4], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=k + 1)
    sc = res.scores.reshape(Hkv, L)
    np.testing.assert_allclose(sc.sum(-1), 1.0, rtol=0, atol=1e-14)
    res1 = _topk_of(lg[:1, 2:3], lse[:1, 2:3], [L], [4], Hq=1, Hkv=1, k=0, row_lo=0, row_hi=1)
    np.testing.assert_allclose(res1.scores, np.exp(lg[0, 2] - lse[0, 2]), rtol=1e-15, atol=0)


def test_topk_uses_exactly_the_averaged_rows_and_group_heads():
    rng = np.random.default_rng(21)
    Hq, Hkv, k, L = 4, 2, 3, 15
    lg = rng.standard_normal((Hq, k + 1, L))
    lse = np.log(np.exp(lg).sum(-1))
    base = _topk_of(lg, lse, [L], [5], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=k + 1)
    lg2 = lg.copy()
    lg2[:, 0, :] = rng.standard_normal((Hq, L)) * 10     # row 0 is not averaged
    r2 = _topk_of(lg2, lse, [L], [5], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=k + 1)
    np.testing.assert_array_equal(r2.scores, base.scores)
    lg3 = lg.copy()
    lg3[3] = rng.standard_normal((k + 1, L)) * 10        # head 3 is in group 1 only
    r3 = _topk_of(lg3, lse, [L], [5], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=k + 1)
    np.testing.assert_array_equal(r3.scores[:L], base.scores[:L])
    assert np.abs(r3.scores[L:] - base.scores[L:]).max() > 1e-6
    # masked (-inf) entries contribute zero
    lg4 = lg.copy()
    lg4[0, 1, 7] = -np.inf
    r4 = _topk_of(lg4, lse, [L], [5], Hq=Hq, Hkv=Hkv, k=k, row_lo=1, row_hi=k + 1)
    expect = base.scores[7] - np.exp(lg[0, 1, 7] - lse[0, 1]) / (k * 2)
    assert abs(r4.scores[7] - expect) < 1e-15


def test_topk_budget_edges():
    lg = np.log(np.arange(1, 7, dtype=np.float64))[None, None, :]
    lse = np.log(np.exp(lg).sum(-1))
    r = _topk_of(lg, lse, [6], [9], max_topk=9)       # K > L keeps everything
    assert r.next_cnt[0, 0] == 6 and list(r.next_idx[0, 0, :6]) == list(range(6))
    r = _topk_of(lg, lse, [6], [0], max_topk=1)
    assert r.next_cnt[0, 0] == 0
    r = _topk_of(lg, lse, [6], [2])
    assert list(r.next_idx[0, 0, :2]) == [4, 5]


def test_topk_of_a_real_verify_recovers_planted_pillars():
    """Informational recall check on the tiny workload: the planted columns
    dominate the verify scores well above chance."""
    w = W.generate("tiny")
    kp, vp = w.pool("k"), w.pool("v")
    r = oracle.attn_unified(Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, scale=1 / math.sqrt(w.D), q=w.q, k_pool=kp,
                            v_pool=vp, slot_table=w.slot_table, req_mode=w.req_mode, req_len=w.req_len,
                            sparse_idx=w.sparse_idx, sparse_cnt=w.sparse_cnt)
    lse = oracle.verify_lse_of(r, w.req_mode, w.k, w.Hq)
    t = oracle.topk_select(Hq=w.Hq, Hkv=w.Hkv, k=w.k, row_lo=1, row_hi=w.k + 1, logits=r.logits, lse=lse,
                           L=w.verify_len, K=w.topk_K, max_topk=int(w.topk_K.max()))
    hits = tot = 0
    base = 0.0
    for vi, b in enumerate(w.verify_batch_index):
        off = int(w.kv_off[b])
        L = int(w.req_len[b])
        pil = w.pillar[off:off + L, 0]
        sel = t.next_idx[vi, 0, :t.next_cnt[vi, 0]]
        hits += int(pil[sel].sum())
        tot += len(sel)
        base += pil.mean() * len(sel)
    assert hits > 3 * base


def test_kv_append_pins():
    """The append writes exactly the listed slots with the new rows, leaves
    every other row as it was, skips out-of-range slots, and appending the
    pool's own rows to their own slots changes nothing."""
    rng = np.random.default_rng(3)
    k = rng.integers(-9, 9, (12, 2, 4)).astype(np.int16)
    v = rng.integers(-9, 9, (12, 2, 4)).astype(np.int16)
    kn = rng.integers(20, 29, (3, 2, 4)).astype(np.int16)
    vn = rng.integers(30, 39, (3, 2, 4)).astype(np.int16)
    k2, v2, skipped = oracle.kv_append(k, v, kn, vn, np.array([5, 12, 0], np.int32))
    assert skipped
    for s in range(12):
        want_k = kn[0] if s == 5 else kn[2] if s == 0 else k[s]
        want_v = vn[0] if s == 5 else vn[2] if s == 0 else v[s]
        assert np.array_equal(k2[s], want_k) and np.array_equal(v2[s], want_v)
    assert np.array_equal(k, k2) is False and k.shape == k2.shape  # the inputs are not modified in place
    same = np.arange(12, dtype=np.int32)
    k3, v3, skipped = oracle.kv_append(k, v, k, v, same)
    assert not skipped and np.array_equal(k3, k) and np.array_equal(v3, v)


def test_kv_offload_pins():
    """The offload gathers the listed slot blocks in list order (a repeated
    slot gives the same row twice), reports out-of-range slots with their
    rows left zero, and appending its rows back to the same slots restores the
    pools; appending them to other slots moves the request's KV there."""
    rng = np.random.default_rng(4)
    k = rng.integers(-9, 9, (10, 3, 4)).astype(np.int16)
    v = rng.integers(-9, 9, (10, 3, 4)).astype(np.int16)
    slots = np.array([7, 2, 2, 9, 0], np.int32)
    ko, vo, skipped = oracle.kv_offload(k, v, slots)
    assert not skipped and ko.shape == (5, 3, 4)
    for i, s in enumerate(slots):
        assert np.array_equal(ko[i], k[s]) and np.array_equal(vo[i], v[s])
    k2, v2, _ = oracle.kv_append(np.zeros_like(k), np.zeros_like(v), ko, vo, slots)
    for s in set(slots.tolist()):
        assert np.array_equal(k2[s], k[s]) and np.array_equal(v2[s], v[s])
    kb, vb, skipped = oracle.kv_offload(k, v, np.array([3, 10, -1], np.int32))
    assert skipped and np.array_equal(kb[0], k[3]) and not kb[1:].any() and not vb[1:].any()
    moved = np.array([1, 4, 5, 6, 8], np.int32)  # the same rows, new slots
    k3, v3, _ = oracle.kv_append(k, v, ko, vo, moved)
    for i, s in enumerate(moved):
        assert np.array_equal(k3[s], k[slots[i]]) and np.array_equal(v3[s], v[slots[i]])


def test_draft_lists_after_topk_rebuild_the_generator_lists():
    """The workload generator builds each draft request's list independently
    (a critical subset of [0, L-p) plus the p newest positions); feeding the
    oracle that critical subset as the Top-K of a verify step of length L-p
    gives back exactly the generator's list, and the slots are the slot
    table's entries for those positions."""
    import workloads as W
    w = W.generate(W.scaled("qwen3_8b", B=20, length_scale=0.05, seed_offset=9))
    for b in np.nonzero(w.req_mode == 0)[0]:
        p, L = int(w.phase[b]), int(w.req_len[b])
        gen = [w.sparse_idx[b, h, :w.sparse_cnt[b, h]] for h in range(w.Hkv)]
        crit = [g[g < L - p] for g in gen]
        kmax = max(1, max(len(c) for c in crit))
        nidx = np.zeros((1, w.Hkv, kmax), np.int32)
        ncnt = np.zeros((1, w.Hkv), np.int32)
        for h, c in enumerate(crit):
            nidx[0, h, :len(c)] = c[::-1]  # any order in: the list comes out ascending
            ncnt[0, h] = len(c)
        lists, counts, slots = oracle.draft_lists_after_topk(nidx, ncnt, [L - p], p, slot_table=w.slot_table,
                                                             kv_off=[w.kv_off[b]])
        for h in range(w.Hkv):
            assert np.array_equal(lists[0, h, :counts[0, h]], gen[h])
            for i in range(counts[0, h]):
                assert slots[0, h, i] == w.slot_table[w.kv_off[b] + lists[0, h, i]]


def test_draft_lists_after_topk_shape_rules():
    nidx = np.array([[[7, 2, 9], [0, 0, 0]], [[4, 0, 0], [1, 3, 0]]], np.int32)
    ncnt = np.array([[3, 0], [1, 2]], np.int32)
    lists, counts, slots = oracle.draft_lists_after_topk(nidx, ncnt, [10, 6], [2, 0])
    assert slots is None
    assert counts.tolist() == [[5, 2], [1, 2]]
    assert lists[0, 0, :5].tolist() == [2, 7, 9, 10, 11]  # Top-K ascending, then the two appended positions
    assert lists[0, 1, :2].tolist() == [10, 11]            # an empty Top-K keeps the appended positions
    assert lists[1, 0, :1].tolist() == [4] and lists[1, 1, :2].tolist() == [1, 3]  # phase 0: the Top-K alone
    ident = np.arange(64, dtype=np.int32)
    _, _, s2 = oracle.draft_lists_after_topk(nidx, ncnt, [10, 6], 3, slot_table=ident, kv_off=[0, 20])
    l3, c3, _ = oracle.draft_lists_after_topk(nidx, ncnt, [10, 6], 3)
    for h in range(2):
        assert s2[0, h, :c3[0, h]].tolist() == l3[0, h, :c3[0, h]].tolist()  # request 0's slots start at 0
        assert s2[1, h, :c3[1, h]].tolist() == [20 + x for x in l3[1, h, :c3[1, h]]]  # request 1's at 20
