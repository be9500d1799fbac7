"""The seeded inputs have the stated shapes and structure."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b"])
def test_structure(name):
    w = W.generate(name)
    r = w.recipe
    assert w.q.shape == (int(np.where(w.req_mode == 1, r.k + 1, 1).sum()), r.Hq, r.D)
    assert w.k_logical.shape == (int(w.req_len.sum()), r.Hkv, r.D)
    st = w.slot_table
    assert len(np.unique(st)) == len(st) and st.min() >= 0 and st.max() < w.num_slots
    assert w.num_slots >= 1.25 * len(st)
    assert np.all(w.req_len[w.req_mode == 1] >= r.k + 1)
    for b in range(w.B):
        if w.req_mode[b] == 1:
            assert np.all(w.sparse_cnt[b] == 0)
            continue
        p, L = int(w.phase[b]), int(w.req_len[b])
        for h in range(w.Hkv):
            lst = w.sparse_idx[b, h, :w.sparse_cnt[b, h]]
            assert np.all(np.diff(lst) > 0) and lst[0] >= 0 and lst[-1] < L
            assert set(range(L - p, L)) <= set(lst.tolist())
            kb = -(-(L - p) * r.s_num // r.s_den)
            assert len(lst) == kb + p
    np.testing.assert_array_equal(w.topk_K, -(-w.verify_len.astype(np.int64) * r.s_num // r.s_den))


def test_deterministic_and_phase_mix():
    a = W.generate(W.scaled("qwen3_8b", B=18, length_scale=0.05))
    b = W.generate(W.scaled("qwen3_8b", B=18, length_scale=0.05))
    for f in ("q", "k_logical", "v_logical", "slot_table", "sparse_idx", "req_len"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert a.V == 2 and list(np.nonzero(a.req_mode)[0]) == [0, 9]


def test_degenerate_mixes():
    d = W.generate(W.scaled("stress_all_draft", B=13, length_scale=0.05))
    v = W.generate(W.scaled("stress_all_verify", B=5, length_scale=0.05))
    assert d.V == 0 and v.V == 5


def test_bf16_rounding_roundtrip():
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    b = W.f32_to_bf16_bits(x)
    y = W.bf16_bits_to_f32(b)
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)
