"""GPU check of pillar_kv_append against the oracle's kv_append (the pools
after the append hold the new rows in the given slots, every other row
unchanged), with out-of-range slots skipped and flagged."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import sparse_self_speculative_pillar_gb300 as P  # noqa: E402


@pytest.mark.parametrize("D,Hkv,n,num_slots", [(128, 8, 1152, 4096), (64, 3, 37, 257), (128, 1, 1, 5)])
def test_append_scatters_rows_into_slots(D, Hkv, n, num_slots):
    rng = np.random.default_rng(D * 1000 + n)
    k_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    v_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    k_new = rng.integers(-2**15, 2**15, (n, Hkv, D), dtype=np.int16)
    v_new = rng.integers(-2**15, 2**15, (n, Hkv, D), dtype=np.int16)
    slots = rng.permutation(num_slots)[:n].astype(np.int32)
    expect_k, expect_v, skipped = oracle.kv_append(k_pool, v_pool, k_new, v_new, slots)
    assert not skipped
    dk, dv = torch.from_numpy(k_pool).cuda(), torch.from_numpy(v_pool).cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = P.make_shape(B=1, Hq=Hkv, Hkv=Hkv, D=D, k=1, max_sparse=0, max_len=1, num_slots=num_slots)
    P.pillar_kv_append(shape, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(),
                       torch.from_numpy(slots).cuda(), dk, dv, device_flags=flags)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dk.cpu().numpy(), expect_k)
    np.testing.assert_array_equal(dv.cpu().numpy(), expect_v)
    assert int(flags.item()) == 0


def test_out_of_range_slot_is_skipped_and_flagged():
    D, Hkv, num_slots = 128, 2, 64
    rng = np.random.default_rng(5)
    k_pool = rng.integers(-2**15, 2**15, (num_slots, Hkv, D), dtype=np.int16)
    k_new = rng.integers(-2**15, 2**15, (4, Hkv, D), dtype=np.int16)
    slots = np.array([3, num_slots, -1, 10], np.int32)
    expect, _, skipped = oracle.kv_append(k_pool, k_pool, k_new, k_new, slots)
    assert skipped
    dk, dv = torch.from_numpy(k_pool).cuda(), torch.from_numpy(k_pool.copy()).cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = P.make_shape(B=1, Hq=Hkv, Hkv=Hkv, D=D, k=1, max_sparse=0, max_len=1, num_slots=num_slots)
    nk = torch.from_numpy(k_new).cuda()
    P.pillar_kv_append(shape, nk, nk, torch.from_numpy(slots).cuda(), dk, dv, device_flags=flags)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dk.cpu().numpy(), expect)
    np.testing.assert_array_equal(dv.cpu().numpy(), expect)
    assert int(flags.item()) == P.FLAG_SLOT
