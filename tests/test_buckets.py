"""Host-side phase buckets of the unified batch ("SparseSpec-MLSys26",
Unified batch scheduler + fused attention kernel, load balancing): a new
request joins the least loaded of the k+1 buckets, so each step verifies
about B/(k+1) requests and carries about (2k+1)/(k+1)*B query rows.  These
checks call the C ABI; no GPU is needed."""
import numpy as np
import pytest

import sparse_self_speculative_pillar_gb300 as P
import workloads as W


@pytest.mark.parametrize("name", ["qwen3_1p7b", "qwen3_8b", "stress"])
def test_admission_in_order_gives_the_workload_phases(name):
    """Admitting a workload's requests in batch order puts request i in bucket
    i mod (k+1); at step 0 the modes and phases are the ones the workload
    generator assigns (phase i mod (k+1), phase 0 verifies)."""
    w = W.generate(W.scaled(name, B=min(W.RECIPES[name].B, 40), length_scale=0.01))
    pb = P.pillar_buckets_init(w.k)
    buckets = [P.pillar_buckets_admit(pb) for _ in range(w.B)]
    assert buckets == [i % (w.k + 1) for i in range(w.B)]
    mode, phase, rows = P.pillar_buckets_step(pb, buckets, 0)
    np.testing.assert_array_equal(mode, w.req_mode)
    np.testing.assert_array_equal(phase, w.phase)
    assert rows == w.q.shape[0]  # the step's T_q


def _least_loaded(count):
    return min(range(len(count)), key=lambda c: (count[c], c))


def test_admission_always_takes_a_least_loaded_bucket():
    rng = np.random.default_rng(11)
    for k in (0, 1, 4, 8, 12, 63):
        pb = P.pillar_buckets_init(k)
        live = []  # buckets of the requests in flight
        for _ in range(600):
            if live and rng.random() < 0.4:
                b = live.pop(int(rng.integers(len(live))))
                P.pillar_buckets_retire(pb, b)
            else:
                expect = _least_loaded([pb.count[c] for c in range(k + 1)])
                b = P.pillar_buckets_admit(pb)
                assert b == expect
                live.append(b)
            assert [pb.count[c] for c in range(k + 1)] == [live.count(c) for c in range(k + 1)]


def test_step_rows_average_2k_plus_1_over_k_plus_1_times_B():
    """Over one cycle every request verifies once (k+1 rows) and drafts k
    times (one row): the mean step carries (2k+1)/(k+1)*B rows, and with
    balanced buckets no step strays from it by more than k rows, where a
    batch whose requests all verify together alternates between B and
    (k+1)*B."""
    for k, B in ((8, 128), (12, 256), (3, 7), (8, 5)):
        pb = P.pillar_buckets_init(k)
        buckets = [P.pillar_buckets_admit(pb) for _ in range(B)]
        rows = [P.pillar_buckets_step(pb, buckets, t)[2] for t in range(k + 1)]
        assert sum(rows) == B * (2 * k + 1)
        lo, hi = B + k * (B // (k + 1)), B + k * (-(-B // (k + 1)))
        assert all(lo <= r <= hi for r in rows)
        same = [0] * B  # every request in one bucket
        naive = [P.pillar_buckets_step(pb, same, t)[2] for t in range(k + 1)]
        assert sorted(set(naive)) == sorted({B, (k + 1) * B})
        assert max(rows) <= max(naive)


def test_phase_advances_one_step_at_a_time():
    pb = P.pillar_buckets_init(5)
    buckets = [P.pillar_buckets_admit(pb) for _ in range(17)]
    prev = P.pillar_buckets_step(pb, buckets, -7)[1]
    for t in range(-6, 20):
        mode, phase, _ = P.pillar_buckets_step(pb, buckets, t)
        assert phase == [(p + 1) % 6 for p in prev]
        assert mode == [int(p == 0) for p in phase]
        prev = phase


def test_bucket_argument_checks():
    with pytest.raises(P.PillarError):
        P.pillar_buckets_init(64)  # more than 64 buckets
    with pytest.raises(P.PillarError):
        P.pillar_buckets_init(-1)
    pb = P.pillar_buckets_init(2)
    with pytest.raises(P.PillarError):
        P.pillar_buckets_retire(pb, 0)  # empty
    b = P.pillar_buckets_admit(pb)
    with pytest.raises(P.PillarError):
        P.pillar_buckets_retire(pb, 3)  # no such bucket
    with pytest.raises(P.PillarError):
        P.pillar_buckets_step(pb, [b, 3], 0)
    assert [pb.count[c] for c in range(3)] == [1, 0, 0]  # nothing changed by the failed calls
    lib = P.load()
    assert lib.pillar_buckets_admit(None, None) == -1
    assert lib.pillar_buckets_step(None, None, 0, 0, None, None, None) == -1
    assert P.pillar_buckets_step(pb, [], 4) == ([], [], 0)
