"""A device wait that runs out, on the GPU.

With a wait bound of one microsecond -- far below the time the persistent
kernel's roles need to hand work to one another (every hand-off waits on a
global-memory round trip) -- some pipeline wait of every CTA gives up.  The
kernel must then record PILLAR_FLAG_TIMEOUT, let the copies and tensor-core
work already in flight finish (those drains keep their one-second bound),
free its tensor memory and return; the CUDA context stays usable, and the
next call on the same buffers with the default bound must be exact against
the oracle.  Nothing here faults, traps or hangs: every wait involved is
bounded."""
import math

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import sparse_self_speculative_pillar_gb300 as P  # noqa: E402
from tests._gpu_common import Gpu, compare_attn, run_oracle  # noqa: E402


def test_short_wait_bound_reports_timeout_and_the_next_call_is_exact():
    w = W.generate(W.scaled("qwen3_8b", B=12, length_scale=0.05, seed_offset=9))
    g = Gpu(w, wait_timeout_us=1)
    g.attn()
    flags = g.attn_flags()
    assert flags & P.FLAG_TIMEOUT, f"device flags 0x{flags:x}: no wait ran out"
    assert flags & ~(P.FLAG_TIMEOUT) == 0, f"device flags 0x{flags:x}"
    # the same buffers, the default bound
    g.shape.wait_timeout_us = 0
    g.out.zero_()
    g.logits.fill_(math.nan)
    g.lse.fill_(math.nan)
    g.attn()
    assert g.attn_flags() == 0
    res = g.host()
    compare_attn(w, res, run_oracle(w))


def test_wait_bound_is_checked_on_the_host():
    w = W.generate(W.scaled("qwen3_8b", B=4, length_scale=0.02, seed_offset=10))
    g = Gpu(w)
    g.shape.wait_timeout_us = -5
    with pytest.raises(P.PillarError):
        g.attn()
    g.shape.wait_timeout_us = 50_000  # a 50 ms bound: ample for this step
    g.attn()
    assert g.attn_flags() == 0
    np.testing.assert_equal(np.isfinite(g.host()["out"]).all(), True)
