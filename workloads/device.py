"""Device copies of one seeded workload and the C-ABI calls on them.

A harness for the tests and the benchmark: it uploads a workload's inputs
(the page-size-1 pools are built on the device by scattering the logical K/V
rows into their slots), allocates the outputs and workspaces the entry points
need, and calls them through the binding.  It holds none of the method's
arithmetic and does not touch the fp64 oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import sparse_self_speculative_pillar_gb300 as P

from . import Workload


def to_device(a: np.ndarray) -> torch.Tensor:
    """A numpy array on cuda:current (bf16 bit patterns travel as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


class Gpu:
    """Device inputs, outputs and workspaces of one workload."""

    def __init__(self, w: Workload, **shape_kw):
        self.w = w
        self.q = to_device(w.q)
        st = to_device(w.slot_table).long()
        self.k_pool = torch.zeros((w.num_slots, w.Hkv, w.D), dtype=torch.int16, device="cuda")
        self.v_pool = torch.zeros_like(self.k_pool)
        self.k_pool[st] = to_device(w.k_logical)
        self.v_pool[st] = to_device(w.v_logical)
        self.slot_table = to_device(w.slot_table)
        self.req_mode = to_device(w.req_mode)
        self.req_len = to_device(w.req_len)
        self.sparse_idx = to_device(w.sparse_idx)
        self.sparse_cnt = to_device(w.sparse_cnt)
        self.group_map = to_device(w.verify_batch_index)
        self.K = to_device(w.topk_K)
        self.V = w.V
        kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, max_sparse=w.max_sparse,
                  max_len=int(max(1, w.req_len.max())), num_slots=w.num_slots,
                  max_topk=int(w.topk_K.max()) if w.V else 1)
        kw.update(shape_kw)
        self.shape = P.make_shape(**kw)
        T_q = w.q.shape[0]
        n_logits = int(w.Hq * (w.k + 1) * w.verify_len.astype(np.int64).sum())
        self.out = torch.empty((T_q, w.Hq, w.D), dtype=torch.int16, device="cuda")
        self.logits = torch.full((max(1, n_logits),), float("nan"), dtype=torch.float32, device="cuda")
        self.lse = torch.full((max(1, w.V), w.Hq, w.k + 1), float("nan"), dtype=torch.float32, device="cuda")
        self.ws = torch.empty(P.pillar_attn_workspace_bytes(self.shape), dtype=torch.uint8, device="cuda")
        self.tws = torch.empty(P.pillar_topk_workspace_bytes(self.shape, max(1, w.V)), dtype=torch.uint8,
                               device="cuda")
        self.next_idx = torch.full((max(1, w.V), w.Hkv, self.shape.max_topk), -1, dtype=torch.int32, device="cuda")
        self.next_cnt = torch.full((max(1, w.V), w.Hkv), -1, dtype=torch.int32, device="cuda")

    def attn(self, stream=None):
        P.pillar_attn_unified(self.shape, self.q, self.k_pool, self.v_pool, self.slot_table, self.req_mode,
                              self.req_len, self.sparse_idx, self.sparse_cnt, self.out, self.logits, self.lse,
                              self.ws, stream=stream)

    def plan(self, stream=None):
        P.pillar_attn_plan(self.shape, self.req_mode, self.req_len, self.sparse_cnt, self.ws, stream=stream)

    def run(self, stream=None):
        P.pillar_attn_run(self.shape, self.q, self.k_pool, self.v_pool, self.slot_table, self.sparse_idx, self.out,
                          self.logits, self.lse, self.ws, stream=stream)

    def topk(self, stream=None):
        P.pillar_topk_select(self.shape, self.V, self.logits, self.lse, self.req_len, self.group_map, self.K,
                             self.next_idx, self.next_cnt, self.tws, stream=stream)

    def attn_flags(self):
        return P.pillar_get_error(self.ws)

    def topk_flags(self):
        return P.pillar_get_error(self.tws)

    def host(self, logits_f64=True):
        """Outputs on the host: out widened to fp64 from its bf16 bits; logits as fp64 (or kept fp32,
        for the largest dumps), LSE as fp64; the next lists as int32."""
        from . import bf16_bits_to_f32
        torch.cuda.synchronize()
        out = bf16_bits_to_f32(self.out.cpu().numpy().view(np.uint16)).astype(np.float64)
        lg = self.logits.cpu().numpy()
        return dict(out=out, logits=lg.astype(np.float64) if logits_f64 else lg,
                    lse=self.lse.cpu().numpy().astype(np.float64),
                    next_idx=self.next_idx.cpu().numpy(), next_cnt=self.next_cnt.cpu().numpy())
