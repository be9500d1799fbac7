"""Seeded synthetic inputs for the PillarAttn unified step.

This module holds the input recipes only -- shapes, length mixes, value
distributions, the planted "pillar" structure and the page-size-1 slot
permutation -- and none of the method's arithmetic.  Both the GPU path and
the fp64 oracle take their inputs from here.

Recipe (shared by every workload, stated once):
  * Q, K, V ~ N(0, 1) drawn in fp32 and rounded to bf16 (round to nearest,
    ties to even).
  * Pillars: each KV head h gets a seeded unit vector u_h.  In every request
    a seeded subset of positions (the workload's pillar fraction) gets
    key = 2*u_h + N(0, 1); every query row of the heads in group h is
    3*u_h + N(0, 1).  These columns are what verify attention concentrates
    on ("SparseSpec-MLSys26", 核心方法 / PillarAttn; the blog post's
    section 4.1 names the column shape "pillars").
  * Request i has phase i mod (k+1); phase 0 is a verify request with k+1
    query rows, phase p >= 1 a draft request with one query row (the unified
    batch of "SparseSpec-MLSys26", Unified batch scheduler section, with k+1
    phase buckets filled round robin).
  * A draft request in phase p of length L holds, per KV head, a critical
    list of ceil(s*(L-p)) positions from [0, L-p) -- the planted pillar
    positions of that head, trimmed or padded with random positions to
    size -- plus the p positions [L-p, L) appended since the last verify.
    Lists are ascending.  This stands in for "Top-K of a prior verify": the
    same size and structure, without computing anything of the method.
  * The slot table is the first sum(L) entries of a seeded random
    permutation of the pool, pool = max(stated, 2**ceil(log2(1.25*sum(L)))).
  * Top-K budget of verify request v: K_v = ceil(s * L_v) in integers.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 0x5EED0000


def f32_to_bf16_bits(x: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    if out is None:
        return r.astype(np.uint16)
    out[...] = r.reshape(out.shape)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Recipe:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    k: int
    s_num: int
    s_den: int
    lengths: tuple            # ("fixed", [..]) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    pillar_frac: tuple        # ("fixed", f) | ("uniform", lo, hi)  -- per KV head
    pool_min: int = 0
    mode_rule: str = "phase"  # "phase" | "all_draft" | "all_verify" | "explicit"
    explicit_modes: tuple = ()
    explicit_phases: tuple = ()
    seed: int = 0


def _recipes():
    r = {}
    r["tiny"] = Recipe("tiny", 4, 4, 1, 64, 4, 1, 10, ("fixed", [256, 320, 448, 512]), ("fixed", 0.03),
                       pool_min=2048, mode_rule="explicit", explicit_modes=(0, 0, 1, 1),
                       explicit_phases=(1, 2, 0, 0), seed=SEED_BASE + 0)
    r["qwen3_1p7b"] = Recipe("qwen3_1p7b", 64, 16, 8, 128, 8, 1, 20, ("uniform", 2048, 8192), ("fixed", 0.03),
                             pool_min=1 << 20, seed=SEED_BASE + 1)
    r["qwen3_8b"] = Recipe("qwen3_8b", 128, 32, 8, 128, 8, 1, 20, ("uniform", 6144, 10240), ("fixed", 0.05),
                           seed=SEED_BASE + 2)
    r["qwen3_14b"] = Recipe("qwen3_14b", 128, 40, 8, 128, 8, 1, 20, ("lognormal", 13500, 0.5, 4096, 24576),
                            ("fixed", 0.05), seed=SEED_BASE + 3)
    r["stress"] = Recipe("stress", 256, 32, 8, 128, 12, 1, 20, ("lognormal", 5793, 0.69, 1024, 32768),
                         ("uniform", 0.02, 0.08), seed=SEED_BASE + 4)
    r["stress_all_draft"] = Recipe("stress_all_draft", 256, 32, 8, 128, 12, 1, 20,
                                   ("lognormal", 5793, 0.69, 1024, 32768), ("uniform", 0.02, 0.08),
                                   mode_rule="all_draft", seed=SEED_BASE + 4)
    r["stress_all_verify"] = Recipe("stress_all_verify", 256, 32, 8, 128, 12, 1, 20,
                                    ("lognormal", 5793, 0.69, 1024, 32768), ("uniform", 0.02, 0.08),
                                    mode_rule="all_verify", seed=SEED_BASE + 4)
    return r


RECIPES = _recipes()


def scaled(name: str, B: int | None = None, length_scale: float = 1.0, seed_offset: int = 0,
           **over) -> Recipe:
    """A smaller variant of a recipe (fewer requests and/or shorter contexts)."""
    base = RECIPES[name]
    d = dict(base.__dict__)
    if B is not None:
        d["B"] = B
    ln = base.lengths
    if length_scale != 1.0:
        if ln[0] == "fixed":
            ln = ("fixed", [max(1, int(x * length_scale)) for x in ln[1]])
        elif ln[0] == "uniform":
            ln = ("uniform", max(1, int(ln[1] * length_scale)), max(1, int(ln[2] * length_scale)))
        else:
            ln = ("lognormal", ln[1] * length_scale, ln[2], max(1, int(ln[3] * length_scale)),
                  max(1, int(ln[4] * length_scale)))
    d["lengths"] = ln
    d["seed"] = base.seed + seed_offset
    d["name"] = f"{base.name}_scaled"
    d.update(over)
    return Recipe(**d)


@dataclass
class Workload:
    recipe: Recipe
    req_mode: np.ndarray          # [B] int32, 0 draft / 1 verify
    req_len: np.ndarray           # [B] int32
    phase: np.ndarray             # [B] int32
    num_slots: int
    slot_table: np.ndarray        # [sum L] int32
    q: np.ndarray                 # [T_q, Hq, D] uint16 (bf16 bits)
    k_logical: np.ndarray         # [sum L, Hkv, D] uint16: K of request b's position t at kv_off[b]+t
    v_logical: np.ndarray         # [sum L, Hkv, D] uint16
    sparse_idx: np.ndarray        # [B, Hkv, max_sparse] int32
    sparse_cnt: np.ndarray        # [B, Hkv] int32
    topk_K: np.ndarray            # [V] int32
    pillar: np.ndarray            # [sum L, Hkv] bool: planted pillar positions
    extra: dict = field(default_factory=dict)

    # convenience -----------------------------------------------------------
    @property
    def B(self): return self.recipe.B

    @property
    def Hq(self): return self.recipe.Hq

    @property
    def Hkv(self): return self.recipe.Hkv

    @property
    def D(self): return self.recipe.D

    @property
    def k(self): return self.recipe.k

    @property
    def G(self): return self.recipe.Hq // self.recipe.Hkv

    @property
    def V(self): return int((self.req_mode == 1).sum())

    @property
    def kv_off(self):
        return np.concatenate([[0], np.cumsum(self.req_len.astype(np.int64))[:-1]]).astype(np.int64)

    @property
    def q_off(self):
        n = np.where(self.req_mode == 1, self.k + 1, 1).astype(np.int64)
        return np.concatenate([[0], np.cumsum(n)[:-1]]).astype(np.int64)

    @property
    def max_sparse(self): return int(self.sparse_idx.shape[2])

    @property
    def verify_len(self): return self.req_len[self.req_mode == 1].astype(np.int32)

    @property
    def verify_batch_index(self): return np.nonzero(self.req_mode == 1)[0].astype(np.int32)

    def pool(self, which: str) -> np.ndarray:
        """The page-size-1 pool [num_slots, Hkv, D]: logical rows placed at their slots,
        unreferenced slots zero."""
        src = self.k_logical if which == "k" else self.v_logical
        p = np.zeros((self.num_slots, self.Hkv, self.D), np.uint16)
        p[self.slot_table] = src
        return p


def _draw_lengths(rec: Recipe, rng: np.random.Generator) -> np.ndarray:
    ln = rec.lengths
    if ln[0] == "fixed":
        L = np.array(ln[1], np.int64)
        assert len(L) == rec.B
    elif ln[0] == "uniform":
        L = rng.integers(ln[1], ln[2] + 1, size=rec.B)
    else:
        _, med, sig, lo, hi = ln
        L = np.clip(np.rint(np.exp(rng.normal(math.log(med), sig, size=rec.B))), lo, hi)
    return L.astype(np.int32)


def _modes(rec: Recipe):
    i = np.arange(rec.B)
    if rec.mode_rule == "explicit":
        return np.array(rec.explicit_modes, np.int32), np.array(rec.explicit_phases, np.int32)
    if rec.mode_rule == "all_draft":
        ph = (i % rec.k) + 1
    elif rec.mode_rule == "all_verify":
        ph = np.zeros(rec.B, np.int64)
    else:
        ph = i % (rec.k + 1)
    return (ph == 0).astype(np.int32), ph.astype(np.int32)


def _threads():
    return max(1, min(16, os.cpu_count() or 1))


def generate(rec: Recipe | str, max_sparse_pad: int = 16) -> Workload:
    """Build one seeded workload.  Deterministic in the recipe's seed."""
    if isinstance(rec, str):
        rec = RECIPES[rec]
    ss = np.random.SeedSequence(rec.seed)
    s_meta, s_q, s_k, s_v, s_list = ss.spawn(5)
    rng = np.random.default_rng(s_meta)
    B, Hq, Hkv, D, k = rec.B, rec.Hq, rec.Hkv, rec.D, rec.k
    G = Hq // Hkv
    L = _draw_lengths(rec, rng)
    mode, phase = _modes(rec)
    L = np.where(mode == 1, np.maximum(L, k + 1), L).astype(np.int32)
    total = int(L.astype(np.int64).sum())
    pool = max(rec.pool_min, 1 << int(math.ceil(math.log2(max(2, 1.25 * total)))))
    slot_table = rng.permutation(pool)[:total].astype(np.int32)

    # pillar directions and per-head pillar fraction
    u = rng.standard_normal((Hkv, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    u = u.astype(np.float32)
    pf = rec.pillar_frac
    frac = np.full(Hkv, pf[1]) if pf[0] == "fixed" else rng.uniform(pf[1], pf[2], size=Hkv)

    kv_off = np.concatenate([[0], np.cumsum(L.astype(np.int64))[:-1]])
    pillar = np.zeros((total, Hkv), bool)
    for b in range(B):
        for h in range(Hkv):
            n = int(round(frac[h] * L[b]))
            if n:
                pos = rng.choice(L[b], size=n, replace=False)
                pillar[kv_off[b] + pos, h] = True

    # K and V, generated request by request in parallel (independent streams)
    k_log = np.empty((total, Hkv, D), np.uint16)
    v_log = np.empty((total, Hkv, D), np.uint16)
    k_seeds = s_k.spawn(B)
    v_seeds = s_v.spawn(B)

    def fill(b):
        lo, n = int(kv_off[b]), int(L[b])
        g = np.random.default_rng(k_seeds[b])
        x = g.standard_normal((n, Hkv, D), dtype=np.float32)
        pm = pillar[lo:lo + n]
        for h in range(Hkv):
            x[pm[:, h], h, :] += 2.0 * u[h]
        f32_to_bf16_bits(x, out=k_log[lo:lo + n])
        g = np.random.default_rng(v_seeds[b])
        x = g.standard_normal((n, Hkv, D), dtype=np.float32)
        f32_to_bf16_bits(x, out=v_log[lo:lo + n])

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(B)))

    # queries: every row of group h is 3*u_h + N(0,1)
    nq = np.where(mode == 1, k + 1, 1)
    T_q = int(nq.sum())
    gq = np.random.default_rng(s_q)
    xq = gq.standard_normal((T_q, Hq, D), dtype=np.float32)
    xq += 3.0 * np.repeat(u, G, axis=0)[None, :, :]
    q = f32_to_bf16_bits(xq).reshape(T_q, Hq, D)

    # critical lists of draft requests
    lr = np.random.default_rng(s_list)
    lists = {}
    max_n = 1
    for b in range(B):
        if mode[b] != 0:
            continue
        p = int(phase[b])
        p = min(p, int(L[b]))
        prefix = int(L[b]) - p
        kb = -(-prefix * rec.s_num // rec.s_den) if prefix > 0 else 0
        kb = min(kb, prefix)
        for h in range(Hkv):
            pil = np.nonzero(pillar[kv_off[b]:kv_off[b] + prefix, h])[0]
            if len(pil) >= kb:
                crit = lr.choice(pil, size=kb, replace=False) if kb else pil[:0]
            else:
                rest = np.setdiff1d(np.arange(prefix), pil, assume_unique=True)
                crit = np.concatenate([pil, lr.choice(rest, size=kb - len(pil), replace=False)])
            lst = np.sort(np.concatenate([crit, np.arange(prefix, int(L[b]))])).astype(np.int32)
            lists[(b, h)] = lst
            max_n = max(max_n, len(lst))
    max_sparse = -(-max_n // max_sparse_pad) * max_sparse_pad
    sparse_idx = np.zeros((B, Hkv, max_sparse), np.int32)
    sparse_cnt = np.zeros((B, Hkv), np.int32)
    for (b, h), lst in lists.items():
        sparse_idx[b, h, :len(lst)] = lst
        sparse_cnt[b, h] = len(lst)

    Lv = L[mode == 1].astype(np.int64)
    topk_K = np.clip(-(-Lv * rec.s_num // rec.s_den), 1, Lv).astype(np.int32)
    return Workload(rec, mode.astype(np.int32), L, phase, pool, slot_table, q, k_log, v_log,
                    sparse_idx, sparse_cnt, topk_K, pillar, extra={"u": u, "pillar_frac": frac})


def query_rows(w: Workload, n: int, seed: int) -> np.ndarray:
    """n extra query tokens [n, Hq, D] (bf16 bits) drawn like the workload's own
    queries (3*u_h + N(0,1) for the heads of group h)."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, w.Hq, w.D), dtype=np.float32)
    x += 3.0 * np.repeat(w.extra["u"], w.G, axis=0)[None, :, :]
    return f32_to_bf16_bits(x).reshape(n, w.Hq, w.D)


def algorithmic_bytes(w: Workload) -> dict:
    """Bytes the step must move: verify reads every K/V row of its context,
    draft reads only the listed rows; plus logits/LSE writes, Q/O, indices and
    slots.  (Counts only; no arithmetic of the method.)"""
    D, Hkv, Hq, k = w.D, w.Hkv, w.Hq, w.k
    ver = w.req_mode == 1
    row = D * 2
    kv_verify = int(w.req_len[ver].astype(np.int64).sum()) * Hkv * row * 2
    kv_draft = int(w.sparse_cnt[~ver].astype(np.int64).sum()) * row * 2
    logits = int(w.req_len[ver].astype(np.int64).sum()) * Hq * (k + 1) * 4
    lse = int(ver.sum()) * Hq * (k + 1) * 4
    qo = int(w.q.shape[0]) * Hq * D * 2 * 2
    idx = int(w.sparse_cnt[~ver].astype(np.int64).sum()) * 4 * 2 + int(w.req_len[ver].astype(np.int64).sum()) * 4
    Kv = w.topk_K.astype(np.int64)
    # Top-K reads the averaged rows (k of the k+1) of every head: k*Hq fp32 per position
    topk_read = int(w.req_len[ver].astype(np.int64).sum()) * Hq * k * 4
    topk_write = int(Kv.sum()) * Hkv * 4
    return dict(kv_verify=kv_verify, kv_draft=kv_draft, kv=kv_verify + kv_draft, logits=logits, lse=lse,
                qo=qo, idx=idx, attn_total=kv_verify + kv_draft + logits + lse + qo + idx,
                topk_read=topk_read, topk_write=topk_write, step_total=kv_verify + kv_draft + logits + lse + qo
                + idx + topk_read + topk_write)
