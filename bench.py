"""Benchmark of the PillarAttn unified step on GB300.

One step = pillar_attn_unified (planner + persistent unified draft/verify
kernel, with the logits/LSE dump) + pillar_topk_select (score
rematerialisation, averaging, Top-K) over one batch of the Qwen3-8B-shaped
workload: 128 requests (1/9 verify with 9 query rows, 8/9 draft), 32 query
heads, 8 KV heads, head_dim 128, bf16, contexts uniform in [6144, 10240],
k = 8, s = 0.05, a randomly permuted page-size-1 KV pool.  Inputs are seeded
synthetic data of that shape (see workloads/).

Prints one JSON line (rank 0).  value = microseconds per layer-step (lower
is better); under torchrun every rank runs its own replica of the workload
(weak scaling) and value = max-over-ranks time / layer-steps of all ranks.
Consecutive steps rotate over --layers (default 4) copies of the KV pools and
logit/LSE buffers, as consecutive layers of a model would.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "PillarAttn unified step: µs/layer-step, KV-read GB/s and % of HBM peak"
UNIT = "us/layer-step"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["pillar_attn.cu", "pillar_plan.cu", "pillar_device.cuh", "pillar_internal.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="qwen3_8b")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--length-scale", type=float, default=1.0, help="shorter contexts (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="fewer requests (profiling runs)")
    ap.add_argument("--quick", action="store_true",
                    help="headline loop only: no CPU baseline, no breakdown, no end-to-end pass")
    ap.add_argument("--layers", type=int, default=4,
                    help="KV pools (with their logit and LSE buffers) rotated over the timed steps")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text):
    """C/CUDA source without comments and blank space: edits to comments do not
    change the kernels a profile was taken on."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_self_speculative_pillar_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """dram bytes per launch of the unified kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"unified_attn_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_sha") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the samples go to a scratch file; PILLAR_CLOCKS_CSV names a place to keep them instead
        self.path = os.environ.get("PILLAR_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"pillar_clocks_{os.getpid()}_{index}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- oracle timing (CPU)

def _kv_bytes(w, mask):
    row = w.D * 2 * 2
    vm = mask & (w.req_mode == 1)
    dm = mask & (w.req_mode == 0)
    return (int(w.req_len[vm].astype(np.int64).sum()) * w.Hkv * row +
            int(w.sparse_cnt[dm].astype(np.int64).sum()) * row)


def oracle_step(w, sel, nthreads):
    """The fp64 oracle over the selected requests of one step: attention, then
    Top-K of the selected verify requests.  Returns seconds."""
    import oracle
    t0 = time.perf_counter()
    r = oracle.attn_unified(Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, scale=1 / math.sqrt(w.D), q=w.q, k_pool=w.k_logical,
                            v_pool=w.v_logical, slot_table=np.arange(len(w.slot_table), dtype=np.int32),
                            req_mode=w.req_mode, req_len=w.req_len, sparse_idx=w.sparse_idx,
                            sparse_cnt=w.sparse_cnt, select=sel, nthreads=nthreads)
    vsel = [v for v, b in enumerate(w.verify_batch_index) if sel[b]]
    if vsel:
        oracle.topk_select(Hq=w.Hq, Hkv=w.Hkv, k=w.k, row_lo=1, row_hi=w.k + 1, logits=r.logits,
                           lse=oracle.verify_lse_of(r, w.req_mode, w.k, w.Hq, select=sel),
                           L=w.verify_len[vsel], K=w.topk_K[vsel], max_topk=int(w.topk_K[vsel].max()),
                           nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_baseline(w, nthreads, min_s=10.0, max_s=30.0):
    """Whole oracle steps of the workload, repeated until about min_s seconds."""
    sel = np.ones(w.B, bool)
    times = []
    t_start = time.perf_counter()
    while True:
        times.append(oracle_step(w, sel, nthreads))
        el = time.perf_counter() - t_start
        if el >= min_s or el + times[-1] > max_s:
            break
    us = statistics.mean(times) * 1e6
    desc = (f"fp64 oracle, the whole {w.recipe.name} layer-step (attention of all {w.B} requests + Top-K of all "
            f"{w.V} verify requests) repeated {len(times)} times, {sum(times):.1f} s of CPU work")
    return us, desc


# --------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = W.generate(args.workload)
    nthreads = os.cpu_count() or 1
    full = np.ones(w.B, bool)
    total = _kv_bytes(w, full)
    t_full = oracle_step(w, full, nthreads)           # calibration, untimed
    n_all = max(1, args.warmup + args.steps)
    frac = min(1.0, (150.0 / n_all) / max(t_full, 1e-6))
    order = np.argsort(-w.req_mode, kind="stable")     # verify requests first, then drafts, in rotation
    n_req = max(1, int(round(frac * w.B)))
    per_step, samp_bytes = [], []
    pos = 0
    for i in range(n_all):
        sel = np.zeros(w.B, bool)
        sel[order[(pos + np.arange(n_req)) % w.B]] = True
        pos = (pos + n_req) % w.B
        dt = oracle_step(w, sel, nthreads)
        if i >= args.warmup:
            per_step.append(dt)
            samp_bytes.append(_kv_bytes(w, sel))
    value = sum(per_step) / max(1, sum(samp_bytes)) * total * 1e6 if per_step else None
    desc = (f"fp64 oracle; each step computed {n_req} of the {w.B} requests of the {w.recipe.name} batch in "
            f"rotation (with the Top-K of the verify requests among them); time scaled to the full layer-step "
            f"by algorithmic KV bytes ({sum(samp_bytes) / 1e6:.0f} MB sampled over {len(per_step)} steps)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3 if value else None,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.recipe.name, "global_batch": int(w.B), "seq_len": int(w.req_len.mean()),
                   "parallelism": "single"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- replicas (N > 1)
# The path shards by request and KV head with no exchange step, so N GPUs run
# N replicas: each rank times its own seeded replica, the ranks meet only at
# the timing barriers, and the whole-job value divides the slowest rank's time
# by the layer-steps of all ranks.

def replica_recipe(args, rank):
    """The workload recipe of one rank: the named one on rank 0 (unless scaled
    for a profiling run), a distinct seed of the same shape elsewhere."""
    if rank or args.length_scale != 1.0 or args.batch:
        return W.scaled(args.workload, B=args.batch, length_scale=args.length_scale, seed_offset=1000 * rank)
    return W.RECIPES[args.workload]


def max_over_ranks(x, world, device):
    """The maximum of a per-rank float over the process group (x itself when alone)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us(max_elapsed_ms, steps, world):
    """Microseconds per layer-step of the whole job: every rank ran `steps`
    layer-steps of its replica in at most max_elapsed_ms."""
    return max_elapsed_ms * 1e3 / (steps * world)


# --------------------------------------------------------------------------- GPU arm

def fusion_ablation(g, P, stream, n):
    """The attention call under the unified schedule and under the schedules
    it replaces ("SparseSpec-MLSys26", Unified batch scheduler + fused
    attention kernel: a sequential pair of launches, and a naive joint batch;
    uniform_rows is the joint batch with only the per-mode row layout taken
    away), each timed over n calls on the launching stream.  Every schedule
    computes the same outputs; `*_same_out` says whether the out tensor came
    back bit for bit equal to the unified pass's (the naive joint batch splits
    long contexts differently, so its rows agree within rounding only)."""
    import torch
    plans = (("unified", (P.SCHEDULE_UNIFIED,)),
             ("sequential", (P.SCHEDULE_DRAFT_ONLY, P.SCHEDULE_VERIFY_ONLY)),
             ("uniform_rows", (P.SCHEDULE_UNIFORM_ROWS,)),
             ("naive_joint", (P.SCHEDULE_NAIVE_JOINT,)))

    def run(scheds):
        for sch in scheds:
            g.shape.schedule = sch
            g.attn(stream)
        g.shape.schedule = P.SCHEDULE_UNIFIED

    run(plans[0][1])
    torch.cuda.synchronize()
    ref = g.out.clone()
    res = {"calls": n}
    for name, scheds in plans:
        for _ in range(3):
            run(scheds)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            run(scheds)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name + "_attn_us"] = e0.elapsed_time(e1) * 1e3 / n
        res[name + "_same_out"] = bool(torch.equal(g.out, ref))
        res[name + "_flags"] = g.attn_flags()
    run(plans[0][1])
    torch.cuda.synchronize()
    for name, _ in plans[1:]:
        res[name + "_vs_unified"] = res[name + "_attn_us"] / res["unified_attn_us"]
    return res


def kv_append_timing(g, w, P, stream, n):
    """pillar_kv_append for the new tokens of one step of the workload's mix (k+1
    per verify request, 1 per draft request), timed over n calls.  The rows
    written are the pool's own rows at those slots, so the pool is unchanged."""
    import torch
    from workloads.device import to_device
    kvo = w.kv_off
    idx = []
    for b in range(w.B):
        n_new = w.k + 1 if w.req_mode[b] == 1 else 1
        L = int(w.req_len[b])
        idx.extend(int(kvo[b]) + t for t in range(L - n_new, L))
    idx = np.asarray(idx, np.int64)
    k_new, v_new = to_device(w.k_logical[idx]), to_device(w.v_logical[idx])
    slots = to_device(w.slot_table[idx].astype(np.int32))
    dflag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        P.pillar_kv_append(g.shape, k_new, v_new, slots, g.k_pool, g.v_pool, dflag, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        P.pillar_kv_append(g.shape, k_new, v_new, slots, g.k_pool, g.v_pool, dflag, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    moved = 2 * len(idx) * w.Hkv * w.D * 2 * 2  # K and V rows read and written
    return {"tokens": int(len(idx)), "us": us, "gbs": moved / (us * 1e-6) / 1e9, "bytes_moved": moved,
            "calls": n, "flags": int(dflag.item())}


def kv_offload_timing(g, w, P, stream, n, n_req=4):
    """The dynamic KV manager's copies ("SparseSpec-MLSys26", 动态 KV 管理):
    the whole KV of the first n_req requests packed into page-locked host
    memory by pillar_kv_offload and put back into the same slots by
    pillar_kv_reload (so the pool is unchanged), each timed over n calls; the
    host side is written and read by the kernels themselves (NVLink-C2C on a
    Grace-Blackwell node)."""
    import torch
    from workloads.device import to_device
    kvo = w.kv_off
    idx = np.concatenate([np.arange(int(kvo[b]), int(kvo[b]) + int(w.req_len[b])) for b in range(min(n_req, w.B))])
    slots = to_device(w.slot_table[idx].astype(np.int32))
    hk = torch.empty((len(idx), w.Hkv, w.D), dtype=torch.int16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    dflag = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {"tokens": int(len(idx)), "bytes_each_way": int(len(idx) * w.Hkv * w.D * 2 * 2), "calls": n}
    for name, call in (("offload", lambda: P.pillar_kv_offload(g.shape, g.k_pool, g.v_pool, slots, hk, hv, dflag,
                                                                stream=stream)),
                       ("reload", lambda: P.pillar_kv_reload(g.shape, hk, hv, slots, g.k_pool, g.v_pool, dflag,
                                                              stream=stream))):
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n
        res[name + "_us"] = us
        res[name + "_gbs"] = res["bytes_each_way"] / (us * 1e-6) / 1e9
    res["flags"] = int(dflag.item())
    return res


def draft_slots_timing(g, w, P, stream, n):
    """The draft lists with their pool slots already translated (as
    pillar_draft_lists writes them after a verify step's Top-K): the attention
    call through pillar_attn_unified_slotted against pillar_attn_unified on the
    same lists, n calls each, out compared bit for bit; and pillar_draft_lists
    itself on this step's Top-K (each verify request one token further on)."""
    import torch
    from workloads.device import to_device
    kvo = w.kv_off
    ss = np.zeros_like(w.sparse_idx)
    for b in np.nonzero(w.req_mode == 0)[0]:
        for h in range(w.Hkv):
            c = int(w.sparse_cnt[b, h])
            ss[b, h, :c] = w.slot_table[kvo[b] + w.sparse_idx[b, h, :c]]
    ss_d = to_device(ss.astype(np.int32))

    def call(slotted):
        args = (g.shape, g.q, g.k_pool, g.v_pool, g.slot_table, g.req_mode, g.req_len, g.sparse_idx, g.sparse_cnt)
        if slotted:
            P.pillar_attn_unified_slotted(*args, ss_d, g.out, g.logits, g.lse, g.ws, stream=stream)
        else:
            P.pillar_attn_unified(*args, g.out, g.logits, g.lse, g.ws, stream=stream)

    res = {"calls": n}
    outs = {}
    for name, slotted in (("positions", False), ("slotted", True)):
        for _ in range(3):
            call(slotted)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call(slotted)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name + "_attn_us"] = e0.elapsed_time(e1) * 1e3 / n
        outs[name] = g.out.clone()
    res["same_out"] = bool(torch.equal(outs["positions"], outs["slotted"]))
    res["slotted_vs_positions"] = res["slotted_attn_us"] / res["positions_attn_us"]
    if w.V:
        max_sparse = max(w.max_sparse, g.shape.max_topk + w.k)
        shape = P.make_shape(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, k=w.k, max_sparse=max_sparse,
                             max_len=g.shape.max_len, num_slots=w.num_slots, max_topk=g.shape.max_topk)
        si = torch.zeros((w.B, w.Hkv, max_sparse), dtype=torch.int32, device="cuda")
        sc = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device="cuda")
        sl = torch.zeros_like(si)
        lv = to_device((w.verify_len - 1).astype(np.int32))  # each verify request one token further on
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")

        def lists():
            P.pillar_draft_lists(shape, w.V, g.next_idx, g.next_cnt, g.group_map, lv, g.req_len, g.slot_table,
                                 si, sc, sl, flags, stream=stream)

        for _ in range(3):
            lists()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            lists()
        e1.record(stream)
        torch.cuda.synchronize()
        res["draft_lists_us"] = e0.elapsed_time(e1) * 1e3 / n
        res["draft_lists_flags"] = int(flags.item())
    return res


def run_gpu(args):
    import torch
    import sparse_self_speculative_pillar_gb300 as P
    from workloads.device import Gpu

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    P.load()

    w = W.generate(replica_recipe(args, rank))  # each rank: its own replica of the workload
    g = Gpu(w)
    ab = W.algorithmic_bytes(w)
    stream = torch.cuda.current_stream()
    # Layer rotation: consecutive steps read the KV pools of different layers (copies of the same
    # rows at other addresses) and write other logit/LSE buffers, as a model's layers do, so that
    # no step finds the previous step's pool or dump in L2.
    n_layers = max(1, args.layers)
    layers = [(g.k_pool, g.v_pool, g.logits, g.lse)]
    for _ in range(n_layers - 1):
        layers.append((g.k_pool.clone(), g.v_pool.clone(), torch.empty_like(g.logits), torch.empty_like(g.lse)))
    layer_bytes = sum(t.numel() * t.element_size() for t in layers[0])

    def use_layer(i):
        g.k_pool, g.v_pool, g.logits, g.lse = layers[i % n_layers]

    def step(i):
        use_layer(i)
        g.attn(stream)
        g.topk(stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    flags = g.attn_flags() | g.topk_flags()
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x} during warm-up")

    # headline: K steps bracketed by events on the launching stream
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, "cuda")
    us_per_step = whole_job_us(elapsed_ms, args.steps, world)
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": us_per_step, "unit": UNIT, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "quick": True,
                              "config": {"workload": w.recipe.name, "B": int(w.B)}}), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    # breakdown: the same steps with events around each call (the dominant
    # call's duration, live, on the launching stream)
    nb = max(10, min(args.steps, 1000))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nb)]
    torch.cuda.synchronize()
    for i in range(nb):
        use_layer(i)
        ev[i][0].record(stream)
        g.attn(stream)
        ev[i][1].record(stream)
        g.topk(stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    attn_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    topk_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    # the same steps with the attention call in its two halves (pillar_attn_plan, then
    # pillar_attn_run: the unified kernel and the merge of split units), so that the
    # kernel that reads the K/V rows is timed without the planner in front of it
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb)]
    torch.cuda.synchronize()
    for i in range(nb):
        use_layer(i)
        ev2[i][0].record(stream)
        g.plan(stream)
        ev2[i][1].record(stream)
        g.run(stream)
        ev2[i][2].record(stream)
        g.topk(stream)
        ev2[i][3].record(stream)
    torch.cuda.synchronize()
    plan_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev2)
    run_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev2)
    split_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in ev2)

    # end to end: per-step inputs from pinned host memory, results back to host,
    # as a serving loop runs it -- the next step's inputs are uploaded while
    # the current step computes.  Two device sets of the per-step inputs and
    # outputs alternate; a copy stream carries the transfers, the launching
    # stream the two calls.  Every step's uploads and its result download are
    # inside the timed region (from the first upload to the last download).
    e2e_steps = args.e2e_steps or max(10, min(args.steps, 500))
    IN = ("q", "slot_table", "req_mode", "req_len", "sparse_idx", "sparse_cnt", "group_map", "K")
    OUT = ("out", "next_idx", "next_cnt")
    # Each direction is one packed buffer (every tensor at a 256-byte aligned offset): one copy per
    # direction and step instead of one per tensor, whose per-copy cost would dominate small steps.

    def packed(names, device):
        offs, n = {}, 0
        for nm in names:
            t = getattr(g, nm)
            offs[nm] = n
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device, pin_memory=(device == "cpu"))
        views = {nm: buf[offs[nm]:offs[nm] + getattr(g, nm).numel() * getattr(g, nm).element_size()]
                 .view(getattr(g, nm).dtype).view(getattr(g, nm).shape) for nm in names}
        return buf, views

    h_in_buf, h_in = packed(IN, "cpu")
    for n in IN:
        h_in[n].copy_(getattr(g, n).cpu())
    h_out = [packed(OUT, "cpu") for _ in range(2)]
    d_in = [packed(IN, "cuda") for _ in range(2)]
    d_out = [packed(OUT, "cuda") for _ in range(2)]
    # the output sets start as copies of the device-resident run's outputs: entries a step leaves
    # untouched (lists past their count, all of them when there is no verify request) then agree
    for _, o in d_out:
        for n in OUT:
            o[n].copy_(getattr(g, n))
    h2d = h_in_buf.numel()
    d2h = h_out[0][0].numel()
    copy = torch.cuda.Stream()
    ev_in, ev_out = [torch.cuda.Event() for _ in range(2)], [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        with torch.cuda.stream(copy):
            d_in[b][0].copy_(h_in_buf, non_blocking=True)
        ev_in[b].record(copy)

    def compute(b, s_i=0):
        use_layer(s_i)
        i, o = d_in[b][1], d_out[b][1]
        P.pillar_attn_unified(g.shape, i["q"], g.k_pool, g.v_pool, i["slot_table"], i["req_mode"], i["req_len"],
                              i["sparse_idx"], i["sparse_cnt"], o["out"], g.logits, g.lse, g.ws, stream=stream)
        P.pillar_topk_select(g.shape, g.V, g.logits, g.lse, i["req_len"], i["group_map"], i["K"], o["next_idx"],
                             o["next_cnt"], g.tws, stream=stream)
        ev_out[b].record(stream)

    def download(b):
        copy.wait_event(ev_out[b])
        with torch.cuda.stream(copy):
            h_out[b][0].copy_(d_out[b][0], non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0.record(copy)
    upload(0)
    for s_i in range(e2e_steps):
        b = s_i & 1
        stream.wait_event(ev_in[b])  # this step's inputs have landed (and its output set was read back)
        compute(b, s_i)
        if s_i + 1 < e2e_steps:
            if s_i >= 1:
                copy.wait_event(ev_out[1 - b])  # the step before has finished reading the other input set
            upload(1 - b)
        download(b)
    e1.record(copy)
    torch.cuda.synchronize()
    # the same steps with every transfer serialised on the launching stream
    # (no overlap), reported beside the pipelined number
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for s_i in range(e2e_steps):
        d_in[0][0].copy_(h_in_buf, non_blocking=True)
        compute(0, s_i)
        h_out[0][0].copy_(d_out[0][0], non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    serial_us = whole_job_us(max_over_ranks(e2.elapsed_time(e3), world, "cuda"), e2e_steps, world)
    use_layer(0)
    last = h_out[(e2e_steps - 1) & 1][1]
    if not (torch.equal(last["next_cnt"], g.next_cnt.cpu()) and torch.equal(last["out"], g.out.cpu())):
        raise RuntimeError("end-to-end results differ from the device-resident run")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    e2e_us = whole_job_us(e2e_ms, e2e_steps, world)
    flags = g.attn_flags() | g.topk_flags()
    ablation = fusion_ablation(g, P, stream, max(10, min(args.steps, 500)))
    append = kv_append_timing(g, w, P, stream, max(10, min(args.steps, 500)))
    offload = kv_offload_timing(g, w, P, stream, max(10, min(args.steps, 100)))
    slots = draft_slots_timing(g, w, P, stream, max(10, min(args.steps, 500)))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_kind = measured_peak()
    attn_s, run_s = attn_ms / 1e3, run_ms / 1e3
    achieved = ab["attn_total"] / run_s / 1e9  # the unified kernel and its merge (the planner is another kernel)
    kv_gbs = ab["kv"] / run_s / 1e9
    call_kv_gbs = ab["kv"] / attn_s / 1e9
    step_gbs = ab["step_total"] / (us_per_step * world / 1e6) / 1e9 if world == 1 else None
    traffic = profiled_traffic(w.recipe.name)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        est_us, desc = oracle_baseline(w, os.cpu_count() or 1)
        cpu = {"value": est_us, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": us_per_step, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_per_step / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.recipe.name, "global_batch": int(w.B) * world, "seq_len": int(w.req_len.mean()),
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "verify_requests": int(w.V), "draft_requests": int(w.B - w.V),
                   "heads": f"{w.Hq}q/{w.Hkv}kv", "head_dim": int(w.D), "k": int(w.k),
                   "l2": "inputs larger than L2 (KV read per step %.0f MB), %d layers' pools rotated"
                         % (ab["kv"] / 1e6, n_layers)},
        "attn_us": attn_ms * 1e3, "topk_us": topk_ms * 1e3,
        "attn_split_us": {"plan": plan_ms * 1e3, "run": run_ms * 1e3, "step": split_ms * 1e3,
                          "note": "pillar_attn_plan + pillar_attn_run (the unified kernel and the merge) in "
                                  "place of the one pillar_attn_unified call, then the Top-K: the same work"},
        "kv_read_gbs": kv_gbs, "kv_read_frac_of_peak": kv_gbs / peak,
        "kv_read_frac_of_nominal": kv_gbs / NOMINAL_HBM_GBS,
        "kv_read_over": "pillar_attn_run (the unified kernel and the merge of split units)",
        "attn_call_kv_read_gbs": call_kv_gbs, "attn_call_kv_read_frac_of_peak": call_kv_gbs / peak,
        "step_algorithmic_gbs": step_gbs,
        "algorithmic_bytes": ab,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "unified_attn_kernel + merge_kernel (pillar_attn_run), event-timed per call; "
                               "over the whole pillar_attn_unified call (planner included) the fraction is "
                               "%.3f" % (ab["attn_total"] / attn_s / 1e9 / peak),
                     "peak_kind": peak_kind},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "pipeline": "every step uploads its inputs from pinned host memory and downloads its result, one "
                            "packed buffer each way; "
                            "double-buffered device sets, transfers on a copy stream overlapping the previous "
                            "or next step's compute",
                "serial_value": serial_us},
        "fusion_ablation": ablation,
        "kv_append": append,
        "kv_offload": offload,
        "draft_slots": slots,
        "layers": {"pools": n_layers, "bytes_per_layer": layer_bytes,
                   "rotation": "step i reads layer i mod pools: its own K/V pools (the same rows at other "
                               "addresses) and logit/LSE buffers"},
        "gpu_launches": 5 * args.steps,
        "breakdown_steps": nb,
        "clocks": clk,
        "device_flags": flags,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
