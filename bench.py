#!/usr/bin/env python3
"""Benchmark of the lookahead sparse decode hot path on one GB300.

Workload (default): the Qwen3-235B-A22B attention shape - 94 layers, batch 64,
64 q / 4 KV heads (GQA 16), d_h 128, 32,768-token context = 2,048 blocks of
16, K = 128, 4 draft queries, fetch ratio 0.05 -> cap 7 - with heavy blocks
drifting by +-2 blocks per decode step over 8 simulated steps.  A step is one
decode step: for each of the 94 layers (each with its own summaries, slot
pool, tables and outputs in HBM), the compressed-key update of the newest
block, draft-query block scoring, top-K selection with capped eviction,
staging of the admitted blocks from pinned host memory, and sparse decode
attention - every step in liboasis.so's kernels, layer-pipelined on CUDA
streams ordered by events and replayed as one CUDA graph per decode step.
Tables advance from step to step (each step starts from the resident sets
the previous one selected), and the queries of step i are those of drift step
i mod 8, so the cap admits new blocks at every step.

Metric: HBM GB/s = (summaries read + selected K/V read + fp32 outputs written)
per step / step time; also microseconds per layer-step and the fraction of
the measured HBM copy bandwidth reached by the dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own copy of the workload (weak scaling; the
segments are independent, no data-path collective) and rank 0 prints one JSON
line with the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "lookahead select + sparse decode-attn: HBM GB/s, µs/step, % of GB300 roofline"
WORKLOAD_ID = 5


def _args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40, help="decode steps timed (one graph replay each)")
    p.add_argument("--warmup", type=int, default=5, help="decode steps run before timing")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=0,
                   help="layers per decode step, each with its own buffers (default: the workload's layer count; "
                        "36 for the single-layer Qwen3-8B-shaped workload)")
    p.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=[1, 2, 3, 4, 5],
                   help="workload id (5 = the Qwen3-235B-A22B attention shape, the largest that fits one GPU)")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget (CPU baseline)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-kernels", action="store_true", help="skip the per-kernel timings")
    p.add_argument("--other-workloads", default="2,3",
                   help="workload ids also measured (layer-step and kernels, under other_workloads; '' for none)")
    p.add_argument("--bg-streams", type=int, default=3, help="background streams, taken by the layers in turn")
    p.add_argument("--xf-streams", type=int, default=3, help="staging streams, taken by the layers in turn")
    p.add_argument("--fg-priority", type=int, default=0, help="CUDA priority of the foreground stream (lower = higher)")
    p.add_argument("--attn", choices=["cluster", "balanced", "tc"], default="cluster",
                   help="attention: per-head thread-block clusters (mma.sync), SM-balanced with a workspace, or the "
                        "tcgen05 kernel (per-head clusters, both products on the 5th-generation tensor cores)")
    p.add_argument("--scoring", choices=["tc", "exact"], default="tc",
                   help="tc: tensor-core estimates + certified selection; exact: fixed-order fp32 scores of every "
                        "block (both give the same tables and plans)")
    return p.parse_args(argv)


def _layers(args, w):
    if args.layers > 0:
        return args.layers
    return 36 if w.layers == 1 and w.name == "qwen3-8b-layer" else w.layers


def _drift_steps(w):
    """Distinct query sets the decode steps cycle through (the drift steps)."""
    return w.steps if w.drift else 1


def _fp32_peak_tfma():
    """Nominal FP32 FMA rate of the GB300 from its unit counts and maximum SM
    clock (no measured figure exists for it): 152 SMs x 128 lanes x 2.07 GHz."""
    return 152 * 128 * 2.07e9 / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _config(w, R, extra=None):
    c = {"workload": f"{w.name}: {R} layers per decode step, batch {w.B}, {w.Hq} q / {w.Hkv} KV heads, "
                     f"d_h {w.D}, context {w.L} ({w.Nb} blocks of 16), K={w.K}, W={w.W}, {w.Nd} drafts, "
                     f"fetch_ratio {w.fetch_ratio} (cap {w.cap})"
                     + (f", heavy blocks drifting +-{w.drift} blocks per step over {w.steps} steps" if w.drift else "")
                     + ", bf16 KV, fp32 scores/out",
         "layers_per_decode_step": R,
         "bytes_per_layer_step": w.headline_bytes_per_layer(),
         "bytes_per_step": R * w.headline_bytes_per_layer(),
         "segments_per_layer": w.S}
    if extra:
        c.update(extra)
    return c


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        import shutil
        import threading
        self.proc, self.lines = None, []
        cmd = ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if shutil.which("stdbuf"):
            cmd = ["stdbuf", "-oL"] + cmd
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.reader = threading.Thread(target=lambda: self.lines.extend(iter(self.proc.stdout.readline, "")),
                                       daemon=True)
        self.reader.start()
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        out = "".join(self.lines)
        sms, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sms.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# --------------------------------------------------------------------------- CPU (oracle) side

def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_setup(w, segs):
    """Oracle inputs of some segments (untimed): tiles, summaries, prior table,
    and the queries of every drift step."""
    import numpy as np
    import torch

    from oracle.score import score_blocks
    from oracle.select import top_k
    from oracle.summary import block_summary
    from synth import workload as wl

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    T = _drift_steps(w)
    qd = [u16(wl.drafts(w, 0, t)) for t in range(T)]
    qt = [u16(wl.q_true(w, 0, t)) for t in range(T)]
    prep = []
    for seg in segs:
        b, h = divmod(seg, w.Hkv)
        tiles = u16(wl.kv_tiles(w, 0, [seg])[0])
        kmin, kmax, _ = block_summary(tiles[:, 0], w.L)
        tk = top_k(score_blocks(kmin[:w.nc], kmax[:w.nc], qt[0][b, h * w.G:(h + 1) * w.G]), w.K)
        prep.append((seg, tiles, kmin, kmax, wl.prior_from_topk(w, 0, seg, tk).tolist()))
    return qd, qt, prep


def _oracle_sample(w, seconds, setup, start=0):
    """Run the oracle's decode step on the prepared segments, cycling over them
    and over the drift steps, until `seconds` of wall time are spent; returns
    (headline bytes, seconds, segment-steps)."""
    import numpy as np

    from oracle import pipeline as opipe
    from oracle.score import segment_queries

    qd, qt, prep = setup
    scale = float(np.float32(1.0 / math.sqrt(w.D)))
    per_seg = w.headline_bytes_per_layer() // w.S
    done, i = 0, start
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        seg, tiles, kmin, kmax, table = prep[i % len(prep)]
        t = i % len(qd)
        b, h = divmod(seg, w.Hkv)
        opipe.run_segment(tiles, w.L, segment_queries(qd[t], b, h, w.G), qt[t][b, h * w.G:(h + 1) * w.G], table,
                          w.K, w.W, w.cap, scale, kmin=kmin.copy(), kmax=kmax.copy(), update_blocks=[w.Nb - 1])
        done += 1
        i += 1
    return done * per_seg, time.perf_counter() - t0, done


def _oracle_worker(wid, n_workers, workload_id, rounds, budget, barrier, out):
    """One host core's share of the oracle baseline: its own segment, then
    `rounds` rounds of `budget` seconds, in step with the other workers."""
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    try:
        import torch
        torch.set_num_threads(1)
        from synth import workload as wl
        w = wl.WORKLOADS[workload_id]
        seg = (wid * w.S) // n_workers
        setup = _oracle_setup(w, [seg])
        res = []
        barrier.wait(timeout=600)
        for r in range(rounds):
            _, secs, n = _oracle_sample(w, budget, setup, start=r)
            res.append((n, secs))
            barrier.wait(timeout=600)
        out.put((wid, res, None))
    except Exception as e:  # reported by the parent
        out.put((wid, None, repr(e)))


def _oracle_parallel(workload_id, rounds, budget):
    """Run the oracle on every host core (one spawned process per core, one
    segment each); returns (cores, per-round segment-steps, per-round seconds)."""
    import multiprocessing as mp
    n = _cores()
    ctx = mp.get_context("spawn")           # the parent may hold a CUDA context: never fork it
    barrier = ctx.Barrier(n)
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(i, n, workload_id, rounds, budget, barrier, q), daemon=True)
             for i in range(n)]
    for p_ in procs:
        p_.start()
    got = [q.get(timeout=900) for _ in procs]
    for p_ in procs:
        p_.join(timeout=60)
    errs = [e for _, _, e in got if e]
    if errs:
        raise RuntimeError(f"oracle worker failed: {errs[0]}")
    segs = [sum(r[k][0] for _, r, _ in got) for k in range(rounds)]
    secs = [max(r[k][1] for _, r, _ in got) for k in range(rounds)]
    return n, segs, secs


def _cpu_baseline(w, workload_id, seconds):
    per_seg = w.headline_bytes_per_layer() // w.S
    n, segs, secs = _oracle_parallel(workload_id, 1, seconds)
    value = segs[0] * per_seg / secs[0] / 1e9
    return {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle", "cpu_model": _cpu_model(),
            "sample": f"{segs[0]} segment-steps in {secs[0]:.1f} s on {n} host cores ({_cpu_model()}), one "
                      f"process per core, each on its own segment of the workload cycling through the drift "
                      f"steps: newest-block summary update, scoring, capped selection, staging and attention "
                      f"of one (sequence, KV head) per segment-step, numpy oracle; value = headline bytes of "
                      f"the segment-steps / time",
            "us_per_layer_step_equiv": secs[0] / max(1, segs[0]) * w.S * 1e6}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import workload as wl
    w = wl.WORKLOADS[args.workload]
    R = _layers(args, w)
    budget = max(1.0, min(5.0, 90.0 / max(1, args.steps + args.warmup)))
    n, segs, secs = _oracle_parallel(args.workload, args.warmup + args.steps, budget)
    tseg, tsec = sum(segs[args.warmup:]), sum(secs[args.warmup:])
    per_seg = w.headline_bytes_per_layer() // w.S
    value = tseg * per_seg / tsec / 1e9
    ms = tsec / max(1, tseg) * w.S * R * 1e3               # one decode step: R layers x S segments
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "us_per_layer_step": ms * 1e3 / R, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": _config(w, R, {"step": "the oracle on the host cores: each step a bounded sample "
                                             f"({budget:.1f} s) of segment-steps of the decode step, one process "
                                             "per core, one segment each",
                                     "parallelism": f"{n} host cores"}),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle", "cpu_model": _cpu_model(),
                             "sample": f"{tseg} segment-steps over {args.steps} timed steps of {budget:.1f} s on "
                                       f"{n} cores, numpy oracle"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- multi-rank host logic

def max_over_ranks(x, device=None):
    """The largest of the ranks' values of x (x itself without a process group).
    Each rank times its own replica; the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step, ms_per_step, world):
    """Whole-job throughput: every rank moves its own step's bytes in the
    (max-over-ranks) step time."""
    return bytes_per_rank_step * world / (ms_per_step / 1e3) / 1e9


# --------------------------------------------------------------------------- GPU side

def _gpu_prior(w, lay, sl, q):
    """Prior resident tables (about 90 % of the true-query top-K), computed with the kernels."""
    import torch

    import sparse_kv_cache_quest_gb300 as okv
    from synth import workload as wl
    S = w.S
    scores = torch.zeros((S, w.Nb), dtype=torch.float32, device=sl.device)
    okv.oasis_score_blocks(lay.kmin, lay.kmax, w.Nb, q.view(w.B, 1, w.Hq, w.D), w.B, w.Hkv, w.G, 1, w.D, sl, w.W,
                           scores, lay.status)
    empty = torch.full((S, w.slots), -1, dtype=torch.int32, device=sl.device)
    if w.W:
        empty[:, w.K:] = torch.tensor(wl.window_blocks(w), dtype=torch.int32, device=sl.device)
    tout = torch.empty_like(empty)
    plan = torch.empty((S, w.K, 2), dtype=torch.int32, device=sl.device)
    cnt = torch.empty((S,), dtype=torch.int32, device=sl.device)
    okv.oasis_select_topk_capped(scores, w.Nb, sl, w.B, w.Hkv, w.K, w.W, w.K, empty, tout, plan, cnt, lay.status)
    t = tout.cpu()
    rows = [wl.prior_from_topk(w, 0, s, [b for b in t[s, :w.K].tolist() if b >= 0]) for s in range(S)]
    return torch.stack(rows)


class Workbench:
    """The benchmarked state on one GPU: R layers of device buffers filled from
    one synthetic layer, the pinned host tier, and the queries of every drift
    step.  reset() puts every layer back to the prior tables and pools."""

    def __init__(self, w, R, dev, balanced_attn=False, scoring="tc", tc_attn=False):
        import torch

        import sparse_kv_cache_quest_gb300 as okv
        from synth import workload as wl
        self.w, self.R, self.dev = w, R, dev
        tiles = torch.empty((w.S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16, device=dev)
        for s0 in range(0, w.S, 16):
            tiles[s0:s0 + 16] = wl.kv_tiles(w, 0, list(range(s0, min(w.S, s0 + 16))), device=dev)
        self.host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
        self.host.copy_(tiles)
        self.seg_stride = self.host[0].numel() * 2
        self.sl = wl.seq_lens(w).to(dev)
        T = _drift_steps(w)
        self.q = [wl.q_true(w, 0, t).to(dev) for t in range(T)]
        self.qd = [wl.drafts(w, 0, t).to(dev) for t in range(T)]
        shape = okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
        self.strides = (tiles.stride(0), tiles.stride(1), tiles.stride(3))
        self.layers = []
        for _ in range(R):
            lay = okv.DecodeLayer(shape, device=dev, balanced_attn=balanced_attn, scoring=scoring, tc_attn=tc_attn)
            lay.build_summary(tiles, self.sl, 0, w.Nb, strides=self.strides)
            self.layers.append(lay)
        self.table0 = _gpu_prior(w, self.layers[0], self.sl, self.q[0]).to(dev)
        self.pool0 = tiles[torch.arange(w.S, device=dev)[:, None], self.table0.long().clamp(min=0)]
        self.new_keys = tiles[:, w.Nb - 1:w.Nb, 0].contiguous()   # keys of the newest block, [S][1][16][D]
        self.tiles = tiles                                        # kept for the full-build timing
        self.reset()

    def reset(self):
        import torch
        for lay in self.layers:
            lay.table.copy_(self.table0)
            lay.table_next.copy_(self.table0)
            lay.pool.copy_(self.pool0)
            lay.status.zero_()
        torch.cuda.synchronize(self.dev)

    def graphs(self, args, host_io=False):
        """One DecodeStepGraph per drift step, tables advancing.  Each graph is
        launched once here: a graph's first launch (which uploads it to the
        device) is slower than its replays, and no timed region should hold one.
        Those launches are decode steps too (one drift period, so the drift order
        of later steps is unchanged); callers that time from the starting state
        reset it afterwards."""
        import torch

        import sparse_kv_cache_quest_gb300 as okv
        w = self.w
        gs = [okv.DecodeStepGraph(self.layers, self.q[t], self.qd[t], self.sl, self.host, self.seg_stride, w.Nb,
                                  new_keys=self.new_keys, new_block=w.Nb - 1, n_bg=args.bg_streams,
                                  fg_priority=args.fg_priority, n_xf=args.xf_streams, advance=True,
                                  host_io=host_io, share_host_inputs=host_io, warmup=(t == 0))
              for t in range(len(self.q))]
        for g in gs:
            g.replay()
        torch.cuda.synchronize(self.dev)
        return gs

    def status(self):
        import torch
        return int(torch.stack([lay.status for lay in self.layers]).max().item())


def _time_steps(graphs, first, n, dev):
    """Replay decode steps first .. first + n - 1 (graph of drift step i mod T)
    between two events on the replay stream; returns ms in total."""
    import torch
    st = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(first, first + n):
        graphs[i % len(graphs)].replay()
    e1.record(st)
    e1.synchronize()
    return e0.elapsed_time(e1)


def _kernel_times(wb, dev, n_rep=20):
    """Per-kernel durations: a CUDA graph of back-to-back launches of one kernel
    over the layers' buffer sets, replayed between events on the replay stream
    (us per launch)."""
    import torch
    w = wb.w
    q, qd, sl = wb.q[0], wb.qd[0], wb.sl
    import sparse_kv_cache_quest_gb300 as okv
    sh = wb.layers[0].shape

    def exact_score(lay, st_):
        okv.oasis_score_blocks(lay.kmin, lay.kmax, sh.Nb_max, qd, sh.B, sh.Hkv, sh.G, sh.Nd, sh.D, sl, sh.W,
                               lay.scores, lay.status, st_)

    calls = {"score": lambda lay, st_: lay.score(qd, sl, stream=st_),
             "attn": lambda lay, st_: lay.attend(q, sl, stream=st_),
             "select": lambda lay, st_: lay.select(sl, stream=st_, qdraft=qd),
             "stage": lambda lay, st_: lay.stage(wb.host, wb.seg_stride, w.Nb, stream=st_),
             "summary_update": lambda lay, st_: lay.build_summary(wb.new_keys, sl, blk_begin=w.Nb - 1, blk_count=1,
                                                                  stream=st_),
             # the full build at sparsification time (not part of a decode step): every block's keys
             "summary_full_build": lambda lay, st_: lay.build_summary(wb.tiles, sl, 0, w.Nb, strides=wb.strides,
                                                                      stream=st_)}
    if wb.layers[0].scoring == "tc":
        calls["score_exact"] = exact_score      # the fixed-order kernel alone, for comparison
    kern = {}
    n_launch = max(8, wb.R)
    for name, fn in calls.items():
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        kg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kg, stream=side):
            for i in range(n_launch):
                fn(wb.layers[i % wb.R], side)
        kg.replay()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(n_rep):
            kg.replay()
        e1.record(st)
        e1.synchronize()
        kern[name] = e0.elapsed_time(e1) / n_rep / n_launch * 1e3
    return kern


def _roofline(w, kern, scoring="tc", attn="cluster"):
    peak, peak_kind = _peaks()
    fp32_peak = _fp32_peak_tfma()
    score_bytes = w.summary_bytes_per_layer()
    attn_bytes = w.kv_bytes_per_layer() + w.out_bytes_per_layer()
    # one FMA per (block, query vector, dim) term of the score's definition
    score_fma = w.S * w.nc * w.Nq * w.D
    k_gbs = {"score": score_bytes / (kern["score"] * 1e-6) / 1e9, "attn": attn_bytes / (kern["attn"] * 1e-6) / 1e9}
    dom = "attn" if kern["attn"] >= kern["score"] else "score"
    kname = {"attn": "k_attn_tc" if attn == "tc" else "k_attn", "score": "k_score_tc" if scoring == "tc" else "k_score"}
    sname = ("k_score_tc (oasis_score_blocks_tc, tensor cores)" if scoring == "tc"
             else "k_score (oasis_score_blocks)")
    score_tfma = score_fma / (kern["score"] * 1e-6) / 1e12
    # the fixed-order kernel is bound by whichever of its bytes and its FMAs takes longer at peak;
    # the tensor-core kernel by its bytes (its MMA work is a small fraction of the tensor roof)
    score_alu_bound = scoring == "exact" and score_fma / (fp32_peak * 1e12) > score_bytes / (peak * 1e9)
    score_fp32 = {"achieved": score_tfma, "peak": fp32_peak, "unit": "TFMA/s", "frac": score_tfma / fp32_peak,
                  "algorithmic_fma_per_launch": score_fma,
                  "peak_kind": "nominal: 152 SMs x 128 FP32 lanes x 2,070 MHz (unit counts and maximum SM clock)",
                  "note": "the kernel issues two FMAs per term (one adds an exact zero), so it can reach at most 0.5"}
    if scoring == "tc":
        ex = kern.get("score_exact")
        score_fp32 = None if ex is None else {
            "kernel": "k_score (oasis_score_blocks, fixed-order fp32, for comparison)", "us": ex,
            "achieved_tfma": score_fma / (ex * 1e-6) / 1e12, "peak_tfma": fp32_peak,
            "frac": score_fma / (ex * 1e-6) / 1e12 / fp32_peak, "gbs": score_bytes / (ex * 1e-6) / 1e9}
    timing = "CUDA graph of back-to-back launches over the layers' buffer sets, CUDA events on the replay stream"
    pk = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind
    if dom == "score" and score_alu_bound:
        roof = {"kernel": sname, "bound": "alu", **score_fp32,
                "traffic": _traffic("k_score", w), "timing": timing,
                "other": {"attn": {"us": kern["attn"], "gbs": k_gbs["attn"], "frac": k_gbs["attn"] / peak,
                                   "traffic": _traffic(kname["attn"], w)},
                          "score_hbm": {"gbs": k_gbs["score"], "frac": k_gbs["score"] / peak}}}
    else:
        aname = ("k_attn_tc (oasis_sparse_decode_attn_tc, tcgen05)" if attn == "tc"
                 else "k_attn (oasis_sparse_decode_attn)")
        roof = {"kernel": {"attn": aname, "score": sname}[dom],
                "bound": "hbm", "achieved": k_gbs[dom], "peak": peak, "unit": "GB/s", "frac": k_gbs[dom] / peak,
                "peak_kind": pk, "traffic": _traffic(kname[dom], w),
                "algorithmic_bytes_per_launch": attn_bytes if dom == "attn" else score_bytes, "timing": timing,
                "other": {k: {"us": kern[k], "gbs": k_gbs[k], "frac": k_gbs[k] / peak, "traffic": _traffic(kname[k], w)}
                          for k in k_gbs if k != dom}}
        if score_fp32 is not None:
            roof["other"]["score_fixed_order" if scoring == "tc" else "score_fp32"] = score_fp32
    # full summary build: reads the keys of every block (16 tokens x D bf16), writes kmin and kmax
    build_bytes = w.S * w.Nb * (16 * w.D * 2 + 2 * w.D * 2)
    build_gbs = build_bytes / (kern["summary_full_build"] * 1e-6) / 1e9
    roof["other"]["summary_full_build"] = {"us": kern["summary_full_build"], "gbs": build_gbs,
                                           "frac": build_gbs / peak, "algorithmic_bytes_per_launch": build_bytes,
                                           "traffic": _traffic("k_build_summary_full", w)}
    return roof


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_kv_cache_quest_gb300 as okv
    from synth import workload as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    okv.load()
    w = wl.WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    R = _layers(args, w)
    K, Wm = args.steps, max(args.warmup, 0)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- setup (untimed): KV cache, summaries, prior tables, pools, pinned host tier
    wb = Workbench(w, R, dev, balanced_attn=args.attn == "balanced", scoring=args.scoring, tc_attn=args.attn == "tc")
    graphs = wb.graphs(args)
    wb.reset()                                  # the capture's warm-up ran one step: start from the prior again

    # ---- the timed region: K decode steps (graph replays), tables advancing
    for i in range(Wm):
        graphs[i % len(graphs)].replay()
    barrier()
    clocks = ClockSampler(local) if rank == 0 else None
    barrier()
    torch.cuda.nvtx.range_push("oasis_timed")
    total_ms = _time_steps(graphs, Wm, K, dev)
    torch.cuda.nvtx.range_pop()
    barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(total_ms / max(1, K), dev)                # per decode step, slowest rank
    st = wb.status()
    assert st == 0, okv.strerror(st)
    admitted = int(sum(int(lay.plan_count.sum().item()) for lay in wb.layers))   # the last step's admissions

    # ---- one layer alone (no pipelining across layers): a StepGraph per buffer set
    iso = [okv.StepGraph(lay, wb.q[0], wb.qd[0], wb.sl, wb.host, wb.seg_stride, w.Nb, new_keys=wb.new_keys,
                         new_block=w.Nb - 1) for lay in wb.layers[:4]]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(50):
        for g in iso:
            g.replay()
    e1.record()
    e1.synchronize()
    iso_us = e0.elapsed_time(e1) / 50 / len(iso) * 1e3
    del iso

    kern = None if args.no_kernels else _kernel_times(wb, dev)

    per_layer = w.headline_bytes_per_layer()
    value = job_gbs(per_layer * R, ms, world)
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, wb, world, dev, Wm + K)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(w, args.workload, args.cpu_seconds)
    others = {}
    ids = [int(x) for x in args.other_workloads.split(",") if x.strip()] if args.other_workloads else []
    ids = [i for i in ids if i != args.workload] if world == 1 else []
    n_drift = len(graphs)
    if ids:
        del graphs, wb                      # free the headline state before the other workloads
        torch.cuda.empty_cache()
        for i in ids:
            others[wl.WORKLOADS[i].name] = _other_workload(args, i, dev)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms, "us_per_layer_step": ms * 1e3 / R,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": _config(w, R, {
                    "background_streams": args.bg_streams,
                    "staging_streams": args.xf_streams,
                    "foreground_priority": args.fg_priority,
                    "attention_split": args.attn,
                    "scoring": args.scoring,
                    "step": f"one decode step: the whole path (summary update, scoring, capped selection, staging, "
                            f"attention) over each of the {R} layers, layer-pipelined in one CUDA graph; tables "
                            f"advance from step to step, step i uses the queries of drift step i mod "
                            f"{n_drift}",
                    "l2": f"{R} per-layer buffer sets ({R * per_layer / 1e9:.1f} GB read per step > L2)",
                    "timed_region_s": total_ms / 1e3,
                    "blocks_admitted_last_step": admitted,
                    "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
                "single_layer_step_us": iso_us,
                "gpu_launches": 5 * R * K,
                "e2e": e2e, "cpu_baseline": cpu, "clocks": clk}
        if kern is not None:
            line["roofline"] = _roofline(w, kern, args.scoring, args.attn)
            line["kernels_us"] = kern
        if others:
            line["other_workloads"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


TRAFFIC_WORKLOAD = "qwen3-235b-attn"  # the workload the committed DRAM-traffic record was captured on


def _traffic(kernel, w):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and on the kernel's current source (else None)."""
    import hashlib
    if w.name != TRAFFIC_WORKLOAD:
        return None
    path = os.path.join(ROOT, "profiles", f"ncu_dram_traffic_{TRAFFIC_WORKLOAD}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "sparse_kv_cache_quest_gb300", "csrc", rec["source"])
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
            return None
    return rec["dram_bytes_per_launch"]


def _other_workload(args, wid, dev, steps=10, warmup=3):
    """Layer-step and per-kernel times of another workload (its own layer count,
    the same layer-pipelined graph), for the line's other_workloads key."""
    import torch

    from synth import workload as wl
    w = wl.WORKLOADS[wid]
    R = w.layers if w.layers > 1 else 36
    wb = Workbench(w, R, dev, balanced_attn=args.attn == "balanced", scoring=args.scoring, tc_attn=args.attn == "tc")
    graphs = wb.graphs(args)
    wb.reset()
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize(dev)
    ms = _time_steps(graphs, warmup, steps, dev) / steps
    st = wb.status()
    assert st == 0, st
    kern = _kernel_times(wb, dev)
    roof = _roofline(w, kern, args.scoring, args.attn)
    out = {"workload": _config(w, R)["workload"], "layers": R, "us_per_layer_step": ms * 1e3 / R,
           "value_gbs": w.headline_bytes_per_layer() / (ms * 1e-3 / R) / 1e9, "steps": steps,
           "kernels_us": kern,
           "frac_of_measured_hbm": {"score": w.summary_bytes_per_layer() / (kern["score"] * 1e-6) / 1e9 / roof["peak"],
                                    "attn": (w.kv_bytes_per_layer() + w.out_bytes_per_layer()) /
                                    (kern["attn"] * 1e-6) / 1e9 / roof["peak"]}}
    del graphs, wb
    torch.cuda.empty_cache()
    return out


def _e2e(args, wb, world, dev, first_step):
    """Same metric through the public call with host buffers: every decode step
    is one DecodeStepGraph(host_io=True) replay that copies each layer's inputs
    (queries, drafts, newest block's keys) from pinned host memory before the
    layer's work and each layer's results (outputs, lse, new table, plan,
    counts) back to pinned host memory once they exist; tables advance."""
    import torch
    import torch.distributed as dist
    graphs = wb.graphs(args, host_io=True)
    R = wb.R
    for i in range(2):
        graphs[(first_step + i) % len(graphs)].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    total = _time_steps(graphs, first_step + 2, K, dev)
    ms = max_over_ranks(total / max(1, K), dev)
    st = wb.status()
    assert st == 0, st
    g = graphs[0]
    return {"value": job_gbs(wb.w.headline_bytes_per_layer() * R, ms, world), "unit": "GB/s", "ms_per_step": ms,
            "us_per_layer_step": ms * 1e3 / R, "h2d_bytes_per_step": g.h2d_bytes, "d2h_bytes_per_step": g.d2h_bytes,
            "timed_region_s": total / 1e3,
            "how": "DecodeStepGraph(host_io=True).replay() per decode step: every layer copies its inputs from "
                   "pinned host memory (one copy) before its work and its results back after it, on copy streams "
                   "that overlap the other layers' kernels; tables advance"}


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
