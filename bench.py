#!/usr/bin/env python3
"""Benchmark of the lookahead sparse decode hot path on one GB300.

A step is one decode step of one layer of the Qwen3-8B-shaped workload
(batch 8, 32 q / 8 KV heads, d_h 128, 32,768-token context = 2,048 blocks of
16, K = 128, 3 draft queries, fetch ratio 0.05 -> cap 7): compressed-key
update of the newest block, draft-query block scoring, top-K selection with
capped eviction, staging of the admitted blocks from pinned host memory, and
sparse decode attention - every step in liboasis.so's kernels, on three CUDA
streams ordered by events.

Metric: HBM GB/s = (summaries read + selected K/V read + fp32 outputs written)
per step / step time; also microseconds per step and the fraction of the
measured HBM copy bandwidth reached by the dominant kernel.

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
WORKLOAD_ID = 2


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=14400, help="layer-steps timed (a multiple of --layers)")
    p.add_argument("--warmup", type=int, default=72, help="layer-steps run before timing")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=0,
                   help="layers per decode step, each with its own buffers (default: 36 for the Qwen3-8B-shaped "
                        "layer, else the workload's own layer count)")
    p.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=[1, 2, 3, 4, 5],
                   help="workload id (2 = the Qwen3-8B-shaped layer the metric is quoted on; the others for "
                        "per-workload kernel timings)")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget (CPU baseline)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--bg-streams", type=int, default=3, help="background streams, taken by the layers in turn")
    p.add_argument("--xf-streams", type=int, default=2, help="staging streams, taken by the layers in turn")
    p.add_argument("--fg-priority", type=int, default=0, help="CUDA priority of the foreground stream (lower = higher)")
    p.add_argument("--attn", choices=["cluster", "balanced"], default="cluster",
                   help="attention split: per-head thread-block clusters, or SM-balanced with a workspace")
    return p.parse_args()


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


def _config(w, extra=None):
    c = {"workload": f"{w.name}: 1 layer, batch {w.B}, {w.Hq} q / {w.Hkv} KV heads, d_h {w.D}, context {w.L} "
                     f"({w.Nb} blocks of 16), K={w.K}, W={w.W}, {w.Nd} drafts, fetch_ratio {w.fetch_ratio} "
                     f"(cap {w.cap}), bf16 KV, fp32 scores/out",
         "bytes_per_step": w.headline_bytes_per_layer(),
         "segments": w.S}
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

def _oracle_setup(w, n_seg):
    """Inputs of n_seg segments for the oracle (untimed): tiles, summaries, prior table."""
    import numpy as np
    import torch

    from oracle.score import score_blocks
    from oracle.select import top_k
    from oracle.summary import block_summary
    from synth import workload as wl

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    qd, qt = u16(wl.drafts(w, 0)), u16(wl.q_true(w, 0))
    segs = sorted({int(round(i * (w.S - 1) / max(1, n_seg - 1))) for i in range(n_seg)})
    prep = []
    for seg in segs:
        b, h = divmod(seg, w.Hkv)
        tiles = u16(wl.kv_tiles(w, 0, [seg])[0])
        kmin, kmax, _ = block_summary(tiles[:, 0], w.L)
        tk = top_k(score_blocks(kmin[:w.nc], kmax[:w.nc], qt[b, h * w.G:(h + 1) * w.G]), w.K)
        prep.append((seg, tiles, kmin, kmax, wl.prior_from_topk(w, 0, seg, tk).tolist()))
    return qd, qt, prep


def _oracle_sample(w, seconds, setup, start=0):
    """Run the oracle's decode step on the prepared segments, cycling, until
    `seconds` of CPU time are spent; returns (headline bytes, seconds, segment-steps)."""
    import numpy as np

    from oracle import pipeline as opipe
    from oracle.score import segment_queries

    qd, qt, prep = setup
    scale = float(np.float32(1.0 / math.sqrt(w.D)))
    per_seg = w.headline_bytes_per_layer() // w.S
    done, elapsed, i = 0, 0.0, start
    while elapsed < seconds:
        seg, tiles, kmin, kmax, table = prep[i % len(prep)]
        b, h = divmod(seg, w.Hkv)
        t0 = time.perf_counter()
        opipe.run_segment(tiles, w.L, segment_queries(qd, b, h, w.G), qt[b, h * w.G:(h + 1) * w.G], table,
                          w.K, w.W, w.cap, scale, kmin=kmin.copy(), kmax=kmax.copy(), update_blocks=[w.Nb - 1])
        elapsed += time.perf_counter() - t0
        done += 1
        i += 1
    return done * per_seg, elapsed, done


def _cpu_baseline(w, seconds):
    setup = _oracle_setup(w, 4)
    nbytes, secs, nseg = _oracle_sample(w, seconds, setup)
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{nseg} segment-steps cycling over {len(setup[2])} of the {w.S} segments of one decode "
                      f"step (newest-block summary update, scoring, capped selection, staging, attention); "
                      f"single-threaded numpy oracle, {secs:.1f} s; value = headline bytes of the sample / time",
            "us_per_step_equiv": secs / nseg * w.S * 1e6}


def run_reference(args):
    from synth import workload as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    setup = _oracle_setup(w, 4)
    budget = min(5.0, max(0.5, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        _oracle_sample(w, budget / 4, setup)
    total_b, total_s, segs = 0, 0.0, 0
    for i in range(args.steps):
        nb, s, n = _oracle_sample(w, budget, setup, start=i)
        total_b, total_s, segs = total_b + nb, total_s + s, segs + n
    value = total_b / total_s / 1e9
    ms = total_s / segs * w.S * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": _config(w, {"layers_per_decode_step": args.layers if args.layers > 0 else
                                  (36 if args.workload == WORKLOAD_ID else w.layers),
                                  "step": "one pass of the whole path (summary update, scoring, capped selection, "
                                          "staging, attention) over one layer, by the oracle on the host, one "
                                          "segment after another",
                                  "sample": f"{segs} segments over {args.steps} steps"}),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{segs} segment-steps cycling over {len(setup[2])} segments, "
                                       f"single-threaded numpy oracle, {total_s:.1f} s timed"},
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

def _gpu_prior(w, lay, tiles, sl, q):
    """Prior resident tables (about 90 % of the true-query top-K), computed with the kernels."""
    import torch

    import sparse_kv_cache_quest_gb300 as okv
    from synth import workload as wl
    S = w.S
    scores = torch.zeros((S, w.Nb), dtype=torch.float32, device="cuda")
    okv.oasis_score_blocks(lay.kmin, lay.kmax, w.Nb, q.view(w.B, 1, w.Hq, w.D), w.B, w.Hkv, w.G, 1, w.D, sl, w.W,
                           scores, lay.status)
    empty = torch.full((S, w.slots), -1, dtype=torch.int32, device="cuda")
    if w.W:
        empty[:, w.K:] = torch.tensor(wl.window_blocks(w), dtype=torch.int32, device="cuda")
    tout = torch.empty_like(empty)
    plan = torch.empty((S, w.K, 2), dtype=torch.int32, device="cuda")
    cnt = torch.empty((S,), dtype=torch.int32, device="cuda")
    okv.oasis_select_topk_capped(scores, w.Nb, sl, w.B, w.Hkv, w.K, w.W, w.K, empty, tout, plan, cnt, lay.status)
    t = tout.cpu()
    rows = [wl.prior_from_topk(w, 0, s, [b for b in t[s, :w.K].tolist() if b >= 0]) for s in range(S)]
    return torch.stack(rows)


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
    R = args.layers if args.layers > 0 else (36 if args.workload == WORKLOAD_ID else w.layers)

    # ---- setup (untimed): KV cache, summaries, prior tables, pool, pinned host tier.
    # Every layer gets its own device buffers (summaries, pool, tables, outputs) filled
    # from the same synthetic layer; the host tier is shared.
    tiles = torch.empty((w.S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16, device=dev)
    for s0 in range(0, w.S, 8):
        tiles[s0:s0 + 8] = wl.kv_tiles(w, 0, list(range(s0, min(w.S, s0 + 8))), device=dev)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)
    sl = wl.seq_lens(w).to(dev)
    q = wl.q_true(w, 0).to(dev)
    qd = wl.drafts(w, 0).to(dev)
    shape = okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
    strides = (tiles.stride(0), tiles.stride(1), tiles.stride(3))
    insts = []
    for i in range(R):
        lay = okv.DecodeLayer(shape, device=dev, balanced_attn=args.attn == "balanced")
        lay.build_summary(tiles, sl, 0, w.Nb, strides=strides)
        insts.append(lay)
    table0 = _gpu_prior(w, insts[0], tiles, sl, q).to(dev)
    pool0 = tiles[torch.arange(w.S, device=dev)[:, None], table0.long().clamp(min=0)]
    for lay in insts:
        lay.table.copy_(table0)
        lay.pool.copy_(pool0)
    del pool0
    new_keys = tiles[:, w.Nb - 1:w.Nb, 0].contiguous()     # keys of the newest block, [S][1][16][D]
    seg_stride = host[0].numel() * 2
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def time_replays(replay, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n                       # ms per replay

    # ---- the timed region: decode steps through R layers, one CUDA graph each
    step_graph = okv.DecodeStepGraph(insts, q, qd, sl, host, seg_stride, w.Nb, new_keys=new_keys,
                                     new_block=w.Nb - 1, n_bg=args.bg_streams, fg_priority=args.fg_priority,
                                     n_xf=args.xf_streams)
    reps = max(1, -(-args.steps // R))
    layer_steps = reps * R
    for _ in range(max(1, -(-args.warmup // R))):
        step_graph.replay()
    barrier()
    clocks = ClockSampler(local) if rank == 0 else None
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("oasis_timed")
    e0.record()
    for _ in range(reps):
        step_graph.replay()
    e1.record()
    torch.cuda.nvtx.range_pop()
    barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(e0.elapsed_time(e1) / layer_steps, dev)          # per layer-step, slowest rank
    st = torch.stack([lay.status for lay in insts]).max().item()
    assert st == 0, okv.strerror(int(st))

    # ---- one layer alone (no pipelining across layers): a StepGraph per buffer set
    iso = [okv.StepGraph(lay, q, qd, sl, host, seg_stride, w.Nb, new_keys=new_keys, new_block=w.Nb - 1)
           for lay in insts[:4]]
    iso_ms = time_replays(lambda: [g.replay() for g in iso], 100) / len(iso)

    # ---- per-kernel durations: a CUDA graph of back-to-back launches of one kernel
    # over the layers' buffer sets, replayed between events on the replay stream
    kern = {}
    calls = {"score": lambda lay, st_: lay.score(qd, sl, stream=st_),
             "attn": lambda lay, st_: lay.attend(q, sl, stream=st_),
             "select": lambda lay, st_: lay.select(sl, stream=st_),
             "stage": lambda lay, st_: lay.stage(host, seg_stride, w.Nb, stream=st_),
             "summary_update": lambda lay, st_: lay.build_summary(new_keys, sl, blk_begin=w.Nb - 1, blk_count=1,
                                                                  stream=st_),
             # the full build at sparsification time (not part of a decode step): every block's keys
             "summary_full_build": lambda lay, st_: lay.build_summary(tiles, sl, 0, w.Nb, strides=strides,
                                                                      stream=st_)}
    n_launch = max(8, R)
    for name, fn in calls.items():
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        kg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kg, stream=side):
            for i in range(n_launch):
                fn(insts[i % R], side)
        kg.replay()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push(f"oasis_kernel_{name}")
        kern[name] = time_replays(kg.replay, 20) / n_launch * 1e3          # us per launch
        torch.cuda.nvtx.range_pop()

    per_layer = w.headline_bytes_per_layer()
    value = job_gbs(per_layer, ms, world)
    peak, peak_kind = _peaks()
    fp32_peak = _fp32_peak_tfma()
    score_bytes = w.summary_bytes_per_layer()
    attn_bytes = w.kv_bytes_per_layer() + w.out_bytes_per_layer()
    # one FMA per (block, query vector, dim) term of the score's definition
    score_fma = w.S * w.nc * w.Nq * w.D
    k_gbs = {"score": score_bytes / (kern["score"] * 1e-6) / 1e9, "attn": attn_bytes / (kern["attn"] * 1e-6) / 1e9}
    dom = "attn" if kern["attn"] >= kern["score"] else "score"
    kname = {"attn": "k_attn", "score": "k_score"}
    score_tfma = score_fma / (kern["score"] * 1e-6) / 1e12
    # the scoring kernel is bound by whichever of its bytes and its FMAs takes longer at peak
    score_alu_bound = score_fma / (fp32_peak * 1e12) > score_bytes / (peak * 1e9)
    score_fp32 = {"achieved": score_tfma, "peak": fp32_peak, "unit": "TFMA/s", "frac": score_tfma / fp32_peak,
                  "algorithmic_fma_per_launch": score_fma,
                  "peak_kind": "nominal: 152 SMs x 128 FP32 lanes x 2,070 MHz (unit counts and maximum SM clock)",
                  "note": "the kernel issues two FMAs per term (one adds an exact zero), so it can reach at most 0.5"}
    if dom == "score" and score_alu_bound:
        roof = {"kernel": "k_score (oasis_score_blocks)", "bound": "alu", **score_fp32,
                "traffic": _traffic("k_score", w),
                "timing": "CUDA graph of back-to-back launches over the layers' buffer sets, CUDA events",
                "other": {"attn": {"us": kern["attn"], "gbs": k_gbs["attn"], "frac": k_gbs["attn"] / peak,
                                   "traffic": _traffic("k_attn", w)},
                          "score_hbm": {"gbs": k_gbs["score"], "frac": k_gbs["score"] / peak}}}
    else:
        roof = {"kernel": {"attn": "k_attn (oasis_sparse_decode_attn)", "score": "k_score (oasis_score_blocks)"}[dom],
                "bound": "hbm", "achieved": k_gbs[dom], "peak": peak, "unit": "GB/s", "frac": k_gbs[dom] / peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "traffic": _traffic(kname[dom], w),
                "algorithmic_bytes_per_launch": attn_bytes if dom == "attn" else score_bytes,
                "timing": "CUDA graph of back-to-back launches over the layers' buffer sets, CUDA events",
                "other": {k: {"us": kern[k], "gbs": k_gbs[k], "frac": k_gbs[k] / peak, "traffic": _traffic(kname[k], w)}
                          for k in k_gbs if k != dom}}
        roof["other"]["score_fp32"] = score_fp32
    # full summary build: reads the keys of every block (16 tokens x D bf16), writes kmin and kmax
    build_bytes = w.S * w.Nb * (16 * w.D * 2 + 2 * w.D * 2)
    build_gbs = build_bytes / (kern["summary_full_build"] * 1e-6) / 1e9
    roof["other"]["summary_full_build"] = {"us": kern["summary_full_build"], "gbs": build_gbs,
                                           "frac": build_gbs / peak, "algorithmic_bytes_per_launch": build_bytes,
                                           "traffic": _traffic("k_build_summary_full", w)}

    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, w, insts, host, seg_stride, q, qd, sl, new_keys, world, dev, time_replays)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": layer_steps,
                "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": _config(w, {
                    "layers_per_decode_step": R,
                    "background_streams": args.bg_streams,
                    "staging_streams": args.xf_streams,
                    "foreground_priority": args.fg_priority,
                    "attention_split": args.attn,
                    "step": "one pass of the whole path (summary update, scoring, capped selection, staging, "
                            "attention) over one layer; decode steps of R such layers run as one CUDA graph, "
                            "layer-pipelined (background of layer l overlaps the attention of later layers)",
                    "l2": f"{R} per-layer buffer sets ({R * per_layer / 1e9:.1f} GB of step inputs > L2)",
                    "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
                "single_layer_step_us": iso_ms * 1e3,
                "roofline": roof, "kernels_us": kern, "gpu_launches": 5 * layer_steps,
                "e2e": e2e, "cpu_baseline": cpu, "clocks": clk}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


TRAFFIC_WORKLOAD = "qwen3-8b-layer"  # the workload the committed DRAM-traffic record was captured on


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


def _e2e(args, w, insts, host, seg_stride, q, qd, sl, new_keys, world, dev, time_replays):
    """Same metric through the public call with host buffers: every decode step
    is one DecodeStepGraph(host_io=True) replay that copies each layer's inputs
    (queries, drafts, newest block's keys) from pinned host memory before the
    layer's work and each layer's results (outputs, lse, new table, plan,
    counts) back to pinned host memory once they exist."""
    import torch
    import torch.distributed as dist

    import sparse_kv_cache_quest_gb300 as okv
    g = okv.DecodeStepGraph(insts, q, qd, sl, host, seg_stride, w.Nb, new_keys=new_keys, new_block=w.Nb - 1,
                            host_io=True, n_bg=args.bg_streams, fg_priority=args.fg_priority,
                            n_xf=args.xf_streams)
    R = len(insts)
    g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    reps = max(1, min(200, -(-args.steps // R)))
    ms = max_over_ranks(time_replays(g.replay, reps) / R, dev)
    return {"value": job_gbs(w.headline_bytes_per_layer(), ms, world), "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": g.h2d_bytes // R, "d2h_bytes_per_step": g.d2h_bytes // R,
            "how": "DecodeStepGraph(host_io=True).replay(): every layer-step copies its inputs from pinned host "
                   "memory (one copy) before its work and its results back after it, on copy streams that "
                   "overlap the other layers' kernels"}


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
