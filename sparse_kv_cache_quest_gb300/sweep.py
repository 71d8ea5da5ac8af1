"""Synthetic analogs of studies in the OasisKV paper review (xllm-io): the
fetch-ratio ablation (§6, Table 2: transfer volume per step against the cap),
the draft-vs-true top-K agreement (§4, Figs. 4 and 6), and the size of the
admission set a request brings when its KV comes from another node (§3 decode
flow and §4 innovations table, remote partial fetching: the union over KV heads
of the first step's top-K, against the full cache; the review reports a 6.5-9.7x
smaller admission transfer).  No accuracy
claim: the inputs are the seeded synthetic Qwen3-8B-shaped layer whose heavy
blocks drift by +-2 blocks per decode step, so the resident set has to follow
them.

Every selection runs in liboasis.so's kernels (summary rebuild, draft scoring,
capped selection); the true-query scores come from the same scoring kernel
with the true query as the only "draft".  The statistics (set overlaps, the
rate at which the cap binds) are computed afterwards with torch on the device.

    python -m sparse_kv_cache_quest_gb300.sweep [--ratios 0.01,0.02,0.05,0.1,0.2]
                                              [--ks 64,128,192] [--steps 8]

Prints one JSON line per (fetch ratio, K) and a markdown table.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_kv_cache_quest_gb300 import binding as ob  # noqa: E402
from sparse_kv_cache_quest_gb300.layer import DecodeLayer, LayerShape  # noqa: E402
from synth import workload as wl  # noqa: E402


def _topk_sets(scores: torch.Tensor, nc: int, k: int) -> torch.Tensor:
    """bool [S][nc]: the first k candidates by (score desc, block asc)."""
    order = torch.sort(-scores[:, :nc], dim=1, stable=True).indices[:, :k]
    sel = torch.zeros((scores.shape[0], nc), dtype=torch.bool, device=scores.device)
    sel.scatter_(1, order, True)
    return sel


def _resident(table: torch.Tensor, K: int, nc: int) -> torch.Tensor:
    t = table[:, :K].long()
    r = torch.zeros((table.shape[0], nc + 1), dtype=torch.bool, device=table.device)
    r.scatter_(1, torch.where(t >= 0, t, torch.full_like(t, nc)), True)
    return r[:, :nc]


def run(ratio: str, K: int, steps: int, dev) -> dict:
    w = wl.WORKLOADS[2].with_(K=K, fetch_ratio=ratio, drift=2, steps=steps, plant_gain=8.0)
    nc, S = w.nc, w.S
    shape = LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
    lay = DecodeLayer(shape, device=dev)
    sl = wl.seq_lens(w).to(dev)
    true_scores = torch.empty((S, w.Nb), dtype=torch.float32, device=dev)
    tiles = torch.empty((S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16, device=dev)
    for s0 in range(0, S, 8):
        tiles[s0:s0 + 8] = wl.kv_tiles(w, 0, list(range(s0, min(S, s0 + 8))), device=dev)
    lay.build_summary(tiles, sl, 0, w.Nb, strides=(tiles.stride(0), tiles.stride(1), tiles.stride(3)))
    stats = {"fetched": [], "cap_binds": [], "draft_true_overlap": [], "resident_recall": [], "admission": []}
    for step in range(steps):
        q = wl.q_true(w, 0, step).to(dev)
        ob.oasis_score_blocks(lay.kmin, lay.kmax, w.Nb, q.view(w.B, 1, w.Hq, w.D), w.B, w.Hkv, w.G, 1, w.D, sl,
                              w.W, true_scores, lay.status)
        t_true = _topk_sets(true_scores, nc, K)
        if step == 0:
            # admission set of a request whose KV arrives from elsewhere: the union over its KV
            # heads of the first step's top-K blocks, against the full cache of the sequence
            union = t_true.view(w.B, w.Hkv, nc).any(dim=1)
            stats["admission"].append((union.sum(1).float() / nc).mean().item())
            # the resident set at the start: the true query's top-K (cold start, cap = K)
            empty = torch.full((S, w.slots), -1, dtype=torch.int32, device=dev)
            plan = torch.empty((S, K, 2), dtype=torch.int32, device=dev)
            cnt = torch.empty((S,), dtype=torch.int32, device=dev)
            ob.oasis_select_topk_capped(true_scores, w.Nb, sl, w.B, w.Hkv, K, w.W, K, empty, lay.table, plan, cnt,
                                        lay.status)
        r_in = _resident(lay.table, K, nc)
        lay.score(wl.drafts(w, 0, step=step).to(dev), sl)
        t_draft = _topk_sets(lay.scores, nc, K)
        lay.select(sl)
        torch.cuda.synchronize(dev)
        assert lay.status.item() == 0, ob.strerror(int(lay.status.item()))
        r_out = _resident(lay.table_next, K, nc)
        if step > 0:
            stats["fetched"].append(lay.plan_count.float().mean().item())
            stats["cap_binds"].append(((t_draft & ~r_in).sum(1) > w.cap).float().mean().item())
        stats["draft_true_overlap"].append(((t_draft & t_true).sum(1).float() / K).mean().item())
        stats["resident_recall"].append(((r_out & t_true).sum(1).float() / K).mean().item())
        lay.swap_tables()
    mean = {k: sum(v) / len(v) for k, v in stats.items() if v}
    tile_bytes = 64 * w.D
    return {"fetch_ratio": ratio, "K": K, "cap": w.cap, "steps": steps,
            "blocks_fetched_per_head_step": mean["fetched"],
            "MB_per_layer_step": mean["fetched"] * S * tile_bytes / 1e6,
            "cap_binding_rate": mean["cap_binds"],
            "draft_true_topk_overlap": mean["draft_true_overlap"],
            "resident_true_topk_recall": mean["resident_recall"],
            "admission_set_fraction": mean["admission"]}


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--ratios", default="0.01,0.02,0.05,0.1,0.2")
    p.add_argument("--ks", default="64,128,192")
    p.add_argument("--steps", type=int, default=8)
    a = p.parse_args()
    ob.load()
    dev = torch.device("cuda", 0)
    rows = []
    for K in [int(x) for x in a.ks.split(",")]:
        for r in a.ratios.split(","):
            res = run(r, K, a.steps, dev)
            print(json.dumps(res), flush=True)
            rows.append(res)
    print("| K | fetch ratio | cap C | blocks fetched / head / step | MB / layer-step | cap binds | "
          "draft-vs-true top-K overlap | resident recall of true top-K | admission set / full cache |")
    print("|---|---|---|---|---|---|---|---|---|")
    for x in rows:
        print(f"| {x['K']} | {x['fetch_ratio']} | {x['cap']} | {x['blocks_fetched_per_head_step']:.2f} | "
              f"{x['MB_per_layer_step']:.2f} | {x['cap_binding_rate']:.2f} | {x['draft_true_topk_overlap']:.3f} | "
              f"{x['resident_true_topk_recall']:.3f} | {x['admission_set_fraction']:.3f} |")


if __name__ == "__main__":
    main()
