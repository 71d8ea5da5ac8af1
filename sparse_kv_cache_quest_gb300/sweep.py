"""Synthetic analogs of studies in the OasisKV paper review (xllm-io): the
fetch-ratio ablation (§6, Table 2: transfer volume per step against the cap),
the draft-vs-true top-K agreement (§4, Figs. 4 and 6), and the size of the
admission set a request brings when its KV comes from another node (§3 decode
flow and §4 innovations table, remote partial fetching: the union over KV heads
of the first step's top-K, against the full cache; the review reports a 6.5-9.7x
smaller admission transfer).  No accuracy claim: the inputs are the seeded
synthetic Qwen3-8B-shaped layer whose heavy blocks drift by +-2 blocks per
decode step (the drafts of step t stand in for the queries of step t + 1).

Every step of the method runs in liboasis.so's kernels: the summaries
(oasis_build_summary), the draft and true-query scores (oasis_score_blocks),
every top-K set (oasis_select_topk_capped with cap = K on an empty table, which
admits exactly the first K candidates) and the capped selection that carries
the resident set from step to step.  What is left is counting set sizes of
those outputs (torch on the device), reported per (step, segment) so that a
test can compare the counts with the oracle's exactly:

  fetched[t][s]     blocks admitted by the capped selection (the plan count)
  binds[t][s]       1 if the draft top-K held more non-resident blocks than the cap
  overlap[t][s]     |draft top-K of step t  n  true top-K of step t + 1|
  recall[t][s]      |resident set after step t  n  true top-K of step t + 1|
  admission[b]      |union over the KV heads of sequence b of the step-0 true top-K|

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


def sweep_workload(ratio: str, K: int, steps: int, base=None):
    """The drifting Qwen3-8B-shaped layer with a given fetch ratio and K."""
    w = base if base is not None else wl.WORKLOADS[2]
    return w.with_(K=K, fetch_ratio=ratio, drift=2, steps=steps, plant_gain=8.0)


def _member(table: torch.Tensor, K: int, nc: int) -> torch.Tensor:
    """bool [S][nc]: the blocks held in slots 0..K-1 of each segment's table."""
    t = table[:, :K].long()
    r = torch.zeros((table.shape[0], nc + 1), dtype=torch.bool, device=table.device)
    r.scatter_(1, torch.where(t >= 0, t, torch.full_like(t, nc)), True)
    return r[:, :nc]


class _TopK:
    """The first K candidates by score of every segment, from the selection
    kernel: cap = K on an empty table admits exactly T."""

    def __init__(self, w, dev):
        self.w = w
        S = w.S
        self.empty = torch.full((S, w.slots), -1, dtype=torch.int32, device=dev)
        if w.W:
            self.empty[:, w.K:] = torch.tensor(wl.window_blocks(w), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.empty)
        self.plan = torch.empty((S, w.K, 2), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((S,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def __call__(self, scores, sl):
        w = self.w
        ob.oasis_select_topk_capped(scores, w.Nb, sl, w.B, w.Hkv, w.K, w.W, w.K, self.empty, self.out, self.plan,
                                    self.cnt, self.status)
        return _member(self.out, w.K, w.nc)


def run_counts(w, dev, table0=None):
    """Per-(step, segment) integer counts of the study on workload w (see the
    module docstring).  table0: int32 [S][K+W] resident tables at step 0
    (default: the step-0 true top-K, a cold start with cap = K)."""
    S, nc, K = w.S, w.nc, w.K
    shape = LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=K, W=w.W, cap=w.cap, Nd=w.Nd)
    lay = DecodeLayer(shape, device=dev)
    sl = wl.seq_lens(w).to(dev)
    tiles = torch.empty((S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16, device=dev)
    for s0 in range(0, S, 8):
        tiles[s0:s0 + 8] = wl.kv_tiles(w, 0, list(range(s0, min(S, s0 + 8))), device=dev)
    lay.build_summary(tiles, sl, 0, w.Nb, strides=(tiles.stride(0), tiles.stride(1), tiles.stride(3)))
    del tiles
    topk = _TopK(w, dev)
    true_scores = torch.empty((S, w.Nb), dtype=torch.float32, device=dev)

    def true_topk(step):
        q = wl.q_true(w, 0, step).to(dev)
        ob.oasis_score_blocks(lay.kmin, lay.kmax, w.Nb, q.view(w.B, 1, w.Hq, w.D), w.B, w.Hkv, w.G, 1, w.D, sl,
                              w.W, true_scores, lay.status)
        return topk(true_scores, sl)

    t_true = true_topk(0)
    admission = t_true.view(w.B, w.Hkv, nc).any(dim=1).sum(1)
    if table0 is None:
        table0 = topk.out.clone()                          # cold start: the true top-K of step 0
    lay.table.copy_(table0)
    counts = {k: [] for k in ("fetched", "binds", "overlap", "recall")}
    for step in range(w.steps):
        r_in = _member(lay.table, K, nc)
        qd = wl.drafts(w, 0, step).to(dev)
        lay.score(qd, sl)
        t_draft = topk(lay.scores, sl)
        lay.select(sl)
        t_next = true_topk((step + 1) % w.steps)
        r_out = _member(lay.table_next, K, nc)
        counts["fetched"].append(lay.plan_count.clone())
        counts["binds"].append(((t_draft & ~r_in).sum(1) > w.cap).to(torch.int32))
        counts["overlap"].append((t_draft & t_next).sum(1).to(torch.int32))
        counts["recall"].append((r_out & t_next).sum(1).to(torch.int32))
        lay.swap_tables()
    torch.cuda.synchronize(dev)
    bad = int(torch.maximum(lay.status, topk.status).item())
    assert bad == 0, ob.strerror(bad)
    out = {k: torch.stack(v).cpu() for k, v in counts.items()}
    out["admission"] = admission.cpu()
    return out


def summarize(w, c) -> dict:
    """Means of the counts (steps 1 .. of the fetch statistics: step 0 admits the
    blocks the cold start left out)."""
    K, nc, S = w.K, w.nc, w.S
    tile_bytes = 64 * w.D
    fetched = c["fetched"][1:].float().mean().item() if w.steps > 1 else float("nan")
    return {"fetch_ratio": w.fetch_ratio, "K": K, "cap": w.cap, "steps": w.steps,
            "blocks_fetched_per_head_step": fetched,
            "MB_per_layer_step": fetched * S * tile_bytes / 1e6,
            "cap_binding_rate": c["binds"][1:].float().mean().item() if w.steps > 1 else float("nan"),
            "draft_true_topk_overlap": c["overlap"].float().mean().item() / K,
            "resident_true_topk_recall": c["recall"].float().mean().item() / K,
            "admission_set_fraction": c["admission"].float().mean().item() / nc}


def run(ratio: str, K: int, steps: int, dev) -> dict:
    w = sweep_workload(ratio, K, steps)
    return summarize(w, run_counts(w, dev))


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
          "draft-vs-next-true top-K overlap | resident recall of next true top-K | admission set / full cache |")
    print("|---|---|---|---|---|---|---|---|---|")
    for x in rows:
        print(f"| {x['K']} | {x['fetch_ratio']} | {x['cap']} | {x['blocks_fetched_per_head_step']:.2f} | "
              f"{x['MB_per_layer_step']:.2f} | {x['cap_binding_rate']:.2f} | {x['draft_true_topk_overlap']:.3f} | "
              f"{x['resident_true_topk_recall']:.3f} | {x['admission_set_fraction']:.3f} |")


if __name__ == "__main__":
    main()
