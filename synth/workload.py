"""Seeded synthetic workloads: shapes, value distributions and structure.

The five workloads mirror the shapes the OasisKV pages evaluate (Qwen3-8B,
Llama-3.1-8B and Qwen3-235B-A22B attention shapes; 16-token blocks, K = 128
blocks per KV head, fetch ratio 0.05: OasisKV paper review (xllm-io), §6
"Benchmarks", default parameters).  No dataset or model weight is used: keys,
values and queries are seeded Irwin-Hall(4) stand-ins for N(0, 1) from
``synth.rng``, with the structure each workload names (outlier key channels,
planted heavy blocks, draft queries = true query + noise).

This module only draws and arranges random numbers.  It contains none of the
method's arithmetic.  The one structural input that needs the method - a prior
resident set that overlaps the true-query top-K by about 90 % - is assembled by
``prior_from_topk`` from a top-K list that the caller computes with its own
implementation (the oracle in tests, the kernels in the benchmark).

Drift over decode steps (workloads with ``drift > 0``).  Keys and values are
written once, as in a real decode where the cache never changes after a token
is written; what moves is where the current query looks.  Step t of the
``steps`` simulated steps has its own heavy-block positions P_t (each block of
P_{t-1} moved by +drift or -drift) and its own random unit direction u_t per
(sequence, KV head).  Every key of a block in P_t gets ``plant_gain * u_t``;
the true query of step t leans towards u_t (``query_lean * u_t`` added to every
query head of the group), so the blocks of P_t are the heavy ones at step t.
The drafts of step t stand in for the speculative queries of the next token:
they are the true query of step t + 1 (cyclically) plus noise.

Tensor layouts (bf16 tensors use torch.bfloat16):
    keys / values      [S_sel][Nb][16][D]   (S_sel = the requested segments)
    kv tiles           [S_sel][Nb][2][16][D] (K tile, then V tile, per block)
    q_true             [B][Hq][D]
    drafts             [B][Nd][Hq][D]
    table (prior)      [S][K + W] int32, slot -> logical block id, -1 = empty
A segment is one (sequence b, KV head h) pair, s = b * Hkv + h.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from fractions import Fraction

import torch

from . import rng

BLOCK = 16  # tokens per logical KV block

# stream tags
T_KEYS, T_VALUES, T_QTRUE, T_QNOISE, T_PLANTS, T_OUTLIERS, T_PRIOR, T_DRIFT, T_MISC, T_DIRECTION = range(1, 11)


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    B: int
    Hkv: int
    G: int
    D: int
    L: int
    K: int
    W: int
    Nd: int
    fetch_ratio: str          # decimal string, so the cap is computed exactly
    plants: int               # planted heavy blocks per segment
    outliers: int             # outlier key channels per (layer, KV head)
    outlier_scale: float      # keys on outlier channels are multiplied by this (a power of 2)
    prior: str                # "random" or "topk90"
    seed: int
    steps: int = 1            # simulated decode steps
    drift: int = 0            # heavy blocks move by +-drift blocks per step
    draft_noise: float = 0.3  # std of the noise added to the true query for each draft
    plant_gain: float = 2.0   # planted keys get += plant_gain * unit(sum of the group's true q)
    query_lean: float = 2.0   # drifting workloads: the true query of step t gets += query_lean * u_t

    @property
    def Hq(self) -> int:
        return self.Hkv * self.G

    @property
    def S(self) -> int:
        return self.B * self.Hkv

    @property
    def Nb(self) -> int:
        return -(-self.L // BLOCK)

    @property
    def nc(self) -> int:
        return self.Nb - self.W

    @property
    def Nq(self) -> int:
        return self.G * self.Nd

    @property
    def slots(self) -> int:
        return self.K + self.W

    @property
    def cap(self) -> int:
        """C = ceil(fetch_ratio * K), computed in exact rational arithmetic."""
        return math.ceil(Fraction(self.fetch_ratio) * self.K)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    # per-layer byte counts of the headline metric
    def summary_bytes_per_layer(self) -> int:
        return self.S * 2 * self.D * self.Nb * 2

    def kv_bytes_per_layer(self) -> int:
        return self.S * self.slots * 2 * BLOCK * self.D * 2

    def out_bytes_per_layer(self) -> int:
        return self.B * self.Hq * self.D * 4

    def headline_bytes_per_layer(self) -> int:
        return self.summary_bytes_per_layer() + self.kv_bytes_per_layer() + self.out_bytes_per_layer()


WORKLOADS = {
    1: Workload("tiny", layers=1, B=1, Hkv=2, G=2, D=64, L=1024, K=8, W=0, Nd=1,
                fetch_ratio="0.25", plants=4, outliers=0, outlier_scale=1.0, prior="random", seed=1001),
    2: Workload("qwen3-8b-layer", layers=1, B=8, Hkv=8, G=4, D=128, L=32768, K=128, W=0, Nd=3,
                fetch_ratio="0.05", plants=64, outliers=4, outlier_scale=8.0, prior="topk90", seed=1002),
    3: Workload("qwen3-8b-step", layers=36, B=32, Hkv=8, G=4, D=128, L=32768, K=128, W=0, Nd=3,
                fetch_ratio="0.05", plants=64, outliers=4, outlier_scale=8.0, prior="topk90", seed=1003),
    4: Workload("llama3.1-8b-long", layers=32, B=16, Hkv=8, G=4, D=128, L=131072, K=128, W=4, Nd=4,
                fetch_ratio="0.05", plants=64, outliers=4, outlier_scale=8.0, prior="topk90", seed=1004),
    5: Workload("qwen3-235b-attn", layers=94, B=64, Hkv=4, G=16, D=128, L=32768, K=128, W=0, Nd=4,
                fetch_ratio="0.05", plants=64, outliers=0, outlier_scale=1.0, prior="topk90", seed=1005,
                steps=8, drift=2, plant_gain=8.0),
}


def seq_lens(w: Workload) -> torch.Tensor:
    """Valid token count of every sequence (int32 [B]); all equal to L."""
    return torch.full((w.B,), w.L, dtype=torch.int32)


def ragged_seq_lens(w: Workload, min_len: int) -> torch.Tensor:
    """Per-sequence lengths drawn uniformly from [min_len, L] (int32 [B])."""
    u = rng.uniform_u32(w.seed, T_MISC, torch.arange(w.B, dtype=torch.int64))
    return (min_len + u % (w.L - min_len + 1)).to(torch.int32)


# ----------------------------------------------------------------------------- queries

def _q_base(w: Workload, layer: int) -> torch.Tensor:
    n = w.B * w.Hq * w.D
    idx = torch.arange(n, dtype=torch.int64) + layer * n
    return rng.normal_bf16(w.seed, T_QTRUE, idx).view(w.B, w.Hq, w.D)


def q_true(w: Workload, layer: int, step: int = 0) -> torch.Tensor:
    """True decode query, bf16 [B][Hq][D] (CPU).

    Without drift the same at every step.  With drift, step t's query is
    bf16(fp32(base) + query_lean * u_t) with u_t = ``drift_direction(w, layer, t)``
    of the query head's KV head (t taken modulo ``steps``).
    """
    base = _q_base(w, layer)
    if w.drift == 0:
        return base
    u = drift_direction(w, layer, step % w.steps).repeat_interleave(w.G, dim=1)      # [B][Hq][D]
    lean = torch.tensor(w.query_lean, dtype=torch.float32)
    return (base.to(torch.float32) + lean * u).to(torch.bfloat16)


def drafts(w: Workload, layer: int, step: int = 0) -> torch.Tensor:
    """Draft queries bf16 [B][Nd][Hq][D]: bf16(fp32(target) + draft_noise * noise) (CPU).

    Draft j of step ``step`` draws its own noise.  The target is the true query
    of the same step without drift, and of the next step (cyclically) with
    drift: the drafts look one token ahead.
    """
    target = q_true(w, layer, (step + 1) % w.steps if w.drift else 0).to(torch.float32)
    n = w.B * w.Nd * w.Hq * w.D
    idx = torch.arange(n, dtype=torch.int64) + (layer * w.steps + step) * n
    noise = rng.normal_f32(w.seed, T_QNOISE, idx).view(w.B, w.Nd, w.Hq, w.D)
    return (target[:, None, :, :] + torch.tensor(w.draft_noise, dtype=torch.float32) * noise).to(torch.bfloat16)


def drift_direction(w: Workload, layer: int, step: int) -> torch.Tensor:
    """Random unit directions u_t, fp32 [B][Hkv][D] (CPU): one per (sequence, KV
    head) and step; normalised in float64, then rounded once to fp32."""
    n = w.B * w.Hkv * w.D
    idx = torch.arange(n, dtype=torch.int64) + (layer * w.steps + step) * n
    v = rng.normal_f32(w.seed, T_DIRECTION, idx).to(torch.float64).view(w.B, w.Hkv, w.D)
    return (v / torch.linalg.vector_norm(v, dim=-1, keepdim=True)).to(torch.float32)


def plant_direction(w: Workload, layer: int) -> torch.Tensor:
    """Unit vector of the sum of each KV head's true group queries, fp32 [B][Hkv][D] (CPU).

    Computed in float64 from the bf16 queries, then rounded once to fp32.
    """
    qt = _q_base(w, layer).to(torch.float64).view(w.B, w.Hkv, w.G, w.D).sum(dim=2)
    nrm = torch.linalg.vector_norm(qt, dim=-1, keepdim=True)
    return (qt / nrm).to(torch.float32)


# ----------------------------------------------------------------------------- structure

def planted_blocks(w: Workload, layer: int, s: int, step: int = 0) -> torch.Tensor:
    """Sorted candidate block ids of segment ``s`` that carry planted heavy keys.

    At step 0 these are a uniform random ``plants``-subset of the candidates.
    With ``drift > 0`` each later step moves every heavy block by +drift or
    -drift (a random sign per block and step), clamped into [0, nc); a block
    that would land on another heavy block of the same step stays where it is.
    """
    return planted_blocks_steps(w, layer, s, step + 1)[step]


def planted_blocks_steps(w: Workload, layer: int, s: int, n_steps: int) -> list:
    """``planted_blocks`` of steps 0 .. n_steps - 1 of segment ``s``, in one pass."""
    if w.plants == 0 or w.nc <= 0:
        return [torch.zeros(0, dtype=torch.int64)] * n_steps
    p = min(w.plants, w.nc)
    cur = rng.random_subset(w.seed, T_PLANTS, (layer * w.S + s) * w.Nb, w.nc, p)
    out = [cur]
    for st in range(1, n_steps):
        base = ((layer * w.S + s) * w.steps + st) * w.plants
        signs = rng.random_signs(w.seed, T_DRIFT, torch.arange(base, base + p, dtype=torch.int64))
        taken = set(cur.tolist())
        nxt = []
        for blk, sg in zip(cur.tolist(), signs.tolist()):
            cand = min(max(blk + sg * w.drift, 0), w.nc - 1)
            if cand != blk and cand not in taken:
                taken.discard(blk)
                taken.add(cand)
                nxt.append(cand)
            else:
                nxt.append(blk)
        cur = torch.tensor(sorted(nxt), dtype=torch.int64)
        out.append(cur)
    return out


def outlier_channels(w: Workload, layer: int, h: int) -> torch.Tensor:
    """Sorted key channels of (layer, KV head h) that are scaled by outlier_scale."""
    if w.outliers == 0:
        return torch.zeros(0, dtype=torch.int64)
    return rng.random_subset(w.seed, T_OUTLIERS, (layer * w.Hkv + h) * w.D, w.D, w.outliers)


# ----------------------------------------------------------------------------- KV cache

def _segment_index(w: Workload, layer: int, segs: torch.Tensor, device) -> torch.Tensor:
    per_seg = w.Nb * BLOCK * w.D
    base = (layer * w.S + segs.to(torch.int64)).to(device) * per_seg
    return base[:, None] + torch.arange(per_seg, dtype=torch.int64, device=device)[None, :]


def keys(w: Workload, layer: int, segs, device="cpu") -> torch.Tensor:
    """Keys bf16 [len(segs)][Nb][16][D] of the requested segments, on ``device``.

    Base values are N(0, 1) stand-ins; on the outlier channels of the segment's
    KV head they are multiplied by ``outlier_scale`` (exact: a power of 2); every
    key of a planted block then gets ``plant_gain * u`` added in fp32 and is
    rounded to bf16.  Without drift u is ``plant_direction`` and the planted
    blocks are those of step 0; with drift, for every step t the blocks of step
    t get ``plant_gain * u_t`` (``drift_direction``), added in step order.
    Tokens past L in a partial last block are generated like the others.
    """
    segs = torch.as_tensor(segs, dtype=torch.int64).reshape(-1)
    idx = _segment_index(w, layer, segs, device)
    k = rng.normal_bf16(w.seed, T_KEYS, idx).view(len(segs), w.Nb, BLOCK, w.D)
    if w.outliers == 0 and w.plants == 0:
        return k
    if w.plants:
        dirs = ([drift_direction(w, layer, t) for t in range(w.steps)] if w.drift
                else [plant_direction(w, layer)])
    kf = k.to(torch.float32)
    gain = torch.tensor(w.plant_gain, dtype=torch.float32)
    for i, s in enumerate(segs.tolist()):
        b, h = divmod(s, w.Hkv)
        ch = outlier_channels(w, layer, h)
        if len(ch):
            kf[i, :, :, ch.to(device)] *= w.outlier_scale
        if w.plants:
            pbs = planted_blocks_steps(w, layer, s, len(dirs))
            for u, pb in zip(dirs, pbs):
                pb = pb.to(device)
                if len(pb):
                    kf[i, pb] = kf[i, pb] + (gain * u[b, h]).to(device)
    return kf.to(torch.bfloat16)


def values(w: Workload, layer: int, segs, device="cpu") -> torch.Tensor:
    """Values bf16 [len(segs)][Nb][16][D]: N(0, 1) stand-ins."""
    segs = torch.as_tensor(segs, dtype=torch.int64).reshape(-1)
    idx = _segment_index(w, layer, segs, device)
    return rng.normal_bf16(w.seed, T_VALUES, idx).view(len(segs), w.Nb, BLOCK, w.D)


def kv_tiles(w: Workload, layer: int, segs, device="cpu") -> torch.Tensor:
    """Full KV cache of the segments in tile layout, bf16 [len(segs)][Nb][2][16][D]."""
    return torch.stack([keys(w, layer, segs, device), values(w, layer, segs, device)], dim=2)


# ----------------------------------------------------------------------------- resident sets

def window_blocks(w: Workload) -> list[int]:
    """Blocks nc .. nc + W - 1: the local window, always resident in slots K .. K + W - 1."""
    return list(range(w.nc, w.nc + w.W))


def prior_random(w: Workload, layer: int, s: int) -> torch.Tensor:
    """Prior table of segment s: K uniform random distinct candidates in ascending
    order (fewer, with -1 padding, when nc < K), then the window blocks."""
    k = min(w.K, max(w.nc, 0))
    blocks = rng.random_subset(w.seed, T_PRIOR, (layer * w.S + s) * w.Nb, max(w.nc, 0), k).tolist()
    blocks += [-1] * (w.K - k)
    return torch.tensor(blocks + window_blocks(w), dtype=torch.int32)


def prior_from_topk(w: Workload, layer: int, s: int, topk: list[int], keep_frac: str = "0.9") -> torch.Tensor:
    """Prior table that keeps about 90 % of a given top-K list.

    ``topk`` is the segment's top-K candidate set under the true query (computed
    by the caller).  round(keep_frac * K) of its members (a random choice) are
    kept and the rest of the K slots get random candidates outside ``topk``;
    slots hold the blocks in ascending order, followed by the window blocks.
    """
    topk = sorted(int(b) for b in topk)
    k = len(topk)
    keep = int(Fraction(keep_frac) * k + Fraction(1, 2))
    off = (layer * w.S + s) * w.Nb
    order = rng.random_order(w.seed, T_PRIOR, off, k).tolist()
    kept = [topk[i] for i in order[:keep]]
    tset = set(topk)
    rest = [b for b in rng.random_order(w.seed, T_PRIOR + 100, off, max(w.nc, 0)).tolist() if b not in tset]
    blocks = sorted(kept + rest[: w.K - keep])
    blocks += [-1] * (w.K - len(blocks))
    return torch.tensor(blocks + window_blocks(w), dtype=torch.int32)
