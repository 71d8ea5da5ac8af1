"""Test-side glue: device inputs from the shared generator, oracle references.

Inputs for both sides come from ``synth``; expected values come only from
``oracle``.  Nothing here performs the method's arithmetic itself.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from conftest import bits
from oracle import pipeline as opipe
from oracle.score import score_blocks, segment_queries
from oracle.select import top_k
from oracle.summary import block_summary
from synth import workload as wl

RTOL_L2 = 1e-3     # relative L2 bound for attention outputs (fp32 vs float64 oracle)
ATOL_MAX = 1e-2    # max-abs bound for attention outputs


def sample_segments(w, n_extra=1):
    """First, last and a few seeded interior segments."""
    S = w.S
    picks = {0, S - 1}
    rs = np.random.default_rng(w.seed)
    for _ in range(n_extra):
        picks.add(int(rs.integers(0, S)))
    return sorted(picks)


def chunk_major_to_blocks(t: torch.Tensor) -> np.ndarray:
    """[S][D/8][Nb][8] bf16 summary -> numpy uint16 [S][Nb][D]."""
    S, C, Nb, _ = t.shape
    return bits(t.permute(0, 2, 1, 3).reshape(S, Nb, C * 8))


def device_tiles(w, layer, device="cuda", chunk=8):
    """The layer's full KV cache in tile layout on the device, bf16 [S][Nb][2][16][D]."""
    out = torch.empty((w.S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16, device=device)
    for s0 in range(0, w.S, chunk):
        segs = list(range(s0, min(w.S, s0 + chunk)))
        out[s0:s0 + len(segs)] = wl.kv_tiles(w, layer, segs, device=device)
    return out


def oracle_topk_true(w, layer, s, tiles_np, L):
    """Top-K candidate list of segment s under the true query (oracle arithmetic)."""
    kmin, kmax, _ = block_summary(tiles_np[:, 0], L)
    nc = max(0, -(-L // 16) - w.W)
    b, h = divmod(s, w.Hkv)
    q = bits(wl.q_true(w, layer))[b, h * w.G:(h + 1) * w.G]
    sc = score_blocks(kmin[:nc], kmax[:nc], q)
    return top_k(sc, w.K)


def prior_tables(w, layer, oracle_segs, tiles_of, seq_len):
    """int32 [S][K+W]: the workload's prior for the oracle-checked segments, random for the rest."""
    rows = []
    for s in range(w.S):
        if w.prior == "topk90" and s in oracle_segs:
            L = int(seq_len[s // w.Hkv])
            rows.append(wl.prior_from_topk(w, layer, s, oracle_topk_true(w, layer, s, tiles_of(s), L)))
        else:
            rows.append(wl.prior_random(w, layer, s))
    return torch.stack(rows)


def gather_pool(tiles: torch.Tensor, table: torch.Tensor) -> torch.Tensor:
    """pool[s][i] = tiles[s][table[s][i]] (zeros for empty slots), on tiles' device."""
    S, slots = table.shape
    t = table.to(tiles.device).long()
    idx = t.clamp(min=0)
    pool = tiles[torch.arange(S, device=tiles.device)[:, None], idx]
    pool[t < 0] = 0
    return pool


def run_oracle_segment(w, layer, s, tiles_np, L, table_in, scale, drafts_np, qtrue_np):
    b, h = divmod(s, w.Hkv)
    qd = segment_queries(drafts_np, b, h, w.G)
    qt = qtrue_np[b, h * w.G:(h + 1) * w.G]
    return opipe.run_segment(tiles_np, L, qd, qt, table_in, w.K, w.W, w.cap, scale)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_attention_close(out_gpu, out_ref, lse_gpu=None, lse_ref=None):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    err = np.abs(out_gpu - out_ref).max() if out_ref.size else 0.0
    assert err <= ATOL_MAX, f"max-abs {err}"
    if np.linalg.norm(out_ref) > 0:
        r = rel_l2(out_gpu, out_ref)
        assert r <= RTOL_L2, f"rel-L2 {r}"
    if lse_gpu is not None:
        lg = np.asarray(lse_gpu, dtype=np.float64)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lg), fin)
        if fin.any():
            assert np.abs(lg[fin] - lse_ref[fin]).max() <= 1e-3 * max(1.0, np.abs(lse_ref[fin]).max())


def default_scale(D):
    return float(np.float32(1.0 / math.sqrt(D)))
