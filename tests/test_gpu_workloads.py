"""Whole-path parity on the five workloads at their full per-layer sizes, run
through DecodeLayer.step (the launch configuration the benchmark times), with
sampled segments checked against the oracle: summaries, scores, tables, plans
and the staged pool bit-exact; attention within tolerance.  Every other
segment is checked for the selection invariants."""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import (assert_attention_close, chunk_major_to_blocks, default_scale, device_tiles, gather_pool,
                     prior_tables, run_oracle_segment, sample_segments)
import sparse_kv_cache_quest_gb300 as okv
from synth import workload as wl

pytestmark = pytest.mark.gpu


def _shape(w):
    return okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)


def test_device_generator_matches_cpu():
    w = wl.WORKLOADS[2]
    g = wl.kv_tiles(w, 0, [5, 63], device="cuda").cpu()
    c = wl.kv_tiles(w, 0, [5, 63])
    assert torch.equal(g.view(torch.int16), c.view(torch.int16))


# the tensor-core scoring pair at 64 and 256 segments: the second runs the selection
# at the width it takes when the segments outnumber the SMs; "tc+attn" adds the
# tcgen05 attention (clusters of 4 CTAs at 64 segments, 2 at 128, one CTA at 256)
@pytest.mark.parametrize("cfg,scoring", [(1, "exact"), (2, "exact"), (3, "exact"), (4, "exact"), (5, "exact"),
                                         (2, "tc"), (3, "tc"), (5, "tc"),
                                         (2, "tc+attn"), (4, "tc+attn"), (5, "tc+attn")])
def test_workload_layer_parity(cfg, scoring):
    okv.load()
    tc_attn = scoring == "tc+attn"
    scoring = "tc" if tc_attn else scoring
    w = wl.WORKLOADS[cfg]
    layer = 0
    segs = sample_segments(w)
    tiles = device_tiles(w, layer)                                  # [S][Nb][2][16][D], generated on the GPU
    seq_len = wl.seq_lens(w)
    cpu_tiles = {s: bits(wl.kv_tiles(w, layer, [s])[0]) for s in segs}
    table0 = prior_tables(w, layer, set(segs), lambda s: cpu_tiles[s], seq_len)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)

    lay = okv.DecodeLayer(_shape(w), scoring=scoring, tc_attn=tc_attn)
    sl = seq_len.cuda()
    lay.build_summary(tiles, sl, 0, w.Nb, strides=(tiles.stride(0), tiles.stride(1), tiles.stride(3)))
    lay.table.copy_(table0.cuda())
    lay.pool.copy_(gather_pool(tiles, table0))
    q = wl.q_true(w, layer).cuda()
    qd = wl.drafts(w, layer).cuda()
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    out, lse = lay.step(q, qd, sl, host, host[0].numel() * 2, w.Nb, streams=streams)
    torch.cuda.synchronize()
    assert lay.status.item() == 0

    kmin, kmax = chunk_major_to_blocks(lay.kmin), chunk_major_to_blocks(lay.kmax)
    scores = lay.scores.cpu().numpy()
    radius = lay.radius.cpu().numpy() if scoring == "tc" else None
    table_out = lay.table.cpu().numpy()            # swapped: the new table
    plan = lay.plan.cpu().numpy()
    cnt = lay.plan_count.cpu().numpy()
    pool = bits(lay.pool)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    drafts_np, qtrue_np = bits(qd), bits(q)
    scale = default_scale(w.D)
    for s in segs:
        L = int(seq_len[s // w.Hkv])
        ref = run_oracle_segment(w, layer, s, cpu_tiles[s], L, table0[s].tolist(), scale, drafts_np, qtrue_np)
        nbv = -(-L // 16)
        nc = nbv - w.W
        assert np.array_equal(kmin[s, :nbv], ref["kmin"][:nbv]) and np.array_equal(kmax[s, :nbv], ref["kmax"][:nbv])
        if scoring == "exact":
            assert np.array_equal(scores[s, :nc].view(np.uint32), ref["scores"].view(np.uint32))
        else:  # estimates within their radii (recomputed blocks hold the exact score, radius kept)
            assert np.all(np.abs(scores[s, :nc].astype(np.float64) - ref["scores"].astype(np.float64))
                          <= radius[s, :nc].astype(np.float64))
        assert table_out[s].tolist() == ref["table_out"]
        n = len(ref["plan"])
        assert int(cnt[s]) == n and [tuple(x) for x in plan[s, :n].tolist()] == ref["plan"]
        assert np.array_equal(pool[s], ref["pool_after"])
        b, h = divmod(s, w.Hkv)
        assert_attention_close(go[b, h * w.G:(h + 1) * w.G], ref["out"], gl[b, h * w.G:(h + 1) * w.G], ref["lse"])
    # invariants on every segment: K distinct blocks, at most cap new ones, window untouched
    t0 = table0.numpy()
    for s in range(w.S):
        new = set(table_out[s, :w.K].tolist()) - {-1}
        old = set(t0[s, :w.K].tolist()) - {-1}
        assert len(new) == min(w.K, w.nc) or len(new) == len(old) + int(cnt[s])
        assert len(new - old) == int(cnt[s]) <= w.cap
        assert np.array_equal(table_out[s, w.K:], t0[s, w.K:])
