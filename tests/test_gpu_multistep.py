"""Parity over several decode steps and several layers, with the resident set
carried forward:

* the Qwen3-235B-shaped layer for all of its decode steps, heavy blocks
  drifting by +-2 blocks per step (the keys are written once; step t's queries
  look at step t's heavy blocks): each step starts from the table and the pool
  the previous step left - the pool changes only through the staging of the
  admitted blocks, so attention at step t reads what the staging of earlier
  steps wrote;
* the Qwen3-8B-shaped step across consecutive layers, each layer's prior
  being the table the previous layer produced.

Sampled segments are checked against the oracle bit for bit (tables, plans,
staged pool) and within tolerance (attention); every segment is checked for the
selection invariants."""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import (assert_attention_close, default_scale, device_tiles, gather_pool, prior_tables,
                     run_oracle_segment, sample_segments)
import sparse_kv_cache_quest_gb300 as okv
from synth import workload as wl

pytestmark = pytest.mark.gpu


def _shape(w):
    return okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)


def _check_step(w, layer, step, lay, tiles_cpu, seq_len, table_in, q, qd, out, lse, segs):
    torch.cuda.synchronize()
    assert lay.status.item() == 0
    table_out = lay.table.cpu().numpy()
    plan = lay.plan.cpu().numpy()
    cnt = lay.plan_count.cpu().numpy()
    pool = bits(lay.pool)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    scale = default_scale(w.D)
    for s in segs:
        L = int(seq_len[s // w.Hkv])
        ref = run_oracle_segment(w, layer, s, tiles_cpu[s], L, table_in[s].tolist(), scale, bits(qd), bits(q))
        assert table_out[s].tolist() == ref["table_out"], (step, s)
        n = len(ref["plan"])
        assert int(cnt[s]) == n and [tuple(x) for x in plan[s, :n].tolist()] == ref["plan"], (step, s)
        assert np.array_equal(pool[s], ref["pool_after"]), (step, s)
        b, h = divmod(s, w.Hkv)
        assert_attention_close(go[b, h * w.G:(h + 1) * w.G], ref["out"], gl[b, h * w.G:(h + 1) * w.G], ref["lse"])
    t0 = table_in.numpy()
    for s in range(w.S):
        new = set(table_out[s, :w.K].tolist()) - {-1}
        old = set(t0[s, :w.K].tolist()) - {-1}
        assert len(new - old) == int(cnt[s]) <= w.cap
        assert np.array_equal(table_out[s, w.K:], t0[s, w.K:])
    return int(cnt.sum())


def test_drifting_heavy_blocks_over_decode_steps():
    okv.load()
    w = wl.WORKLOADS[5]
    assert w.steps > 1 and w.drift > 0
    layer = 0
    segs = sample_segments(w)
    seq_len = wl.seq_lens(w)
    sl = seq_len.cuda()
    lay = okv.DecodeLayer(_shape(w))
    tiles = device_tiles(w, layer)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)
    tiles_cpu = {s: bits(host[s]) for s in segs}
    table = prior_tables(w, layer, set(segs), lambda s: tiles_cpu[s], seq_len)
    lay.build_summary(tiles, sl, 0, w.Nb, strides=(tiles.stride(0), tiles.stride(1), tiles.stride(3)))
    lay.table.copy_(table.cuda())
    lay.pool.copy_(gather_pool(tiles, table))
    del tiles
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    admitted = []
    for step in range(w.steps):
        q = wl.q_true(w, layer, step).cuda()
        qd = wl.drafts(w, layer, step).cuda()
        out, lse = lay.step(q, qd, sl, host, host[0].numel() * 2, w.Nb, streams=streams, advance=True)
        admitted.append(_check_step(w, layer, step, lay, tiles_cpu, seq_len, table, q, qd, out, lse, segs))
        table = lay.table.cpu()
    # the heavy blocks move, so the cap admits blocks at every step
    assert all(a > 0 for a in admitted)


def test_resident_set_carried_across_layers():
    okv.load()
    w = wl.WORKLOADS[3]
    n_layers = 3
    segs = sample_segments(w)
    seq_len = wl.seq_lens(w)
    sl = seq_len.cuda()
    host = torch.empty((w.S, w.Nb, 2, 16, w.D), dtype=torch.bfloat16).pin_memory()
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    table = None
    for layer in range(n_layers):
        lay = okv.DecodeLayer(_shape(w))
        tiles = device_tiles(w, layer)
        host.copy_(tiles)
        tiles_cpu = {s: bits(host[s]) for s in segs}
        if table is None:
            table = prior_tables(w, layer, set(segs), lambda s: tiles_cpu[s], seq_len)
        lay.build_summary(tiles, sl, 0, w.Nb, strides=(tiles.stride(0), tiles.stride(1), tiles.stride(3)))
        lay.table.copy_(table.cuda())
        lay.pool.copy_(gather_pool(tiles, table))
        del tiles
        q = wl.q_true(w, layer).cuda()
        qd = wl.drafts(w, layer).cuda()
        out, lse = lay.step(q, qd, sl, host, host[0].numel() * 2, w.Nb, streams=streams, advance=True)
        _check_step(w, layer, 0, lay, tiles_cpu, seq_len, table, q, qd, out, lse, segs)
        table = lay.table.cpu()
        del lay
