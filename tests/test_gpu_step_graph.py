"""Parity of the launch configuration the benchmark times: a decode step over
several layers captured as one CUDA graph (``DecodeStepGraph``), layer-pipelined
on several streams, with and without the host I/O of the end-to-end
measurement.  Each layer's new table, plan, staged pool and attention output
are checked against the oracle on sampled segments of the Qwen3-8B-shaped layer
at full size."""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import (assert_attention_close, default_scale, device_tiles, gather_pool, prior_tables,
                     run_oracle_segment, sample_segments)
import sparse_kv_cache_quest_gb300 as okv
from synth import workload as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("host_io", [False, True])
def test_decode_step_graph_parity(host_io):
    okv.load()
    w = wl.WORKLOADS[2]
    R = 3
    layer = 0
    segs = sample_segments(w)
    tiles = device_tiles(w, layer)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)
    tiles_cpu = {s: bits(host[s]) for s in segs}
    seq_len = wl.seq_lens(w)
    sl = seq_len.cuda()
    table0 = prior_tables(w, layer, set(segs), lambda s: tiles_cpu[s], seq_len).cuda()
    pool0 = gather_pool(tiles, table0)
    shape = okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
    strides = (tiles.stride(0), tiles.stride(1), tiles.stride(3))
    lays = []
    for _ in range(R):
        lay = okv.DecodeLayer(shape)
        lay.build_summary(tiles, sl, 0, w.Nb, strides=strides)
        lay.table.copy_(table0)
        lays.append(lay)
    q = wl.q_true(w, layer).cuda()
    qd = wl.drafts(w, layer).cuda()
    new_keys = tiles[:, w.Nb - 1:w.Nb, 0].contiguous()
    g = okv.DecodeStepGraph(lays, q, qd, sl, host, host[0].numel() * 2, w.Nb, new_keys=new_keys,
                            new_block=w.Nb - 1, host_io=host_io)
    del tiles
    for lay in lays:                      # the graph's warm-up pass staged into the pools: start afresh
        lay.pool.copy_(pool0)
        lay.status.zero_()
    g.replay()
    torch.cuda.synchronize()
    scale = default_scale(w.D)
    refs = {s: run_oracle_segment(w, layer, s, tiles_cpu[s], int(seq_len[s // w.Hkv]), table0[s].tolist(), scale,
                                  bits(qd), bits(q)) for s in segs}
    for i, lay in enumerate(lays):
        assert lay.status.item() == 0
        if host_io:
            out, lse, tout, plan, cnt = g.host_out[i]
        else:
            out, lse, tout, plan, cnt = lay.out.cpu(), lay.lse.cpu(), lay.table_next.cpu(), lay.plan.cpu(), \
                lay.plan_count.cpu()
        out, lse, tout, plan, cnt = (x.numpy() for x in (out, lse, tout, plan, cnt))
        pool = bits(lay.pool)
        for s in segs:
            ref = refs[s]
            assert tout[s].tolist() == ref["table_out"], (i, s)
            n = len(ref["plan"])
            assert int(cnt[s]) == n and [tuple(x) for x in plan[s, :n].tolist()] == ref["plan"], (i, s)
            assert np.array_equal(pool[s], ref["pool_after"]), (i, s)
            b, h = divmod(s, w.Hkv)
            assert_attention_close(out[b, h * w.G:(h + 1) * w.G], ref["out"], lse[b, h * w.G:(h + 1) * w.G],
                                   ref["lse"])
    if host_io:
        assert g.h2d_bytes >= R * (q.numel() + qd.numel() + new_keys.numel()) * 2


@pytest.mark.parametrize("host_io,scoring", [(False, "exact"), (True, "exact"), (False, "tc"), (True, "tc")])
def test_decode_steps_advance_over_drift_steps(host_io, scoring):
    """The benchmarked form: one graph per drift step, tables advancing, the
    graphs replayed in drift order; after several decode steps every layer's
    table, plan, pool and attention output equal the oracle chained over the
    same steps (each step starting from the table the previous one produced)."""
    okv.load()
    w = wl.WORKLOADS[5].with_(B=4)
    R, n_steps = 3, 4
    layer = 0
    segs = sample_segments(w)
    tiles = device_tiles(w, layer)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)
    tiles_cpu = {s: bits(host[s]) for s in segs}
    seq_len = wl.seq_lens(w)
    sl = seq_len.cuda()
    table0 = prior_tables(w, layer, set(segs), lambda s: tiles_cpu[s], seq_len).cuda()
    pool0 = gather_pool(tiles, table0)
    shape = okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
    strides = (tiles.stride(0), tiles.stride(1), tiles.stride(3))
    lays = []
    for _ in range(R):
        lay = okv.DecodeLayer(shape, scoring=scoring)
        lay.build_summary(tiles, sl, 0, w.Nb, strides=strides)
        lays.append(lay)
    new_keys = tiles[:, w.Nb - 1:w.Nb, 0].contiguous()
    qs = [wl.q_true(w, layer, t) for t in range(n_steps)]
    qds = [wl.drafts(w, layer, t) for t in range(n_steps)]
    graphs = [okv.DecodeStepGraph(lays, qs[t].cuda(), qds[t].cuda(), sl, host, host[0].numel() * 2, w.Nb,
                                  new_keys=new_keys, new_block=w.Nb - 1, host_io=host_io, advance=True,
                                  share_host_inputs=host_io, warmup=(t == 0)) for t in range(n_steps)]
    for lay in lays:                      # the warm-up pass ran a step: start from the prior again
        lay.table.copy_(table0)
        lay.pool.copy_(pool0)
        lay.status.zero_()
    del tiles
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    scale = default_scale(w.D)
    admitted = 0
    for s in segs:
        table = table0[s].tolist()
        for t in range(n_steps):
            ref = run_oracle_segment(w, layer, s, tiles_cpu[s], int(seq_len[s // w.Hkv]), table, scale,
                                     bits(qds[t]), bits(qs[t]))
            table = ref["table_out"]
            admitted += len(ref["plan"])
        b, h = divmod(s, w.Hkv)
        for i, lay in enumerate(lays):
            assert lay.status.item() == 0
            if host_io:
                out, lse, tnext, plan, cnt = (x.numpy() for x in graphs[-1].host_out[i])
            else:
                out, lse, tnext, plan, cnt = (x.cpu().numpy() for x in (lay.out, lay.lse, lay.table_next, lay.plan,
                                                                        lay.plan_count))
            assert lay.table[s].tolist() == table == tnext[s].tolist(), (i, s)
            n = len(ref["plan"])
            assert int(cnt[s]) == n and [tuple(x) for x in plan[s, :n].tolist()] == ref["plan"], (i, s)
            assert np.array_equal(bits(lay.pool[s]), ref["pool_after"]), (i, s)
            assert_attention_close(out[b, h * w.G:(h + 1) * w.G], ref["out"], lse[b, h * w.G:(h + 1) * w.G],
                                   ref["lse"])
    assert admitted >= len(segs) * n_steps     # the cap admits blocks at every step
