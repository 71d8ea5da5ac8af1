"""Decode-time append: the context grows one token per decode step, so the
newest block's summary is refreshed from its valid tokens every step (the
compressed-key update of the OasisKV paper review (xllm-io), §5), the local
window slides when a block fills, and the block leaving the window becomes a
candidate.  Every step of every segment is checked against the oracle: the
incrementally maintained summaries against a full rebuild at that length, and
scores, table, plan, staged pool and attention as in the single-step tests."""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import assert_attention_close, chunk_major_to_blocks, default_scale, gather_pool
from oracle import pipeline as opipe
from oracle.score import segment_queries
import sparse_kv_cache_quest_gb300 as okv
from synth import workload as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W", [0, 2])
def test_token_by_token_append(W):
    okv.load()
    L0, n_steps = 1000, 44                       # crosses the block boundaries at 1008, 1024 and 1040
    w = wl.WORKLOADS[1].with_(L=1056, W=W, steps=n_steps)
    layer = 0
    tiles = wl.kv_tiles(w, layer, list(range(w.S))).cuda()        # the final cache; validity comes from L
    tiles_np = bits(tiles)
    host = torch.empty(tiles.shape, dtype=torch.bfloat16).pin_memory()
    host.copy_(tiles)
    shape = okv.LayerShape(B=w.B, Hkv=w.Hkv, G=w.G, D=w.D, Nb_max=w.Nb, K=w.K, W=w.W, cap=w.cap, Nd=w.Nd)
    lay = okv.DecodeLayer(shape)
    q = wl.q_true(w, layer).cuda()
    qt_np = bits(q)
    scale = default_scale(w.D)
    strides = (tiles.stride(0), tiles.stride(1), tiles.stride(3))

    def window(L):
        nc = -(-L // 16) - W
        return list(range(nc, nc + W))

    sl = torch.full((w.B,), L0, dtype=torch.int32, device="cuda")
    lay.build_summary(tiles, sl, 0, w.Nb, strides=strides)           # sparsification: full build at L0
    nc0 = -(-L0 // 16) - W
    rs = np.random.default_rng(7)
    table = torch.tensor([sorted(rs.choice(nc0, size=w.K, replace=False).tolist()) + window(L0)
                          for _ in range(w.S)], dtype=torch.int32)
    admitted = 0
    for t in range(n_steps):
        L = L0 + t
        sl.fill_(L)
        newest = (L - 1) // 16
        # the model writes the new token's K/V: the window slots follow the newest blocks
        table[:, w.K:] = torch.tensor(window(L), dtype=torch.int32)
        lay.table.copy_(table.cuda())
        lay.pool.copy_(gather_pool(tiles, table))
        qd = wl.drafts(w, layer, step=t).cuda()
        out, lse = lay.step(q, qd, sl, host, host[0].numel() * 2, w.Nb,
                            new_keys=tiles[:, newest:newest + 1, 0].contiguous(), new_block=newest)
        torch.cuda.synchronize()
        assert lay.status.item() == 0
        kmin, kmax = chunk_major_to_blocks(lay.kmin), chunk_major_to_blocks(lay.kmax)
        scores = lay.scores.cpu().numpy()
        tout, plan, cnt = lay.table.cpu().numpy(), lay.plan.cpu().numpy(), lay.plan_count.cpu().numpy()
        pool = bits(lay.pool)
        go, gl = out.cpu().numpy(), lse.cpu().numpy()
        qd_np = bits(qd)
        nbv = -(-L // 16)
        nc = nbv - W
        for s in range(w.S):
            b, h = divmod(s, w.Hkv)
            ref = opipe.run_segment(tiles_np[s], L, segment_queries(qd_np, b, h, w.G),
                                    qt_np[b, h * w.G:(h + 1) * w.G], table[s].tolist(), w.K, w.W, w.cap, scale)
            assert np.array_equal(kmin[s, :nbv], ref["kmin"][:nbv]), (t, s)
            assert np.array_equal(kmax[s, :nbv], ref["kmax"][:nbv]), (t, s)
            assert np.array_equal(scores[s, :nc].view(np.uint32), ref["scores"].view(np.uint32)), (t, s)
            assert tout[s].tolist() == ref["table_out"], (t, s)
            n = len(ref["plan"])
            assert int(cnt[s]) == n and [tuple(x) for x in plan[s, :n].tolist()] == ref["plan"], (t, s)
            assert np.array_equal(pool[s], ref["pool_after"]), (t, s)
            assert_attention_close(go[b, h * w.G:(h + 1) * w.G], ref["out"], gl[b, h * w.G:(h + 1) * w.G],
                                   ref["lse"])
            admitted += n
        table = lay.table.cpu()
    assert admitted > 0
