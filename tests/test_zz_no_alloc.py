"""The no-allocation attention entry point (scratch in a static device array)
against the workspace entry point it wraps: same shapes, two calls in a row of
each, bit-identical outputs, and the oracle's tolerance.  Collected last, and
passes alone as well as after the other tests (the scratch is shared by the
process, its counters are cleared by every call)."""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import assert_attention_close, default_scale
from oracle import attention as oattn
import sparse_kv_cache_quest_gb300 as okv
from sparse_kv_cache_quest_gb300 import binding as ob

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(rng, B, Hkv, G, D, slots, Nb):
    S = B * Hkv
    lens = np.array([16 * Nb - 5 - 7 * b for b in range(B)], dtype=np.int32)
    q = torch.randn((B, Hkv * G, D), generator=rng).to(torch.bfloat16)
    tiles = torch.randn((S, Nb, 2, 16, D), generator=rng).to(torch.bfloat16)
    table = torch.stack([torch.randperm(Nb, generator=rng)[:slots] for _ in range(S)]).to(torch.int32)
    table[torch.rand((S, slots), generator=rng) < 0.1] = -1
    pool = tiles[torch.arange(S)[:, None], table.long().clamp(min=0)]
    pool[table < 0] = 0
    return lens, q, pool, table


@pytest.mark.parametrize("B,Hkv,G,D,slots,Nb", [(8, 8, 4, 128, 128, 256), (2, 3, 16, 128, 37, 64),
                                                (1, 2, 2, 64, 8, 16), (4, 4, 5, 64, 300, 320)])
def test_noalloc_matches_workspace_entry(B, Hkv, G, D, slots, Nb):
    okv.load()
    rng = torch.Generator().manual_seed(B * 1000 + slots)
    lens, q, pool, table = _case(rng, B, Hkv, G, D, slots, Nb)
    args = (q.to(DEV), pool.to(DEV), table.to(DEV), slots, torch.from_numpy(lens).to(DEV), B, Hkv, G, D,
            default_scale(D))
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    ws = okv.attn_workspace(B, Hkv, G, D, slots, device=DEV)
    outs = []
    for call in range(2):
        o1 = torch.full((B, Hkv * G, D), 7.0, device=DEV)
        l1 = torch.zeros((B, Hkv * G), device=DEV)
        okv.oasis_sparse_decode_attn_noalloc(*args, o1, l1, st)
        o2 = torch.full_like(o1, 5.0)
        l2 = torch.zeros_like(l1)
        okv.oasis_sparse_decode_attn_ws(*args, o2, l2, ws, ws.numel(), st)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        outs.append((o1, l1))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert st.item() == 0
    go, gl = outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy()
    qn, pn, tn = bits(q), bits(pool), table.numpy()
    for s in (0, B * Hkv - 1):
        b, h = divmod(s, Hkv)
        ro, rl = oattn.sparse_decode_attention(qn[b, h * G:(h + 1) * G], pn[s], tn[s], int(lens[b]),
                                               default_scale(D))
        assert_attention_close(go[b, h * G:(h + 1) * G], ro, gl[b, h * G:(h + 1) * G], rl)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    okv.load()
    # 16 query heads per KV head, D = 128, 2^20 slot tiles: the workspace needs more than 8 MiB
    B, Hkv, G, D, slots = 64, 8, 16, 128, 2048
    assert okv.oasis_attn_workspace_bytes(B, Hkv, G, D, slots) > (8 << 20)
    # real buffers of the shape's sizes, every table entry empty: were the host
    # check to let the call through, the kernel would load no tile and write zeros
    q = torch.zeros((B, Hkv * G, D), dtype=torch.bfloat16, device=DEV)
    table = torch.full((B * Hkv, slots), -1, dtype=torch.int32, device=DEV)
    pool = torch.zeros((1, 1, 2, 16, D), dtype=torch.bfloat16, device=DEV)
    lens = torch.full((B,), 16 * slots, dtype=torch.int32, device=DEV)
    out = torch.empty((B, Hkv * G, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, Hkv * G), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    with pytest.raises(ob.OasisError) as e:
        okv.oasis_sparse_decode_attn_noalloc(q, pool, table, slots, lens, B, Hkv, G, D, 0.1, out, lse, st)
    assert e.value.code == ob.EINVAL
    torch.cuda.synchronize()
    assert st.item() == 0
