"""Seeded random shapes against the oracle: scoring and selection bit for bit,
attention within tolerance.  Each case draws its own dimensions (head size,
group size, drafts, window, capacity, slots, cap) and ragged sequence
lengths, including empty sequences and lengths that leave no candidate, so the
launch geometry of every kernel (units per warp, phases of a scoring CTA,
cluster size and per-rank merge share of the attention) varies from case to
case."""
import numpy as np
import pytest
import torch

from helpers import assert_attention_close, default_scale
from oracle import attention as oattn
from oracle import score as oscore
from oracle import select as osel
import sparse_kv_cache_quest_gb300 as okv
from test_gpu_kernels import _bf16_rand, _dev_bf16, _random_summaries, _select_gpu, _status, _to_chunk_major

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    okv.load()


def _lengths(rng, B, Nb):
    lens = rng.integers(0, 16 * Nb + 1, B)
    if B > 1:
        lens[rng.integers(B)] = rng.choice([0, 1, 16 * Nb, 16 * Nb - 1])  # an edge in every case
    return lens.astype(np.int32)


@pytest.mark.parametrize("seed", range(16))
def test_scores_random_shapes(seed):
    rng = np.random.default_rng(7000 + seed)
    D = int(rng.choice([64, 128]))
    G = int(rng.integers(1, 17))
    Nd = int(rng.integers(1, min(4, 64 // G) + 1))
    B, Hkv = int(rng.integers(1, 4)), int(rng.integers(1, 6))
    Nb, W = int(rng.integers(1, 400)), int(rng.integers(0, 4))
    S = B * Hkv
    lo, hi = _random_summaries(rng, S, Nb, D)
    qd = _bf16_rand(rng, (B, Nd, Hkv * G, D), zeros=0.05)
    lens = _lengths(rng, B, Nb)
    scores = torch.full((S, Nb), -123.0, dtype=torch.float32, device=DEV)
    st = _status()
    okv.oasis_score_blocks(_to_chunk_major(lo), _to_chunk_major(hi), Nb, _dev_bf16(qd), B, Hkv, G, Nd, D,
                           torch.from_numpy(lens).to(DEV), W, scores, st)
    torch.cuda.synchronize()
    got = scores.cpu().numpy()
    for s in range(S):
        b, h = divmod(s, Hkv)
        nc = max(0, -(-int(lens[b]) // 16) - W)
        ref = oscore.score_blocks(lo[s, :nc], hi[s, :nc], oscore.segment_queries(qd, b, h, G))
        assert np.array_equal(got[s, :nc].view(np.uint32), ref.view(np.uint32)), f"segment {s}"
        assert np.all(got[s, nc:] == -123.0)
    assert st.item() == 0


@pytest.mark.parametrize("seed", range(12))
def test_select_random_shapes(seed):
    rng = np.random.default_rng(8000 + seed)
    K, W = int(rng.integers(1, 97)), int(rng.integers(0, 4))
    cap = int(rng.integers(0, K + 1))
    Nb_max = int(rng.integers(K + W + 1, 600))
    B, Hkv = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    S = B * Hkv
    lens = _lengths(rng, B, Nb_max)
    rows, tables, refs = [], [], []
    for s in range(S):
        nc = max(0, -(-int(lens[s // Hkv]) // 16) - W)
        row = rng.integers(-30, 30, nc).astype(np.float32) * 0.25          # ties
        row[rng.random(nc) < 0.05] = -0.0
        resident = [int(x) for x in rng.choice(nc, size=min(K, nc), replace=False)] if nc else []
        resident = [x if rng.random() > 0.2 else -1 for x in resident] + [-1] * (K - len(resident))
        rng.shuffle(resident)
        table = resident + list(range(nc, nc + W))
        rows.append(row)
        tables.append(table)
        refs.append(osel.select_topk_capped(row, table, K, W, cap))
    tout, plan, cnt, st = _select_gpu(rows, tables, lens, Nb_max, K, W, cap, Hkv)
    for s in range(S):
        t_ref, p_ref, _ = refs[s]
        assert tout[s].tolist() == t_ref, f"segment {s}"
        assert int(cnt[s]) == len(p_ref)
        assert [tuple(x) for x in plan[s, :len(p_ref)].tolist()] == p_ref
        assert np.all(plan[s, len(p_ref):cap] == -1)
    assert st == 0


@pytest.mark.parametrize("seed", range(12))
def test_attention_random_shapes(seed):
    rng = np.random.default_rng(9000 + seed)
    D = int(rng.choice([64, 128]))
    G = int(rng.integers(1, 17))
    slots = int(rng.integers(1, 49))
    B, Hkv = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    Nb = int(rng.integers(slots, 200))
    S = B * Hkv
    lens = _lengths(rng, B, Nb)
    q = _bf16_rand(rng, (B, Hkv * G, D))
    pool = _bf16_rand(rng, (S, slots, 2, 16, D))
    tables = np.full((S, slots), -1, np.int32)
    for s in range(S):
        blocks = rng.choice(Nb, size=slots, replace=False)      # some beyond the sequence
        tables[s] = np.where(rng.random(slots) > 0.2, blocks, -1)
    out = torch.full((B, Hkv * G, D), 9.0, dtype=torch.float32, device=DEV)
    lse = torch.zeros((B, Hkv * G), dtype=torch.float32, device=DEV)
    scale = default_scale(D)
    args = (_dev_bf16(q), _dev_bf16(pool), torch.from_numpy(tables).to(DEV), slots, torch.from_numpy(lens).to(DEV),
            B, Hkv, G, D, scale, out, lse)
    st = _status()
    if seed % 2:
        work = okv.attn_workspace(B, Hkv, G, D, slots, device=DEV)
        okv.oasis_sparse_decode_attn_ws(*args, work, work.numel(), st)
    else:
        okv.oasis_sparse_decode_attn(*args, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    if D == 128:  # the tcgen05 kernel on the same shape must agree with the oracle as well
        out_tc, lse_tc = torch.full_like(out, 9.0), torch.zeros_like(lse)
        okv.oasis_sparse_decode_attn_tc(*args[:10], out_tc, lse_tc, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        gt, glt = out_tc.cpu().numpy(), lse_tc.cpu().numpy()
        for s in range(S):
            b, h = divmod(s, Hkv)
            ro, rl = oattn.sparse_decode_attention(q[b, h * G:(h + 1) * G], pool[s], tables[s], int(lens[b]), scale)
            assert_attention_close(gt[b, h * G:(h + 1) * G], ro, glt[b, h * G:(h + 1) * G], rl)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for s in range(S):
        b, h = divmod(s, Hkv)
        ro, rl = oattn.sparse_decode_attention(q[b, h * G:(h + 1) * G], pool[s], tables[s], int(lens[b]), scale)
        assert_attention_close(go[b, h * G:(h + 1) * G], ro, gl[b, h * G:(h + 1) * G], rl)
