"""Kernel-level parity: each C-ABI entry point against the oracle, bit-exact for
summaries, scores, tables and plans, within tolerance for attention; edge
cases (ragged lengths, signed zeros, ties, empty slots, invalid tables)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN, bits, from_f32
from helpers import assert_attention_close, chunk_major_to_blocks, default_scale
from oracle import attention as oattn
from oracle import score as oscore
from oracle import select as osel
from oracle import stage as ostage
from oracle import summary as osum
import sparse_kv_cache_quest_gb300 as okv

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    okv.load()


def _bf16_rand(rng, shape, zeros=0.0, scale=1.0):
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = (v.view(np.uint32) >> 16).astype(np.uint16)
    if zeros:
        m = rng.random(shape)
        u[m < zeros / 2] = 0x0000
        u[(m >= zeros / 2) & (m < zeros)] = 0x8000
    return u


def _dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(u16.astype(np.int16)).view(torch.bfloat16).to(DEV)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ------------------------------------------------------------------ summaries

@pytest.mark.parametrize("D", [64, 128])
def test_summary_full_build_ragged_and_signed_zeros(D):
    rng = np.random.default_rng(D)
    B, Hkv, Nb = 2, 3, 37
    keys = _bf16_rand(rng, (B * Hkv, Nb, 16, D), zeros=0.3)
    lens = np.array([16 * Nb - 5, 16 * 20 + 1], dtype=np.int32)
    kmin = torch.full((B * Hkv, D // 8, Nb, 8), 7.0, dtype=torch.bfloat16, device=DEV)
    kmax = kmin.clone()
    st = _status()
    kd = _dev_bf16(keys)
    okv.oasis_build_summary(kd, Nb * 16 * D, 16 * D, D, B, Hkv, D, torch.from_numpy(lens).to(DEV), 0, Nb,
                            kmin, kmax, Nb, st)
    torch.cuda.synchronize()
    gmn, gmx = chunk_major_to_blocks(kmin), chunk_major_to_blocks(kmax)
    sentinel = bits(torch.tensor([7.0], dtype=torch.bfloat16))[0]
    for s in range(B * Hkv):
        L = int(lens[s // Hkv])
        mn, mx, ids = osum.block_summary(keys[s], L)
        assert np.array_equal(gmn[s, :len(ids)], mn) and np.array_equal(gmx[s, :len(ids)], mx)
        assert np.all(gmn[s, len(ids):] == sentinel)
    assert st.item() == 0


def test_summary_update_range_from_tile_layout():
    rng = np.random.default_rng(9)
    B, Hkv, D, Nb = 1, 2, 128, 10
    tiles = _bf16_rand(rng, (B * Hkv, Nb, 2, 16, D), zeros=0.1)
    lens = torch.tensor([16 * 7 + 3], dtype=torch.int32, device=DEV)
    kmin = torch.zeros((B * Hkv, D // 8, Nb, 8), dtype=torch.bfloat16, device=DEV)
    kmax = torch.zeros_like(kmin)
    td = _dev_bf16(tiles)
    # blocks 5..8 from a view that starts at block 5 (block 8 has no valid token)
    view = td[:, 5:]
    okv.oasis_build_summary(view, view.stride(0), view.stride(1), view.stride(3), B, Hkv, D, lens, 5, 4,
                            kmin, kmax, Nb, None)
    torch.cuda.synchronize()
    gmn, gmx = chunk_major_to_blocks(kmin), chunk_major_to_blocks(kmax)
    for s in range(B * Hkv):
        mn, mx, ids = osum.block_summary(tiles[s, :, 0], 16 * 7 + 3, blocks=[5, 6, 7, 8])
        assert ids == [5, 6, 7]
        assert np.array_equal(gmn[s, 5:8], mn) and np.array_equal(gmx[s, 5:8], mx)
        assert np.all(gmn[s, :5] == 0) and np.all(gmn[s, 8:] == 0)


# ------------------------------------------------------------------ scores

def _random_summaries(rng, S, Nb, D):
    a = _bf16_rand(rng, (S, Nb, D), zeros=0.05)
    b = _bf16_rand(rng, (S, Nb, D), zeros=0.05)
    fa, fb = from_bits(a), from_bits(b)
    lo = np.where(fa <= fb, a, b)
    hi = np.where(fa <= fb, b, a)
    return lo, hi


def from_bits(u):
    return (u.astype(np.uint32) << 16).view(np.float32)


def _to_chunk_major(x):  # [S][Nb][D] uint16 -> device [S][D/8][Nb][8]
    S, Nb, D = x.shape
    return _dev_bf16(np.ascontiguousarray(x.reshape(S, Nb, D // 8, 8).transpose(0, 2, 1, 3)))


@pytest.mark.parametrize("D,G,Nd,W", [(128, 4, 3, 0), (64, 2, 1, 0), (128, 1, 1, 3), (128, 16, 4, 0),
                                      (64, 3, 2, 2), (128, 16, 1, 0), (128, 5, 3, 1), (128, 8, 3, 0),
                                      (128, 10, 4, 1), (64, 13, 1, 2), (64, 16, 4, 0)])
def test_scores_bit_exact(D, G, Nd, W):
    rng = np.random.default_rng(100 + D + G * 7 + Nd)
    B, Hkv, Nb = 2, 2, 700
    S = B * Hkv
    lo, hi = _random_summaries(rng, S, Nb, D)
    qd = _bf16_rand(rng, (B, Nd, Hkv * G, D), zeros=0.05)
    lens = np.array([16 * Nb - 9, 16 * 300 + 4], dtype=np.int32)
    scores = torch.full((S, Nb), -123.0, dtype=torch.float32, device=DEV)
    st = _status()
    okv.oasis_score_blocks(_to_chunk_major(lo), _to_chunk_major(hi), Nb, _dev_bf16(qd), B, Hkv, G, Nd, D,
                           torch.from_numpy(lens).to(DEV), W, scores, st)
    torch.cuda.synchronize()
    got = scores.cpu().numpy()
    for s in range(S):
        b, h = divmod(s, Hkv)
        nc = -(-int(lens[b]) // 16) - W
        ref = oscore.score_blocks(lo[s, :nc], hi[s, :nc], oscore.segment_queries(qd, b, h, G))
        assert np.array_equal(got[s, :nc].view(np.uint32), ref.view(np.uint32)), f"segment {s}"
        assert np.all(got[s, nc:] == -123.0)
    assert st.item() == 0


def test_scores_configuration_changes_keep_launching():
    """Launches of one scoring kernel with more, then less, then more dynamic
    shared memory (query groups of different widths): each must still launch and
    match the oracle, i.e. the kernel's shared-memory limit never drops below a
    size an earlier configuration needs."""
    rng = np.random.default_rng(77)
    B, Hkv, Nb, D = 1, 2, 200, 128
    S = B * Hkv
    lo, hi = _random_summaries(rng, S, Nb, D)
    lens = torch.tensor([16 * Nb], dtype=torch.int32, device=DEV)
    for G, Nd in [(10, 4), (16, 4), (10, 4), (6, 3), (16, 4)]:
        qd = _bf16_rand(rng, (B, Nd, Hkv * G, D))
        scores = torch.zeros((S, Nb), dtype=torch.float32, device=DEV)
        okv.oasis_score_blocks(_to_chunk_major(lo), _to_chunk_major(hi), Nb, _dev_bf16(qd), B, Hkv, G, Nd, D, lens,
                               0, scores, None)
        torch.cuda.synchronize()
        got = scores.cpu().numpy()
        for s in range(S):
            ref = oscore.score_blocks(lo[s], hi[s], oscore.segment_queries(qd, 0, s, G))
            assert np.array_equal(got[s].view(np.uint32), ref.view(np.uint32)), (G, Nd, s)


def test_scores_golden_toy_and_order_case():
    with open(os.path.join(GOLDEN, "score_toy.json")) as f:
        g = json.load(f)
    D = 64
    kmin = np.zeros((1, 2, D), np.float32)
    kmax = np.zeros((1, 2, D), np.float32)
    kmin[0, :, :4] = g["kmin"]
    kmax[0, :, :4] = g["kmax"]
    q = np.zeros((1, 2, 1, D), np.float32)            # B=1, Nd=2 drafts, Hq=1 (G=1)
    q[0, :, 0, :4] = g["queries"]
    scores = torch.zeros((1, 2), dtype=torch.float32, device=DEV)
    lens = torch.tensor([32], dtype=torch.int32, device=DEV)
    okv.oasis_score_blocks(_to_chunk_major(from_f32(kmin)), _to_chunk_major(from_f32(kmax)), 2,
                           _dev_bf16(from_f32(q)), 1, 1, 1, 2, D, lens, 0, scores, None)
    torch.cuda.synchronize()
    assert scores.cpu().tolist()[0] == g["expected_scores"]
    c = g["order_case"]
    k = np.zeros((1, 1, D), np.float32)
    k[0, 0, :4] = c["k"]
    q1 = np.zeros((1, 1, 1, D), np.float32)
    q1[0, 0, 0, :4] = c["query"]
    sc = torch.zeros((1, 1), dtype=torch.float32, device=DEV)
    okv.oasis_score_blocks(_to_chunk_major(from_f32(k)), _to_chunk_major(from_f32(k)), 1,
                           _dev_bf16(from_f32(q1)), 1, 1, 1, 1, D, torch.tensor([16], dtype=torch.int32,
                                                                                device=DEV), 0, sc, None)
    torch.cuda.synchronize()
    assert sc.item() == c["expected_score"]


# ------------------------------------------------------------------ selection

def _select_gpu(scores_rows, tables, lens, Nb_max, K, W, cap, Hkv=1):
    S = len(tables)
    sc = torch.full((S, Nb_max), float("nan"), dtype=torch.float32)
    for s, row in enumerate(scores_rows):
        sc[s, :len(row)] = torch.as_tensor(np.asarray(row, dtype=np.float32))
    tin = torch.as_tensor(np.asarray(tables, dtype=np.int32)).to(DEV)
    tout = torch.full_like(tin, -7)
    plan = torch.full((S, max(cap, 1), 2), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((S,), -7, dtype=torch.int32, device=DEV)
    st = _status()
    okv.oasis_select_topk_capped(sc.to(DEV), Nb_max, torch.as_tensor(np.asarray(lens, np.int32)).to(DEV),
                                 S // Hkv, Hkv, K, W, cap, tin, tout, plan, cnt, st)
    torch.cuda.synchronize()
    return tout.cpu().numpy(), plan.cpu().numpy(), cnt.cpu().numpy(), st.item()


def _golden_select_cases():
    with open(os.path.join(GOLDEN, "select_toy.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_select_cases(), ids=lambda c: c["name"])
def test_select_golden_cases(case):
    nc = len(case["scores"])
    W = case["W"]
    tout, plan, cnt, st = _select_gpu([case["scores"]], [case["table_in"]], [16 * (nc + W)], nc + W + 3,
                                      case["K"], W, case["C"])
    assert tout[0].tolist() == case["table_out"]
    n = int(cnt[0])
    assert plan[0, :n].tolist() == case["plan"]
    assert np.all(plan[0, n:case["C"]] == -1)
    assert st == case["status"]


@pytest.mark.parametrize("K,W,cap,Nb_max", [(128, 0, 7, 3000), (128, 4, 7, 3000), (64, 0, 0, 900),
                                            (32, 2, 32, 900), (200, 0, 13, 180), (1024, 0, 51, 4000)])
def test_select_random_bit_exact(K, W, cap, Nb_max):
    rng = np.random.default_rng(K * 7 + cap + W)
    B, Hkv = 2, 4
    S = B * Hkv
    lens = [16 * Nb_max - 11, max(0, 16 * (Nb_max // 2) + 3)]
    rows, tables, refs = [], [], []
    for s in range(S):
        L = lens[s // Hkv]
        nc = max(0, -(-L // 16) - W)
        row = rng.integers(-40, 40, nc).astype(np.float32) * 0.5      # many ties
        row[rng.random(nc) < 0.05] = -0.0
        resident = list(rng.choice(nc, size=min(K, nc), replace=False)) if nc else []
        resident = [int(x) if rng.random() > 0.1 else -1 for x in resident]
        resident += [-1] * (K - len(resident))
        table = resident + list(range(nc, nc + W))
        rows.append(row)
        tables.append(table)
        refs.append(osel.select_topk_capped(row, table, K, W, cap))
    tout, plan, cnt, st = _select_gpu(rows, tables, lens, Nb_max, K, W, cap, Hkv)
    for s in range(S):
        t_ref, p_ref, st_ref = refs[s]
        assert tout[s].tolist() == t_ref, f"segment {s}"
        assert int(cnt[s]) == len(p_ref)
        assert [tuple(x) for x in plan[s, :len(p_ref)].tolist()] == p_ref
        assert np.all(plan[s, len(p_ref):cap] == -1)
    assert st == 0


def test_select_invalid_tables_and_nan():
    K, W, cap, Nb = 4, 0, 2, 16
    rows = [np.arange(10, dtype=np.float32)] * 3
    tables = [[1, 1, 2, 3], [1, 12, 2, 3], [0, 1, 2, 3]]
    rows = [rows[0], rows[1], np.array([1, np.nan, 3, 4, 5, 6, 7, 8, 9, 10], np.float32)]
    tout, plan, cnt, st = _select_gpu(rows, tables, [160, 160, 160], Nb, K, W, cap, Hkv=3)
    assert tout[0].tolist() == [1, 1, 2, 3] and cnt[0] == 0
    assert tout[1].tolist() == [1, 12, 2, 3] and cnt[1] == 0
    t_ref, p_ref, st_ref = osel.select_topk_capped(rows[2], tables[2], K, W, cap)
    assert tout[2].tolist() == t_ref and int(cnt[2]) == len(p_ref)
    assert st == osel.STATUS_TABLE_DUP | osel.STATUS_TABLE_RANGE | osel.STATUS_NAN_SCORE


def test_select_in_place_and_empty_sequence():
    K, W, cap, Nb = 8, 0, 3, 64
    rows = [np.linspace(0, 1, 64, dtype=np.float32), np.zeros(0, np.float32)]
    tables = [[5, -1, 9, -1, -1, 40, -1, 2], [-1] * 8]
    sc = torch.zeros((2, Nb), dtype=torch.float32)
    sc[0] = torch.from_numpy(rows[0])
    t = torch.tensor(tables, dtype=torch.int32, device=DEV)
    plan = torch.zeros((2, cap, 2), dtype=torch.int32, device=DEV)
    cnt = torch.zeros(2, dtype=torch.int32, device=DEV)
    st = _status()
    okv.oasis_select_topk_capped(sc.to(DEV), Nb, torch.tensor([1024, 0], dtype=torch.int32, device=DEV), 2, 1,
                                 K, W, cap, t, t, plan, cnt, st)
    torch.cuda.synchronize()
    ref = osel.select_topk_capped(rows[0], tables[0], K, W, cap)
    assert t[0].tolist() == ref[0] and t[1].tolist() == [-1] * 8 and cnt.tolist() == [len(ref[1]), 0]


# ------------------------------------------------------------------ staging

def test_stage_copies_exactly_the_plan():
    rng = np.random.default_rng(21)
    B, Hkv, D, Nb, slots, cap = 2, 2, 128, 50, 12, 5
    S = B * Hkv
    host = torch.from_numpy(rng.integers(-30000, 30000, (S, Nb, 2, 16, D), dtype=np.int16)).pin_memory()
    pool0 = torch.from_numpy(rng.integers(-30000, 30000, (S, slots, 2, 16, D), dtype=np.int16))
    pool = pool0.to(DEV).view(torch.bfloat16)
    plans = [[(3, 0), (49, 11), (7, 4)], [], [(0, 5), (1, 6), (2, 7), (3, 8), (4, 9)], [(60, 1), (2, 12)]]
    plan = torch.full((S, cap, 2), -1, dtype=torch.int32)
    cnt = torch.zeros(S, dtype=torch.int32)
    for s, p in enumerate(plans):
        cnt[s] = len(p)
        for i, e in enumerate(p):
            plan[s, i] = torch.tensor(e)
    st = _status()
    okv.oasis_stage_blocks(host, host[0].numel() * 2, Nb, plan.to(DEV), cnt.to(DEV), cap, B, Hkv, D, pool,
                           slots, st)
    torch.cuda.synchronize()
    got = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    for s, p in enumerate(plans):
        ref, rst = ostage.stage_blocks(host[s].numpy().view(np.uint16), p, pool0[s].numpy().view(np.uint16))
        assert np.array_equal(got[s], ref)
    assert st.item() == osel.STATUS_PLAN_RANGE


# ------------------------------------------------------------------ attention

@pytest.mark.parametrize("D,G", [(128, 4), (64, 8), (128, 1)])
def test_attention_one_cta_of_8_warps(D, G):
    """Between half the SMs and all of them in segments (here 100 segments, or
    the SM count if smaller), the attention runs one 8-warp CTA per segment;
    ragged slot lists, empty slots and a partial last block as elsewhere."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hkv = 4, max(1, min(sms, 100)) // 4
    S = B * Hkv
    rng = np.random.default_rng(700 + D + G)
    Nb, slots = 64, 21
    lens = np.array([16 * Nb - 3, 16 * 40 + 7, 16 * Nb, 5], dtype=np.int32)
    tiles = _bf16_rand(rng, (S, Nb, 2, 16, D))
    q = _bf16_rand(rng, (B, Hkv * G, D))
    tables = np.full((S, slots), -1, np.int32)
    for s in range(S):
        blocks = rng.choice(Nb, size=slots, replace=False)
        tables[s] = np.where(rng.random(slots) > 0.1, blocks, -1)
    pool = np.zeros((S, slots, 2, 16, D), np.uint16)
    for s in range(S):
        for i, blk in enumerate(tables[s]):
            if blk >= 0:
                pool[s, i] = tiles[s, blk]
    out = torch.full((B, Hkv * G, D), 9.0, dtype=torch.float32, device=DEV)
    lse = torch.zeros((B, Hkv * G), dtype=torch.float32, device=DEV)
    scale = default_scale(D)
    st = _status()
    okv.oasis_sparse_decode_attn(_dev_bf16(q), _dev_bf16(pool), torch.from_numpy(tables).to(DEV), slots,
                                 torch.from_numpy(lens).to(DEV), B, Hkv, G, D, scale, out, lse, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for s in range(S):
        b, h = divmod(s, Hkv)
        ro, rl = oattn.sparse_decode_attention(q[b, h * G:(h + 1) * G], pool[s], tables[s], int(lens[b]), scale)
        assert_attention_close(go[b, h * G:(h + 1) * G], ro, gl[b, h * G:(h + 1) * G], rl)


@pytest.mark.parametrize("mode", ["cluster", "ws", "tc"])
# G > 8 runs the head-split kernel: (64, 12) its d_h 64 form, (128, 9) a second half
# with one head, (128, 16, 3) slot partitions left empty.  The tcgen05 kernel (d_h
# 128 only) splits the 6 segments over clusters of 4 CTAs (3 at 3 slots, 1 at one
# slot), and its tiles of 8 slots end ragged at 5, 33, 37 and 3 listed slots.
@pytest.mark.parametrize("D,G,slots", [(128, 4, 128), (64, 2, 37), (128, 1, 5), (128, 8, 64), (128, 16, 128),
                                       (64, 5, 20), (128, 3, 1), (64, 12, 40), (128, 9, 33), (128, 16, 3)])
def test_attention_within_tolerance(D, G, slots, mode):
    if mode == "tc" and D != 128:
        pytest.skip("the tcgen05 kernel takes d_h 128")
    ws = mode == "ws"
    rng = np.random.default_rng(D + G * 13 + slots)
    B, Hkv, Nb = 2, 3, 300
    S = B * Hkv
    lens = np.array([16 * Nb - 7, 16 * 150 + 9], dtype=np.int32)
    tiles = _bf16_rand(rng, (S, Nb, 2, 16, D))
    q = _bf16_rand(rng, (B, Hkv * G, D))
    tables = np.full((S, slots), -1, np.int32)
    for s in range(S):
        nb_valid = -(-int(lens[s // Hkv]) // 16)
        blocks = rng.choice(Nb, size=slots, replace=False)          # some beyond the sequence
        keep = rng.random(slots) > 0.15
        tables[s] = np.where(keep, blocks, -1)
        if s == 1:
            tables[s] = -1                                          # nothing resident
        if s == 2:
            tables[s, 0] = nb_valid - 1                             # the partial last block
    pool = np.zeros((S, slots, 2, 16, D), np.uint16)
    for s in range(S):
        for i, blk in enumerate(tables[s]):
            if blk >= 0:
                pool[s, i] = tiles[s, blk]
    out = torch.full((B, Hkv * G, D), 9.0, dtype=torch.float32, device=DEV)
    lse = torch.zeros((B, Hkv * G), dtype=torch.float32, device=DEV)
    scale = default_scale(D)
    args = (_dev_bf16(q), _dev_bf16(pool), torch.from_numpy(tables).to(DEV), slots, torch.from_numpy(lens).to(DEV),
            B, Hkv, G, D, scale, out, lse)
    st = _status()
    if ws:
        # the balanced split: two calls in a row on one workspace (its counters must come back to zero)
        work = okv.attn_workspace(B, Hkv, G, D, slots, device=DEV)
        okv.oasis_sparse_decode_attn_ws(*args, work, work.numel(), st)
        torch.cuda.synchronize()
        first = out.clone()
        out.fill_(9.0)
        okv.oasis_sparse_decode_attn_ws(*args, work, work.numel(), st)
        torch.cuda.synchronize()
        assert torch.equal(out, first)
        counters = work[-4 * S:].view(torch.int32)
        assert int(counters.abs().sum()) == 0
    elif mode == "tc":
        okv.oasis_sparse_decode_attn_tc(*args, st)
    else:
        okv.oasis_sparse_decode_attn(*args, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for s in range(S):
        b, h = divmod(s, Hkv)
        ro, rl = oattn.sparse_decode_attention(q[b, h * G:(h + 1) * G], pool[s], tables[s], int(lens[b]), scale)
        assert_attention_close(go[b, h * G:(h + 1) * G], ro, gl[b, h * G:(h + 1) * G], rl)
