"""Per-layer device state and one decode step, built on the C ABI.

This is orchestration only (buffers, streams, events, argument marshalling):
every step of the path runs in liboasis.so's kernels.

Step order, after the OasisKV paper review (xllm-io), §3 decode flow and
Fig. 8 (asynchronous prefetch pipeline): the foreground attends the true
query over the blocks resident now, while the background scores the blocks
with the draft queries and selects the next resident set; the transfer of the
admitted blocks starts once both are done (the slots it overwrites may still
be read by the attention of this step) and must finish before the next
step's attention.  Foreground and background run on separate CUDA streams
ordered by events ([XR] §5).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import binding as ob

BLOCK = 16


@dataclass
class LayerShape:
    B: int
    Hkv: int
    G: int
    D: int
    Nb_max: int
    K: int
    W: int
    cap: int
    Nd: int

    @property
    def S(self) -> int:
        return self.B * self.Hkv

    @property
    def Hq(self) -> int:
        return self.Hkv * self.G

    @property
    def slots(self) -> int:
        return self.K + self.W


class DecodeLayer:
    """Device buffers of one layer: summaries, scores, tables, plan, pool, outputs.

    balanced_attn: run the attention as the SM-balanced split with a workspace
    of this layer's own (oasis_sparse_decode_attn_ws) instead of the per-head
    cluster split (oasis_sparse_decode_attn).
    tc_attn: run the attention on the tcgen05 tensor cores
    (oasis_sparse_decode_attn_tc; d_h 128 only).
    scoring: "exact" - every score in the fixed-order fp32 arithmetic
    (oasis_score_blocks, then oasis_select_topk_capped); "tc" - tensor-core
    estimates with radii (oasis_score_blocks_tc), then the certified selection
    (oasis_select_topk_capped_tc), which recomputes the fixed-order scores the
    decisions need.  Both give the same tables and plans; with "tc" the scores
    buffer holds fixed-order values only for the recomputed blocks."""

    def __init__(self, shape: LayerShape, device="cuda", balanced_attn: bool = False, scoring: str = "exact",
                 tc_attn: bool = False):
        if balanced_attn and tc_attn:
            raise ValueError("balanced_attn and tc_attn are alternatives")
        self.tc_attn = tc_attn
        self.shape = sh = shape
        dev = torch.device(device)
        self.device = dev
        self.kmin = torch.zeros((sh.S, sh.D // 8, sh.Nb_max, 8), dtype=torch.bfloat16, device=dev)
        self.kmax = torch.zeros_like(self.kmin)
        self.scores = torch.zeros((sh.S, sh.Nb_max), dtype=torch.float32, device=dev)
        self.table = torch.full((sh.S, sh.slots), -1, dtype=torch.int32, device=dev)
        self.table_next = torch.full_like(self.table, -1)
        self.plan = torch.full((sh.S, max(sh.cap, 1), 2), -1, dtype=torch.int32, device=dev)
        self.plan_count = torch.zeros((sh.S,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.pool = torch.zeros((sh.S, sh.slots, 2, BLOCK, sh.D), dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros((sh.B, sh.Hq, sh.D), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((sh.B, sh.Hq), dtype=torch.float32, device=dev)
        self.scale = 1.0 / math.sqrt(sh.D)
        self.attn_ws = ob.attn_workspace(sh.B, sh.Hkv, sh.G, sh.D, sh.slots, device=dev) if balanced_attn else None
        if scoring not in ("exact", "tc"):
            raise ValueError(f"scoring must be 'exact' or 'tc', not {scoring!r}")
        self.scoring = scoring
        self.radius = torch.zeros_like(self.scores) if scoring == "tc" else None
        # per-block sums of the summary values on the wrong side of zero, kept by the
        # summary build for the tensor-core scoring's error bound
        self.wsum = torch.zeros_like(self.scores) if scoring == "tc" else None
        self._qdraft = None                   # the drafts the last score() call read (the tc selection rereads them)

    # -- individual steps ---------------------------------------------------
    def build_summary(self, keys, seq_len, blk_begin=0, blk_count=None, strides=None, stream=None):
        """keys: bf16 [S][n][16][D] (or a tile array [S][n][2][16][D] with strides) of blocks
        blk_begin .. blk_begin + n - 1."""
        sh = self.shape
        if strides is None:
            seg, blk, tok = keys.stride(0), keys.stride(1), keys.stride(-2)
        else:
            seg, blk, tok = strides
        n = keys.shape[1] if blk_count is None else blk_count
        ob.oasis_build_summary(keys, seg, blk, tok, sh.B, sh.Hkv, sh.D, seq_len, blk_begin, n,
                               self.kmin, self.kmax, sh.Nb_max, self.status, stream, wsum=self.wsum)

    def score(self, qdraft, seq_len, stream=None):
        sh = self.shape
        self._qdraft = qdraft
        if self.scoring == "tc":
            ob.oasis_score_blocks_tc(self.kmin, self.kmax, sh.Nb_max, qdraft, sh.B, sh.Hkv, sh.G, sh.Nd, sh.D,
                                     seq_len, sh.W, self.scores, self.radius, self.status, stream, wsum=self.wsum)
            return
        ob.oasis_score_blocks(self.kmin, self.kmax, sh.Nb_max, qdraft, sh.B, sh.Hkv, sh.G, sh.Nd, sh.D,
                              seq_len, sh.W, self.scores, self.status, stream)

    def select(self, seq_len, stream=None, qdraft=None):
        """qdraft: the drafts of the preceding score() call (the default); the
        tensor-core path recomputes the scores its decisions need from them."""
        sh = self.shape
        if self.scoring == "tc":
            qd = qdraft if qdraft is not None else self._qdraft
            if qd is None:
                raise RuntimeError("select() before score(): the tc selection needs the draft queries")
            ob.oasis_select_topk_capped_tc(self.scores, self.radius, self.kmin, self.kmax, qd, sh.G, sh.Nd, sh.D,
                                           sh.Nb_max, seq_len, sh.B, sh.Hkv, sh.K, sh.W, sh.cap, self.table,
                                           self.table_next, self.plan, self.plan_count, self.status, stream)
            return
        ob.oasis_select_topk_capped(self.scores, sh.Nb_max, seq_len, sh.B, sh.Hkv, sh.K, sh.W, sh.cap,
                                    self.table, self.table_next, self.plan, self.plan_count, self.status, stream)

    def stage(self, host_kv, host_seg_stride_bytes, host_nb, stream=None):
        sh = self.shape
        ob.oasis_stage_blocks(host_kv, host_seg_stride_bytes, host_nb, self.plan, self.plan_count, sh.cap,
                              sh.B, sh.Hkv, sh.D, self.pool, sh.slots, self.status, stream)

    def attend(self, q, seq_len, stream=None):
        sh = self.shape
        if self.attn_ws is not None:
            ob.oasis_sparse_decode_attn_ws(q, self.pool, self.table, sh.slots, seq_len, sh.B, sh.Hkv, sh.G, sh.D,
                                           self.scale, self.out, self.lse, self.attn_ws, self.attn_ws.numel(),
                                           self.status, stream)
            return
        fn = ob.oasis_sparse_decode_attn_tc if self.tc_attn else ob.oasis_sparse_decode_attn
        fn(q, self.pool, self.table, sh.slots, seq_len, sh.B, sh.Hkv, sh.G, sh.D, self.scale, self.out, self.lse,
           self.status, stream)

    def swap_tables(self):
        self.table, self.table_next = self.table_next, self.table

    # -- one decode step ----------------------------------------------------
    def step(self, q, qdraft, seq_len, host_kv, host_seg_stride_bytes, host_nb, new_keys=None,
             new_block: Optional[int] = None, streams=None, advance: bool = True, timers=None):
        """One decode step of this layer; returns (out, lse) of the attention.

        new_keys (optional): bf16 [S][1][16][D] keys of block ``new_block`` whose
        summary is refreshed first (the compressed-key update of a decode step).
        streams: (foreground, background, transfer) CUDA streams; the current
        stream for all three when None.  The caller's current stream is made
        to wait for the whole step.
        advance: make the new table current (False keeps the old table current,
        so repeated steps start from the same resident set).
        timers: optional dict; CUDA event pairs around the attention ("attn",
        foreground stream) and the scoring ("score", background stream) are
        appended to timers[name].
        """
        cur = torch.cuda.current_stream(self.device)
        fg, bg, xf = streams if streams is not None else (cur, cur, cur)
        start = torch.cuda.Event()
        start.record(cur)
        for s_ in (fg, bg, xf):
            s_.wait_event(start)
        if new_keys is not None:
            self.build_summary(new_keys, seq_len, blk_begin=new_block, blk_count=1, stream=bg)
        def timed(name, st, fn):
            if timers is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            timers.setdefault(name, []).append((a, b))

        timed("attn", fg, lambda: self.attend(q, seq_len, stream=fg))
        timed("score", bg, lambda: self.score(qdraft, seq_len, stream=bg))
        timed("select", bg, lambda: self.select(seq_len, stream=bg, qdraft=qdraft))
        e_fg, e_bg = torch.cuda.Event(), torch.cuda.Event()
        e_fg.record(fg)
        e_bg.record(bg)
        xf.wait_event(e_fg)
        xf.wait_event(e_bg)
        timed("stage", xf, lambda: self.stage(host_kv, host_seg_stride_bytes, host_nb, stream=xf))
        done = torch.cuda.Event()
        done.record(xf)
        cur.wait_event(done)
        if advance:
            self.swap_tables()
        return self.out, self.lse


class StepGraph:
    """One decode step of a DecodeLayer captured as a CUDA graph.

    The graph reads its inputs from static device buffers owned by this object
    (copy new values into ``q``, ``qdraft``, ``seq_len``, ``new_keys`` or, with
    host_io=True, into the pinned host staging tensors ``host_in``) and writes
    the layer's outputs; ``replay()`` runs the whole step - and with host_io,
    the host->device copies of the step's inputs and the device->host copies
    of its results (out, lse, new table, plan, plan counts into ``host_out``) -
    as one graph launch, without per-kernel launch overhead.  The step keeps
    the layer's current table (the new table is left in ``layer.table_next``).
    """

    def __init__(self, layer: DecodeLayer, q, qdraft, seq_len, host_kv, host_seg_stride_bytes, host_nb,
                 new_keys=None, new_block: Optional[int] = None, host_io: bool = False):
        dev = layer.device
        self.layer = layer
        self.q = q.detach().to(dev).clone()
        self.qdraft = qdraft.detach().to(dev).clone()
        self.seq_len = seq_len.detach().to(dev).clone()
        self.new_keys = new_keys.detach().to(dev).contiguous().clone() if new_keys is not None else None
        ins = [self.q, self.qdraft, self.seq_len] + ([self.new_keys] if self.new_keys is not None else [])
        outs = [layer.out, layer.lse, layer.table_next, layer.plan, layer.plan_count]
        self.host_in = [t.cpu().pin_memory() for t in ins] if host_io else []
        self.host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] if host_io else []
        self.streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        args = (host_kv, host_seg_stride_bytes, host_nb)

        def body():
            for d, h in zip(ins, self.host_in):
                d.copy_(h, non_blocking=True)
            layer.step(self.q, self.qdraft, self.seq_len, *args, new_keys=self.new_keys, new_block=new_block,
                       streams=self.streams, advance=False)
            for h, d in zip(self.host_out, outs):
                h.copy_(d, non_blocking=True)

        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()                                   # warm-up outside capture (lazy initialisation)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            body()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host_in)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.host_out)

    def replay(self):
        self.graph.replay()


def _arena(tensors, dev):
    """One uint8 device buffer holding copies of ``tensors`` (each at a 256-byte
    aligned offset) and typed views of it in the tensors' shapes."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    arena = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        v = arena[o:o + n].view(t.dtype).view(t.shape)
        v.copy_(t.detach())
        views.append(v)
    return arena, views


class DecodeStepGraph:
    """One decode step through several layers as one CUDA graph, pipelined
    across layers as in the asynchronous prefetch pipeline of the OasisKV paper
    review (xllm-io), §3 Fig. 8 and eq. (4): the foreground attends layer after
    layer on one stream; the background of layer l (summary update, scoring and
    selection on one stream, then staging) starts once the foreground has reached layer l
    (its draft queries exist) and overlaps the attention of the following
    layers; the staging of layer l waits for layer l's attention (it overwrites
    slots that attention reads) and must end before the next step, where the
    graph ends.

    Each layer gets static input buffers (q, qdraft, new_keys, packed in one
    device buffer per layer; seq_len is shared); with host_io=True the graph
    copies each layer's inputs from a pinned host buffer (``host_in[i]``, one
    copy) before that layer's work and each layer's results (out, lse, new
    table, plan, plan counts) back to pinned host memory (``host_out[i]``) once
    they exist, on two copy streams, so the copies overlap other layers'
    kernels.  share_host_inputs: all layers copy their inputs from one pinned
    host buffer (``host_in[0]``; the bytes moved are the same, the host memory
    held is one layer's).
    advance: after its staging, each layer's new table becomes its current
    table (a device copy of ``table_next`` into ``table``), so that successive
    replays are successive decode steps; without it the tables do not advance
    (the new tables stay in ``table_next``).
    n_bg: background streams, taken by the layers in turn; fg_priority: CUDA
    stream priority of the foreground stream (lower is higher; 0 = default);
    n_xf: staging streams, taken by the layers in turn.
    warmup: run the step once outside the capture first (the step then really
    runs: with advance, the tables move on by one step).
    """

    def __init__(self, layers, q, qdraft, seq_len, host_kv, host_seg_stride_bytes, host_nb, new_keys=None,
                 new_block: Optional[int] = None, host_io: bool = False, n_bg: int = 3, fg_priority: int = 0,
                 n_xf: int = 3, advance: bool = False, share_host_inputs: bool = False, warmup: bool = True):
        dev = layers[0].device
        self.layers = layers
        self.seq_len = seq_len.detach().to(dev).clone()
        # per layer, one contiguous device buffer holds that layer's inputs (q, qdraft,
        # new keys), so host I/O moves them with a single copy
        srcs = [q, qdraft] + ([new_keys] if new_keys is not None else [])
        self.in_dev, self.in_host, views = [], [], []
        for i, _ in enumerate(layers):
            arena, v = _arena(srcs, dev)
            self.in_dev.append(arena)
            views.append(v)
            if host_io and (i == 0 or not share_host_inputs):
                self.in_host.append(arena.cpu().pin_memory())
        self.q = [v[0] for v in views]
        self.qdraft = [v[1] for v in views]
        self.new_keys = [v[2] if new_keys is not None else None for v in views]
        outs = [[l.out, l.lse, l.table_next, l.plan, l.plan_count] for l in layers]
        self.host_in = self.in_host if host_io else None
        self.host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in x] for x in outs] \
            if host_io else None
        fg = torch.cuda.Stream(dev, priority=fg_priority)
        # staging streams taken by the layers in turn (three by default): the
        # staging of layer l+1 may start while layer l's still runs, hiding each
        # copy's start-up and tail behind its neighbours (the copies are bound by
        # the host link, and a chain of them on one stream sets the step's pace)
        xfs = [torch.cuda.Stream(dev) for _ in range(n_xf)]
        # host I/O on copy streams of its own, per layer, so that the copies of one
        # layer overlap the kernels of the others
        h2d, d2h = (torch.cuda.Stream(dev) for _ in range(2)) if host_io else (None, None)
        # background streams taken by the layers in turn (three by default): the
        # background of layer l+1 needs only the foreground to have passed layer
        # l, so it may start while layer l's scoring or selection still runs,
        # which hides each kernel's start-up and tail behind its neighbours
        bgs = [torch.cuda.Stream(dev) for _ in range(n_bg)]
        stage_args = (host_kv, host_seg_stride_bytes, host_nb)

        copy_streams = (h2d, d2h) if host_io else ()

        def body(cur):
            start = torch.cuda.Event()
            start.record(cur)
            for st in (fg, *xfs, *bgs, *copy_streams):
                st.wait_event(start)
            prev_fg = None
            for i, lay in enumerate(layers):
                bg = bgs[i % len(bgs)]
                xf = xfs[i % len(xfs)]
                if host_io:
                    with torch.cuda.stream(h2d):
                        self.in_dev[i].copy_(self.in_host[0 if share_host_inputs else i], non_blocking=True)
                    e_in = torch.cuda.Event()
                    e_in.record(h2d)
                    bg.wait_event(e_in)
                    fg.wait_event(e_in)
                if prev_fg is not None:
                    bg.wait_event(prev_fg)                     # the forward pass has reached layer i
                if new_keys is not None:
                    lay.build_summary(self.new_keys[i], self.seq_len, blk_begin=new_block, blk_count=1, stream=bg)
                lay.score(self.qdraft[i], self.seq_len, stream=bg)
                lay.select(self.seq_len, stream=bg, qdraft=self.qdraft[i])
                e_sel = torch.cuda.Event()
                e_sel.record(bg)
                lay.attend(self.q[i], self.seq_len, stream=fg)
                e_fg = torch.cuda.Event()
                e_fg.record(fg)
                prev_fg = e_fg
                xf.wait_event(e_sel)
                xf.wait_event(e_fg)
                lay.stage(*stage_args, stream=xf)
                if host_io:
                    d2h.wait_event(e_sel)
                    d2h.wait_event(e_fg)
                    with torch.cuda.stream(d2h):
                        for h, d in zip(self.host_out[i], outs[i]):
                            h.copy_(d, non_blocking=True)
                if advance:                                    # after this layer's attention and staging
                    with torch.cuda.stream(xf):
                        lay.table.copy_(lay.table_next, non_blocking=True)
            for st in (fg, *xfs, *bgs, *copy_streams):
                e = torch.cuda.Event()
                e.record(st)
                cur.wait_event(e)

        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        if warmup:
            with torch.cuda.stream(side):
                body(side)                               # warm-up outside capture
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            body(side)
        self.h2d_bytes = sum(t.numel() for t in self.in_dev) if host_io else 0
        self.d2h_bytes = sum(t.numel() * t.element_size() for x in (self.host_out or []) for t in x)

    def replay(self):
        self.graph.replay()
