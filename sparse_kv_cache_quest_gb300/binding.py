"""Thin ctypes binding of liboasis.so (include/oasis.h).

Argument marshalling only: every function forwards to the C entry point of
the same name; torch tensors are passed as their data pointers, the stream
defaults to torch's current CUDA stream.  All arithmetic runs in the
library's kernels.  There is no fallback: if liboasis.so is missing or a
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liboasis.so")

OK, EINVAL, ECUDA = 0, -1, -2
STATUS_TABLE_RANGE, STATUS_TABLE_DUP, STATUS_NAN_SCORE = 1, 2, 4
STATUS_PLAN_RANGE, STATUS_SEQ_LEN, STATUS_TIMEOUT = 8, 16, 32

EXPORTS = (
    "oasis_strerror", "oasis_abi_version", "oasis_build_summary", "oasis_score_blocks", "oasis_score_blocks_tc",
    "oasis_select_topk_capped", "oasis_select_topk_capped_tc", "oasis_stage_blocks", "oasis_sparse_decode_attn",
    "oasis_attn_workspace_bytes", "oasis_sparse_decode_attn_ws", "oasis_sparse_decode_attn_noalloc",
    "oasis_sparse_decode_attn_tc",
)


class OasisError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} returned {code}: {text}")
        self.code = code


class XferT(ctypes.Structure):
    """oasis_xfer_t: one transfer of the plan (host block -> pool slot)."""
    _fields_ = [("src_block", ctypes.c_int32), ("dst_slot", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "oasis_strerror": (ctypes.c_char_p, [_I]),
    "oasis_abi_version": (_I, []),
    "oasis_build_summary": (_I, [_P, _I64, _I64, _I64, _I, _I, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P]),
    "oasis_score_blocks": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "oasis_score_blocks_tc": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P]),
    "oasis_select_topk_capped": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "oasis_select_topk_capped_tc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                        _P]),
    "oasis_stage_blocks": (_I, [_P, _I64, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P]),
    "oasis_sparse_decode_attn": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "oasis_attn_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "oasis_sparse_decode_attn_ws": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, ctypes.c_size_t, _P,
                                         _P]),
    "oasis_sparse_decode_attn_noalloc": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "oasis_sparse_decode_attn_tc": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
}


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liboasis.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int address or None, got {type(x)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, rc: int) -> int:
    if rc != OK:
        raise OasisError(fn, rc, load().oasis_strerror(rc).decode())
    return rc


def strerror(code: int) -> str:
    return load().oasis_strerror(code).decode()


def abi_version() -> int:
    return load().oasis_abi_version()


def oasis_build_summary(k, seg_stride, blk_stride, tok_stride, B, Hkv, D, seq_len, blk_begin, blk_count,
                        kmin, kmax, Nb_max, status=None, stream=None, wsum=None):
    return _check("oasis_build_summary", load().oasis_build_summary(
        _ptr(k), seg_stride, blk_stride, tok_stride, B, Hkv, D, _ptr(seq_len), blk_begin, blk_count,
        _ptr(kmin), _ptr(kmax), _ptr(wsum), Nb_max, _ptr(status), _stream(stream)))


def oasis_score_blocks(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status=None,
                       stream=None):
    return _check("oasis_score_blocks", load().oasis_score_blocks(
        _ptr(kmin), _ptr(kmax), Nb_max, _ptr(qdraft), B, Hkv, G, Nd, D, _ptr(seq_len), W, _ptr(scores),
        _ptr(status), _stream(stream)))


def oasis_score_blocks_tc(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, radius, status=None,
                          stream=None, wsum=None):
    return _check("oasis_score_blocks_tc", load().oasis_score_blocks_tc(
        _ptr(kmin), _ptr(kmax), _ptr(wsum), Nb_max, _ptr(qdraft), B, Hkv, G, Nd, D, _ptr(seq_len), W, _ptr(scores),
        _ptr(radius), _ptr(status), _stream(stream)))


def oasis_select_topk_capped(scores, Nb_max, seq_len, B, Hkv, K, W, cap, table_in, table_out, plan,
                             plan_count, status, stream=None):
    return _check("oasis_select_topk_capped", load().oasis_select_topk_capped(
        _ptr(scores), Nb_max, _ptr(seq_len), B, Hkv, K, W, cap, _ptr(table_in), _ptr(table_out), _ptr(plan),
        _ptr(plan_count), _ptr(status), _stream(stream)))


def oasis_select_topk_capped_tc(scores, radius, kmin, kmax, qdraft, G, Nd, D, Nb_max, seq_len, B, Hkv, K, W, cap,
                                table_in, table_out, plan, plan_count, status, stream=None):
    return _check("oasis_select_topk_capped_tc", load().oasis_select_topk_capped_tc(
        _ptr(scores), _ptr(radius), _ptr(kmin), _ptr(kmax), _ptr(qdraft), G, Nd, D, Nb_max, _ptr(seq_len), B, Hkv,
        K, W, cap, _ptr(table_in), _ptr(table_out), _ptr(plan), _ptr(plan_count), _ptr(status), _stream(stream)))


def oasis_stage_blocks(host_kv, host_seg_stride_bytes, host_nb, plan, plan_count, cap, B, Hkv, D, pool,
                       slots_per_seg, status, stream=None):
    return _check("oasis_stage_blocks", load().oasis_stage_blocks(
        _ptr(host_kv), host_seg_stride_bytes, host_nb, _ptr(plan), _ptr(plan_count), cap, B, Hkv, D,
        _ptr(pool), slots_per_seg, _ptr(status), _stream(stream)))


def oasis_sparse_decode_attn(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse=None,
                             status=None, stream=None):
    return _check("oasis_sparse_decode_attn", load().oasis_sparse_decode_attn(
        _ptr(q), _ptr(pool), _ptr(table), slots_per_seg, _ptr(seq_len), B, Hkv, G, D, float(scale),
        _ptr(out), _ptr(lse), _ptr(status), _stream(stream)))


def oasis_attn_workspace_bytes(B, Hkv, G, D, slots_per_seg) -> int:
    return int(load().oasis_attn_workspace_bytes(B, Hkv, G, D, slots_per_seg))


def oasis_sparse_decode_attn_ws(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse, ws,
                                ws_bytes, status=None, stream=None):
    return _check("oasis_sparse_decode_attn_ws", load().oasis_sparse_decode_attn_ws(
        _ptr(q), _ptr(pool), _ptr(table), slots_per_seg, _ptr(seq_len), B, Hkv, G, D, float(scale),
        _ptr(out), _ptr(lse), _ptr(ws), int(ws_bytes), _ptr(status), _stream(stream)))


def oasis_sparse_decode_attn_noalloc(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse=None,
                                     status=None, stream=None):
    return _check("oasis_sparse_decode_attn_noalloc", load().oasis_sparse_decode_attn_noalloc(
        _ptr(q), _ptr(pool), _ptr(table), slots_per_seg, _ptr(seq_len), B, Hkv, G, D, float(scale),
        _ptr(out), _ptr(lse), _ptr(status), _stream(stream)))


def oasis_sparse_decode_attn_tc(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse=None,
                                status=None, stream=None):
    return _check("oasis_sparse_decode_attn_tc", load().oasis_sparse_decode_attn_tc(
        _ptr(q), _ptr(pool), _ptr(table), slots_per_seg, _ptr(seq_len), B, Hkv, G, D, float(scale),
        _ptr(out), _ptr(lse), _ptr(status), _stream(stream)))


def attn_workspace(B, Hkv, G, D, slots_per_seg, device=None):
    """A zero-filled device workspace for oasis_sparse_decode_attn_ws (uint8 tensor)."""
    import torch
    n = oasis_attn_workspace_bytes(B, Hkv, G, D, slots_per_seg)
    if n == 0:
        raise ValueError("oasis_attn_workspace_bytes rejected the arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")
