"""GB300-native lookahead sparse decode hot path of OasisKV.

The kernels live in liboasis.so (C ABI: include/oasis.h); ``binding`` wraps
each entry point under the same name, ``layer`` chains them into one decode
step of one layer on CUDA streams.  Build the library with ``build.build()``.
"""
from .binding import (  # noqa: F401
    EXPORTS, OasisError, abi_version, attn_workspace, load, oasis_attn_workspace_bytes, oasis_build_summary,
    oasis_score_blocks, oasis_score_blocks_tc, oasis_select_topk_capped, oasis_select_topk_capped_tc,
    oasis_sparse_decode_attn, oasis_sparse_decode_attn_noalloc, oasis_sparse_decode_attn_tc,
    oasis_sparse_decode_attn_ws,
    oasis_stage_blocks, strerror,
)
from .layer import DecodeLayer, DecodeStepGraph, LayerShape, StepGraph  # noqa: F401
