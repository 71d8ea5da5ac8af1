"""KV transfer: copy the planned blocks from the host cache into HBM slots.

What the pages fix:
  * [XR] §3 Fig. 5: a KV transfer worker copies CPU -> GPU; the full KV cache
    lives in host memory.
  * [XR] §3 decode flow: the transfer plan is carried out by an asynchronous
    copy into the GPU working set; [XR] §5: persistent workers on background
    CUDA streams, ordered by CUDA events.
  * [XR] §4: only head-wise mapping entries change; the page table does not.

Reading: a byte copy of whole block tiles (K tile then V tile); plan entries
whose source block or destination slot is out of range are skipped and set
STATUS_PLAN_RANGE.

Pin (tests/test_oracle_stage.py): the result equals the input pool with
exactly the planned slots replaced by the named host tiles.
"""
import numpy as np

STATUS_PLAN_RANGE = 8


def stage_blocks(host_tiles, plan, pool):
    """host_tiles uint16 [Nb][2][16][D]; plan [(src_block, dst_slot)];
    pool uint16 [slots][2][16][D].  Returns (new pool, status)."""
    out = np.array(pool, dtype=np.uint16, copy=True)
    status = 0
    for src, dst in plan:
        if 0 <= src < host_tiles.shape[0] and 0 <= dst < out.shape[0]:
            out[dst] = host_tiles[src]
        else:
            status |= STATUS_PLAN_RANGE
    return out, status
