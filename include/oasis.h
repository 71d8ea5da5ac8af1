/*
 * oasis.h - C ABI of liboasis.so: the lookahead sparse decode hot path of
 * OasisKV on one NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [XR] "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
 *        Sparse Prefetching", paper review on xllm-io.github.io: §2 core idea,
 *        §3 architecture (Fig. 5, eqs. (1)-(4), component table, decode flow),
 *        §4 innovations (Figs. 6-9), §5 implementation, §6 experiments.
 *   [LP] "Scaling KV Cache Beyond Memory Limits", legiblepapers.com: Key
 *        Takeaways, FAQ Q4 and Q7.
 *
 * One decode step of one layer, per KV head ("segment" s = b * Hkv + h of
 * sequence b and KV head h):
 *   oasis_build_summary       per-block min/max key summaries (update path)
 *   oasis_score_blocks        draft queries scan the summaries -> block scores
 *   oasis_select_topk_capped  top-K, capped admission, eviction, plan, table
 *   oasis_stage_blocks        host-resident KV tiles -> HBM slots (the plan)
 *   oasis_sparse_decode_attn  attention of the true query over the slots
 *                             (oasis_sparse_decode_attn_ws: SM-balanced, with a
 *                             caller workspace; oasis_sparse_decode_attn_tc:
 *                             both products on the tcgen05 tensor cores)
 * and the tensor-core scoring path that replaces the second and third calls
 * with the same selections:
 *   oasis_score_blocks_tc        score estimates with certified error radii
 *   oasis_select_topk_capped_tc  the exact selection from those estimates
 *
 * Conventions shared by every entry point
 *   Memory.     The caller allocates and owns every buffer.  The library
 *               allocates no memory and keeps no state between calls, except
 *               per process: that each kernel's shared-memory limit was
 *               raised, the driver's tensor-map encoder entry point, and for
 *               oasis_sparse_decode_attn_noalloc a static 8 MiB device scratch
 *               array and its address.  Device pointers must be device memory
 *               or, where stated, host memory the GPU can address (pinned and
 *               mapped).
 *   Execution.  Every call enqueues kernels on `stream` (NULL = the legacy
 *               default stream) and returns without synchronising.  Outputs
 *               are valid once the stream reaches that point.
 *   Errors.     OASIS_EINVAL: an argument failed host-side validation; nothing
 *               was launched.  OASIS_ECUDA: a launch failed (the CUDA error is
 *               left for cudaGetLastError to report).  Faults that only the
 *               device can see (an invalid table, a NaN score, a plan entry
 *               out of range, a sequence longer than the summary capacity) are
 *               OR-ed into the caller's int32 status word as OASIS_STATUS_*
 *               bits; kernels never trap or assert.  The library never clears
 *               the status word; pass NULL where the call allows it to skip
 *               reporting.
 *   Types.      bf16 is passed as uint16_t (the bit pattern of __nv_bfloat16);
 *               fp32 as float; block ids and slots as int32_t.
 *   Blocks.     A logical block holds 16 consecutive tokens; token t of block
 *               b of sequence i is valid when 16*b + t < seq_len[i]
 *               ([XR] §6 default parameters: block size 16).
 *
 * Where the interface departs from the plain five-call form (one call per
 * step, every shape rule checked on the host before a launch), and why:
 *   - Lengths are per sequence (seq_len[B]) in every call, with B and Hkv in
 *     place of S = B*Hkv: all KV heads of a sequence share its length, so a
 *     per-segment copy would only repeat it Hkv times.
 *   - Rules that depend on the lengths are not host errors: seq_len lives in
 *     device memory, and checking it on the host would synchronise every call.
 *     A length beyond the summary capacity (seq_len > 16*Nb_max) or below 0
 *     sets OASIS_STATUS_SEQ_LEN and is clamped; fewer candidates than K
 *     (K > nc) is not an error - the rule takes the first min(K, nc).  C > K
 *     stays a host error.  This is why oasis_build_summary and
 *     oasis_score_blocks take a status word as well.
 *   - oasis_stage_blocks takes host_nb, the blocks per segment of the host
 *     copy, so that a plan entry naming a block outside it is skipped and
 *     reported (OASIS_STATUS_PLAN_RANGE) instead of read out of bounds.
 *   - oasis_sparse_decode_attn needs no workspace: the CTAs of a cluster merge
 *     their partial results in distributed shared memory.  The workspace form
 *     (ws, ws_bytes, oasis_attn_workspace_bytes) belongs to the SM-balanced
 *     variant oasis_sparse_decode_attn_ws.
 *   - oasis_build_summary can also write wsum, and oasis_score_blocks_tc with
 *     oasis_select_topk_capped_tc are a second scoring path: tensor-core
 *     estimates with certified radii, from which the selection is exactly the
 *     one of the fixed-order scores.  oasis_sparse_decode_attn_noalloc and
 *     oasis_abi_version are conveniences with no counterpart in the pages.
 *   - No status code is returned for device faults (there is no
 *     OASIS_EDEVICE): the calls return before the kernels run, so only the
 *     caller, reading its status word after the stream, can see them.
 *
 * Layouts (element counts; all arrays dense and row-major)
 *   KV tile     [2][16][D] bf16: the block's 16 keys, then its 16 values.
 *               8 KiB at D = 128.  Both the host copy of the full cache and
 *               the HBM slot pool are arrays of tiles.
 *   pool        [S][slots_per_seg][2][16][D] bf16, slots_per_seg = K + W.
 *   summary     kmin, kmax: [S][D/8][Nb_max][8] bf16 each ("chunk-major":
 *               the 8 dims d = 8c .. 8c+7 of consecutive blocks are
 *               consecutive in memory).
 *   table       [S][K + W] int32: slot -> logical block id, -1 = empty.  Slots
 *               0..K-1 hold the selected blocks, K..K+W-1 the local window.
 *   queries     q [B][Hq][D] bf16 and qdraft [B][Nd][Hq][D] bf16, Hq = Hkv*G;
 *               query head h*G + g (g < G) belongs to KV head h.
 */
#ifndef OASIS_H
#define OASIS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers (it is this same type). */
typedef struct CUstream_st *oasis_stream_t;

#define OASIS_ABI_VERSION 3

/* Return codes. */
#define OASIS_OK 0
#define OASIS_EINVAL (-1)
#define OASIS_ECUDA (-2)

/* Bits of the device status word. */
#define OASIS_STATUS_TABLE_RANGE 1  /* a resident block is not a candidate (outside [0, nc)) */
#define OASIS_STATUS_TABLE_DUP 2    /* a block is resident in two slots of one segment */
#define OASIS_STATUS_NAN_SCORE 4    /* a candidate's score is NaN (it ranks below all numbers) */
#define OASIS_STATUS_PLAN_RANGE 8   /* a plan entry names a block or slot out of range; skipped */
#define OASIS_STATUS_SEQ_LEN 16     /* seq_len < 0 or beyond 16 * Nb_max; clamped */
#define OASIS_STATUS_TIMEOUT 32     /* a bounded device wait gave up; the output is incomplete */

/* One transfer of the plan: host block src_block -> pool slot dst_slot. */
typedef struct {
  int32_t src_block;
  int32_t dst_slot;
} oasis_xfer_t;

/* Text of a return code or of one status bit. */
const char *oasis_strerror(int code);

/* OASIS_ABI_VERSION of the loaded library. */
int oasis_abi_version(void);

/*
 * Min/max key summaries of blocks [blk_begin, blk_begin + blk_count) of every
 * segment - the full build at sparsification (blk_begin = 0, blk_count =
 * Nb_max) or the per-step update of the newest blocks.
 * [XR] §3 component table "Compressed Key Cache" (per-dimension min/max per
 * logical block, 1/16 of the full KV); §5 compressed-key update.
 *
 * k:        bf16 keys; key d of token t of block blk_begin + j of segment s is
 *           k[s*seg_stride + j*blk_stride + t*tok_stride + d].  16-byte
 *           aligned; the three strides (elements) non-negative multiples of 8.
 *           A KV tile array (full cache or pool) has tok_stride = D,
 *           blk_stride = 32*D.
 * seq_len:  int32 [B] valid tokens per sequence (device).
 * kmin/kmax: summary arrays (layout above), written for every block of the
 *           range that holds a valid token; other entries are not touched.
 * wsum:     optional (NULL: not written) float32 [S][Nb_max]: for the same
 *           blocks, an upper bound (within a relative 2^-14) of the sum over
 *           the dims of the summary values on the wrong side of zero, |kmax_d|
 *           where kmax_d < 0 plus kmin_d where kmin_d > 0.  Not part of the
 *           method: oasis_score_blocks_tc reads it to bound its rounding.
 * Per dim, over the block's valid tokens: kmin = IEEE minimum, kmax = IEEE
 * maximum, with -0 below +0.  Exact (no rounding).  NaN keys: undefined.
 * EINVAL: a NULL pointer, D not 64 or 128, B or Hkv < 1, Nb_max < 1,
 * blk_begin < 0, blk_count < 0, blk_begin + blk_count > Nb_max, a misaligned
 * pointer or stride.  status may be NULL.
 */
int oasis_build_summary(const uint16_t *k, int64_t seg_stride, int64_t blk_stride, int64_t tok_stride,
                        int B, int Hkv, int D, const int32_t *seq_len, int blk_begin, int blk_count,
                        uint16_t *kmin, uint16_t *kmax, float *wsum, int Nb_max, int32_t *status,
                        oasis_stream_t stream);

/*
 * Look-ahead block scores: the draft queries of each KV head scan its
 * summaries ([XR] §3 decode flow; §4 Fig. 7).
 *
 * scores[s][b], float32 [S][Nb_max], is written for the candidate blocks
 * b < nc = ceil(seq_len/16) - W of segment s (the W newest blocks form the
 * always-resident window and are not scored); other entries are not touched.
 *   score = max over the G query heads of KV head h and the Nd drafts of
 *           sum_{d = 0..D-1, in this order, from +0, fp32 round-to-nearest}
 *               q_d * (q_d >= 0 ? kmax_d : kmin_d)
 * (each term is an exact fp32 product of two bf16 values, so the result is
 * reproducible bit for bit).
 * EINVAL: a NULL or misaligned pointer (kmin, kmax and qdraft need 16-byte
 * alignment, seq_len, scores and status 4-byte), D not 64 or 128, G not in
 * [1, 16], Nd < 1, G*Nd > 64, B or Hkv < 1, W < 0, Nb_max < 1.  status may be
 * NULL.
 */
int oasis_score_blocks(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft,
                       int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                       float *scores, int32_t *status, oasis_stream_t stream);

/*
 * The same look-ahead scores on the tensor cores, each with a certified error
 * radius ([XR] §3 decode flow; §4 Fig. 7).  Per segment the scan is a dense
 * product of the candidate blocks' summaries [kmax | kmin] (2D values per
 * block) with the head's split queries [q+ ; q-] (q+ = q where q >= 0, q- =
 * q where q < 0, +0 elsewhere), run as tcgen05 MMAs with fp32 accumulation;
 * the block score is the max over the query columns.
 *
 * scores[s][b] = s~, radius[s][b] = r (both float32 [S][Nb_max]), written
 * for the same candidate blocks as oasis_score_blocks, such that the score s
 * that oasis_score_blocks computes for the block satisfies |s~ - s| <= r.
 *   r = 2^-12 (|s~| + 2 C) + 2^-110,  C >= sum_d Q_d c_d,
 * Q_d = max over the head's query vectors of |q_d|, c_d = |kmax_d| where
 * kmax_d < 0 plus kmin_d where kmin_d > 0, else 0.  The sum of the absolute
 * terms of any query is at most |s~| + 2C (up to rounding), and both the
 * fixed-order fp32 sum and the tensor cores' fp32 accumulation of 2D terms
 * stay within 2^-16 of it, so r carries a margin of 16.  A NaN score gets
 * radius +inf.
 * wsum:     optional; the sums oasis_build_summary keeps for these summaries.
 *           Given: C = (max_d Q_d) * wsum[s][b].  NULL: C = sum_d Q_d c_d,
 *           read from the summaries (slower when many blocks have a dim on the
 *           wrong side of zero).
 * oasis_select_topk_capped_tc turns these into the exact selection.
 * Host-side checks, alignment and EINVAL cases: as oasis_score_blocks, plus
 * radius (4-byte aligned, not NULL).  Two CTAs per SM with up to 113 KB of
 * shared memory each; every internal wait is bounded (OASIS_STATUS_TIMEOUT).
 */
int oasis_score_blocks_tc(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                          const uint16_t *qdraft, int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                          float *scores, float *radius, int32_t *status, oasis_stream_t stream);

/*
 * Per-KV-head top-K with capped admission ([XR] §3 decode flow and component
 * table "Capped Eviction Policy" and "Head-wise Mapping"; §4 innovations;
 * [LP] FAQ Q7).  One segment, nc = ceil(seq_len/16) - W candidates:
 *   T  = the first min(K, nc) candidates by (score desc, block id asc); -0
 *        equals +0; a NaN score ranks below every number.
 *   R  = the blocks in table_in slots 0..K-1 (-1 = empty slot).
 *   A  = the first `cap` blocks of T that are not in R, in the same order.
 *   R' = the first K of R and A in that order, empty slots ranking below every
 *        block: empty slots are filled first (lowest slot first), then the
 *        lowest-ranked residents are evicted.
 *   A in ascending block id takes the freed slots in ascending order; all
 *   other slots, and the window slots K..K+W-1, keep their entries.
 * table_out [S][K+W] receives the new table (it may alias table_in).
 * plan [S][cap] receives plan_count[s] = |A| entries in ascending dst_slot;
 * entries past plan_count[s] are set to {-1, -1}.
 * A table whose slots 0..K-1 hold a block outside [0, nc) or the same block
 * twice sets OASIS_STATUS_TABLE_RANGE / _DUP: that segment's table passes
 * through unchanged and its plan is empty.
 * EINVAL: a NULL pointer (status may not be NULL), B or Hkv < 1, K not in
 * [1, 1024], W not in [0, 256], cap not in [0, K], Nb_max not in [1, 32768].
 */
int oasis_select_topk_capped(const float *scores, int Nb_max, const int32_t *seq_len, int B, int Hkv,
                             int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                             oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, oasis_stream_t stream);

/*
 * The same selection from tensor-core estimates (oasis_score_blocks_tc): the
 * outputs table_out, plan and plan_count are exactly those that
 * oasis_select_topk_capped gives on the fixed-order scores of
 * oasis_score_blocks ([XR] §3 decode flow, component table "Capped Eviction
 * Policy"; the certification is this library's own).
 * Each of the rule's three decisions splits a set into its first m members
 * and the rest: T (the first K candidates), A (the first cap of T \ R) and
 * the evicted (the last max(0, |A| - empty slots) of R \ T).  With the
 * intervals [s~ - r, s~ + r], a member whose interval lies above every
 * interval of the members ranked after the first m by the estimates (or below
 * every interval of the first m) is settled; every other member's score is
 * recomputed with the oasis_score_blocks arithmetic from kmin, kmax and
 * qdraft, and the selection runs on the mixed scores.
 * scores:  in: the estimates s~ [S][Nb_max]; out: the recomputed blocks hold
 *          their fixed-order scores, the others keep their estimates.
 * radius:  [S][Nb_max], any r with |s~ - s| <= r (a larger r only means more
 *          recomputation; +inf recomputes every candidate).
 * kmin, kmax, qdraft, G, Nd, D: as for oasis_score_blocks.
 * Other arguments, outputs and status bits: as oasis_select_topk_capped.
 * EINVAL: as oasis_select_topk_capped, or a NULL or misaligned summary / query
 * / radius pointer, D not 64 or 128, G not in [1, 16], Nd < 1, G*Nd > 64,
 * Nb_max > 16384, or shared memory beyond 200 KB for the shape.
 */
int oasis_select_topk_capped_tc(float *scores, const float *radius, const uint16_t *kmin, const uint16_t *kmax,
                                const uint16_t *qdraft, int G, int Nd, int D, int Nb_max, const int32_t *seq_len,
                                int B, int Hkv, int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                                oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, oasis_stream_t stream);

/*
 * Carry out the transfer plan: copy each planned block's KV tile from the host
 * tier into its HBM slot ([XR] §3 Fig. 5 KV transfer worker; decode flow
 * "asynchronous transfer").  Meant for a side stream ordered by events.
 *
 * host_kv:  device-addressable pointer to pinned, mapped host memory (on a
 *           unified-address system the host pointer of cudaHostAlloc memory);
 *           the tile of block blk of segment s starts at byte
 *           s*host_seg_stride_bytes + blk*(64*D).  16-byte aligned, stride a
 *           multiple of 16.  host_nb: blocks per segment in the host copy.
 * plan, plan_count: as written by oasis_select_topk_capped (cap per segment).
 * pool:     [S][slots_per_seg][2][16][D] bf16; slot dst_slot of segment s
 *           receives the tile; other slots are not touched.
 * An entry with src_block outside [0, host_nb) or dst_slot outside
 * [0, slots_per_seg) is skipped and sets OASIS_STATUS_PLAN_RANGE.
 * EINVAL: a NULL or misaligned pointer (status may not be NULL), D not 64 or
 * 128, B or Hkv < 1, cap < 0, host_nb < 1, slots_per_seg < 1.
 */
int oasis_stage_blocks(const void *host_kv, int64_t host_seg_stride_bytes, int host_nb,
                       const oasis_xfer_t *plan, const int32_t *plan_count, int cap, int B, int Hkv, int D,
                       uint16_t *pool, int slots_per_seg, int32_t *status, oasis_stream_t stream);

/*
 * Sparse paged decode attention of the true queries over each KV head's
 * resident slots ([XR] §3 Fig. 5 foreground sparse attention; Fig. 9
 * head-wise mapping).  For query head h*G + g of sequence b:
 *   out = sum_i p_i v_i,  p = softmax_i(scale * q . k_i)
 * over every valid token i of every slot whose table entry is >= 0.
 * out: float32 [B][Hq][D].  lse (may be NULL): float32 [B][Hq], the natural
 * log of sum_i exp(scale * q . k_i).  No valid token: out = 0, lse = -inf.
 * Products on the tensor cores with fp32 accumulation (p is carried as a
 * bf16 hi + lo pair); against a float64 evaluation the error is within 1e-2
 * max-abs and 1e-3 relative L2 on N(0,1)-like bf16 data.
 * EINVAL: a NULL or misaligned pointer, D not 64 or 128, G not in [1, 16],
 * B or Hkv < 1, slots_per_seg not in [1, 4096], B*Hkv*slots_per_seg*32 >= 2^31
 * (pool rows).  status may be NULL.
 */
int oasis_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                             const int32_t *seq_len, int B, int Hkv, int G, int D, float scale,
                             float *out, float *lse, int32_t *status, oasis_stream_t stream);

/*
 * The same attention with the work balanced over the SMs: all segments' slots
 * form one range split evenly over the CTAs, so the SMs stream equal byte
 * counts whatever the number of segments.  A segment whose slots are spread
 * over several CTAs is merged by the CTA that finishes its part last, through
 * partial results (running max, sum, output) and one arrival counter per
 * segment kept in the caller's workspace (the same split-K merge as the
 * cluster path, [XR] §4 Fig. 9 names only the attention, not its split).
 * Results equal oasis_sparse_decode_attn's within rounding.
 *
 * ws:  device memory of at least oasis_attn_workspace_bytes(B, Hkv, G, D,
 *      slots_per_seg) bytes, 16-byte aligned, ZERO-FILLED before its first
 *      use.  It holds the partial results (scratch) and the per-segment
 *      arrival counters; every call that completes leaves the counters at zero
 *      again, so the workspace can be reused without clearing.  Calls that may
 *      run at the same time (other streams) need workspaces of their own.
 *      After a call that set OASIS_STATUS_TIMEOUT it must be zero-filled again.
 * oasis_attn_workspace_bytes returns 0 for arguments the call would reject.
 * EINVAL: as oasis_sparse_decode_attn, or ws NULL / misaligned, or ws_bytes
 * smaller than the workspace size.
 */
size_t oasis_attn_workspace_bytes(int B, int Hkv, int G, int D, int slots_per_seg);
int oasis_sparse_decode_attn_ws(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                                const int32_t *seq_len, int B, int Hkv, int G, int D, float scale,
                                float *out, float *lse, void *ws, size_t ws_bytes, int32_t *status,
                                oasis_stream_t stream);

/*
 * oasis_sparse_decode_attn_ws without caller memory: the partial results and
 * arrival counters live in a scratch array of 8 MiB that the library holds in
 * device memory per device (a static device variable whose address is looked
 * up once per CUDA context - a context made after a device reset gets its own
 * lookup; nothing is allocated or freed by the call).  The paper has no
 * counterpart: this is a convenience of this library for callers that cannot
 * provide a workspace.  Same arguments and results as oasis_sparse_decode_attn.
 * The counters are cleared at the start of every call (a 4-byte-per-segment
 * memset on `stream`).  Calls that may overlap in time on one device (other
 * streams, other host threads) race on the shared scratch: serialise them on
 * one stream or use oasis_sparse_decode_attn_ws with separate workspaces.
 * The first call in a context should not be inside a stream capture (it looks
 * up the scratch's device address).
 * EINVAL: as oasis_sparse_decode_attn, or a shape whose workspace
 * (oasis_attn_workspace_bytes) exceeds the 8 MiB scratch.
 */
int oasis_sparse_decode_attn_noalloc(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                     int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                     float scale, float *out, float *lse, int32_t *status, oasis_stream_t stream);

/*
 * The same attention with both products on the tcgen05 tensor cores (the
 * calls above use warp-level mma.sync): per CTA, tiles of 8 slots (128
 * tokens) land by TMA; S^T = K . Q^T and O^T = V^T . P^T (P as a bf16 hi + lo
 * pair) run as tcgen05 MMAs into tensor memory, and the softmax warps read S
 * and O back from it.  A segment is split over a cluster of up to 4 CTAs as in
 * oasis_sparse_decode_attn.  Same arguments, outputs, status bits and error
 * bound.  It is slower than the mma.sync kernels (it keeps a whole tile's
 * values in shared memory through the softmax, so each CTA looks one tile
 * ahead), and its 113 KB CTAs leave no room beside them for the selection and
 * staging kernels of a layer-pipelined step, so it is not the default.
 * EINVAL: as oasis_sparse_decode_attn, or D not 128.
 */
int oasis_sparse_decode_attn_tc(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                                const int32_t *seq_len, int B, int Hkv, int G, int D, float scale,
                                float *out, float *lse, int32_t *status, oasis_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OASIS_H */
