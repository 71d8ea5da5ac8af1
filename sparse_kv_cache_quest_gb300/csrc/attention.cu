// Sparse paged decode attention over the head-wise logical-to-logical table.
//
// OasisKV paper review (xllm-io), §3 Fig. 5: the foreground forward pass runs
// sparse attention of the true query over the working set resident in HBM;
// §4 / Fig. 9: each KV head addresses its own resident blocks through the
// head-wise mapping.  For query head h*G + g of sequence b:
//     out = sum_i softmax_i(scale * q . k_i) v_i
// over the valid tokens of the slots whose table entry is >= 0.
//
// Data path.  A segment's pool is slots_per_seg contiguous 8 KiB tiles (16
// key rows, then 16 value rows, D = 128).  The segment is split over a
// thread-block cluster of CL CTAs (split-K); the CL*4 warps of the cluster
// take the slots round-robin.  Each warp first lists its non-empty slots in
// shared memory (one table read per slot), then streams their tiles through a
// private two-stage ring with 2-D TMA tensor copies (cp.async.bulk.tensor, one
// mbarrier per stage, lane 0 issues).  The tensor map views the pool as rows
// of D bf16 and uses the 128-byte swizzle, so the tensor-core fragment loads
// below are bank-conflict free.  Empty slots are never loaded.
//
// Math, per warp and 16-token slot, on the tensor cores (mma.sync m16n8k16,
// bf16 inputs, fp32 accumulation):
//   S^T[16 tokens x 8n queries] = K[16 x D] . Q^T[D x 8n]   (Q fragments in registers)
//   online softmax over tokens in the log2 domain (scale*log2(e) applied in fp32)
//   O^T[D x 8n] += V^T[D x 16] . P^T[16 x 8n]
// The query heads of the GQA group fill the N dimension (8 or 16 columns; unused
// columns are zero).  P^T reaches the B-fragment layout with one in-register
// 8x8 transpose per half (movmatrix), and is split into bf16 hi + lo parts so
// that the PV product keeps about 16 significant bits of p.  Each thread owns
// whole output elements, so no cross-lane reduction is needed per slot.
// Warps combine through shared memory (reusing the rings), then every CTA of
// the cluster combines a 1/CL share of the outputs from all CL CTAs' totals
// through distributed shared memory and writes it to out and lse; a segment
// on one CTA (CL = 1) writes its outputs straight from the warp merge, with no
// cluster barrier.  No global scratch memory is used.  With more than 8 query heads per KV head the heads
// are split over warp pairs that share a partition's ring (k_attn_hs, further
// down), so that each warp carries the math of 8 heads.
//
// k_attn_bal (further down) is the alternative split over all segments' slots
// with a caller workspace; it measured slower than the cluster split on the
// shapes benchmarked and is only used when a caller asks for it.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cfloat>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace oasis {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kNST = 2;                    // ring stages per warp
constexpr int kListMax = 512;              // listed slots per warp
constexpr int kMaxCluster = 8;             // CTAs per segment in the cluster split
constexpr uint32_t kWaitTries = 1u << 22;  // bounded mbarrier polls (far beyond any real copy)
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a . b  (m16n8k16, bf16 x bf16 -> fp32)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// {lo, hi} -> bf16x2 with `lo` in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// A slot tile is read once per step, so its copy marks the L2 lines evict-first:
// the half gigabyte a decode step streams through L2 then does not push out what
// other kernels of the step reuse (tiles just staged for a later layer's
// attention, the scores and radii the selection reads).  Measured on the
// 235B-shaped decode step with the same hint on the scorer's copies: 92.8 / 93.0
// -> 89.8 / 90.1 us per layer-step (this kernel alone 45.1 -> 45.6 us).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// Shared-memory plan (offsets in bytes from a 1024-aligned base).
template <int D, int GQ, int W = kWarps>
struct Plan {
  static constexpr int kTile = 64 * D;                    // one slot: 32 rows of D bf16
  static constexpr int kRing = W * kNST * kTile;
  static constexpr int kBars = kRing;                      // W * kNST mbarriers
  static constexpr int kLists = kBars + 8 * W * kNST;      // W * kListMax int32
  static constexpr int kEnd = kLists + 4 * W * kListMax;
  // combine scratch (floats), aliased onto the ring once every stage is drained
  // (per-warp output rows padded to D + 4 floats: the fragment-order stores of
  // lanes with different t then fall in different banks)
  static constexpr int kOS = D + 4;
  static constexpr int kWarpM = 0, kWarpL = W * GQ, kWarpO = 2 * W * GQ;
  static constexpr int kCtaM = kWarpO + W * GQ * kOS, kCtaL = kCtaM + GQ, kCtaO = kCtaL + GQ;
  // per query column: each warp's merge factor 2^(m_w - M), then 1 / l
  static constexpr int kHeadF = kCtaO + GQ * D, kHeadInv = kHeadF + GQ * W;
  static constexpr int kScratchBytes = 4 * (kHeadInv + GQ);
  static_assert(kScratchBytes <= kRing, "combine scratch must fit in the ring");
};

// One 16-token slot tile in shared memory (swizzled as the tensor map writes it)
// folded into a warp's online softmax state, on the tensor cores:
//   S^T = K . Q^T, log2-domain online softmax over the tile's nv valid tokens,
//   O^T += V^T . P^T with P^T split into bf16 hi + lo parts.
template <int KS, int NT>
__device__ __forceinline__ void attend_tile(uint32_t tile, int nv, const uint32_t (&qb)[NT][KS][2], float scale_log2,
                                            float (&o)[NT][KS][4], float (&m)[NT][2], float (&l)[NT][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  // fragment addressing inside a swizzled tile: row r, 16-byte chunk j of the D-wide row
  auto frag_addr = [](uint32_t tile, int r, int j) {
    return tile + (j >> 3) * 4096 + r * 128 + (((j & 7) ^ (r & 7)) << 4);
  };
  const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);  // K rows 0..15 for ldmatrix
  const int khalf = lane >> 4;
  const int vrow = 16 + (lane & 7) + 8 * (lane >> 4);   // V rows 16..31 for ldmatrix.trans
  const int vhalf = (lane >> 3) & 1;

  // ---- S^T = K . Q^T
  float sacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.0f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a[4];
    ldsm_x4(frag_addr(tile, krow, 2 * ks + khalf), a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma16816(sacc[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
  }
  // ---- online softmax over the slot's tokens (rows g and g + 8), per query column
  const bool v0 = g < nv, v1 = g + 8 < nv;
  uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float p0[2], p1[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float x0 = v0 ? sacc[nt][j] * scale_log2 : -INFINITY;
      const float x1 = v1 ? sacc[nt][2 + j] * scale_log2 : -INFINITY;
      float mx = fmaxf(x0, x1);
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float mn = fmaxf(m[nt][j], mx);
      const float corr = exp2f(m[nt][j] - mn);
      m[nt][j] = mn;
      p0[j] = exp2f(x0 - mn);
      p1[j] = exp2f(x1 - mn);
      l[nt][j] = l[nt][j] * corr + p0[j] + p1[j];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[nt][mt][j] *= corr;
        o[nt][mt][2 + j] *= corr;
      }
    }
    // P^T B-fragments: hi and lo bf16 parts, transposed 8x8 per token half
    const uint32_t h0 = pack_bf16(p0[0], p0[1]), h1 = pack_bf16(p1[0], p1[1]);
    const uint32_t l0 = pack_bf16(p0[0] - bf16_lo(h0), p0[1] - bf16_hi(h0));
    const uint32_t l1 = pack_bf16(p1[0] - bf16_lo(h1), p1[1] - bf16_hi(h1));
    bh[nt][0] = transpose8x8(h0);
    bh[nt][1] = transpose8x8(h1);
    bl[nt][0] = transpose8x8(l0);
    bl[nt][1] = transpose8x8(l1);
  }
  // ---- O^T += V^T . P^T
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    uint32_t a[4];
    ldsm_x4_t(frag_addr(tile, vrow, 2 * mt + vhalf), a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(o[nt][mt], a, bh[nt][0], bh[nt][1]);
      mma16816(o[nt][mt], a, bl[nt][0], bl[nt][1]);
    }
  }
}

// KS = D / 16 (k-steps of the QK product and m-tiles of the PV product);
// NT = query tiles of 8 heads (GQ = 8 * NT columns); W = warps per CTA (slot
// partitions): 4, two CTAs per SM; 8, one CTA per SM with twice the copies in
// flight, for layers with no more segments than SMs.
template <int KS, int NT, int W>
__global__ void __launch_bounds__(32 * W)
    k_attn(const __grid_constant__ CUtensorMap tmap, const uint16_t *__restrict__ q,
           const int32_t *__restrict__ table, int slots, const int32_t *__restrict__ seq_len, int Hkv, int G,
           float scale_log2, float *__restrict__ out, float *__restrict__ lse, int32_t *status) {
  constexpr int D = 16 * KS;
  constexpr int GQ = 8 * NT;
  constexpr int kBoxes = D / 64;  // 64-dim boxes (128 bytes per row) per tile
  using P = Plan<D, GQ, W>;
  constexpr int kW = W, kT = 32 * W;
  extern __shared__ unsigned char sm_raw[];
  const uint32_t raw_addr = smem_addr(sm_raw);
  unsigned char *sm = sm_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  cg::cluster_group cluster = cg::this_cluster();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int s = blockIdx.y;
  const int bseq = s / Hkv, h = s % Hkv;
  const int Hq = Hkv * G;

  int L = seq_len[bseq];
  if (L < 0) {
    if (tid == 0 && rank == 0 && h == 0) report(status, OASIS_STATUS_SEQ_LEN);
    L = 0;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + P::kBars) + warp * kNST;
  int32_t *list = reinterpret_cast<int32_t *>(sm + P::kLists) + warp * kListMax;
  const uint32_t ring = sbase + warp * kNST * P::kTile;
  if (lane == 0) {
    for (int i = 0; i < kNST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }

  float o[NT][KS][4];
  float m[NT][2], l[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      m[nt][j] = -INFINITY;
      l[nt][j] = 0.0f;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[nt][mt][i] = 0.0f;
  }

  // this warp's non-empty slots, as (slot << 5 | valid tokens)
  const int nw = CL * kW, gw = rank * kW + warp;
  const int nk = slots > gw ? (slots - gw + nw - 1) / nw : 0;
  const int32_t *trow = table + static_cast<int64_t>(s) * slots;
  int count = 0;
  for (int base = 0; base < nk; base += 32) {
    const int k = base + lane;
    int nv = 0, slot = 0;
    if (k < nk) {
      slot = gw + nw * k;
      const int blk = trow[slot];
      const int64_t n = blk < 0 ? 0 : static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
      nv = n <= 0 ? 0 : (n >= kBlockTokens ? kBlockTokens : static_cast<int>(n));
    }
    const unsigned mk = __ballot_sync(0xFFFFFFFFu, nv > 0);
    if (nv > 0) list[count + __popc(mk & ((1u << lane) - 1u))] = (slot << 5) | nv;
    count += __popc(mk);
  }
  __syncwarp();
  const int row_base = s * slots;  // tile index of slot 0 of this segment
  auto issue = [&](int c, int stg) {
    mbar_arrive_expect_tx(&bars[stg], P::kTile);
    const int y = (row_base + (list[c] >> 5)) * 32;
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_load_2d(ring + stg * P::kTile + bx * 4096, &tmap, bx * 64, y, &bars[stg]);
  };
  if (lane == 0)
    for (int c = 0; c < kNST && c < count; ++c) issue(c, c);

  // Q^T B-fragments: column n = query head nt*8 + g, rows k = dims 16ks + 2t (+1, +8, +9);
  // loaded once the first tile copies are in flight, so they overlap the copies
  uint32_t qb[NT][KS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = nt * 8 + g;
    const uint32_t *row =
        reinterpret_cast<const uint32_t *>(q + (static_cast<int64_t>(bseq) * Hq + h * G + qi) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[nt][ks][0] = qi < G ? row[(16 * ks + 2 * t) >> 1] : 0u;
      qb[nt][ks][1] = qi < G ? row[(16 * ks + 8 + 2 * t) >> 1] : 0u;
    }
  }
  int issued = min(kNST, count), consumed = 0;
  bool timed_out = false;

  for (int c = 0; c < count; ++c) {
    const int stg = c % kNST;
    const bool ok = mbar_wait_bounded(&bars[stg], static_cast<uint32_t>(c / kNST) & 1u, kWaitTries);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      timed_out = true;
      break;
    }
    const int nv = list[c] & 31;
    const uint32_t tile = ring + stg * P::kTile;

    attend_tile<KS, NT>(tile, nv, qb, scale_log2, o, m, l);
    __syncwarp();
    ++consumed;
    if (c + kNST < count) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(c + kNST, stg);
      }
      ++issued;
    }
  }
  if (timed_out) {
    if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
    for (int c = consumed; c < issued; ++c)
      mbar_wait_bounded(&bars[c % kNST], static_cast<uint32_t>(c / kNST) & 1u, kWaitTries);
  }

  // ---- warp totals: l over the token rows (lanes with equal t); o is complete per thread
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l[nt][j];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      l[nt][j] = v;
    }
  __syncthreads();  // every warp is past its ring: the scratch may alias it
  float *scratch = reinterpret_cast<float *>(sm);
  float *wm = scratch + P::kWarpM, *wl = scratch + P::kWarpL, *wo = scratch + P::kWarpO;
  float *cm = scratch + P::kCtaM, *cl = scratch + P::kCtaL, *co = scratch + P::kCtaO;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (g == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        wm[warp * GQ + nt * 8 + 2 * t + j] = m[nt][j];
        wl[warp * GQ + nt * 8 + 2 * t + j] = l[nt][j];
      }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int qc = nt * 8 + 2 * t + (i & 1), dim = 16 * mt + g + 8 * (i >> 1);
        wo[(warp * GQ + qc) * P::kOS + dim] = o[nt][mt][i];
      }
  }
  __syncthreads();
  // per query column (once, not once per output): the warps' merge factors
  // 2^(m_w - M), the CTA's M and l, and 1 / l
  float *hf = scratch + P::kHeadF, *hinv = scratch + P::kHeadInv;
  for (int qc = tid; qc < G; qc += kT) {  // the padded columns qc >= G are never read
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, wm[w * GQ + qc]);
    float ls = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const float f = M > -INFINITY ? exp2f(wm[w * GQ + qc] - M) : 0.0f;
      hf[qc * kW + w] = f;
      ls += f * wl[w * GQ + qc];
    }
    cm[qc] = M;
    cl[qc] = ls;
    hinv[qc] = ls > 0.0f ? 1.0f / ls : 0.0f;
    if (CL == 1 && lse != nullptr)
      lse[static_cast<int64_t>(bseq) * Hq + h * G + qc] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kT) {
    const int qc = idx / D, d = idx % D;
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) acc += hf[qc * kW + w] * wo[(w * GQ + qc) * P::kOS + d];
    if (CL == 1)  // one CTA: its totals are the results
      out[(static_cast<int64_t>(bseq) * Hq + h * G + qc) * D + d] = hinv[qc] > 0.0f ? acc * hinv[qc] : 0.0f;
    else
      co[qc * D + d] = acc;
  }
  if (CL == 1) return;  // no other CTA reads this one's shared memory
  cluster.sync();
  // Cluster merge: every rank combines its share of the G*D outputs, reading all
  // ranks' CTA totals through distributed shared memory with a thread's remote
  // loads issued together (one round trip per output, spread over the cluster).
  {
    const int n_out = G * D, per = (n_out + CL - 1) / CL;
    const int e1 = min(n_out, (rank + 1) * per);
    for (int idx = rank * per + tid; idx < e1; idx += kT) {
      const int qc = idx / D, d = idx % D;
      float mr[kMaxCluster], lr[kMaxCluster], orr[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < CL) {
          mr[r] = cluster.map_shared_rank(cm, r)[qc];
          lr[r] = cluster.map_shared_rank(cl, r)[qc];
          orr[r] = cluster.map_shared_rank(co, r)[qc * D + d];
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < CL) M = fmaxf(M, mr[r]);
      float acc = 0.0f, ls = 0.0f;
      if (M > -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (r < CL) {
            const float f = exp2f(mr[r] - M);
            acc += f * orr[r];
            ls += f * lr[r];
          }
        }
      }
      const int64_t row = static_cast<int64_t>(bseq) * Hq + h * G + qc;
      out[row * D + d] = ls > 0.0f ? acc / ls : 0.0f;
      if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ---- 9 to 16 query heads per KV head: the heads split over warp pairs ---------
// With more than 8 query heads per KV head a warp's chain per tile (S = K.Q^T
// over 16 heads, their online softmax, O^T += V^T.P^T) is four times that of a
// 4-head layer, and 4 warps per CTA no longer hide it.  This kernel runs 8
// warps: warp w takes the slots of partition w % 4 (the slots warp w % 4 of
// k_attn takes) for the 8 query heads of tile w / 4, so every head's arithmetic
// and merge order are those of k_attn<KS, 2>.  The two warps of a partition
// share its slot tiles: the first issues each tile's tensor copy into the pair's
// ring, both read it, and each releases the stage through an "empty" mbarrier
// of two arrivals, which the first waits on (bounded) before it copies the next
// tile into the stage.
constexpr int kThreadsHS = 256;
constexpr int kWarpsHS = kThreadsHS / 32;
constexpr int kPairs = kWarpsHS / 2;  // slot partitions per CTA (as many as k_attn's warps)
static_assert(kPairs == kWarps, "a pair takes the slots of one k_attn warp");

template <int D>
struct PlanHS {
  static constexpr int kNS = 2;                              // ring stages per pair
  static constexpr int kTile = 64 * D;
  static constexpr int kRing = kPairs * kNS * kTile;
  static constexpr int kFull = kRing;                        // kPairs * kNS mbarriers
  static constexpr int kEmpty = kFull + 8 * kPairs * kNS;    // kPairs * kNS mbarriers
  static constexpr int kLists = kEmpty + 8 * kPairs * kNS;   // kWarpsHS * kListMax int32
  static constexpr int kEnd = kLists + 4 * kWarpsHS * kListMax;
  // combine scratch (floats): each warp's 8 heads (m, l, o), then the CTA's 16
  static constexpr int kOS = D + 4;  // padded per-warp output rows, as in Plan
  static constexpr int kWarpM = 0, kWarpL = kWarpsHS * 8, kWarpO = 2 * kWarpsHS * 8;
  static constexpr int kCtaM = kWarpO + kWarpsHS * 8 * kOS, kCtaL = kCtaM + 16, kCtaO = kCtaL + 16;
  static constexpr int kHeadF = kCtaO + 16 * D, kHeadInv = kHeadF + 16 * kPairs;  // as in Plan
  static constexpr int kScratchBytes = 4 * (kHeadInv + 16);
  static_assert(kScratchBytes <= kRing, "combine scratch must fit in the ring");
};

__device__ __forceinline__ void stage_release(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <int KS>
__global__ void __launch_bounds__(kThreadsHS)
    k_attn_hs(const __grid_constant__ CUtensorMap tmap, const uint16_t *__restrict__ q,
              const int32_t *__restrict__ table, int slots, const int32_t *__restrict__ seq_len, int Hkv, int G,
              float scale_log2, float *__restrict__ out, float *__restrict__ lse, int32_t *status) {
  constexpr int D = 16 * KS;
  constexpr int kBoxes = D / 64;
  using P = PlanHS<D>;
  constexpr int NS = P::kNS;
  extern __shared__ unsigned char sm_raw[];
  const uint32_t raw_addr = smem_addr(sm_raw);
  unsigned char *sm = sm_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  cg::cluster_group cluster = cg::this_cluster();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = warp % kPairs, half = warp / kPairs;  // slot partition, query tile
  const bool issuer = half == 0;
  const int g = lane >> 2, t = lane & 3;
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int s = blockIdx.y;
  const int bseq = s / Hkv, h = s % Hkv;
  const int Hq = Hkv * G;

  int L = seq_len[bseq];
  if (L < 0) {
    if (tid == 0 && rank == 0 && h == 0) report(status, OASIS_STATUS_SEQ_LEN);
    L = 0;
  }
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + P::kFull) + pair * NS;
  uint64_t *empty = reinterpret_cast<uint64_t *>(sm + P::kEmpty) + pair * NS;
  int32_t *list = reinterpret_cast<int32_t *>(sm + P::kLists) + warp * kListMax;
  const uint32_t ring = sbase + pair * NS * P::kTile;
  if (issuer && lane == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);  // both warps of the pair
    }
    fence_mbar_init();
  }
  __syncthreads();  // the pair's barriers exist before its second warp waits on them

  float o[1][KS][4];
  float m[1][2], l[1][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    m[0][j] = -INFINITY;
    l[0][j] = 0.0f;
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[0][mt][i] = 0.0f;

  // the partition's non-empty slots, as (slot << 5 | valid tokens); both warps
  // of a pair build the same list
  const int nw = CL * kPairs, gw = rank * kPairs + pair;
  const int nk = slots > gw ? (slots - gw + nw - 1) / nw : 0;
  const int32_t *trow = table + static_cast<int64_t>(s) * slots;
  int count = 0;
  for (int base = 0; base < nk; base += 32) {
    const int k = base + lane;
    int nv = 0, slot = 0;
    if (k < nk) {
      slot = gw + nw * k;
      const int blk = trow[slot];
      const int64_t n = blk < 0 ? 0 : static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
      nv = n <= 0 ? 0 : (n >= kBlockTokens ? kBlockTokens : static_cast<int>(n));
    }
    const unsigned mk = __ballot_sync(0xFFFFFFFFu, nv > 0);
    if (nv > 0) list[count + __popc(mk & ((1u << lane) - 1u))] = (slot << 5) | nv;
    count += __popc(mk);
  }
  __syncwarp();
  const int row_base = s * slots;
  auto issue = [&](int c, int stg) {
    mbar_arrive_expect_tx(&full[stg], P::kTile);
    const int y = (row_base + (list[c] >> 5)) * 32;
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_load_2d(ring + stg * P::kTile + bx * 4096, &tmap, bx * 64, y, &full[stg]);
  };
  if (issuer && lane == 0)
    for (int c = 0; c < NS && c < count; ++c) issue(c, c);

  // Q^T B-fragments of this warp's 8 query heads (half * 8 + g)
  uint32_t qb[1][KS][2];
  {
    const int qi = half * 8 + g;
    const uint32_t *row =
        reinterpret_cast<const uint32_t *>(q + (static_cast<int64_t>(bseq) * Hq + h * G + qi) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[0][ks][0] = qi < G ? row[(16 * ks + 2 * t) >> 1] : 0u;
      qb[0][ks][1] = qi < G ? row[(16 * ks + 8 + 2 * t) >> 1] : 0u;
    }
  }
  int issued = issuer ? min(NS, count) : 0, consumed = 0;
  bool timed_out = false;

  for (int c = 0; c < count; ++c) {
    const int stg = c % NS;
    const bool ok = mbar_wait_bounded(&full[stg], static_cast<uint32_t>(c / NS) & 1u, kWaitTries);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      timed_out = true;
      break;
    }
    attend_tile<KS, 1>(ring + stg * P::kTile, list[c] & 31, qb, scale_log2, o, m, l);
    __syncwarp();
    ++consumed;
    if (lane == 0) stage_release(&empty[stg]);  // this warp is done reading the stage
    if (issuer && c + NS < count) {
      // both warps have read the stage: copy the partition's next tile into it
      int free_ok = 1;
      if (lane == 0) {
        free_ok = mbar_wait_bounded(&empty[stg], static_cast<uint32_t>(c / NS) & 1u, kWaitTries);
        if (free_ok) {
          fence_proxy_async_smem();
          issue(c + NS, stg);
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, free_ok, 0)) {
        timed_out = true;
        break;
      }
      ++issued;
    }
  }
  if (timed_out) {  // never leave with copies in flight
    if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
    for (int c = consumed; c < issued; ++c)
      mbar_wait_bounded(&full[c % NS], static_cast<uint32_t>(c / NS) & 1u, kWaitTries);
  }

  // ---- warp totals: l over the token rows (lanes with equal t); o is complete per thread
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float v = l[0][j];
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
    l[0][j] = v;
  }
  __syncthreads();  // every warp is past the rings: the scratch may alias them
  float *scratch = reinterpret_cast<float *>(sm);
  float *wm = scratch + P::kWarpM, *wl = scratch + P::kWarpL, *wo = scratch + P::kWarpO;
  float *cm = scratch + P::kCtaM, *cl = scratch + P::kCtaL, *co = scratch + P::kCtaO;
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      wm[warp * 8 + 2 * t + j] = m[0][j];
      wl[warp * 8 + 2 * t + j] = l[0][j];
    }
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qc = 2 * t + (i & 1), dim = 16 * mt + g + 8 * (i >> 1);
      wo[(warp * 8 + qc) * P::kOS + dim] = o[0][mt][i];
    }
  __syncthreads();
  // head qc = 8 * half + j was processed by warps half * kPairs + p, p = 0..kPairs-1
  // (combined in that order, as k_attn combines its warps)
  // per query column first (as in k_attn), then the outputs
  float *hf = scratch + P::kHeadF, *hinv = scratch + P::kHeadInv;
  for (int qc = tid; qc < G; qc += kThreadsHS) {
    const int w0 = (qc >> 3) * kPairs, j = qc & 7;
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < kPairs; ++p) M = fmaxf(M, wm[(w0 + p) * 8 + j]);
    float ls = 0.0f;
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      const float f = M > -INFINITY ? exp2f(wm[(w0 + p) * 8 + j] - M) : 0.0f;
      hf[qc * kPairs + p] = f;
      ls += f * wl[(w0 + p) * 8 + j];
    }
    cm[qc] = M;
    cl[qc] = ls;
    hinv[qc] = ls > 0.0f ? 1.0f / ls : 0.0f;
    if (CL == 1 && lse != nullptr)
      lse[static_cast<int64_t>(bseq) * Hq + h * G + qc] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreadsHS) {
    const int qc = idx / D, d = idx % D;
    const int w0 = (qc >> 3) * kPairs, j = qc & 7;
    float acc = 0.0f;
#pragma unroll
    for (int p = 0; p < kPairs; ++p) acc += hf[qc * kPairs + p] * wo[((w0 + p) * 8 + j) * P::kOS + d];
    if (CL == 1)  // one CTA: its totals are the results
      out[(static_cast<int64_t>(bseq) * Hq + h * G + qc) * D + d] = hinv[qc] > 0.0f ? acc * hinv[qc] : 0.0f;
    else
      co[qc * D + d] = acc;
  }
  if (CL == 1) return;  // no other CTA reads this one's shared memory
  cluster.sync();
  // cluster merge, as in k_attn
  {
    const int n_out = G * D, per = (n_out + CL - 1) / CL;
    const int e1 = min(n_out, (rank + 1) * per);
    for (int idx = rank * per + tid; idx < e1; idx += kThreadsHS) {
      const int qc = idx / D, d = idx % D;
      float mr[kMaxCluster], lr[kMaxCluster], orr[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < CL) {
          mr[r] = cluster.map_shared_rank(cm, r)[qc];
          lr[r] = cluster.map_shared_rank(cl, r)[qc];
          orr[r] = cluster.map_shared_rank(co, r)[qc * D + d];
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < CL) M = fmaxf(M, mr[r]);
      float acc = 0.0f, ls = 0.0f;
      if (M > -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (r < CL) {
            const float f = exp2f(mr[r] - M);
            acc += f * orr[r];
            ls += f * lr[r];
          }
        }
      }
      const int64_t row = static_cast<int64_t>(bseq) * Hq + h * G + qc;
      out[row * D + d] = ls > 0.0f ? acc / ls : 0.0f;
      if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ---- balanced split with a caller workspace --------------------------------
// All segments' slots form one flat range of N = S * slots tiles; CTA c of P
// takes [c*N/P, (c+1)*N/P), so every SM streams the same number of tiles
// whatever the segment count.  A CTA walks the segments its range touches
// ("pieces"), each as above (per-warp slot lists, 2-stage TMA rings, tensor-core
// tile math, warp merge in shared memory).  A piece that is a whole segment is
// written to out/lse directly.  A partial piece leaves (m, l, o) in the
// workspace (its CTA's slot 0 for the first piece of its range, 1 for the
// last), then the CTA counts itself in the segment's arrival counter; the CTA
// that arrives last merges all pieces of the segment, writes out/lse and sets
// the counter back to zero.  No CTA ever waits for another.
__host__ __device__ __forceinline__ int64_t cta_of(int64_t x, int64_t N, int64_t P) { return ((x + 1) * P - 1) / N; }

template <int KS, int NT>
__global__ void __launch_bounds__(kThreads)
    k_attn_bal(const __grid_constant__ CUtensorMap tmap, const uint16_t *__restrict__ q,
               const int32_t *__restrict__ table, int slots, const int32_t *__restrict__ seq_len, int Hkv, int G,
               float scale_log2, float *__restrict__ out, float *__restrict__ lse, int32_t *status,
               float *__restrict__ part, int32_t *__restrict__ counter, int64_t N, int P) {
  constexpr int D = 16 * KS;
  constexpr int GQ = 8 * NT;
  constexpr int kBoxes = D / 64;
  using PL = Plan<D, GQ>;
  extern __shared__ unsigned char sm_raw[];
  __shared__ int s_merge;
  const uint32_t raw_addr = smem_addr(sm_raw);
  unsigned char *sm = sm_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int Hq = Hkv * G;
  const int part_floats = G * (D + 2);  // m[G], l[G], o[G][D]
  const int64_t x0 = N * blockIdx.x / P, x1 = N * (blockIdx.x + 1) / P;
  if (x0 >= x1) return;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + PL::kBars) + warp * kNST;
  int32_t *list = reinterpret_cast<int32_t *>(sm + PL::kLists) + warp * kListMax;
  const uint32_t ring = sbase + warp * kNST * PL::kTile;
  if (lane == 0) {
    for (int i = 0; i < kNST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  uint32_t tc = 0;        // tiles this warp has issued and consumed so far (ring position, phase)
  bool dead = false;      // a wait of this warp timed out: it stops streaming
  const int seg_first = static_cast<int>(x0 / slots), seg_last = static_cast<int>((x1 - 1) / slots);

  for (int s = seg_first; s <= seg_last; ++s) {
    const int64_t seg_lo = static_cast<int64_t>(s) * slots;
    const int a = static_cast<int>(std::max(x0, seg_lo) - seg_lo);
    const int b = static_cast<int>(std::min(x1, seg_lo + slots) - seg_lo);  // slots [a, b) of segment s
    const int bseq = s / Hkv, h = s % Hkv;
    int L = seq_len[bseq];
    if (L < 0) {
      if (tid == 0 && a == 0 && h == 0) report(status, OASIS_STATUS_SEQ_LEN);
      L = 0;
    }
    uint32_t qb[NT][KS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int qi = nt * 8 + g;
      const uint32_t *row =
          reinterpret_cast<const uint32_t *>(q + (static_cast<int64_t>(bseq) * Hq + h * G + qi) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[nt][ks][0] = qi < G ? row[(16 * ks + 2 * t) >> 1] : 0u;
        qb[nt][ks][1] = qi < G ? row[(16 * ks + 8 + 2 * t) >> 1] : 0u;
      }
    }
    float o[NT][KS][4];
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m[nt][j] = -INFINITY;
        l[nt][j] = 0.0f;
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[nt][mt][i] = 0.0f;
    }
    // this warp's non-empty slots of the piece, as (slot << 5 | valid tokens)
    const int nk = (b - a) > warp ? (b - a - warp + kWarps - 1) / kWarps : 0;
    const int32_t *trow = table + seg_lo;
    int count = 0;
    for (int base = 0; base < nk; base += 32) {
      const int k = base + lane;
      int nv = 0, slot = 0;
      if (k < nk) {
        slot = a + warp + kWarps * k;
        const int blk = trow[slot];
        const int64_t n = blk < 0 ? 0 : static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
        nv = n <= 0 ? 0 : (n >= kBlockTokens ? kBlockTokens : static_cast<int>(n));
      }
      const unsigned mk = __ballot_sync(0xFFFFFFFFu, nv > 0);
      if (nv > 0) list[count + __popc(mk & ((1u << lane) - 1u))] = (slot << 5) | nv;
      count += __popc(mk);
    }
    __syncwarp();
    if (dead) count = 0;
    const int row_base = s * slots;
    auto issue = [&](int c) {
      const int stg = static_cast<int>((tc + c) % kNST);
      mbar_arrive_expect_tx(&bars[stg], PL::kTile);
      const int y = (row_base + (list[c] >> 5)) * 32;
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_load_2d(ring + stg * PL::kTile + bx * 4096, &tmap, bx * 64, y, &bars[stg]);
    };
    if (lane == 0) {
      fence_proxy_async_smem();  // the ring was last written as merge scratch
      for (int c = 0; c < kNST && c < count; ++c) issue(c);
    }
    int issued = min(kNST, count), consumed = 0;
    for (int c = 0; c < count; ++c) {
      const uint32_t gi = tc + static_cast<uint32_t>(c);
      const int stg = static_cast<int>(gi % kNST);
      const bool ok = mbar_wait_bounded(&bars[stg], (gi / kNST) & 1u, kWaitTries);
      if (__any_sync(0xFFFFFFFFu, !ok)) {
        dead = true;
        break;
      }
      attend_tile<KS, NT>(ring + stg * PL::kTile, list[c] & 31, qb, scale_log2, o, m, l);
      __syncwarp();
      ++consumed;
      if (c + kNST < count) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(c + kNST);
        }
        ++issued;
      }
    }
    if (dead) {
      if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
      for (int c = consumed; c < issued; ++c) {
        const uint32_t gi = tc + static_cast<uint32_t>(c);
        mbar_wait_bounded(&bars[gi % kNST], (gi / kNST) & 1u, kWaitTries);
      }
    }
    tc += static_cast<uint32_t>(dead ? issued : count);

    // ---- warp totals, then the CTA's partial (m, l, o) of the piece in shared memory
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = l[nt][j];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        l[nt][j] = v;
      }
    __syncthreads();  // every warp is past its ring: the scratch may alias it
    float *scratch = reinterpret_cast<float *>(sm);
    float *wm = scratch + PL::kWarpM, *wl = scratch + PL::kWarpL, *wo = scratch + PL::kWarpO;
    float *cm = scratch + PL::kCtaM, *cl = scratch + PL::kCtaL, *co = scratch + PL::kCtaO;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (g == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          wm[warp * GQ + nt * 8 + 2 * t + j] = m[nt][j];
          wl[warp * GQ + nt * 8 + 2 * t + j] = l[nt][j];
        }
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int qc = nt * 8 + 2 * t + (i & 1), dim = 16 * mt + g + 8 * (i >> 1);
          wo[(warp * GQ + qc) * PL::kOS + dim] = o[nt][mt][i];
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int qc = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * GQ + qc]);
      float acc = 0.0f, ls = 0.0f;
      if (M > -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = exp2f(wm[w * GQ + qc] - M);
          acc += f * wo[(w * GQ + qc) * PL::kOS + d];
          ls += f * wl[w * GQ + qc];
        }
      }
      co[qc * D + d] = acc;
      if (d == 0) {
        cm[qc] = M;
        cl[qc] = ls;
      }
    }
    __syncthreads();

    const int64_t c_first = cta_of(seg_lo, N, P), c_last = cta_of(seg_lo + slots - 1, N, P);
    if (c_first == c_last) {  // the whole segment is this CTA's piece
      for (int idx = tid; idx < G * D; idx += kThreads) {
        const int qc = idx / D, d = idx % D;
        const float ls = cl[qc];
        const int64_t row = static_cast<int64_t>(bseq) * Hq + h * G + qc;
        out[row * D + d] = ls > 0.0f ? co[idx] / ls : 0.0f;
        if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (cm[qc] + log2f(ls)) * kLn2 : -INFINITY;
      }
    } else {
      const int which = s == seg_first ? 0 : 1;
      float *pp = part + (static_cast<int64_t>(blockIdx.x) * 2 + which) * part_floats;
      for (int idx = tid; idx < G * D; idx += kThreads) pp[2 * G + idx] = co[(idx / D) * D + idx % D];
      for (int qc = tid; qc < G; qc += kThreads) {
        pp[qc] = cm[qc];
        pp[G + qc] = cl[qc];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int arrived = atomicAdd(&counter[s], 1);
        s_merge = arrived == static_cast<int>(c_last - c_first);
      }
      __syncthreads();
      if (s_merge) {
        __threadfence();
        for (int idx = tid; idx < G * D; idx += kThreads) {
          const int qc = idx / D, d = idx % D;
          // online merge over the pieces, kBatch at a time: each batch's loads go out
          // together, so a merge costs a few L2 round trips, not one per piece
          constexpr int kBatch = 8;
          float M = -INFINITY, acc = 0.0f, ls = 0.0f;
          for (int64_t c0 = c_first; c0 <= c_last; c0 += kBatch) {
            float pm[kBatch], pl[kBatch], po[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int64_t c = c0 + k;
              pm[k] = -INFINITY;
              pl[k] = 0.0f;
              po[k] = 0.0f;
              if (c <= c_last) {
                const int sl = (N * c / P) / slots == s ? 0 : 1;
                const float *pc = part + (c * 2 + sl) * part_floats;
                pm[k] = __ldcg(pc + qc);
                pl[k] = __ldcg(pc + G + qc);
                po[k] = __ldcg(pc + 2 * G + idx);
              }
            }
            float bm = M;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, pm[k]);
            if (bm > -INFINITY) {
              const float r = exp2f(M - bm);  // 0 while nothing was valid yet
              acc *= r;
              ls *= r;
#pragma unroll
              for (int k = 0; k < kBatch; ++k) {
                const float f = exp2f(pm[k] - bm);
                acc += f * po[k];
                ls += f * pl[k];
              }
              M = bm;
            }
          }
          const int64_t row = static_cast<int64_t>(bseq) * Hq + h * G + qc;
          out[row * D + d] = ls > 0.0f ? acc / ls : 0.0f;
          if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
        }
        if (tid == 0) counter[s] = 0;
      }
    }
    __syncthreads();  // scratch and s_merge are reused by the next piece
  }
}

// The pool as a 2-D tensor: rows of D bf16, one 32-row box per 64 dims of a slot.
cudaError_t make_pool_map(CUtensorMap *tmap, const uint16_t *pool, int D, int S, int slots) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S) * slots * 32};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// Cluster size of the split: about two CTAs per SM in all (measured on GB300:
// larger clusters lose more to co-scheduling than they gain, and deeper
// per-warp rings or a persistent SM-balanced split with a separate merge kernel
// were slower), enough that each list of `lists` per CTA fits.
int cluster_size(int sms, int S, int slots, int lists, int ctas_per_sm = 2) {
  int CL = static_cast<int>(
      std::min<int64_t>(4, std::max<int64_t>(1, static_cast<int64_t>(ctas_per_sm) * sms / S)));
  CL = std::min(CL, slots);
  while ((slots + CL * lists - 1) / (CL * lists) > kListMax) ++CL;
  return CL;
}

template <int KS, int NT, int W>
cudaError_t launch_tw(const CUtensorMap &tmap, const uint16_t *q, const int32_t *table, int slots,
                      const int32_t *seq_len, int S, int Hkv, int G, float scale, float *out, float *lse,
                      int32_t *status, cudaStream_t st) {
  constexpr int D = 16 * KS;
  using P = Plan<D, 8 * NT, W>;
  const size_t smem = P::kEnd + 1024;  // + slack for the 1024-byte alignment of the swizzled tiles
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn<KS, NT, W>), 32 * W, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  // split each segment over a cluster of CL CTAs (about 2 CTAs per SM in all at
  // 4 warps, one at 8)
  const int CL = cluster_size(sms, S, slots, W, W == 4 ? 2 : 1);
  if (CL > kMaxCluster) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3(static_cast<unsigned>(CL), static_cast<unsigned>(S)), dim3(32 * W), smem, st);
  cudaLaunchAttribute cl;
  cl.id = cudaLaunchAttributeClusterDimension;
  cl.val.clusterDim.x = static_cast<unsigned>(CL);
  cl.val.clusterDim.y = 1;
  cl.val.clusterDim.z = 1;
  lc.add(cl);
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&lc.cfg, k_attn<KS, NT, W>, tmap, q, table, slots, seq_len, Hkv, G, scale_log2, out,
                            lse, status);
}

// Up to 8 query heads per KV head: 4-warp CTAs, about two per SM in all.  When
// the segments fill more than half of the SMs but do not outnumber them, that
// takes a cluster of two per segment; one CTA of 8 warps (one per SM, as many
// copies in flight) instead needs no cluster merge (measured on GB300 at 128
// segments: 26.8 -> 24.7 us).  With fewer segments the 8-warp CTAs would still
// need clusters, and were slower (64 segments: 15.4 -> 15.5 us).
template <int KS, int NT>
cudaError_t launch_t(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                     const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                     int32_t *status, cudaStream_t st) {
  constexpr int D = 16 * KS;
  const int S = B * Hkv;
  CUtensorMap tmap;
  cudaError_t me = make_pool_map(&tmap, pool, D, S, slots);
  if (me != cudaSuccess) return me;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (S <= sms && 2 * S > sms)
    return launch_tw<KS, NT, 8>(tmap, q, table, slots, seq_len, S, Hkv, G, scale, out, lse, status, st);
  return launch_tw<KS, NT, 4>(tmap, q, table, slots, seq_len, S, Hkv, G, scale, out, lse, status, st);
}

// More than 8 query heads per KV head: the head-split kernel (8 warps per CTA).
template <int KS>
cudaError_t launch_hs(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                      const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                      int32_t *status, cudaStream_t st) {
  constexpr int D = 16 * KS;
  using P = PlanHS<D>;
  const int S = B * Hkv;
  CUtensorMap tmap;
  cudaError_t me = make_pool_map(&tmap, pool, D, S, slots);
  if (me != cudaSuccess) return me;
  const size_t smem = P::kEnd + 1024;  // + slack for the 1024-byte alignment of the swizzled tiles
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn_hs<KS>), kThreadsHS, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int CL = cluster_size(sms, S, slots, kPairs);
  if (CL > kMaxCluster) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3(static_cast<unsigned>(CL), static_cast<unsigned>(S)), dim3(kThreadsHS), smem, st);
  cudaLaunchAttribute cl;
  cl.id = cudaLaunchAttributeClusterDimension;
  cl.val.clusterDim.x = static_cast<unsigned>(CL);
  cl.val.clusterDim.y = 1;
  cl.val.clusterDim.z = 1;
  lc.add(cl);
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&lc.cfg, k_attn_hs<KS>, tmap, q, table, slots, seq_len, Hkv, G, scale_log2, out, lse,
                            status);
}

// Grid of the balanced split: two CTAs per SM, at least enough CTAs that no
// warp's list of a piece exceeds kListMax, never more CTAs than slot tiles
// (so that every CTA owns at least one tile).
int64_t bal_grid(int64_t N) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 1;
  }
  const int64_t per_cta = static_cast<int64_t>(kWarps) * kListMax;
  const int64_t P = std::max<int64_t>(2 * static_cast<int64_t>(sms), (N + per_cta - 1) / per_cta);
  return std::min(P, N);
}

template <int KS, int NT>
cudaError_t launch_bal_t(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                         const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                         int32_t *status, float *part, int32_t *counter, int64_t P, cudaStream_t st) {
  constexpr int D = 16 * KS;
  using PL = Plan<D, 8 * NT>;
  const int S = B * Hkv;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S) * slots * 32};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = PL::kEnd + 1024;
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn_bal<KS, NT>), kThreads, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t N = static_cast<int64_t>(S) * slots;
  if (P < 1 || P > N || P > 0x7FFFFFFF) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3(static_cast<unsigned>(P)), dim3(kThreads), smem, st);
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&lc.cfg, k_attn_bal<KS, NT>, tmap, q, table, slots, seq_len, Hkv, G, scale_log2, out,
                            lse, status, part, counter, N, static_cast<int>(P));
}

}  // namespace

cudaError_t launch_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                      int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                      float scale, float *out, float *lse, int32_t *status, cudaStream_t st) {
  if (D == 128) {
    if (G <= 8) return launch_t<8, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
    return launch_hs<8>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
  }
  if (G <= 8) return launch_t<4, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
  return launch_hs<4>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
}

// Workspace of the balanced split, from one grid size: P pieces' partial
// results (2 per piece: running max and sum, then G x D outputs) and, at a
// 256-byte boundary after them, one arrival counter per segment.
struct BalLayout {
  int64_t P;
  size_t counters_at, total;
};
BalLayout bal_layout(int B, int Hkv, int G, int D, int slots_per_seg) {
  const int64_t N = static_cast<int64_t>(B) * Hkv * slots_per_seg;
  BalLayout L;
  L.P = bal_grid(N);
  const size_t parts = static_cast<size_t>(L.P) * 2 * static_cast<size_t>(G) * (D + 2) * sizeof(float);
  L.counters_at = (parts + 255) / 256 * 256;
  L.total = L.counters_at + static_cast<size_t>(B) * Hkv * sizeof(int32_t);
  return L;
}

size_t attn_workspace_bytes(int B, int Hkv, int G, int D, int slots_per_seg) {
  return bal_layout(B, Hkv, G, D, slots_per_seg).total;
}

// The balanced split on a workspace laid out as L says.
static cudaError_t launch_bal(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                              const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out,
                              float *lse, void *ws, const BalLayout &L, int32_t *status, cudaStream_t st) {
  float *part = static_cast<float *>(ws);
  int32_t *counter = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(ws) + L.counters_at);
  if (D == 128) {
    if (G <= 8)
      return launch_bal_t<8, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, part,
                                counter, L.P, st);
    return launch_bal_t<8, 2>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, part,
                              counter, L.P, st);
  }
  if (G <= 8)
    return launch_bal_t<4, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, part,
                              counter, L.P, st);
  return launch_bal_t<4, 2>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, part,
                            counter, L.P, st);
}

cudaError_t launch_sparse_decode_attn_ws(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                         int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                         float scale, float *out, float *lse, void *ws, int32_t *status,
                                         cudaStream_t st) {
  return launch_bal(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse, ws,
                    bal_layout(B, Hkv, G, D, slots_per_seg), status, st);
}

// ---- the balanced split without caller memory -------------------------------
// Scratch for oasis_sparse_decode_attn_noalloc: a file-scope device array, so
// the call needs no allocation at all.  8 MiB holds the workspace of a split
// into up to 504 CTAs at 16 query heads per KV head and D = 128 (about a
// million slot tiles), more with fewer heads; larger shapes are rejected.  One
// array per device and process: calls that could overlap (different streams)
// race on it.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Identity of the current CUDA context: cuCtxGetId through the runtime's
// driver entry points (no link to the driver library).  A device reset or a
// released and recreated primary context is a new context with a new id.
static bool current_context_id(unsigned long long *id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;  // none before the runtime has made one current
  return get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current context, looked up once per
// context: the address belongs to the module loaded in that context, so a new
// context (after a device reset, say) gets its own lookup, never a stale one.
static void *noalloc_scratch() {
  static std::mutex mu;
  static std::vector<std::pair<unsigned long long, void *>> addr;  // (context id, address)
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(mu);
  if (known)
    for (const auto &e : addr)
      if (e.first == ctx) return e.second;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;  // (makes the context if none)
  if (known || current_context_id(&ctx)) addr.emplace_back(ctx, p);
  return p;
}

cudaError_t launch_sparse_decode_attn_noalloc(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                              int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G,
                                              int D, float scale, float *out, float *lse, int32_t *status,
                                              cudaStream_t st) {
  const BalLayout L = bal_layout(B, Hkv, G, D, slots_per_seg);  // one grid size for the memset and the launch
  if (L.total > kNoAllocScratchBytes) return cudaErrorInvalidValue;
  void *ws = noalloc_scratch();
  if (ws == nullptr) return cudaErrorInvalidDevice;
  // The per-segment arrival counters must start at zero.  Every completed call
  // leaves them at zero, but one that timed out may not, so clear them on every
  // call (a memset of 4 bytes per segment, no allocation).
  cudaError_t e = cudaMemsetAsync(static_cast<unsigned char *>(ws) + L.counters_at, 0,
                                  static_cast<size_t>(B) * Hkv * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  return launch_bal(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse, ws, L, status, st);
}

}  // namespace oasis
