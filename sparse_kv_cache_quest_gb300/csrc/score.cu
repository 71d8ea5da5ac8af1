// Look-ahead block scoring: the draft queries of a KV head scan its min/max
// key summaries (OasisKV paper review (xllm-io), §3 decode flow: "draft query
// scans the compressed key summary -> predicts top-K blocks"; §4 Fig. 7).
//
//   score[s][b] = max over the Nq = G*Nd query vectors of
//                 sum_{d ascending, from +0, fp32 RN} q_d * (q_d >= 0 ? kmax_d : kmin_d)
//
// The max over the query vectors propagates NaN (as the IEEE maximum does), so
// a NaN key or query gives a NaN score, which the selection flags.
//
// Exactness.  Each term is the product of two bf16 values, exact in fp32, so
// the kernel writes the term as two fused multiply-adds,
//     acc = fma(qn_d, kmin_d, acc);  acc = fma(qp_d, kmax_d, acc)
// with qp = q, qn = +0 when q >= 0 and qp = +0, qn = q otherwise: one of the
// two adds an exact zero, which leaves acc unchanged (acc is never -0), and the
// other rounds acc + q*sel once, exactly as the sequential definition does.
// No reassociation, no fast-math: the result is bit-identical to a plain loop.
//
// Work split.  The unit of work is 32*NB consecutive candidate blocks of one
// segment, NB = 2 blocks per lane of a warp.  Units are numbered segment-major
// and each CTA of a persistent grid (SM count x resident CTAs per SM) takes one
// contiguous range of units, so every SM gets the same number of units (+-1)
// whatever the segment count.  A CTA walks the segments of its range in phases
// of at most `qseg` segments whose query operands it holds in shared memory;
// its warps take the units of a phase round-robin.
//
// Inner loop.  Lane b streams its block's 16-byte kmin/kmax chunks (8 dims of
// the chunk-major layout [S][D/8][Nb][8], so a warp reads 512 contiguous bytes
// per load) with kPF chunks in flight.  Per dim it widens kmin/kmax to fp32 and
// runs two packed fp32x2 FMAs (fma.rn.f32x2) per pair of queries and block:
// the query operands sit in shared memory as {qn_j, qn_j+1, qp_j, qp_j+1}, one
// broadcast 16-byte load per pair and dim feeding 2*NB packed FMAs.  Queries
// are padded to NQP by repeating the last one, which leaves the max unchanged.
//
// More than 16 query vectors (e.g. 16 query heads x 4 drafts): the
// accumulators of all of them no longer fit two blocks per lane, so k_score_qg
// splits the query pairs over the warps of a CTA (8 pairs each) and takes the
// max over the groups in shared memory; see below.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 256;  // 8 warps: two CTAs fill the 16 warp slots 128 registers allow
constexpr int kWarps = kThreads / 32;

// Blocks per lane: two while the accumulators fit (each broadcast query load
// then feeds four packed FMAs instead of two), else one.
template <int NQP>
constexpr int blocks_per_lane() { return NQP <= 16 ? 2 : 1; }
// Register cap: 128 keeps two 8-warp CTAs per SM (all 16 warp slots the register
// file allows at 128).  At 16 query vectors the kernel spills a few words under
// that cap and still runs faster than with one CTA of 154 registers per SM.
// (Caps of 112-120, which would leave room beside two CTAs for an attention CTA of
// another layer, spill and did not speed up the pipelined decode step.)
template <int NQP>
constexpr int max_regs() { return 128; }
template <int NQP>
constexpr size_t smem_budget() { return 100 * 1024; }
template <int NQP>
constexpr int prefetch() { return 2; }  // chunks in flight per lane and block

// Summary chunk loads of k_score: read-only path, no L1 allocation (each chunk
// is read by one warp once), L2 fetching 256-byte groups (a warp's load covers
// 512 contiguous bytes).  Measured 0.3 us faster per launch than plain __ldg.
__device__ __forceinline__ uint4 ld_summary(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// CH = D / 8 chunks of 8 dims (8 for D = 64, 16 for D = 128).
template <int NQP, int CH>
__global__ void __launch_bounds__(kThreads) __maxnreg__(max_regs<NQP>())
    k_score(const uint16_t *__restrict__ kmin, const uint16_t *__restrict__ kmax, int Nb_max,
            const uint16_t *__restrict__ qdraft, int S, int Hkv, int G, int Nd, const int32_t *__restrict__ seq_len,
            int W, float *__restrict__ scores, int32_t *status, int units_per_seg, int qseg) {
  constexpr int D = CH * 8;
  constexpr int per_seg_q = D * (NQP / 2);
  constexpr int kPF = prefetch<NQP>();
  constexpr int NB = blocks_per_lane<NQP>();
  constexpr int kUnit = 32 * NB;  // blocks per warp unit
  constexpr int kFill = 2;        // raw query loads in flight per thread while filling qsm
  static_assert(CH % kPF == 0, "the chunk loop steps by kPF: it must divide the chunk count");
  extern __shared__ float4 qsm[];  // [qseg][D][NQP/2] {qn_j, qn_j+1, qp_j, qp_j+1}
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) return;
  const int Nq = G * Nd, Hq = Hkv * G;
  const int s_last = static_cast<int>((u1 - 1) / units_per_seg);

  // State of the warp's current unit.  Its first kPF chunks and its sequence
  // length are requested as soon as the unit is known; the block rows are
  // clamped to the summary capacity (always inside the arrays), so the loads
  // do not wait for the length.  Rows at or past nc are never written.
  int s = 0, base = 0, Lraw = 0;
  int bl[NB];
  const uint4 *pmn = nullptr, *pmx = nullptr;
  uint4 bmn[kPF][NB], bmx[kPF][NB];
  auto start_unit = [&](int64_t u) {
    s = static_cast<int>(u / units_per_seg);
    base = static_cast<int>(u % units_per_seg) * kUnit;
#pragma unroll
    for (int i = 0; i < NB; ++i) bl[i] = min(base + lane + 32 * i, Nb_max - 1);
    pmn = reinterpret_cast<const uint4 *>(kmin) + static_cast<int64_t>(s) * CH * Nb_max;
    pmx = reinterpret_cast<const uint4 *>(kmax) + static_cast<int64_t>(s) * CH * Nb_max;
#pragma unroll
    for (int p = 0; p < kPF; ++p)
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        bmn[p][i] = ld_summary(pmn + static_cast<int64_t>(p) * Nb_max + bl[i]);
        bmx[p][i] = ld_summary(pmx + static_cast<int64_t>(p) * Nb_max + bl[i]);
      }
    Lraw = __ldg(seq_len + s / Hkv);
  };

  for (int s_lo = static_cast<int>(u0 / units_per_seg); s_lo <= s_last; s_lo += qseg) {
    const int s_hi = min(s_last + 1, s_lo + qseg);  // segments [s_lo, s_hi) in this phase
    const int64_t pu0 = std::max(u0, static_cast<int64_t>(s_lo) * units_per_seg);
    const int64_t pu1 = std::min(u1, static_cast<int64_t>(s_hi) * units_per_seg);
    int64_t u = pu0 + warp;
    __syncthreads();  // the previous phase is done with qsm
    if (u < pu1) start_unit(u);

    // Query operands of the phase's segments: 16-byte loads of 8 dims of one
    // (padded) query each, kFill in flight per thread, then split into the
    // {qn, qn', qp, qp'} layout.  Item order (segment, chunk, query) keeps a
    // warp's stores spread over the banks.
    const int n_items = (s_hi - s_lo) * CH * NQP;
    for (int i0 = 0; i0 < n_items; i0 += kFill * kThreads) {
      uint4 raw[kFill];
#pragma unroll
      for (int k = 0; k < kFill; ++k) {
        const int idx = i0 + k * kThreads + tid;
        if (idx < n_items) {
          const int sl = idx / (CH * NQP), rem = idx % (CH * NQP), c = rem / NQP;
          const int j = min(rem % NQP, Nq - 1), jd = j / G, g = j % G;
          const int sq = s_lo + sl, bseq = sq / Hkv, h = sq % Hkv;
          raw[k] = __ldg(reinterpret_cast<const uint4 *>(
              qdraft + ((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + g) * D + c * 8));
        }
      }
#pragma unroll
      for (int k = 0; k < kFill; ++k) {
        const int idx = i0 + k * kThreads + tid;
        if (idx < n_items) {
          const int sl = idx / (CH * NQP), rem = idx % (CH * NQP), c = rem / NQP, j = rem % NQP;
          float *dst = reinterpret_cast<float *>(qsm + sl * per_seg_q + (c * 8) * (NQP / 2) + (j >> 1)) + (j & 1);
          const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float v = (e & 1) ? bf16_hi(w4[e >> 1]) : bf16_lo(w4[e >> 1]);
            const bool pos = v >= 0.0f;
            dst[e * (NQP / 2) * 4] = pos ? 0.0f : v;      // qn
            dst[e * (NQP / 2) * 4 + 2] = pos ? v : 0.0f;  // qp
          }
        }
      }
    }
    __syncthreads();

    for (; u < pu1; u += kWarps) {
      int L = Lraw;
      if (L < 0 || L > Nb_max * kBlockTokens) {
        if (lane == 0 && base == 0 && (s % Hkv) == 0) report(status, OASIS_STATUS_SEQ_LEN);
        L = L < 0 ? 0 : Nb_max * kBlockTokens;
      }
      const int nc = ceil_div(L, kBlockTokens) - W;
      if (base < nc) {  // warp-uniform
        const float4 *qbase = qsm + (s - s_lo) * per_seg_q;
        unsigned long long acc[NB][NQP / 2];
#pragma unroll
        for (int i = 0; i < NB; ++i)
#pragma unroll
          for (int jp = 0; jp < NQP / 2; ++jp) acc[i][jp] = 0ull;  // (+0, +0)
        // unrolled by kPF only (ring indices stay compile-time constants): the fully
        // unrolled body overflows the instruction cache
#pragma unroll 1
        for (int c0 = 0; c0 < CH; c0 += kPF)
#pragma unroll
          for (int cc = 0; cc < kPF; ++cc) {
            const int c = c0 + cc;
            uint4 mn[NB], mx[NB];
#pragma unroll
            for (int i = 0; i < NB; ++i) {
              mn[i] = bmn[cc][i];
              mx[i] = bmx[cc][i];
              if (c + kPF < CH) {
                bmn[cc][i] = ld_summary(pmn + static_cast<int64_t>(c + kPF) * Nb_max + bl[i]);
                bmx[cc][i] = ld_summary(pmx + static_cast<int64_t>(c + kPF) * Nb_max + bl[i]);
              }
            }
            const float4 *qrow = qbase + (c * 8) * (NQP / 2);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              unsigned long long kn2[NB], kx2[NB];
#pragma unroll
              for (int i = 0; i < NB; ++i) {
                const uint32_t wn = e < 2 ? mn[i].x : e < 4 ? mn[i].y : e < 6 ? mn[i].z : mn[i].w;
                const uint32_t wx = e < 2 ? mx[i].x : e < 4 ? mx[i].y : e < 6 ? mx[i].z : mx[i].w;
                const float fn = (e & 1) ? bf16_hi(wn) : bf16_lo(wn);
                const float fx = (e & 1) ? bf16_hi(wx) : bf16_lo(wx);
                kn2[i] = pack2(fn, fn);
                kx2[i] = pack2(fx, fx);
              }
#pragma unroll
              for (int jp = 0; jp < NQP / 2; ++jp) {
                const float4 qv = qrow[e * (NQP / 2) + jp];
                const unsigned long long qn2 = pack2(qv.x, qv.y), qp2 = pack2(qv.z, qv.w);
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                  acc[i][jp] = fma2(qn2, kn2[i], acc[i][jp]);
                  acc[i][jp] = fma2(qp2, kx2[i], acc[i][jp]);
                }
              }
            }
          }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          float best = -FLT_MAX;
#pragma unroll
          for (int jp = 0; jp < NQP / 2; ++jp) {
            float a0, a1;
            unpack2(acc[i][jp], a0, a1);
            best = jp == 0 ? max_nan(a0, a1) : max_nan(best, max_nan(a0, a1));  // NaN propagates
          }
          const int b = base + lane + 32 * i;
          if (b < nc) scores[static_cast<int64_t>(s) * Nb_max + b] = best;
        }
      }
      if (u + kWarps < pu1) start_unit(u + kWarps);
    }
  }
}

// ---- wide query groups (Nq > 16) ------------------------------------------
// The padded query pairs of a KV head are split into NG groups of kQG pairs.
// A round of a CTA takes WB consecutive units of 64 blocks; the NG warps of a
// unit score its blocks against one group each (the same inner loop as above,
// with 2*kQG query vectors), leave their per-block maxima in shared memory,
// and after a barrier the CTA writes the max over the groups.  The summary
// chunks a unit's warps share are read through L1 once per warp.
constexpr int kQG = 8;              // query pairs per warp (4 measured 13 % slower at 64 queries)
constexpr int kWarpsQGMax = 8;      // warps per CTA (NG <= 4 groups of a unit for up to 64 queries)
static_assert((64 / 2 + kQG - 1) / kQG <= kWarpsQGMax, "64 query vectors must fit one CTA's warps");

template <int CH>
__global__ void __maxnreg__(128)
    k_score_qg(const uint16_t *__restrict__ kmin, const uint16_t *__restrict__ kmax, int Nb_max,
               const uint16_t *__restrict__ qdraft, int S, int Hkv, int G, int Nd,
               const int32_t *__restrict__ seq_len, int W, float *__restrict__ scores, int32_t *status,
               int units_per_seg, int qseg, int NG) {
  constexpr int D = CH * 8;
  constexpr int NB = 2, kUnit = 64, kPF = 2;
  static_assert(CH % kPF == 0, "the chunk loop steps by kPF: it must divide the chunk count");
  const int npairs = NG * kQG;             // padded query pairs of a segment
  const int per_seg_q = D * npairs;        // float4 entries per segment
  extern __shared__ float4 qsm[];          // [qseg][D][npairs] {qn_j, qn_j+1, qp_j, qp_j+1}
  float *pm = reinterpret_cast<float *>(qsm + static_cast<int64_t>(qseg) * per_seg_q);  // [warps][64]
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int WB = nwarps / NG;              // units per round
  const int ub = warp / NG, grp = warp % NG;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) return;
  const int Nq = G * Nd, Hq = Hkv * G, nqv = 2 * npairs;
  const int s_last = static_cast<int>((u1 - 1) / units_per_seg);
  const int max_tokens = Nb_max * kBlockTokens;

  // State of the warp's current unit, as in k_score: its first kPF chunks and its
  // sequence length are requested as soon as the unit is known (before the
  // previous round's merge), block rows clamped to the summary capacity.
  int s = 0, base = 0, Lraw = 0;
  int bl[NB];
  const uint4 *pmn = nullptr, *pmx = nullptr;
  uint4 bmn[kPF][NB], bmx[kPF][NB];
  auto start_unit = [&](int64_t u) {
    s = static_cast<int>(u / units_per_seg);
    base = static_cast<int>(u % units_per_seg) * kUnit;
#pragma unroll
    for (int i = 0; i < NB; ++i) bl[i] = min(base + lane + 32 * i, Nb_max - 1);
    pmn = reinterpret_cast<const uint4 *>(kmin) + static_cast<int64_t>(s) * CH * Nb_max;
    pmx = reinterpret_cast<const uint4 *>(kmax) + static_cast<int64_t>(s) * CH * Nb_max;
#pragma unroll
    for (int p = 0; p < kPF; ++p)
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        bmn[p][i] = __ldg(pmn + static_cast<int64_t>(p) * Nb_max + bl[i]);
        bmx[p][i] = __ldg(pmx + static_cast<int64_t>(p) * Nb_max + bl[i]);
      }
    Lraw = __ldg(seq_len + s / Hkv);
  };

  for (int s_lo = static_cast<int>(u0 / units_per_seg); s_lo <= s_last; s_lo += qseg) {
    const int s_hi = min(s_last + 1, s_lo + qseg);
    const int64_t pu0 = std::max(u0, static_cast<int64_t>(s_lo) * units_per_seg);
    const int64_t pu1 = std::min(u1, static_cast<int64_t>(s_hi) * units_per_seg);
    __syncthreads();  // the previous phase is done with qsm
    if (ub < WB && pu0 + ub < pu1) start_unit(pu0 + ub);
    const int n_items = (s_hi - s_lo) * CH * nqv;
    for (int idx = tid; idx < n_items; idx += nthreads) {
      const int sl = idx / (CH * nqv), rem = idx % (CH * nqv), c = rem / nqv, j = rem % nqv;
      const int jq = min(j, Nq - 1), jd = jq / G, gq = jq % G;
      const int sq = s_lo + sl, bseq = sq / Hkv, h = sq % Hkv;
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
          qdraft + ((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + gq) * D + c * 8));
      float *dst = reinterpret_cast<float *>(qsm + sl * per_seg_q + (c * 8) * npairs + (j >> 1)) + (j & 1);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float v = (e & 1) ? bf16_hi(w4[e >> 1]) : bf16_lo(w4[e >> 1]);
        const bool pos = v >= 0.0f;
        dst[e * npairs * 4] = pos ? 0.0f : v;      // qn
        dst[e * npairs * 4 + 2] = pos ? v : 0.0f;  // qp
      }
    }
    __syncthreads();

    for (int64_t r0 = pu0; r0 < pu1; r0 += WB) {
      const int64_t u = r0 + ub;
      float best[NB] = {-FLT_MAX, -FLT_MAX};
      if (ub < WB && u < pu1) {
        int L = Lraw;
        if (L < 0 || L > max_tokens) {
          if (lane == 0 && grp == 0 && base == 0 && (s % Hkv) == 0) report(status, OASIS_STATUS_SEQ_LEN);
          L = L < 0 ? 0 : max_tokens;
        }
        const int nc = ceil_div(L, kBlockTokens) - W;
        if (base < nc) {  // warp-uniform
          const float4 *qbase = qsm + (s - s_lo) * per_seg_q + grp * kQG;
          unsigned long long acc[NB][kQG];
#pragma unroll
          for (int i = 0; i < NB; ++i)
#pragma unroll
            for (int jp = 0; jp < kQG; ++jp) acc[i][jp] = 0ull;  // (+0, +0)
#pragma unroll 1
          for (int c0 = 0; c0 < CH; c0 += kPF)
#pragma unroll
            for (int cc = 0; cc < kPF; ++cc) {
              const int c = c0 + cc;
              uint4 mn[NB], mx[NB];
#pragma unroll
              for (int i = 0; i < NB; ++i) {
                mn[i] = bmn[cc][i];
                mx[i] = bmx[cc][i];
                if (c + kPF < CH) {
                  bmn[cc][i] = __ldg(pmn + static_cast<int64_t>(c + kPF) * Nb_max + bl[i]);
                  bmx[cc][i] = __ldg(pmx + static_cast<int64_t>(c + kPF) * Nb_max + bl[i]);
                }
              }
              const float4 *qrow = qbase + (c * 8) * npairs;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                unsigned long long kn2[NB], kx2[NB];
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                  const uint32_t wn = e < 2 ? mn[i].x : e < 4 ? mn[i].y : e < 6 ? mn[i].z : mn[i].w;
                  const uint32_t wx = e < 2 ? mx[i].x : e < 4 ? mx[i].y : e < 6 ? mx[i].z : mx[i].w;
                  const float fn = (e & 1) ? bf16_hi(wn) : bf16_lo(wn);
                  const float fx = (e & 1) ? bf16_hi(wx) : bf16_lo(wx);
                  kn2[i] = pack2(fn, fn);
                  kx2[i] = pack2(fx, fx);
                }
#pragma unroll
                for (int jp = 0; jp < kQG; ++jp) {
                  const float4 qv = qrow[e * npairs + jp];
                  const unsigned long long qn2 = pack2(qv.x, qv.y), qp2 = pack2(qv.z, qv.w);
#pragma unroll
                  for (int i = 0; i < NB; ++i) {
                    acc[i][jp] = fma2(qn2, kn2[i], acc[i][jp]);
                    acc[i][jp] = fma2(qp2, kx2[i], acc[i][jp]);
                  }
                }
              }
            }
#pragma unroll
          for (int i = 0; i < NB; ++i)
#pragma unroll
            for (int jp = 0; jp < kQG; ++jp) {
              float a0, a1;
              unpack2(acc[i][jp], a0, a1);
              best[i] = max_nan(best[i], max_nan(a0, a1));  // NaN propagates
            }
        }
        // the next round's unit: its loads overlap this round's merge
        if (u + WB < pu1) start_unit(u + WB);
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) pm[warp * kUnit + lane + 32 * i] = best[i];
      __syncthreads();
      for (int t = tid; t < WB * kUnit; t += nthreads) {
        const int64_t uu = r0 + t / kUnit;
        if (uu >= pu1) continue;
        const int su = static_cast<int>(uu / units_per_seg);
        const int b = static_cast<int>(uu % units_per_seg) * kUnit + t % kUnit;
        int Lu = __ldg(seq_len + su / Hkv);
        Lu = Lu < 0 ? 0 : (Lu > max_tokens ? max_tokens : Lu);
        if (b >= ceil_div(Lu, kBlockTokens) - W) continue;
        const float *col = pm + (t / kUnit) * NG * kUnit + t % kUnit;
        float m = col[0];
        for (int gq = 1; gq < NG; ++gq) m = max_nan(m, col[gq * kUnit]);
        scores[static_cast<int64_t>(su) * Nb_max + b] = m;
      }
      __syncthreads();  // pm is rewritten next round
    }
  }
}

template <int CH>
cudaError_t launch_qg(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                      int Hkv, int G, int Nd, const int32_t *seq_len, int W, float *scores, int32_t *status,
                      cudaStream_t st) {
  constexpr int D = CH * 8;
  const int S = B * Hkv;
  const int Nq = G * Nd;
  const int NG = ((Nq + 1) / 2 + kQG - 1) / kQG;
  if (NG < 1 || NG > kWarpsQGMax) return cudaErrorInvalidValue;  // one warp per group, at most kWarpsQGMax
  const int WB = std::max(1, kWarpsQGMax / NG);
  const int threads = 32 * NG * WB;
  const int ncand = std::max(1, Nb_max - W);
  const int units_per_seg = (ncand + 63) / 64;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const size_t per_seg = sizeof(float4) * static_cast<size_t>(D) * NG * kQG;
  const size_t pm_bytes = sizeof(float) * 64 * (threads / 32);  // one row of partial maxima per warp
  const int qseg_max = static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, (100 * 1024) / per_seg)));
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_score_qg<CH>), threads,
                                  per_seg * qseg_max + pm_bytes, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(sms) * per_sm, U));
  const int64_t per_cta = (U + grid - 1) / grid;
  const int qseg = static_cast<int>(std::min<int64_t>(qseg_max, (per_cta + units_per_seg - 1) / units_per_seg + 1));
  LaunchCfg lc(dim3(grid), dim3(threads), per_seg * qseg + pm_bytes, st);
  return cudaLaunchKernelEx(&lc.cfg, k_score_qg<CH>, kmin, kmax, Nb_max, qdraft, S, Hkv, G, Nd, seq_len, W, scores,
                            status, units_per_seg, qseg, NG);
}

template <int NQP, int CH>
cudaError_t launch_nqp_ch(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                          int Hkv, int G, int Nd, const int32_t *seq_len, int W, float *scores, int32_t *status,
                          cudaStream_t st) {
  constexpr int D = CH * 8;
  const int S = B * Hkv;
  const int ncand = std::max(1, Nb_max - W);
  constexpr int kUnit = 32 * blocks_per_lane<NQP>();
  const int units_per_seg = (ncand + kUnit - 1) / kUnit;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const size_t per_seg = sizeof(float4) * static_cast<size_t>(D) * (NQP / 2);
  const int qseg_max = static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, smem_budget<NQP>() / per_seg)));
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_score<NQP, CH>), kThreads, per_seg * qseg_max,
                                  &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(std::min<int64_t>(want, U));  // every CTA gets >= 1 unit
  // segments a CTA's unit range can touch: shared memory for just those (a small
  // footprint leaves room for the kernels running beside this one)
  const int64_t per_cta = (U + grid - 1) / grid;
  const int qseg = static_cast<int>(std::min<int64_t>(qseg_max, (per_cta + units_per_seg - 1) / units_per_seg + 1));
  const size_t smem = per_seg * qseg;
  LaunchCfg lc(dim3(grid), dim3(kThreads), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_score<NQP, CH>, kmin, kmax, Nb_max, qdraft, S, Hkv, G, Nd, seq_len, W, scores,
                            status, units_per_seg, qseg);
}

template <int NQP>
cudaError_t launch_nqp(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                       int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W, float *scores,
                       int32_t *status, cudaStream_t st) {
  if (D == 128)
    return launch_nqp_ch<NQP, 16>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, status, st);
  return launch_nqp_ch<NQP, 8>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, status, st);
}

}  // namespace

cudaError_t launch_score_blocks(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft,
                                int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                                float *scores, int32_t *status, cudaStream_t st) {
  const int Nq = G * Nd;
  // up to 16 query vectors: every query in one warp (measured faster at 16: 208 vs
  // 219 us on the 128-head, 8192-block layer); more: query groups over warps
  // (434 vs 510 us at 64 query vectors on the 256-head layer)
  if (Nq > 16) {
    if (D == 128) return launch_qg<16>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, status, st);
    return launch_qg<8>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, status, st);
  }
#define OASIS_SCORE_CASE(N) \
  if (Nq <= N) return launch_nqp<N>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  OASIS_SCORE_CASE(2)
  OASIS_SCORE_CASE(4)
  OASIS_SCORE_CASE(8)
  OASIS_SCORE_CASE(12)
  OASIS_SCORE_CASE(16)
#undef OASIS_SCORE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace oasis
