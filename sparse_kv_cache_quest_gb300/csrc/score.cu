// Look-ahead block scoring: the draft queries of a KV head scan its min/max
// key summaries (OasisKV paper review (xllm-io), §3 decode flow: "draft query
// scans the compressed key summary -> predicts top-K blocks"; §4 Fig. 7).
//
//   score[s][b] = max over the Nq = G*Nd query vectors of
//                 sum_{d ascending, from +0, fp32 RN} q_d * (q_d >= 0 ? kmax_d : kmin_d)
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
// segment, NB blocks per lane of a warp (NB = 2 while the accumulators fit).  Units are numbered segment-major and
// each CTA of a persistent grid (SM count x resident CTAs per SM) takes one
// contiguous range of units, so every SM gets the same number of units (+-1)
// whatever the segment count.  A CTA walks the segments of its range in phases
// of at most `qseg` segments whose query operands it holds in shared memory;
// its warps take the units of a phase round-robin.
//
// Data path.  Each warp streams the 8-dim chunks of its units (a chunk of a
// 64-block unit is 1 KiB of kmin and 1 KiB of kmax, contiguous in the
// chunk-major layout [S][D/8][Nb][8]) through a private ring of kNS stages
// with 1-D bulk async copies (cp.async.bulk + mbarrier), across unit
// boundaries; a stage is refilled as soon as its data is in registers.  Every
// mbarrier wait is bounded and reports OASIS_STATUS_TIMEOUT instead of hanging.
// Inner loop.  Per dim it widens kmin/kmax to fp32 and
// runs two packed fp32x2 FMAs (fma.rn.f32x2) per pair of queries and block:
// the query operands sit in shared memory as {qn_j, qn_j+1, qp_j, qp_j+1}, one
// broadcast 16-byte load per pair and dim feeding 2*NB packed FMAs.  Queries are padded to NQP by repeating the
// last one, which leaves the max unchanged.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kNB = 2;               // blocks per lane
constexpr int kUnit = 32 * kNB;      // blocks per warp unit
constexpr int kNS = 4;               // ring stages per warp (one 8-dim chunk of a unit each)
constexpr int kStage = 2 * kUnit * 16;  // kmin then kmax: 64 blocks x 16 bytes each
constexpr uint32_t kWaitTries = 1u << 22;
constexpr size_t kQBudget = 40 * 1024;  // query operands of the segments of one phase

// CH = D / 8 chunks of 8 dims (8 for D = 64, 16 for D = 128).
template <int NQP, int CH>
__global__ void __launch_bounds__(kThreads, NQP <= 24 ? 2 : 1)
    k_score(const uint16_t *__restrict__ kmin, const uint16_t *__restrict__ kmax, int Nb_max,
            const uint16_t *__restrict__ qdraft, int S, int Hkv, int G, int Nd, const int32_t *__restrict__ seq_len,
            int W, float *__restrict__ scores, int32_t *status, int units_per_seg, int qseg) {
  constexpr int D = CH * 8;
  constexpr int per_seg_q = D * (NQP / 2);
  extern __shared__ __align__(16) unsigned char smraw[];
  unsigned char *rings = smraw;                                           // [kWarps][kNS][kStage]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smraw + kWarps * kNS * kStage);  // [kWarps][kNS]
  float4 *qsm = reinterpret_cast<float4 *>(bars + kWarps * kNS);        // [qseg][D][NQP/2]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) return;
  const int Nq = G * Nd, Hq = Hkv * G;
  const int s_last = static_cast<int>((u1 - 1) / units_per_seg);
  unsigned char *ring = rings + warp * kNS * kStage;
  uint64_t *wbar = bars + warp * kNS;
  if (lane == 0) {
    for (int i = 0; i < kNS; ++i) mbar_init(&wbar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  uint32_t phase_bits = 0;  // parity of the next completion of each stage (bit per stage)
  bool timed_out = false;

  for (int s_lo = static_cast<int>(u0 / units_per_seg); s_lo <= s_last; s_lo += qseg) {
    const int s_hi = min(s_last + 1, s_lo + qseg);  // segments [s_lo, s_hi) in this phase
    __syncthreads();                                // the previous phase is done with qsm
    for (int idx = tid; idx < (s_hi - s_lo) * per_seg_q; idx += kThreads) {
      const int sl = idx / per_seg_q, rem = idx % per_seg_q;
      const int d = rem / (NQP / 2), jp = rem % (NQP / 2);
      const int s = s_lo + sl, bseq = s / Hkv, h = s % Hkv;
      float qv[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int j = min(2 * jp + t, Nq - 1);
        const int jd = j / G, g = j % G;
        const uint16_t raw = qdraft[((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + g) * D + d];
        qv[t] = __uint_as_float(static_cast<uint32_t>(raw) << 16);
      }
      const bool p0 = qv[0] >= 0.0f, p1 = qv[1] >= 0.0f;
      qsm[idx] = make_float4(p0 ? 0.0f : qv[0], p1 ? 0.0f : qv[1], p0 ? qv[0] : 0.0f, p1 ? qv[1] : 0.0f);
    }
    __syncthreads();

    // this warp's units of the phase: pu0 + warp + j * kWarps; items (j, chunk) in order
    const int64_t pu0 = std::max(u0, static_cast<int64_t>(s_lo) * units_per_seg);
    const int64_t pu1 = std::min(u1, static_cast<int64_t>(s_hi) * units_per_seg);
    const int nunits = pu1 > pu0 + warp ? static_cast<int>((pu1 - pu0 - warp + kWarps - 1) / kWarps) : 0;
    const int nitems = nunits * CH;
    auto issue = [&](int i) {  // lane 0: bulk-copy item i into stage i % kNS
      const int64_t u = pu0 + warp + static_cast<int64_t>(i / CH) * kWarps;
      const int c = i % CH;
      const int s = static_cast<int>(u / units_per_seg);
      const int base = static_cast<int>(u % units_per_seg) * kUnit;
      const uint32_t bytes = static_cast<uint32_t>(min(kUnit, Nb_max - base)) * 16u;
      const int64_t off = ((static_cast<int64_t>(s) * CH + c) * Nb_max + base) * 8;
      unsigned char *dst = ring + (i % kNS) * kStage;
      mbar_arrive_expect_tx(&wbar[i % kNS], 2 * bytes);
      bulk_g2s(dst, kmin + off, bytes, &wbar[i % kNS]);
      bulk_g2s(dst + kUnit * 16, kmax + off, bytes, &wbar[i % kNS]);
    };
    if (lane == 0 && !timed_out)
      for (int i = 0; i < kNS && i < nitems; ++i) issue(i);

    // after a timed-out wait the warp skips its remaining work but still meets
    // every CTA barrier of the later phases
    unsigned long long acc[kNB][NQP / 2];
    for (int j = 0; j < nunits && !timed_out; ++j) {
      const int64_t u = pu0 + warp + static_cast<int64_t>(j) * kWarps;
      const int s = static_cast<int>(u / units_per_seg);
      const int base = static_cast<int>(u % units_per_seg) * kUnit;
      const int L = load_len(seq_len, s / Hkv, Nb_max * kBlockTokens, status,
                             lane == 0 && base == 0 && (s % Hkv) == 0);
      const int nc = ceil_div(L, kBlockTokens) - W;
      const float4 *qbase = qsm + (s - s_lo) * per_seg_q;
#pragma unroll
      for (int i = 0; i < kNB; ++i)
#pragma unroll
        for (int jp = 0; jp < NQP / 2; ++jp) acc[i][jp] = 0ull;  // (+0, +0)
#pragma unroll 1
      for (int c = 0; c < CH; ++c) {
        const int it = j * CH + c, stg = it % kNS;
        const bool ok = mbar_wait_bounded(&wbar[stg], (phase_bits >> stg) & 1u, kWaitTries);
        phase_bits ^= 1u << stg;
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          timed_out = true;
          break;
        }
        const uint4 *st4 = reinterpret_cast<const uint4 *>(ring + stg * kStage);
        uint4 mn[kNB], mx[kNB];
#pragma unroll
        for (int i = 0; i < kNB; ++i) {
          mn[i] = st4[lane + 32 * i];
          mx[i] = st4[kUnit + lane + 32 * i];
        }
        __syncwarp();  // the stage is in registers: refill it at once
        if (lane == 0 && it + kNS < nitems) {
          fence_proxy_async_smem();
          issue(it + kNS);
        }
        if (base >= nc) continue;  // empty unit (warp-uniform): loaded, not scored
        const float4 *qrow = qbase + (c * 8) * (NQP / 2);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          unsigned long long kn2[kNB], kx2[kNB];
#pragma unroll
          for (int i = 0; i < kNB; ++i) {
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
            for (int i = 0; i < kNB; ++i) {
              acc[i][jp] = fma2(qn2, kn2[i], acc[i][jp]);
              acc[i][jp] = fma2(qp2, kx2[i], acc[i][jp]);
            }
          }
        }
      }
      if (timed_out || base >= nc) continue;  // (the j loop ends after a timeout)
#pragma unroll
      for (int i = 0; i < kNB; ++i) {
        float best = -FLT_MAX;
#pragma unroll
        for (int jp = 0; jp < NQP / 2; ++jp) {
          float a0, a1;
          unpack2(acc[i][jp], a0, a1);
          best = jp == 0 ? fmaxf(a0, a1) : fmaxf(best, fmaxf(a0, a1));
        }
        const int b = base + lane + 32 * i;
        if (b < nc) scores[static_cast<int64_t>(s) * Nb_max + b] = best;
      }
    }
  }
  if (timed_out && lane == 0) report(status, OASIS_STATUS_TIMEOUT);
}

template <int NQP, int CH>
cudaError_t launch_nqp_ch(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                          int Hkv, int G, int Nd, const int32_t *seq_len, int W, float *scores, int32_t *status,
                          cudaStream_t st) {
  constexpr int D = CH * 8;
  const int S = B * Hkv;
  const int ncand = std::max(1, Nb_max - W);
  const int units_per_seg = (ncand + kUnit - 1) / kUnit;
  const int64_t U = static_cast<int64_t>(S) * units_per_seg;
  const size_t per_seg = sizeof(float4) * static_cast<size_t>(D) * (NQP / 2);
  const int qseg = static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, kQBudget / per_seg)));
  const size_t smem = static_cast<size_t>(kWarps) * kNS * (kStage + sizeof(uint64_t)) + per_seg * qseg;
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_score<NQP, CH>), kThreads, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(std::min<int64_t>(want, U));  // every CTA gets >= 1 unit
  k_score<NQP, CH><<<grid, kThreads, smem, st>>>(kmin, kmax, Nb_max, qdraft, S, Hkv, G, Nd, seq_len, W, scores,
                                                  status, units_per_seg, qseg);
  return cudaGetLastError();
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
#define OASIS_SCORE_CASE(N) \
  if (Nq <= N) return launch_nqp<N>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  OASIS_SCORE_CASE(2)
  OASIS_SCORE_CASE(4)
  OASIS_SCORE_CASE(8)
  OASIS_SCORE_CASE(12)
  OASIS_SCORE_CASE(16)
  OASIS_SCORE_CASE(24)
  OASIS_SCORE_CASE(32)
  OASIS_SCORE_CASE(48)
  OASIS_SCORE_CASE(64)
#undef OASIS_SCORE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace oasis
