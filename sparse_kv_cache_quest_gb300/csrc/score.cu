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
// Mapping.  A CTA of 128 threads covers 128*NB consecutive candidate blocks of
// one segment; thread t owns blocks base + t + 128*i (i < NB).  The chunk-major
// summary layout [S][D/8][Nb][8] makes every 16-byte load of a warp part of
// one contiguous 512-byte run.  Accumulators of block pairs are packed fp32x2
// registers (fma.rn.f32x2), which halves the issue slots of the FMAs; the
// query operands sit in shared memory pre-split and pre-duplicated as
// {qp, qp, qn, qn}, one broadcast 16-byte load per (query, dim) feeding 2*NB/2
// packed FMAs.  Queries are processed in tiles of QT (padded by repeating the
// last query, which leaves the max unchanged); the next 8-dim chunk is loaded
// while the current one is consumed.
#include <cfloat>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 128;

template <int NB, int QT>
__global__ void __launch_bounds__(kThreads) k_score(const uint16_t *__restrict__ kmin,
                                                    const uint16_t *__restrict__ kmax, int Nb_max,
                                                    const uint16_t *__restrict__ qdraft, int Hkv, int G, int Nd,
                                                    int D, const int32_t *__restrict__ seq_len, int W,
                                                    float *__restrict__ scores, int32_t *status) {
  static_assert(NB % 2 == 0, "blocks are processed in packed pairs");
  extern __shared__ float4 qsm[];  // [D][nqp] {qp, qp, qn, qn}
  const int s = blockIdx.y;
  const int bseq = s / Hkv, h = s % Hkv;
  const int Nq = G * Nd;
  const int nqp = ((Nq + QT - 1) / QT) * QT;
  const int L = load_len(seq_len, bseq, Nb_max * kBlockTokens, status,
                         blockIdx.x == 0 && threadIdx.x == 0 && h == 0);
  const int nc = ceil_div(L, kBlockTokens) - W;
  const int base = blockIdx.x * kThreads * NB;
  if (base >= nc) return;  // uniform across the CTA

  const int Hq = Hkv * G;
  for (int idx = threadIdx.x; idx < D * nqp; idx += kThreads) {
    const int d = idx / nqp;
    const int j = min(idx % nqp, Nq - 1);
    const int jd = j / G, g = j % G;
    const uint16_t raw = qdraft[((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + g) * D + d];
    const float q = __uint_as_float(static_cast<uint32_t>(raw) << 16);
    const bool pos = q >= 0.0f;
    const float qp = pos ? q : 0.0f, qn = pos ? 0.0f : q;
    qsm[idx] = make_float4(qp, qp, qn, qn);
  }
  __syncthreads();

  int blk[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) blk[i] = min(base + static_cast<int>(threadIdx.x) + kThreads * i, nc - 1);
  const int chunks = D >> 3;
  const uint4 *pmin = reinterpret_cast<const uint4 *>(kmin) + static_cast<int64_t>(s) * chunks * Nb_max;
  const uint4 *pmax = reinterpret_cast<const uint4 *>(kmax) + static_cast<int64_t>(s) * chunks * Nb_max;

  float best[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) best[i] = -FLT_MAX;
  bool first_tile = true;

  for (int q0 = 0; q0 < nqp; q0 += QT) {
    unsigned long long acc[NB / 2][QT];
#pragma unroll
    for (int p = 0; p < NB / 2; ++p)
#pragma unroll
      for (int jj = 0; jj < QT; ++jj) acc[p][jj] = 0ull;  // (+0, +0)

    uint4 cmn[NB], cmx[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      cmn[i] = __ldg(pmin + blk[i]);
      cmx[i] = __ldg(pmax + blk[i]);
    }
    for (int c = 0; c < chunks; ++c) {
      uint4 nmn[NB], nmx[NB];
      const int cn = c + 1 < chunks ? c + 1 : c;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        nmn[i] = __ldg(pmin + static_cast<int64_t>(cn) * Nb_max + blk[i]);
        nmx[i] = __ldg(pmax + static_cast<int64_t>(cn) * Nb_max + blk[i]);
      }
      const float4 *qrow = qsm + (c * 8) * nqp + q0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        unsigned long long kn2[NB / 2], kx2[NB / 2];
#pragma unroll
        for (int p = 0; p < NB / 2; ++p) {
          const uint32_t wn0 = (&cmn[2 * p].x)[e >> 1], wn1 = (&cmn[2 * p + 1].x)[e >> 1];
          const uint32_t wx0 = (&cmx[2 * p].x)[e >> 1], wx1 = (&cmx[2 * p + 1].x)[e >> 1];
          if (e & 1) {
            kn2[p] = pack2(bf16_hi(wn0), bf16_hi(wn1));
            kx2[p] = pack2(bf16_hi(wx0), bf16_hi(wx1));
          } else {
            kn2[p] = pack2(bf16_lo(wn0), bf16_lo(wn1));
            kx2[p] = pack2(bf16_lo(wx0), bf16_lo(wx1));
          }
        }
#pragma unroll
        for (int jj = 0; jj < QT; ++jj) {
          const float4 qv = qrow[e * nqp + jj];
          const unsigned long long qp2 = pack2(qv.x, qv.y), qn2 = pack2(qv.z, qv.w);
#pragma unroll
          for (int p = 0; p < NB / 2; ++p) {
            acc[p][jj] = fma2(qn2, kn2[p], acc[p][jj]);
            acc[p][jj] = fma2(qp2, kx2[p], acc[p][jj]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        cmn[i] = nmn[i];
        cmx[i] = nmx[i];
      }
    }
#pragma unroll
    for (int p = 0; p < NB / 2; ++p)
#pragma unroll
      for (int jj = 0; jj < QT; ++jj) {
        float a0, a1;
        unpack2(acc[p][jj], a0, a1);
        if (first_tile && jj == 0) {
          best[2 * p] = a0;
          best[2 * p + 1] = a1;
        } else {
          best[2 * p] = fmaxf(best[2 * p], a0);
          best[2 * p + 1] = fmaxf(best[2 * p + 1], a1);
        }
      }
    first_tile = false;
  }

  float *out = scores + static_cast<int64_t>(s) * Nb_max;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = base + static_cast<int>(threadIdx.x) + kThreads * i;
    if (b < nc) out[b] = best[i];
  }
}

template <int NB, int QT>
cudaError_t launch_nb_qt(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                         int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W, float *scores,
                         int32_t *status, cudaStream_t st) {
  const int Nq = G * Nd;
  const int nqp = ((Nq + QT - 1) / QT) * QT;
  const size_t smem = sizeof(float4) * static_cast<size_t>(D) * nqp;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_score<NB, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>((Nb_max + kThreads * NB - 1) / (kThreads * NB)),
                  static_cast<unsigned>(B * Hkv));
  k_score<NB, QT><<<grid, kThreads, smem, st>>>(kmin, kmax, Nb_max, qdraft, Hkv, G, Nd, D, seq_len, W, scores,
                                                 status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_blocks(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft,
                                int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                                float *scores, int32_t *status, cudaStream_t st) {
  const int Nq = G * Nd;
  if (Nq <= 2) return launch_nb_qt<4, 2>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  if (Nq <= 4) return launch_nb_qt<4, 4>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  if (Nq <= 8) return launch_nb_qt<4, 8>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  if (Nq <= 12) return launch_nb_qt<4, 12>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
  return launch_nb_qt<4, 16>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores, status, st);
}

}  // namespace oasis
