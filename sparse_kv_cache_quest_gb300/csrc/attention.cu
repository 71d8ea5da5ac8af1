// Sparse paged decode attention over the head-wise logical-to-logical table.
//
// OasisKV paper review (xllm-io), §3 Fig. 5: the foreground forward pass runs
// sparse attention of the true query over the working set resident in HBM;
// §4 / Fig. 9: each KV head addresses its own resident blocks through the
// head-wise mapping.  For query head h*G + g of sequence b:
//     out = sum_i softmax_i(scale * q . k_i) v_i
// over the valid tokens of the slots whose table entry is >= 0.
//
// Data path.  A segment's pool is slots_per_seg contiguous 8 KiB tiles (K then
// V, D = 128).  The segment is split over a thread-block cluster of CL CTAs
// (split-K): CTA rank r takes a contiguous slot range, and inside it warp w
// takes every 4th slot.  Each warp streams its tiles through a private ring of
// NST shared-memory stages with 1-D bulk async copies (cp.async.bulk, one
// mbarrier per stage, lane 0 issues), so up to NST tiles per warp are in
// flight.  Empty slots and slots without valid tokens are never loaded.
//
// Math.  A warp works on one 16-token slot at a time: lane (tsub, dpart) owns
// dims dpart*VEC .. dpart*VEC + VEC - 1 of tokens 2u + tsub (u < 8).  Partial
// dots are summed over the 16 lanes of a half with xor shuffles; the online
// softmax runs in the log2 domain (q is pre-multiplied by scale * log2(e),
// exp2f), with per-warp running max m, sum l and output o[g][dims] in fp32.
// Warps combine through shared memory, then the CL CTAs of the cluster
// combine through distributed shared memory into rank 0, which writes out and
// lse.  No global scratch memory is used.
//
// G > 8 is processed in query-head tiles of 8 (separate clusters).
#include <cooperative_groups.h>

#include <cfloat>
#include <cstdlib>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace oasis {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kWaitTries = 1u << 22;  // bounded mbarrier polls (far beyond any real copy)
constexpr float kLn2 = 0.69314718055994530942f;

template <int VEC>
__device__ __forceinline__ void load_row(const uint16_t *p, float (&f)[VEC]) {
  if constexpr (VEC == 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  } else {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  }
}

template <int VEC, int GT, int NST>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn(const uint16_t *__restrict__ q, const uint16_t *__restrict__ pool, const int32_t *__restrict__ table,
           int slots, const int32_t *__restrict__ seq_len, int Hkv, int G, int ntiles, float scale_log2,
           float *__restrict__ out, float *__restrict__ lse, int32_t *status) {
  constexpr int D = 16 * VEC;
  constexpr uint32_t kTileBytes = 64u * D;
  extern __shared__ __align__(128) unsigned char sm[];
  cg::cluster_group cluster = cg::this_cluster();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tsub = lane >> 4, dpart = lane & 15;
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int s = blockIdx.y / ntiles, tile = blockIdx.y % ntiles;
  const int bseq = s / Hkv, h = s % Hkv;
  const int g0 = tile * GT;
  const int gcount = min(GT, G - g0);
  const int Hq = Hkv * G;

  int L = seq_len[bseq];
  if (L < 0) {
    if (tid == 0 && rank == 0 && h == 0 && tile == 0) report(status, OASIS_STATUS_SEQ_LEN);
    L = 0;
  }

  unsigned char *ring = sm + static_cast<size_t>(warp) * NST * kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + static_cast<size_t>(kWarps) * NST * kTileBytes) + warp * NST;
  float *red = reinterpret_cast<float *>(sm + static_cast<size_t>(kWarps) * NST * kTileBytes +
                                         sizeof(uint64_t) * kWarps * NST);
  float *wm = red;                          // [kWarps][GT]
  float *wl = wm + kWarps * GT;             // [kWarps][GT]
  float *wo = wl + kWarps * GT;             // [kWarps][GT][D]
  float *cm = wo + kWarps * GT * D;         // [GT]   CTA partials, read by cluster rank 0
  float *cl = cm + GT;                      // [GT]
  float *co = cl + GT;                      // [GT][D]

  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // queries of this lane's dims, pre-scaled into the log2 domain
  float qr[GT][VEC];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    if (g < gcount) {
      float f[VEC];
      load_row<VEC>(q + (static_cast<int64_t>(bseq) * Hq + h * G + g0 + g) * D + dpart * VEC, f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) qr[g][e] = f[e] * scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) qr[g][e] = 0.0f;
    }
  }
  float m[GT], l[GT], o[GT][VEC];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[g][e] = 0.0f;
  }

  const int per = (slots + CL - 1) / CL;
  const int lo = min(slots, rank * per), hi = min(slots, lo + per);
  const int nk = hi - lo > warp ? (hi - lo - warp + kWarps - 1) / kWarps : 0;
  const int32_t *trow = table + static_cast<int64_t>(s) * slots;
  const uint16_t *prow = pool + static_cast<int64_t>(s) * slots * 32 * D;
  auto slot_of = [&](int k) { return lo + warp + kWarps * k; };
  auto nvalid_of = [&](int k) {
    const int blk = trow[slot_of(k)];
    if (blk < 0) return 0;
    const int64_t n = static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
    return n <= 0 ? 0 : (n >= kBlockTokens ? kBlockTokens : static_cast<int>(n));
  };
  auto next_valid = [&](int k) {
    while (k < nk && nvalid_of(k) == 0) ++k;
    return k;
  };

  int ki = next_valid(0), issued = 0;
  while (issued < NST && ki < nk) {
    if (lane == 0) {
      const int stg = issued % NST;
      mbar_arrive_expect_tx(&bars[stg], kTileBytes);
      bulk_g2s(ring + stg * kTileBytes, prow + static_cast<int64_t>(slot_of(ki)) * 32 * D, kTileBytes, &bars[stg]);
    }
    ++issued;
    ki = next_valid(ki + 1);
  }

  int kc = next_valid(0), consumed = 0;
  bool timed_out = false;
  while (kc < nk) {
    const int stg = consumed % NST;
    const bool ok = mbar_wait_bounded(&bars[stg], static_cast<uint32_t>(consumed / NST) & 1u, kWaitTries);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      timed_out = true;
      break;
    }
    const int nv = nvalid_of(kc);
    const uint16_t *kt = reinterpret_cast<const uint16_t *>(ring + stg * kTileBytes);
    const uint16_t *vt = kt + kBlockTokens * D;

    float sc[GT][8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float kf[VEC];
      load_row<VEC>(kt + (2 * u + tsub) * D + dpart * VEC, kf);
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float a = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a = fmaf(qr[g][e], kf[e], a);
        sc[g][u] = a;
      }
    }
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float a = sc[g][u];
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 8);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 4);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
        sc[g][u] = (2 * u + tsub < nv) ? a : -INFINITY;
      }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float mx = sc[g][0];
#pragma unroll
      for (int u = 1; u < 8; ++u) mx = fmaxf(mx, sc[g][u]);
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float mnew = fmaxf(m[g], mx);
      const float corr = exp2f(m[g] - mnew);
      float ps = 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float p = exp2f(sc[g][u] - mnew);
        sc[g][u] = p;
        ps += p;
      }
      l[g] = l[g] * corr + ps;
      m[g] = mnew;
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[g][e] *= corr;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float vf[VEC];
      load_row<VEC>(vt + (2 * u + tsub) * D + dpart * VEC, vf);
#pragma unroll
      for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[g][e] = fmaf(sc[g][u], vf[e], o[g][e]);
    }
    __syncwarp();
    ++consumed;
    if (ki < nk) {
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[stg], kTileBytes);
        bulk_g2s(ring + stg * kTileBytes, prow + static_cast<int64_t>(slot_of(ki)) * 32 * D, kTileBytes,
                 &bars[stg]);
      }
      ++issued;
      ki = next_valid(ki + 1);
    }
    kc = next_valid(kc + 1);
  }
  if (timed_out) {
    if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
    for (int c = consumed; c < issued; ++c) mbar_wait_bounded(&bars[c % NST], static_cast<uint32_t>(c / NST) & 1u, kWaitTries);
  }

  // combine the two token halves of the warp, then the warps of the CTA
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    l[g] += __shfl_xor_sync(0xFFFFFFFFu, l[g], 16);
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[g][e] += __shfl_xor_sync(0xFFFFFFFFu, o[g][e], 16);
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      wm[warp * GT + g] = m[g];
      wl[warp * GT + g] = l[g];
    }
  }
  if (tsub == 0) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int e = 0; e < VEC; ++e) wo[(warp * GT + g) * D + dpart * VEC + e] = o[g][e];
  }
  __syncthreads();
  for (int idx = tid; idx < GT * D; idx += kThreads) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * GT + g]);
    float acc = 0.0f, ls = 0.0f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(wm[w * GT + g] - M);
        acc += f * wo[(w * GT + g) * D + d];
        ls += f * wl[w * GT + g];
      }
    }
    co[g * D + d] = acc;
    if (d == 0) {
      cm[g] = M;
      cl[g] = ls;
    }
  }
  cluster.sync();
  if (rank == 0) {
    for (int idx = tid; idx < GT * D; idx += kThreads) {
      const int g = idx / D, d = idx % D;
      if (g >= gcount) continue;
      float M = -INFINITY;
      for (int r = 0; r < CL; ++r) M = fmaxf(M, cluster.map_shared_rank(cm, r)[g]);
      float acc = 0.0f, ls = 0.0f;
      if (M > -INFINITY) {
        for (int r = 0; r < CL; ++r) {
          const float f = exp2f(cluster.map_shared_rank(cm, r)[g] - M);
          acc += f * cluster.map_shared_rank(co, r)[g * D + d];
          ls += f * cluster.map_shared_rank(cl, r)[g];
        }
      }
      const int64_t row = static_cast<int64_t>(bseq) * Hq + h * G + g0 + g;
      out[row * D + d] = ls > 0.0f ? acc / ls : 0.0f;
      if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
    }
  }
  cluster.sync();
}

int env_int(const char *name, int dflt) {
  const char *v = std::getenv(name);
  return v != nullptr ? std::atoi(v) : dflt;
}

template <int VEC, int GT, int NST>
cudaError_t launch_t(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                     const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                     int32_t *status, cudaStream_t st) {
  constexpr int D = 16 * VEC;
  const int ntiles = (G + GT - 1) / GT;
  const int units = B * Hkv * ntiles;
  int CL = env_int("OASIS_ATTN_CLUSTER", 0);
  if (CL <= 0) {
    CL = 1;
    while (CL < 8 && units * CL * 2 <= 2 * 152) CL *= 2;
  }
  const size_t smem = static_cast<size_t>(kWarps) * NST * 64 * D + sizeof(uint64_t) * kWarps * NST +
                      sizeof(float) * (2 * kWarps * GT + kWarps * GT * D + 2 * GT + GT * D);
  cudaError_t e = cudaFuncSetAttribute(k_attn<VEC, GT, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_attn<VEC, GT, NST>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(CL), static_cast<unsigned>(units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, k_attn<VEC, GT, NST>, q, pool, table, slots, seq_len, Hkv, G, ntiles,
                            scale_log2, out, lse, status);
}

template <int VEC>
cudaError_t launch_vec(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                       const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                       int32_t *status, cudaStream_t st) {
  constexpr int NST = VEC == 8 ? 3 : 4;
  if (G == 1) return launch_t<VEC, 1, NST>(q, pool, table, slots, seq_len, B, Hkv, G, scale, out, lse, status, st);
  if (G == 2) return launch_t<VEC, 2, NST>(q, pool, table, slots, seq_len, B, Hkv, G, scale, out, lse, status, st);
  if (G <= 4) return launch_t<VEC, 4, NST>(q, pool, table, slots, seq_len, B, Hkv, G, scale, out, lse, status, st);
  return launch_t<VEC, 8, NST>(q, pool, table, slots, seq_len, B, Hkv, G, scale, out, lse, status, st);
}

}  // namespace

cudaError_t launch_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                      int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                      float scale, float *out, float *lse, int32_t *status, cudaStream_t st) {
  if (D == 128)
    return launch_vec<8>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
  return launch_vec<4>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, status, st);
}

}  // namespace oasis
