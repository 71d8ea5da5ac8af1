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
// (split-K): the CL*4 warps of the cluster take the slots round-robin.  Each
// warp first lists its non-empty slots in shared memory (one table read per
// slot, off the streaming loop), then streams their tiles through a ring of
// NST shared-memory stages with 1-D bulk async copies (cp.async.bulk, one
// mbarrier per stage, lane 0 issues), so the next tile is in flight while one
// is consumed.  Empty slots and slots without valid tokens are never loaded.
//
// Math (CUDA cores: a GQA group of a few heads is no dense tensor-core tile).
// A warp works on one 16-token slot at a time.  Lane (tsub = lane/16,
// dpart = lane%16) owns dims dpart*VEC .. +VEC of tokens 2u + tsub (u < 8).
//  * QK: per lane, partial dots of its dims for its 8 tokens and the GT query
//    heads, two heads per packed fp32x2 FMA.  The lane visits its tokens in the
//    order u_i = i ^ rot (rot = dpart bits 3..1) and holds its heads in the
//    order g_k = k ^ (dpart bit 0) * GT/2, so that a butterfly reduce-scatter
//    over the 16 lanes of a half (xor 8, 4, 2 over tokens, xor 1 over heads)
//    always exchanges registers with static indices (GT*7 + GT/2 shuffles
//    instead of an all-reduce's 32*GT); afterwards each lane owns the complete
//    logits of token 2*rot + tsub for heads g_0 .. g_{GT/2-1}.
//  * Online softmax in the log2 domain (q pre-scaled by scale*log2(e), exp2f)
//    on the owned logits only; running max m and sum l per head.
//  * PV: each lane gathers p for its 8 tokens and GT heads with shuffles and
//    accumulates o[g][its dims] with packed fp32x2 FMAs over dim pairs.
// Warps combine through shared memory (reusing the rings), then the CL CTAs of
// the cluster combine through distributed shared memory into rank 0, which
// writes out and lse.  No global scratch memory is used.
//
// G > 8 is processed in query-head tiles of 8 (separate clusters).
#include <cooperative_groups.h>

#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace oasis {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kWaitTries = 1u << 22;  // bounded mbarrier polls (far beyond any real copy)
constexpr float kLn2 = 0.69314718055994530942f;

// Widen VEC bf16 (16 or 8 bytes of shared memory) to fp32.
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

template <int VEC, int GT>
struct Smem {
  static constexpr int D = 16 * VEC;
  static constexpr int kTile = 64 * D;  // bytes per slot tile
  // combine scratch (floats), aliased onto the rings after the main loop
  static constexpr int kWarpM = 0, kWarpL = kWarps * GT, kWarpO = 2 * kWarps * GT;
  static constexpr int kCtaM = kWarpO + kWarps * GT * D, kCtaL = kCtaM + GT, kCtaO = kCtaL + GT;
  static constexpr int kScratchFloats = kCtaO + GT * D;
};

template <int VEC, int GT, int NST>
__global__ void __launch_bounds__(kThreads)
    k_attn(const uint16_t *__restrict__ q, const uint16_t *__restrict__ pool, const int32_t *__restrict__ table,
           int slots, const int32_t *__restrict__ seq_len, int Hkv, int G, int ntiles, float scale_log2,
           float *__restrict__ out, float *__restrict__ lse, int32_t *status, int list_cap) {
  using SM = Smem<VEC, GT>;
  constexpr int D = SM::D;
  constexpr uint32_t kTileBytes = SM::kTile;
  constexpr int H = GT > 1 ? GT / 2 : 1;  // heads owned per lane after the reduce-scatter
  extern __shared__ __align__(128) unsigned char sm[];
  cg::cluster_group cluster = cg::this_cluster();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tsub = lane >> 4, dpart = lane & 15;
  const int rot = (dpart >> 1) & 7;  // token order u_i = i ^ rot
  const int hb = dpart & 1;          // head order  g_k = k ^ hb * GT/2
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
  float *scratch = reinterpret_cast<float *>(sm);  // used only once every ring stage is drained
  int32_t *list = reinterpret_cast<int32_t *>(bars + (kWarps - warp) * NST) + warp * list_cap;

  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // query slot k holds head g_k = k ^ (hb * GT/2); packed in head pairs for fp32x2
  unsigned long long q2[(GT + 1) / 2][VEC];
  {
    float qf[GT][VEC];
#pragma unroll
    for (int k = 0; k < GT; ++k) {
      const int g = GT > 1 ? (k ^ (hb * (GT / 2))) : 0;
      if (g < gcount) {
        float f[VEC];
        load_row<VEC>(q + (static_cast<int64_t>(bseq) * Hq + h * G + g0 + g) * D + dpart * VEC, f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) qf[k][e] = f[e] * scale_log2;
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) qf[k][e] = 0.0f;
      }
    }
#pragma unroll
    for (int kp = 0; kp < (GT + 1) / 2; ++kp)
#pragma unroll
      for (int e = 0; e < VEC; ++e) q2[kp][e] = pack2(qf[2 * kp][e], 2 * kp + 1 < GT ? qf[2 * kp + 1][e] : 0.0f);
  }
  float m[GT], l[H];
  unsigned long long o2[GT][VEC / 2];  // o[k][e], dims packed in pairs
#pragma unroll
  for (int k = 0; k < GT; ++k) {
    m[k] = -INFINITY;
#pragma unroll
    for (int e = 0; e < VEC / 2; ++e) o2[k][e] = 0ull;
  }
#pragma unroll
  for (int k = 0; k < H; ++k) l[k] = 0.0f;

  // this warp's slots: gw, gw + nw, ... over the whole cluster; the non-empty ones
  // (slot << 5 | valid tokens) go to a per-warp list in shared memory, so the
  // streaming loop below makes no global-memory round trip for control flow
  const int nw = CL * kWarps, gw = rank * kWarps + warp;
  const int nk = slots > gw ? (slots - gw + nw - 1) / nw : 0;
  const int32_t *trow = table + static_cast<int64_t>(s) * slots;
  const uint16_t *prow = pool + static_cast<int64_t>(s) * slots * 32 * D;
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
  auto issue = [&](int c, int stg) {
    mbar_arrive_expect_tx(&bars[stg], kTileBytes);
    bulk_g2s(ring + stg * kTileBytes, prow + static_cast<int64_t>(list[c] >> 5) * 32 * D, kTileBytes, &bars[stg]);
  };
  if (lane == 0)
    for (int c = 0; c < NST && c < count; ++c) issue(c, c);
  int issued = min(NST, count), consumed = 0;
  bool timed_out = false;
  for (int c = 0; c < count; ++c) {
    const int stg = c % NST;
    const bool ok = mbar_wait_bounded(&bars[stg], static_cast<uint32_t>(c / NST) & 1u, kWaitTries);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      timed_out = true;
      break;
    }
    const int nv = list[c] & 31;
    const uint16_t *kt = reinterpret_cast<const uint16_t *>(ring + stg * kTileBytes);
    const uint16_t *vt = kt + kBlockTokens * D;

    // ---- QK partials: sc[k][i] for head slot k, token u_i = i ^ rot
    float sc[GT][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float kf[VEC];
      load_row<VEC>(kt + (2 * (i ^ rot) + tsub) * D + dpart * VEC, kf);
#pragma unroll
      for (int kp = 0; kp < (GT + 1) / 2; ++kp) {
        unsigned long long a = 0ull;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a = fma2(q2[kp][e], pack2(kf[e], kf[e]), a);
        float a0, a1;
        unpack2(a, a0, a1);
        sc[2 * kp][i] = a0;
        if (2 * kp + 1 < GT) sc[2 * kp + 1][i] = a1;
      }
    }
    // ---- reduce-scatter over the 16 lanes of the half
#pragma unroll
    for (int k = 0; k < GT; ++k) {
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[k][j] += __shfl_xor_sync(0xFFFFFFFFu, sc[k][j + 4], 8);
#pragma unroll
      for (int j = 0; j < 2; ++j) sc[k][j] += __shfl_xor_sync(0xFFFFFFFFu, sc[k][j + 2], 4);
      sc[k][0] += __shfl_xor_sync(0xFFFFFFFFu, sc[k][1], 2);
    }
    float s_own[H];
    if constexpr (GT > 1) {
#pragma unroll
      for (int k = 0; k < H; ++k) s_own[k] = sc[k][0] + __shfl_xor_sync(0xFFFFFFFFu, sc[k + H][0], 1);
    } else {
      s_own[0] = sc[0][0] + __shfl_xor_sync(0xFFFFFFFFu, sc[0][0], 1);
    }
    const bool tok_ok = 2 * rot + tsub < nv;
    // ---- online softmax on the owned logits
    float mnew[GT];
#pragma unroll
    for (int k = 0; k < H; ++k) {
      float v = tok_ok ? s_own[k] : -INFINITY;
      s_own[k] = v;
      v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 16));
      v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
      mnew[k] = fmaxf(m[k], v);
    }
    if constexpr (GT > 1) {
#pragma unroll
      for (int k = 0; k < H; ++k) mnew[k + H] = __shfl_xor_sync(0xFFFFFFFFu, mnew[k], 1);
    }
    float p_own[H];
#pragma unroll
    for (int k = 0; k < H; ++k) {
      p_own[k] = exp2f(s_own[k] - mnew[k]);
      const float lcorr = exp2f(m[k] - mnew[k]);
      l[k] = l[k] * lcorr + ((GT > 1 || hb == 0) ? p_own[k] : 0.0f);
    }
#pragma unroll
    for (int k = 0; k < GT; ++k) {
      const float corr = exp2f(m[k] - mnew[k]);
      const unsigned long long c2 = pack2(corr, corr);
#pragma unroll
      for (int e = 0; e < VEC / 2; ++e) o2[k][e] = fma2(o2[k][e], c2, 0ull);
      m[k] = mnew[k];
    }
    // ---- PV: gather p of this lane's tokens, accumulate its dims
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float vf[VEC];
      load_row<VEC>(vt + (2 * u + tsub) * D + dpart * VEC, vf);
#pragma unroll
      for (int k = 0; k < GT; ++k) {
        const int src = tsub * 16 + 2 * u + (GT > 1 ? ((k >= H) ^ hb) : 0);
        const float p = __shfl_sync(0xFFFFFFFFu, p_own[GT > 1 ? k % H : 0], src);
        const unsigned long long p2 = pack2(p, p);
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) o2[k][e] = fma2(p2, pack2(vf[2 * e], vf[2 * e + 1]), o2[k][e]);
      }
    }
    __syncwarp();
    ++consumed;
    if (c + NST < count) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(c + NST, stg);
      }
      ++issued;
    }
  }
  if (timed_out) {
    if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
    for (int c = consumed; c < issued; ++c)
      mbar_wait_bounded(&bars[c % NST], static_cast<uint32_t>(c / NST) & 1u, kWaitTries);
  }

  // ---- per-warp totals: l over the owning lanes, o over the two token halves
#pragma unroll
  for (int k = 0; k < H; ++k) {
    float v = l[k];
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    if constexpr (GT == 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    l[k] = v;
  }
  float lfull[GT];
#pragma unroll
  for (int k = 0; k < H; ++k) lfull[k] = l[k];
  if constexpr (GT > 1) {
#pragma unroll
    for (int k = 0; k < H; ++k) lfull[k + H] = __shfl_xor_sync(0xFFFFFFFFu, l[k], 1);
  }
  float of[GT][VEC];
#pragma unroll
  for (int k = 0; k < GT; ++k)
#pragma unroll
    for (int e = 0; e < VEC / 2; ++e) {
      float a, b;
      unpack2(o2[k][e], a, b);
      of[k][2 * e] = a + __shfl_xor_sync(0xFFFFFFFFu, a, 16);
      of[k][2 * e + 1] = b + __shfl_xor_sync(0xFFFFFFFFu, b, 16);
    }
  __syncthreads();  // every warp is past its ring: the scratch may alias it
  float *wm = scratch + SM::kWarpM, *wl = scratch + SM::kWarpL, *wo = scratch + SM::kWarpO;
  float *cm = scratch + SM::kCtaM, *cl = scratch + SM::kCtaL, *co = scratch + SM::kCtaO;
  if (lane == 0) {  // hb = 0 here: slot k holds head k
#pragma unroll
    for (int k = 0; k < GT; ++k) {
      wm[warp * GT + k] = m[k];
      wl[warp * GT + k] = lfull[k];
    }
  }
  if (tsub == 0) {
#pragma unroll
    for (int k = 0; k < GT; ++k) {
      const int g = GT > 1 ? (k ^ (hb * (GT / 2))) : 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) wo[(warp * GT + g) * D + dpart * VEC + e] = of[k][e];
    }
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

template <int VEC, int GT, int NST>
cudaError_t launch_t(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                     const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                     int32_t *status, cudaStream_t st) {
  using SM = Smem<VEC, GT>;
  const int ntiles = (G + GT - 1) / GT;
  const int units = B * Hkv * ntiles;
  const size_t ring = static_cast<size_t>(kWarps) * NST * SM::kTile + sizeof(uint64_t) * kWarps * NST;
  // the shared-memory size (and so the occupancy) is fixed by the rings; the slot
  // lists take a fixed maximum of kListMax entries per warp
  constexpr int kListMax = 512;
  const size_t smem = std::max(ring + sizeof(int32_t) * kWarps * kListMax, sizeof(float) * SM::kScratchFloats);
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn<VEC, GT, NST>), kThreads, smem, &sms,
                                  &per_sm);
  if (e != cudaSuccess) return e;
  // split every segment over a cluster so that the grid fills the resident CTA slots
  int CL = static_cast<int>(std::min<int64_t>(8, std::max<int64_t>(1, static_cast<int64_t>(sms) * per_sm / units)));
  CL = std::min(CL, slots);
  while ((slots + CL * kWarps - 1) / (CL * kWarps) > kListMax) ++CL;  // keep each warp's list within kListMax
  if (CL > 8) return cudaErrorInvalidValue;
  const int list_cap = kListMax;
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
                            scale_log2, out, lse, status, list_cap);
}

template <int VEC>
cudaError_t launch_vec(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                       const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                       int32_t *status, cudaStream_t st) {
  constexpr int NST = 2;
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
