// Sparse paged decode attention over the head-wise logical-to-logical table.
//
// OasisKV paper review (xllm-io), §3 Fig. 5: the foreground forward pass runs
// sparse attention of the true query over the working set resident in HBM;
// §4 / Fig. 9: each KV head addresses its own resident blocks through the
// head-wise mapping.  For query head h*G + g of sequence b:
//     out = sum_i softmax_i(scale * q . k_i) v_i
// over the valid tokens of the slots whose table entry is >= 0.
//
// Work split (split-K, balanced per SM).  All segments' slots are one flat
// range of N = S * slots_per_seg slot tiles (8 KiB each at D = 128).  A
// persistent grid of `grid` CTAs (SM count x resident CTAs per SM, or more for
// very large N) gives every warp an equal contiguous share (+-1 slot), so every
// SM streams the same number of bytes whatever the segment count.  A warp's
// share spans at most two segments (the grid is sized so), giving at most two
// partial results (running max, sum and output of the online softmax); each
// CTA merges its warps' partials per segment and writes one partial per
// (segment, CTA) to the caller's workspace; k_attn_combine merges the partials
// of each segment and writes out and lse.
//
// Data path.  Each warp first lists its non-empty slots in shared memory (one
// table read per slot), then streams their tiles through a private two-stage
// ring with 2-D TMA tensor copies (cp.async.bulk.tensor, one mbarrier per
// stage, lane 0 issues).  The tensor map views the pool as rows of D bf16 and
// uses the 128-byte swizzle, so the tensor-core fragment loads are bank-conflict
// free.  Empty slots are never loaded.  Every mbarrier wait is bounded.
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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cfloat>
#include <mutex>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kListMax = 512;              // listed slots per warp
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
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Shared-memory plan (offsets in bytes from a 1024-aligned base); kNST ring
// stages (slot tiles) per warp.
template <int D, int GQ, int kNST>
struct Plan {
  static constexpr int kTile = 64 * D;                       // one slot: 32 rows of D bf16
  static constexpr int kRing = kWarps * kNST * kTile;
  static constexpr int kRun = GQ * (D + 2) + 1;              // floats: m[GQ], l[GQ], o[GQ][D], segment
  static constexpr int kFirstRuns = kRing;                   // [kWarps] first-run partials (floats)
  static constexpr int kBars = kFirstRuns + 4 * kWarps * kRun;  // kWarps * kNST mbarriers
  static constexpr int kLists = kBars + 8 * kWarps * kNST;   // kWarps * kListMax int32
  static constexpr int kEnd = kLists + 4 * kWarps * kListMax;
  static_assert(4 * kWarps * kRun <= kRing, "the last-run partials reuse the ring");
};

// Split of the flat slot range over CTAs and warps; shared by both kernels and
// the workspace size.
struct Split {
  int64_t N;  // S * slots
  int grid, slots, R;
  __host__ __device__ int64_t cta_begin(int c) const { return N * c / grid; }
  __host__ __device__ int64_t warp_begin(int64_t gw) const { return N * gw / (static_cast<int64_t>(grid) * kWarps); }
  // CTA whose range holds flat slot n
  __host__ __device__ int cta_of(int64_t n) const { return static_cast<int>(((n + 1) * grid - 1) / N); }
  __host__ __device__ bool cta_touches(int c, int s) const {
    const int64_t a = cta_begin(c), b = cta_begin(c + 1);
    return b > a && a < static_cast<int64_t>(s + 1) * slots && b > static_cast<int64_t>(s) * slots;
  }
};

template <int D>
__device__ __forceinline__ float *ws_partial(float *ws, const Split &sp, int s, int r, int G, int q) {
  return ws + ((static_cast<int64_t>(s) * sp.R + r) * G + q) * (D + 2);
}

// KS = D / 16 (k-steps of the QK product and m-tiles of the PV product);
// NT = query tiles of 8 heads (GQ = 8 * NT columns).
template <int KS, int NT, int kNST>
__global__ void __launch_bounds__(kThreads)
    k_attn_part(const __grid_constant__ CUtensorMap tmap, const uint16_t *__restrict__ q,
                const int32_t *__restrict__ table, const int32_t *__restrict__ seq_len, int Hkv, int G,
                float scale_log2, Split sp, float *__restrict__ ws, int32_t *status) {
  constexpr int D = 16 * KS;
  constexpr int GQ = 8 * NT;
  constexpr int kBoxes = D / 64;  // 64-dim boxes (128 bytes per row) per tile
  using P = Plan<D, GQ, kNST>;
  extern __shared__ unsigned char sm_raw[];
  const uint32_t raw_addr = smem_addr(sm_raw);
  unsigned char *sm = sm_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int c = blockIdx.x;
  const int slots = sp.slots;
  const int Hq = Hkv * G;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + P::kBars) + warp * kNST;
  int32_t *list = reinterpret_cast<int32_t *>(sm + P::kLists) + warp * kListMax;
  float *first_run = reinterpret_cast<float *>(sm + P::kFirstRuns) + warp * P::kRun;
  float *last_runs = reinterpret_cast<float *>(sm);  // [kWarps][kRun], reuses the ring after the loop
  // run k < kWarps: warp k's first run; k >= kWarps: warp k - kWarps's last run
  auto run_ptr = [&](int k) -> const float * {
    return k < kWarps ? reinterpret_cast<const float *>(sm + P::kFirstRuns) + k * P::kRun
                      : last_runs + (k - kWarps) * P::kRun;
  };
  const uint32_t ring = sbase + warp * kNST * P::kTile;
  if (lane == 0) {
    for (int i = 0; i < kNST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    first_run[P::kRun - 1] = -1.0f;  // no first run yet
  }

  // this warp's share of the flat slot range; its non-empty slots as (n << 5 | valid tokens)
  const int64_t gw = static_cast<int64_t>(c) * kWarps + warp;
  const int64_t n0 = sp.warp_begin(gw), n1 = sp.warp_begin(gw + 1);
  const int nk = static_cast<int>(n1 - n0);
  int count = 0;
  for (int base = 0; base < nk; base += 32) {
    const int k = base + lane;
    int nv = 0;
    int64_t n = 0;
    if (k < nk) {
      n = n0 + k;
      const int s = static_cast<int>(n / slots);
      int L = seq_len[s / Hkv];
      if (L < 0) {
        report(status, OASIS_STATUS_SEQ_LEN);
        L = 0;
      }
      const int blk = table[n];
      const int64_t rem = blk < 0 ? 0 : static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
      nv = rem <= 0 ? 0 : (rem >= kBlockTokens ? kBlockTokens : static_cast<int>(rem));
    }
    const unsigned mk = __ballot_sync(0xFFFFFFFFu, nv > 0);
    if (nv > 0) list[count + __popc(mk & ((1u << lane) - 1u))] = static_cast<int32_t>((n << 5) | nv);
    count += __popc(mk);
  }
  __syncwarp();
  auto issue = [&](int i, int stg) {
    mbar_arrive_expect_tx(&bars[stg], P::kTile);
    const int y = (list[i] >> 5) * 32;
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_load_2d(ring + stg * P::kTile + bx * 4096, &tmap, bx * 64, y, &bars[stg]);
  };
  if (lane == 0)
    for (int i = 0; i < kNST && i < count; ++i) issue(i, i);
  int issued = min(kNST, count), consumed = 0;
  bool timed_out = false;

  auto frag_addr = [&](uint32_t tile, int r, int j) {
    return tile + (j >> 3) * 4096 + r * 128 + (((j & 7) ^ (r & 7)) << 4);
  };
  const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);  // K rows 0..15 for ldmatrix
  const int khalf = lane >> 4;
  const int vrow = 16 + (lane & 7) + 8 * (lane >> 4);   // V rows 16..31 for ldmatrix.trans
  const int vhalf = (lane >> 3) & 1;

  uint32_t qb[NT][KS][2];
  float o[NT][KS][4];
  float m[NT][2], l[NT][2];
  int s_cur = -1;
  auto reset_state = [&]() {
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
  };
  // run partial -> shared memory: m, l (reduced over the token lanes) and o
  auto store_run = [&](float *dst, int seg) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = l[nt][j];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        if (g == 0) {
          dst[nt * 8 + 2 * t + j] = m[nt][j];
          dst[GQ + nt * 8 + 2 * t + j] = v;
        }
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[2 * GQ + (nt * 8 + 2 * t + (i & 1)) * D + 16 * mt + g + 8 * (i >> 1)] = o[nt][mt][i];
    if (lane == 0) dst[P::kRun - 1] = static_cast<float>(seg);
  };
  reset_state();

  for (int i = 0; i < count; ++i) {
    const int stg = i % kNST;
    const int64_t n = list[i] >> 5;
    const int s = static_cast<int>(n / slots);
    if (s != s_cur) {  // warp-uniform: a new segment (at most once after the first)
      if (s_cur >= 0) {
        store_run(first_run, s_cur);
        reset_state();
      }
      s_cur = s;
      const int bseq = s / Hkv, h = s % Hkv;
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
    }
    const bool ok = mbar_wait_bounded(&bars[stg], static_cast<uint32_t>(i / kNST) & 1u, kWaitTries);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      timed_out = true;
      break;
    }
    const int nv = list[i] & 31;
    const uint32_t tile = ring + stg * P::kTile;

    // ---- S^T = K . Q^T
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.0f;
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
    __syncwarp();
    ++consumed;
    if (i + kNST < count) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(i + kNST, stg);
      }
      ++issued;
    }
  }
  if (timed_out) {
    if (lane == 0) report(status, OASIS_STATUS_TIMEOUT);
    for (int i = consumed; i < issued; ++i)
      mbar_wait_bounded(&bars[i % kNST], static_cast<uint32_t>(i / kNST) & 1u, kWaitTries);
  }

  // ---- merge the warps' runs per segment and write one partial per (segment, CTA)
  __syncthreads();  // every warp is past its ring: run slots may reuse it
  {
    float *mine = last_runs + warp * P::kRun;
    if (s_cur >= 0) {
      store_run(mine, s_cur);
    } else if (lane == 0) {
      mine[P::kRun - 1] = -1.0f;
    }
  }
  __syncthreads();
  const int64_t a = sp.cta_begin(c), b = sp.cta_begin(c + 1);
  if (b > a) {
    const int s_first = static_cast<int>(a / slots), s_last = static_cast<int>((b - 1) / slots);
    for (int s = s_first; s <= s_last; ++s) {
      const int r = c - sp.cta_of(static_cast<int64_t>(s) * slots);
      for (int idx = tid; idx < G * (D + 2); idx += kThreads) {
        const int qc = idx / (D + 2), e = idx % (D + 2);
        float M = -INFINITY;
        for (int k = 0; k < 2 * kWarps; ++k) {
          const float *run = run_ptr(k);
          if (static_cast<int>(run[P::kRun - 1]) == s) M = fmaxf(M, run[qc]);
        }
        float acc = 0.0f;
        if (M > -INFINITY) {
          for (int k = 0; k < 2 * kWarps; ++k) {
            const float *run = run_ptr(k);
            if (static_cast<int>(run[P::kRun - 1]) != s) continue;
            const float f = exp2f(run[qc] - M);
            acc += f * (e == 1 ? run[GQ + qc] : run[2 * GQ + qc * D + (e - 2)]);
          }
        }
        float *dst = ws_partial<D>(ws, sp, s, r, G, qc);
        dst[e] = e == 0 ? M : acc;
      }
    }
  }
}

// Merge the per-CTA partials of each segment: out = sum f_r o_r / sum f_r l_r,
// f_r = 2^(m_r - max m), lse = ln(sum f_r l_r) + max m * ln 2.
template <int D>
__global__ void __launch_bounds__(256) k_attn_combine(const float *__restrict__ ws, Split sp, int Hkv, int G,
                                                      float *__restrict__ out, float *__restrict__ lse) {
  const int s = blockIdx.x;
  const int bseq = s / Hkv, h = s % Hkv;
  const int c_lo = sp.cta_of(static_cast<int64_t>(s) * sp.slots);
  const int c_hi = sp.cta_of(static_cast<int64_t>(s + 1) * sp.slots - 1);
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int qc = idx / D, d = idx % D;
    float M = -INFINITY;
    for (int c = c_lo; c <= c_hi; ++c)
      if (sp.cta_touches(c, s)) M = fmaxf(M, ws_partial<D>(const_cast<float *>(ws), sp, s, c - c_lo, G, qc)[0]);
    float acc = 0.0f, ls = 0.0f;
    if (M > -INFINITY) {
      for (int c = c_lo; c <= c_hi; ++c) {
        if (!sp.cta_touches(c, s)) continue;
        const float *pr = ws_partial<D>(const_cast<float *>(ws), sp, s, c - c_lo, G, qc);
        const float f = exp2f(pr[0] - M);
        ls += f * pr[1];
        acc += f * pr[2 + d];
      }
    }
    const int64_t row = static_cast<int64_t>(bseq) * (Hkv * G) + h * G + qc;
    out[row * D + d] = ls > 0.0f ? acc / ls : 0.0f;
    if (d == 0 && lse != nullptr) lse[row] = ls > 0.0f ? (M + log2f(ls)) * kLn2 : -INFINITY;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

constexpr int kNSTAttn = 2;

template <int KS, int NT>
size_t part_smem() {
  return Plan<16 * KS, 8 * NT, kNSTAttn>::kEnd + 1024;  // + slack for the 1024-byte alignment
}

// The split for S segments of `slots` slots on the current device.
template <int KS, int NT>
cudaError_t make_split(int S, int slots, int G, Split *sp) {
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn_part<KS, NT, kNSTAttn>), kThreads,
                                  part_smem<KS, NT>(), &sms, &per_sm);
  if (e != cudaSuccess) return e;
  sp->N = static_cast<int64_t>(S) * slots;
  sp->slots = slots;
  // each warp's share must fit its list and span at most two segments
  const int64_t cap = std::min(slots, kListMax);
  const int64_t min_grid = (sp->N + kWarps * cap - 1) / (kWarps * cap);
  sp->grid = static_cast<int>(std::max<int64_t>(static_cast<int64_t>(sms) * per_sm, min_grid));
  sp->R = (sp->grid + S - 1) / S + 1;
  (void)G;
  return cudaSuccess;
}

template <int KS, int NT>
size_t workspace_bytes_t(int S, int slots, int G) {
  Split sp;
  if (make_split<KS, NT>(S, slots, G, &sp) != cudaSuccess) return 0;
  return sizeof(float) * static_cast<size_t>(S) * sp.R * G * (16 * KS + 2);
}

template <int KS, int NT>
cudaError_t launch_t(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                     const int32_t *seq_len, int B, int Hkv, int G, float scale, float *out, float *lse,
                     void *ws, size_t ws_bytes, int32_t *status, cudaStream_t st) {
  constexpr int D = 16 * KS;
  const int S = B * Hkv;
  Split sp;
  cudaError_t e = make_split<KS, NT>(S, slots, G, &sp);
  if (e != cudaSuccess) return e;
  if (ws_bytes < sizeof(float) * static_cast<size_t>(S) * sp.R * G * (D + 2)) return cudaErrorInvalidValue;
  // the pool as a 2-D tensor: rows of D bf16, one 32-row box per 64 dims of a slot
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(sp.N) * 32};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const float scale_log2 = scale * 1.4426950408889634f;
  k_attn_part<KS, NT, kNSTAttn><<<sp.grid, kThreads, part_smem<KS, NT>(), st>>>(
      tmap, q, table, seq_len, Hkv, G, scale_log2, sp, static_cast<float *>(ws), status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_attn_combine<D><<<S, 256, 0, st>>>(static_cast<const float *>(ws), sp, Hkv, G, out, lse);
  return cudaGetLastError();
}

}  // namespace

size_t attn_workspace_bytes(int B, int Hkv, int G, int D, int slots_per_seg) {
  const int S = B * Hkv;
  if (D == 128) return G <= 8 ? workspace_bytes_t<8, 1>(S, slots_per_seg, G) : workspace_bytes_t<8, 2>(S, slots_per_seg, G);
  return G <= 8 ? workspace_bytes_t<4, 1>(S, slots_per_seg, G) : workspace_bytes_t<4, 2>(S, slots_per_seg, G);
}

cudaError_t launch_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                      int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                      float scale, float *out, float *lse, void *ws, size_t ws_bytes,
                                      int32_t *status, cudaStream_t st) {
  if (D == 128) {
    if (G <= 8)
      return launch_t<8, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, ws, ws_bytes, status, st);
    return launch_t<8, 2>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, ws, ws_bytes, status, st);
  }
  if (G <= 8)
    return launch_t<4, 1>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, ws, ws_bytes, status, st);
  return launch_t<4, 2>(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, scale, out, lse, ws, ws_bytes, status, st);
}

}  // namespace oasis
