// Per-KV-head top-K selection with capped admission, eviction, transfer plan
// and head-wise table update.
//
// OasisKV paper review (xllm-io): §3 decode flow (predict top-K -> compare with
// the resident set -> build the transfer plan), §3 component table ("Capped
// Eviction Policy": at most C new blocks per head per step, fetch ratio 0.05;
// "Head-wise Mapping": per-KV-head logical-to-logical table), §4 innovations
// (only head-wise mapping entries change).  legiblepapers, FAQ Q7: the cap is
// applied at the KV-selection stage.
//
// Rule (per segment; T = top-K, R = residents, A = admitted, R' = new set):
//   T  = first min(K, nc) candidates by (score desc, block asc)
//   A  = first `cap` blocks of T \ R in that order
//   R' = first K of R u A, empty slots ranking below every block
//   A in ascending id takes the freed slots (filled empties, then the slots of
//   evicted residents) in ascending slot order.
//
// One CTA of 512 threads per segment, everything in shared memory:
//  * scores -> order-preserving 32-bit keys (larger key = larger score; -0 is
//    mapped to +0 so the two tie; NaN maps to 0, below -inf, and is flagged);
//  * T by a 4-pass 8-bit MSB radix select of the K-th largest key (warp-
//    aggregated shared-memory histograms), then ties at the threshold taken in
//    ascending block order through a block-wide prefix count;
//  * T, R as bitmaps; the small lists T\R and R\T are ranked by counting
//    (O(n^2) over <= K entries, no sorting network, few barriers) with the
//    unique 64-bit composite key (key << 32) | ~block.
#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr size_t kStaticSmemBound = 4096;  // >= the kernel's static shared memory (3 KiB of histograms + scalars)

__device__ __forceinline__ uint32_t score_key(float f, bool &nan) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) {
    nan = true;
    return 0u;
  }
  if (u == 0x80000000u) u = 0u;  // -0 ties with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int b) {
  return (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(b));
}
__device__ __forceinline__ int composite_block(uint64_t c) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(c & 0xFFFFFFFFu));
}

__device__ __forceinline__ bool bit(const uint32_t *bm, int b) { return (bm[b >> 5] >> (b & 31)) & 1u; }

// Exclusive prefix sum of v over the CTA (all threads call it).
__device__ int block_exclusive_scan(int v, int *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) warp_tot[lane] = t;  // inclusive totals
  }
  __syncthreads();
  const int before_warp = warp > 0 ? warp_tot[warp - 1] : 0;
  const int r = before_warp + x - v;
  __syncthreads();  // warp_tot may be reused by the caller
  return r;
}

struct SelScalars {
  int err;
  int nN, nE, nF, nEmpty;
  uint32_t digit;
  int remaining;
  int warp_tot[kWarps];
};

static_assert(sizeof(SelScalars) + 3 * 256 * sizeof(uint32_t) <= kStaticSmemBound, "static shared memory bound");

// Sum of v over the CTA (all threads call it, all get the sum).
__device__ int block_sum(int v, int *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();  // warp_tot may still be read by a previous use
  if (lane == 0) warp_tot[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < kWarps; ++w) t += warp_tot[w];
  __syncthreads();
  return t;
}

// T as a bitmap: the first min(K, nc) candidates by (key desc, block asc).
// 4-pass 8-bit MSB radix select of the K-th largest key (warp-aggregated
// shared-memory histograms, triple-buffered so each pass takes one barrier),
// then the keys equal to it taken in ascending block order through a
// block-wide prefix count.  bmT must be clear; all threads call it; the caller
// synchronises before reading bmT.
__device__ void topk_bitmap(const uint32_t *keys, int nc, int K, uint32_t *bmT, uint32_t (*hist)[256],
                            SelScalars &sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (nc <= K) {
    for (int b = tid; b < nc; b += kThreads) atomicOr(&bmT[b >> 5], 1u << (b & 31));
  } else {
    uint32_t prefix = 0u, pmask = 0u;
    int remaining = K;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t *h = hist[pass % 3];
      for (int i = tid; i < 256; i += kThreads) hist[(pass + 1) % 3][i] = 0u;
      for (int b0 = warp * 32; b0 < nc; b0 += kThreads) {
        const int b = b0 + lane;
        int dig = -1;
        if (b < nc) {
          const uint32_t key = keys[b];
          if ((key & pmask) == prefix) dig = static_cast<int>((key >> shift) & 0xFFu);
        }
        const unsigned grp = __match_any_sync(0xFFFFFFFFu, dig);
        if (dig >= 0 && lane == __ffs(grp) - 1) atomicAdd(&h[dig], static_cast<uint32_t>(__popc(grp)));
      }
      // The only barrier of the pass: the counts are complete, the next buffer is
      // clear, and every warp has finished reading the buffer cleared next pass.
      __syncthreads();
      // Every warp finds the digit of the remaining-th largest key on its own.
      // Lane l owns bins 255-8l down to 248-8l (descending digit order).
      // (two 16-byte loads per lane: consecutive lanes read consecutive 16-byte
      // chunks, so every warp's reads are free of bank conflicts)
      const uint4 lo4 = reinterpret_cast<const uint4 *>(h)[62 - 2 * lane];  // bins 248-8l .. 251-8l
      const uint4 hi4 = reinterpret_cast<const uint4 *>(h)[63 - 2 * lane];  // bins 252-8l .. 255-8l
      const uint32_t c[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
      uint32_t sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) sum += c[q];
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t before = incl - sum;
      uint32_t digit = 0u;
      int rem = 0;
      const bool mine = before < static_cast<uint32_t>(remaining) && static_cast<uint32_t>(remaining) <= incl;
      if (mine) {
        uint32_t cum = before;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (cum < static_cast<uint32_t>(remaining) && static_cast<uint32_t>(remaining) <= cum + c[q]) {
            digit = static_cast<uint32_t>(255 - 8 * lane - q);
            rem = remaining - static_cast<int>(cum);
          }
          cum += c[q];
        }
      }
      const unsigned holders = __ballot_sync(0xFFFFFFFFu, mine);  // exactly one lane holds it
      const int src = holders ? __ffs(holders) - 1 : 0;
      digit = __shfl_sync(0xFFFFFFFFu, digit, src);
      rem = __shfl_sync(0xFFFFFFFFu, rem, src);
      prefix |= digit << shift;
      pmask |= 0xFFu << shift;
      remaining = rem;
    }
    const uint32_t tau = prefix;
    const int need = remaining;  // keys equal to tau to take, lowest block id first
    const int per = ceil_div(nc, kThreads);
    const int lo = min(nc, tid * per), hi = min(nc, lo + per);
    int ties = 0;
    for (int b = lo; b < hi; ++b) ties += keys[b] == tau;
    int before = block_exclusive_scan(ties, sc.warp_tot);
    for (int b = lo; b < hi; ++b) {
      const uint32_t key = keys[b];
      bool in = key > tau;
      if (key == tau) {
        in = before < need;
        ++before;
      }
      if (in) atomicOr(&bmT[b >> 5], 1u << (b & 31));
    }
  }
}


// ---- certified selection from tensor-core score estimates ------------------
// The certified kernel receives for every candidate an estimate s~ and a
// radius r with |s~ - s| <= r around the fixed-order score s.  A selection
// decision that splits a set into its first m members and the rest (T: the
// first K candidates; A: the first cap of T \ R; the evicted: the last nEvict
// of R \ T) is settled without s wherever the intervals separate: with X~ the
// first m by the estimates, lo = min over X~ of (s~ - r) and hi = max over the
// rest of (s~ + r), a member with s~ - r > hi is in the first m whatever the
// exact order (at most m - 1 others can rank above it), one with s~ + r < lo is
// not (m others surely rank above it).  Every other member is recomputed with
// the fixed-order arithmetic, and the selection then runs on the mixed scores:
// the settled members keep their side, the recomputed ones are ordered
// exactly, so every set equals the one the exact scores give.
constexpr int kBatch = 32;  // blocks recomputed per pass

// Byte offsets of the certified kernel's extra shared memory, from the start
// of the dynamic allocation; one definition serves the kernel's pointers and
// the launcher's allocation size.
struct CertLayout {
  size_t stage, qsm, res, bmX, xl, rankE, end;
};
__host__ __device__ inline CertLayout cert_layout(size_t base_bytes, int Nb_max, int K, int CH, int Nq) {
  const size_t words = (static_cast<size_t>(Nb_max) + 31) / 32;
  const size_t Nq4 = (static_cast<size_t>(Nq) + 3) & ~static_cast<size_t>(3);
  CertLayout L;
  L.stage = (base_bytes + 15) & ~static_cast<size_t>(15);
  L.qsm = L.stage + 16 * static_cast<size_t>(kBatch) * (2 * CH + 1);      // uint4 [kBatch][2*CH + 1]
  L.res = L.qsm + 4 * static_cast<size_t>(CH) * 8 * Nq4;                 // float [D][Nq4]
  L.bmX = L.res + 4 * static_cast<size_t>(kBatch) * Nq4;                 // float [kBatch][Nq4]
  L.xl = L.bmX + 4 * words;                                              // uint32 [words]
  L.rankE = L.xl + 4 * static_cast<size_t>(Nb_max);                      // int32 [Nb_max]
  L.end = L.rankE + 4 * static_cast<size_t>(K);                          // int32 [K]
  return L;
}

struct CertArgs {
  float *scores;  // in: estimates; out: the recomputed blocks' fixed-order scores
  const float *radius;
  const uint16_t *kmin, *kmax, *qdraft;
  int G, Nd;
};

__device__ float block_reduce(float v, bool is_max, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = is_max ? fmaxf(v, y) : fminf(v, y);
  }
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < kWarps; ++w) r = is_max ? fmaxf(r, red[w]) : fminf(r, red[w]);
  return r;
}

// Fixed-order fp32 scores of the listed blocks (the oasis_score_blocks
// arithmetic: per query, sum over d ascending from +0 of q_d * (q_d >= 0 ?
// kmax_d : kmin_d), one rounding per term; max over the queries, NaN kept).
// Writes them to srow and their keys to keys, marks them in bmX.
// A thread takes one block and four queries (the widened summary values serve
// all four); qsm holds the queries as [d][Nq4], Nq4 = Nq rounded up to 4, the
// padding repeating the last query.
template <int CH>
__device__ void recompute_blocks(const int32_t *xl, int n, const uint4 *gmin, const uint4 *gmax, int Nb_max,
                                 int Nq, const float *qsm, uint4 *stage, float *res, float *srow, uint32_t *keys,
                                 uint32_t *bmX, SelScalars &sc) {
  constexpr int ES = 2 * CH + 1;  // staged entry: kmin chunks, kmax chunks, one pad (bank spread)
  const int tid = threadIdx.x;
  const int Nq4 = (Nq + 3) & ~3, ng = Nq4 / 4;
  for (int e0 = 0; e0 < n; e0 += kBatch) {
    const int nb = min(kBatch, n - e0);
    for (int i = tid; i < nb * 2 * CH; i += kThreads) {
      const int e = i / (2 * CH), k = i % (2 * CH), c = k % CH;
      const int b = xl[e0 + e];
      stage[e * ES + k] = __ldg((k < CH ? gmin : gmax) + static_cast<int64_t>(c) * Nb_max + b);
    }
    __syncthreads();
    for (int i = tid; i < nb * ng; i += kThreads) {
      const int e = i / ng, g = i % ng;
      const uint4 *st = stage + e * ES;
      const float *qg = qsm + 4 * g;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
      for (int c = 0; c < CH; ++c) {
        const uint4 mn = st[c], mx = st[CH + c];
        const uint32_t wn[4] = {mn.x, mn.y, mn.z, mn.w}, wx[4] = {mx.x, mx.y, mx.z, mx.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float kn = (t & 1) ? bf16_hi(wn[t >> 1]) : bf16_lo(wn[t >> 1]);
          const float kx = (t & 1) ? bf16_hi(wx[t >> 1]) : bf16_lo(wx[t >> 1]);
          const float4 q = *reinterpret_cast<const float4 *>(qg + (c * 8 + t) * Nq4);
          acc[0] = fmaf(q.x, q.x >= 0.0f ? kx : kn, acc[0]);  // exact product, one rounding
          acc[1] = fmaf(q.y, q.y >= 0.0f ? kx : kn, acc[1]);
          acc[2] = fmaf(q.z, q.z >= 0.0f ? kx : kn, acc[2]);
          acc[3] = fmaf(q.w, q.w >= 0.0f ? kx : kn, acc[3]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) res[e * Nq4 + 4 * g + k] = acc[k];
    }
    __syncthreads();
    for (int e = tid; e < nb; e += kThreads) {
      float best = -INFINITY;
      bool nan = false;
      for (int j = 0; j < Nq; ++j) {
        const float v = res[e * Nq4 + j];
        nan |= v != v;
        best = fmaxf(best, v);
      }
      const float v = nan ? __uint_as_float(0x7FC00000u) : best;
      const int b = xl[e0 + e];
      srow[b] = v;
      bool isn = false;
      keys[b] = score_key(v, isn);
      if (isn) atomicOr(&sc.err, OASIS_STATUS_NAN_SCORE);
      atomicOr(&bmX[b >> 5], 1u << (b & 31));
    }
    __syncthreads();
  }
}

// interval of block b: recomputed blocks are exact (radius 0)
__device__ __forceinline__ void interval(const float *srow, const float *rrow, const uint32_t *bmX, int b, float &lo,
                                         float &hi) {
  const float v = srow[b];
  const float r = bit(bmX, b) ? 0.0f : rrow[b];
  lo = v - r;
  hi = v + r;
}

// CERTIFY = false: the selection on exact scores.  CERTIFY = true: `scores`
// holds estimates with radii (CertArgs); the decisions the estimates cannot
// settle are settled by recomputing fixed-order scores (see above).
template <bool CERTIFY, int CH>
__global__ void __launch_bounds__(kThreads) k_select(const float *scores, int Nb_max,
                                                     const int32_t *__restrict__ seq_len, int Hkv, int K, int W,
                                                     int cap, const int32_t *table_in, int32_t *table_out,
                                                     oasis_xfer_t *__restrict__ plan, int32_t *__restrict__ plan_count,
                                                     int32_t *status, CertArgs ca) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ SelScalars sc;
  __shared__ __align__(16) uint32_t hist[3][256];  // pass p counts into hist[p % 3], clears hist[(p + 1) % 3]
  __shared__ float red[kWarps];
  __shared__ int nX;

  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slots = K + W;
  const int words = (Nb_max + 31) >> 5;

  uint64_t *listN = reinterpret_cast<uint64_t *>(smraw);       // [K]
  uint64_t *listE = listN + K;                                 // [K]
  uint32_t *keys = reinterpret_cast<uint32_t *>(listE + K);   // [Nb_max]
  uint32_t *bmR = keys + Nb_max;                               // [words]
  uint32_t *bmT = bmR + words;                                 // [words]
  int32_t *tin = reinterpret_cast<int32_t *>(bmT + words);     // [slots]
  int32_t *slotE = tin + slots;                                // [K]
  int32_t *rankN = slotE + K;                                  // [K]
  int32_t *aSorted = rankN + K;                                // [cap]
  int32_t *fList = aSorted + cap;                              // [cap]
  int32_t *fSorted = fList + cap;                              // [cap]
  // certified selection only (sized by cert_smem_bytes)
  constexpr int D = CH * 8;
  const int Nq = CERTIFY ? ca.G * ca.Nd : 0;
  const int Nq4 = (Nq + 3) & ~3;
  const CertLayout cl = cert_layout(reinterpret_cast<unsigned char *>(fSorted + cap) - smraw, Nb_max, K, CH, Nq);
  uint4 *stage = reinterpret_cast<uint4 *>(smraw + cl.stage);      // staged summaries of recomputed blocks
  float *qsm = reinterpret_cast<float *>(smraw + cl.qsm);          // [D][Nq4] queries
  float *res = reinterpret_cast<float *>(smraw + cl.res);          // [kBatch][Nq4] per-query sums
  uint32_t *bmX = reinterpret_cast<uint32_t *>(smraw + cl.bmX);    // [words] recomputed blocks
  int32_t *xl = reinterpret_cast<int32_t *>(smraw + cl.xl);        // [Nb_max] blocks to recompute
  int32_t *rankE = reinterpret_cast<int32_t *>(smraw + cl.rankE);  // [K]
  float *srow_w = CERTIFY ? ca.scores + static_cast<int64_t>(s) * Nb_max : nullptr;
  const float *rrow = CERTIFY ? ca.radius + static_cast<int64_t>(s) * Nb_max : nullptr;
  const uint4 *gmin = CERTIFY ? reinterpret_cast<const uint4 *>(ca.kmin) + static_cast<int64_t>(s) * CH * Nb_max
                              : nullptr;
  const uint4 *gmax = CERTIFY ? reinterpret_cast<const uint4 *>(ca.kmax) + static_cast<int64_t>(s) * CH * Nb_max
                              : nullptr;

  const int L = load_len(seq_len, s / Hkv, Nb_max * kBlockTokens, status, tid == 0 && (s % Hkv) == 0);
  const int nc = max(0, ceil_div(L, kBlockTokens) - W);

  // 1. table, bitmaps, keys
  for (int i = tid; i < slots; i += kThreads) tin[i] = table_in[static_cast<int64_t>(s) * slots + i];
  for (int i = tid; i < words; i += kThreads) {
    bmR[i] = 0u;
    bmT[i] = 0u;
  }
  if (tid == 0) {
    sc.err = 0;
    sc.nN = sc.nE = sc.nF = sc.nEmpty = 0;
  }
  for (int i = tid; i < 256; i += kThreads) hist[0][i] = 0u;
  if constexpr (CERTIFY) {
    for (int i = tid; i < words; i += kThreads) bmX[i] = 0u;
    // the segment's query vectors, widened: qsm[d][j], j = draft * G + head in group,
    // padded to a multiple of 4 by repeating the last one
    const int Hq = Hkv * ca.G, bseq = s / Hkv, h = s % Hkv, Nq4 = (Nq + 3) & ~3;
    for (int i = tid; i < Nq4 * CH; i += kThreads) {
      const int j = i / CH, c = i % CH, jq = min(j, Nq - 1), jd = jq / ca.G, g = jq % ca.G;
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
          ca.qdraft + ((static_cast<int64_t>(bseq) * ca.Nd + jd) * Hq + h * ca.G + g) * D + c * 8));
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int t = 0; t < 8; ++t) qsm[(c * 8 + t) * Nq4 + j] = (t & 1) ? bf16_hi(w4[t >> 1]) : bf16_lo(w4[t >> 1]);
    }
  }
  bool nan = false;
  const float *srow = scores + static_cast<int64_t>(s) * Nb_max;
  for (int b = tid; b < nc; b += kThreads) keys[b] = score_key(srow[b], nan);
  __syncthreads();
  if (nan) atomicOr(&sc.err, OASIS_STATUS_NAN_SCORE);

  // 2. residents: range and duplicate checks, R bitmap, empty count
  for (int i = tid; i < K; i += kThreads) {
    const int blk = tin[i];
    if (blk == -1) {
      atomicAdd(&sc.nEmpty, 1);
    } else if (blk < 0 || blk >= nc) {
      atomicOr(&sc.err, OASIS_STATUS_TABLE_RANGE);
    } else {
      const uint32_t m = 1u << (blk & 31);
      if (atomicOr(&bmR[blk >> 5], m) & m) atomicOr(&sc.err, OASIS_STATUS_TABLE_DUP);
    }
  }
  __syncthreads();
  const int err = sc.err;
  if (err & (OASIS_STATUS_TABLE_RANGE | OASIS_STATUS_TABLE_DUP)) {
    for (int i = tid; i < slots; i += kThreads) table_out[static_cast<int64_t>(s) * slots + i] = tin[i];
    for (int k = tid; k < cap; k += kThreads) plan[static_cast<int64_t>(s) * cap + k] = oasis_xfer_t{-1, -1};
    if (tid == 0) {
      plan_count[s] = 0;
      report(status, err);
    }
    return;
  }

  // 3. T = top-K candidates
  if constexpr (CERTIFY) {
    if (nc > K) {
      // T by the estimates, then the blocks it cannot settle
      topk_bitmap(keys, nc, K, bmT, hist, sc);
      __syncthreads();
      float lo_in = INFINITY, hi_out = -INFINITY;
      for (int b = tid; b < nc; b += kThreads) {
        float lo, hi;
        interval(srow, rrow, bmX, b, lo, hi);
        if (lo != lo || hi != hi) continue;  // NaN estimate: recomputed below
        if (bit(bmT, b))
          lo_in = fminf(lo_in, lo);
        else
          hi_out = fmaxf(hi_out, hi);
      }
      lo_in = block_reduce(lo_in, false, red);
      hi_out = block_reduce(hi_out, true, red);
      if (tid == 0) nX = 0;
      __syncthreads();
      for (int b = tid; b < nc; b += kThreads) {
        float lo, hi;
        interval(srow, rrow, bmX, b, lo, hi);
        if (!(lo > hi_out) && !(hi < lo_in)) xl[atomicAdd(&nX, 1)] = b;  // NaN lands here too
      }
      __syncthreads();
      recompute_blocks<CH>(xl, nX, gmin, gmax, Nb_max, Nq, qsm, stage, res, srow_w, keys, bmX, sc);
      // T = the settled members of the estimated T, and as many of the recomputed
      // ones as the estimated T held, best first by the exact keys
      int need = 0;
      for (int i = tid; i < nX; i += kThreads) need += bit(bmT, xl[i]);
      need = block_sum(need, sc.warp_tot);
      for (int i = warp; i < nX; i += kWarps) {
        const int b = xl[i];
        const uint64_t ci = composite(keys[b], b);
        int r = 0;
        for (int j0 = 0; j0 < nX; j0 += 32) {
          const int j = j0 + lane;
          r += __popc(__ballot_sync(0xFFFFFFFFu, j < nX && composite(keys[xl[j]], xl[j]) > ci));
        }
        if (lane == 0) {
          const uint32_t m = 1u << (b & 31);
          if (r < need)
            atomicOr(&bmT[b >> 5], m);
          else
            atomicAnd(&bmT[b >> 5], ~m);
        }
      }
      __syncthreads();
    }
  } else {
    topk_bitmap(keys, nc, K, bmT, hist, sc);
    __syncthreads();
  }
  if constexpr (CERTIFY) {
    if (nc <= K) {
      topk_bitmap(keys, nc, K, bmT, hist, sc);  // every candidate
      __syncthreads();
    }
  }

  // 4. lists: N = T \ R (candidates to admit), E = R \ T (residents that may go)
  for (int b = tid; b < nc; b += kThreads) {
    if (bit(bmT, b) && !bit(bmR, b)) {
      const int e = atomicAdd(&sc.nN, 1);
      if (e < K) listN[e] = composite(keys[b], b);
    }
  }
  for (int i = tid; i < K; i += kThreads) {
    const int blk = tin[i];
    if (blk >= 0 && !bit(bmT, blk)) {
      const int e = atomicAdd(&sc.nE, 1);
      if (e < K) {
        listE[e] = composite(keys[blk], blk);
        slotE[e] = i;
      }
    }
  }
  __syncthreads();
  const int nN = min(sc.nN, K), nE = min(sc.nE, K), nEmpty = sc.nEmpty;
  const int nA = min(cap, nN);
  const int nEvict = max(0, nA - nEmpty);
  const int nFill = nA - nEvict;

  if constexpr (CERTIFY) {
    // A = the first nA of N, evicted = the last nEvict of E: settle both by the
    // estimates' intervals, recompute what they cannot settle
    const bool certA = nN > nA, certE = nEvict > 0 && nE > nEvict;
    if (certA || certE) {
      for (int i = warp; i < nN; i += kWarps) {  // rank by the estimates (larger first)
        const uint64_t ci = listN[i];
        int r = 0;
        for (int j0 = 0; j0 < nN; j0 += 32) {
          const int j = j0 + lane;
          r += __popc(__ballot_sync(0xFFFFFFFFu, j < nN && listN[j] > ci));
        }
        if (lane == 0) rankN[i] = r;
      }
      for (int i = warp; i < nE; i += kWarps) {  // rank from the bottom (smaller first)
        const uint64_t ci = listE[i];
        int r = 0;
        for (int j0 = 0; j0 < nE; j0 += 32) {
          const int j = j0 + lane;
          r += __popc(__ballot_sync(0xFFFFFFFFu, j < nE && listE[j] < ci));
        }
        if (lane == 0) rankE[i] = r;
      }
      __syncthreads();
      float a_lo = INFINITY, a_hi = -INFINITY, e_lo = INFINITY, e_hi = -INFINITY;
      for (int i = tid; i < nN; i += kThreads) {
        float lo, hi;
        interval(srow, rrow, bmX, composite_block(listN[i]), lo, hi);
        if (rankN[i] < nA)
          a_lo = fminf(a_lo, lo);
        else
          a_hi = fmaxf(a_hi, hi);
      }
      for (int i = tid; i < nE; i += kThreads) {
        float lo, hi;
        interval(srow, rrow, bmX, composite_block(listE[i]), lo, hi);
        if (rankE[i] < nEvict)
          e_hi = fmaxf(e_hi, hi);  // evicted by the estimates
        else
          e_lo = fminf(e_lo, lo);  // kept by the estimates
      }
      a_lo = block_reduce(a_lo, false, red);
      a_hi = block_reduce(a_hi, true, red);
      e_lo = block_reduce(e_lo, false, red);
      e_hi = block_reduce(e_hi, true, red);
      if (tid == 0) nX = 0;
      __syncthreads();
      for (int i = tid; i < nN && certA; i += kThreads) {
        const int b = composite_block(listN[i]);
        float lo, hi;
        interval(srow, rrow, bmX, b, lo, hi);
        if (!bit(bmX, b) && !(lo > a_hi) && !(hi < a_lo)) xl[atomicAdd(&nX, 1)] = b;
      }
      for (int i = tid; i < nE && certE; i += kThreads) {
        const int b = composite_block(listE[i]);
        float lo, hi;
        interval(srow, rrow, bmX, b, lo, hi);
        if (!bit(bmX, b) && !(lo > e_hi) && !(hi < e_lo)) xl[atomicAdd(&nX, 1)] = b;
      }
      __syncthreads();
      recompute_blocks<CH>(xl, nX, gmin, gmax, Nb_max, Nq, qsm, stage, res, srow_w, keys, bmX, sc);
      for (int i = tid; i < nN; i += kThreads) {
        const int b = composite_block(listN[i]);
        listN[i] = composite(keys[b], b);
      }
      for (int i = tid; i < nE; i += kThreads) {
        const int b = composite_block(listE[i]);
        listE[i] = composite(keys[b], b);
      }
      __syncthreads();
    }
  }

  // 5. A = the nA best of N; freed slots = first nFill empty slots + the nEvict worst of E.
  // Every rank is a count over a list of at most K entries: one warp per entry,
  // its lanes splitting the list, a ballot-popcount per 32 entries.
  for (int i = warp; i < nN; i += kWarps) {
    const uint64_t ci = listN[i];
    int r = 0;
    for (int j0 = 0; j0 < nN; j0 += 32) {
      const int j = j0 + lane;
      r += __popc(__ballot_sync(0xFFFFFFFFu, j < nN && listN[j] > ci));
    }
    if (lane == 0) rankN[i] = r;
  }
  for (int i = warp; i < nE; i += kWarps) {
    const uint64_t ci = listE[i];
    int r = 0;
    for (int j0 = 0; j0 < nE; j0 += 32) {
      const int j = j0 + lane;
      r += __popc(__ballot_sync(0xFFFFFFFFu, j < nE && listE[j] < ci));
    }
    if (lane == 0 && r < nEvict) {
      const int f = atomicAdd(&sc.nF, 1);
      if (f < cap) fList[f] = slotE[i];
    }
  }
  if (nFill > 0) {
    for (int i = warp; i < K; i += kWarps) {
      if (tin[i] != -1) continue;  // warp-uniform
      int r = 0;                   // empty slots before slot i
      for (int j0 = 0; j0 < i; j0 += 32) {
        const int j = j0 + lane;
        r += __popc(__ballot_sync(0xFFFFFFFFu, j < i && tin[j] == -1));
      }
      if (lane == 0 && r < nFill) {
        const int f = atomicAdd(&sc.nF, 1);
        if (f < cap) fList[f] = i;
      }
    }
  }
  __syncthreads();
  for (int i = warp; i < nN; i += kWarps) {
    if (rankN[i] >= nA) continue;  // warp-uniform
    const int b = composite_block(listN[i]);
    int r = 0;
    for (int j0 = 0; j0 < nN; j0 += 32) {
      const int j = j0 + lane;
      r += __popc(__ballot_sync(0xFFFFFFFFu, j < nN && rankN[j] < nA && composite_block(listN[j]) < b));
    }
    if (lane == 0 && r < cap) aSorted[r] = b;
  }
  for (int i = tid; i < nA; i += kThreads) {
    const int sl = fList[i];
    int r = 0;
    for (int j = 0; j < nA; ++j) r += fList[j] < sl;
    if (r < cap) fSorted[r] = sl;
  }
  __syncthreads();

  // 6. outputs
  for (int k = tid; k < nA; k += kThreads) {
    const int sl = fSorted[k];
    if (sl >= 0 && sl < K) tin[sl] = aSorted[k];
  }
  __syncthreads();
  for (int i = tid; i < slots; i += kThreads) table_out[static_cast<int64_t>(s) * slots + i] = tin[i];
  for (int k = tid; k < cap; k += kThreads)
    plan[static_cast<int64_t>(s) * cap + k] = k < nA ? oasis_xfer_t{aSorted[k], fSorted[k]} : oasis_xfer_t{-1, -1};
  if (tid == 0) {
    plan_count[s] = nA;
    report(status, err);
  }
}

}  // namespace

size_t select_smem_bytes(int Nb_max, int K, int W, int cap) {
  const size_t words = (static_cast<size_t>(Nb_max) + 31) / 32;
  return 2 * sizeof(uint64_t) * K + sizeof(uint32_t) * (Nb_max + 2 * words) +
         sizeof(int32_t) * (static_cast<size_t>(K + W) + 2 * K + 3 * static_cast<size_t>(cap));
}


cudaError_t launch_select_topk_capped(const float *scores, int Nb_max, const int32_t *seq_len, int B, int Hkv,
                                      int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                                      oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, cudaStream_t st) {
  const size_t smem = select_smem_bytes(Nb_max, K, W, cap);
  // static (histograms, scalars) + dynamic shared memory may pass the 48 KiB
  // default before the dynamic part alone does
  if (smem + kStaticSmemBound > 48 * 1024) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(k_select<false, 1>), smem);
    if (e != cudaSuccess) return e;
  }
  LaunchCfg lc(dim3(B * Hkv), dim3(kThreads), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_select<false, 1>, scores, Nb_max, seq_len, Hkv, K, W, cap, table_in,
                            table_out, plan, plan_count, status, CertArgs{});
}

size_t select_tc_smem_bytes(int Nb_max, int K, int W, int cap, int D, int Nq) {
  return cert_layout(select_smem_bytes(Nb_max, K, W, cap), Nb_max, K, D / 8, Nq).end;
}

cudaError_t launch_select_topk_capped_tc(float *scores, const float *radius, const uint16_t *kmin,
                                         const uint16_t *kmax, const uint16_t *qdraft, int G, int Nd, int D,
                                         int Nb_max, const int32_t *seq_len, int B, int Hkv, int K, int W, int cap,
                                         const int32_t *table_in, int32_t *table_out, oasis_xfer_t *plan,
                                         int32_t *plan_count, int32_t *status, cudaStream_t st) {
  const size_t smem = select_tc_smem_bytes(Nb_max, K, W, cap, D, G * Nd);
  const void *fn = D == 128 ? reinterpret_cast<const void *>(k_select<true, 16>)
                            : reinterpret_cast<const void *>(k_select<true, 8>);
  if (smem + kStaticSmemBound > 48 * 1024) {
    cudaError_t e = raise_smem_limit(fn, smem);
    if (e != cudaSuccess) return e;
  }
  const CertArgs ca{scores, radius, kmin, kmax, qdraft, G, Nd};
  LaunchCfg lc(dim3(B * Hkv), dim3(kThreads), smem, st);
  if (D == 128)
    return cudaLaunchKernelEx(&lc.cfg, k_select<true, 16>, static_cast<const float *>(scores), Nb_max, seq_len, Hkv,
                              K, W, cap, table_in, table_out, plan, plan_count, status, ca);
  return cudaLaunchKernelEx(&lc.cfg, k_select<true, 8>, static_cast<const float *>(scores), Nb_max, seq_len, Hkv, K,
                            W, cap, table_in, table_out, plan, plan_count, status, ca);
}

}  // namespace oasis
