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
// One CTA per segment (512 threads while the segments do not outnumber the
// SMs, else 256 so that the CTAs share SMs with other kernels), the working
// set in shared memory:
//  * scores -> order-preserving 32-bit keys (larger key = larger score; -0 is
//    mapped to +0 so the two tie; NaN maps to 0, below -inf, and is flagged);
//  * T by a 4-pass 8-bit MSB radix select of the K-th largest key (shared-
//    memory histograms, the digit of each pass found by one warp), then ties
//    at the threshold taken in ascending block order;
//  * T, R as bitmaps; the small lists T\R and R\T are ranked by counting
//    (O(n^2) over <= K entries, no sorting network, few barriers) with the
//    unique 64-bit composite key (key << 32) | ~block.
#include "common.cuh"

namespace oasis {
namespace {

constexpr int kMaxWarps = 16;  // 512 threads at most (the thread count NT is a template parameter)
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

// The score a key came from (NaN for the key of a NaN; +0 for the key of -0).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int b) {
  return (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(b));
}
__device__ __forceinline__ int composite_block(uint64_t c) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(c & 0xFFFFFFFFu));
}

__device__ __forceinline__ bool bit(const uint32_t *bm, int b) { return (bm[b >> 5] >> (b & 31)) & 1u; }

// Exclusive prefix sum of v over the CTA of NT threads (all threads call it).
template <int NT>
__device__ int block_exclusive_scan(int v, int *warp_tot) {
  constexpr int kWarps = NT / 32;
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
  uint32_t digit, dcount;  // radix select: the pass's digit and the keys in its bin
  int remaining;
  int warp_tot[kMaxWarps];
};

static_assert(sizeof(SelScalars) + 2 * 256 * sizeof(uint32_t) + 4 * kMaxWarps * sizeof(float) + 64 <= kStaticSmemBound,
              "static shared memory bound");

// Sum of v over the CTA of NT threads (all threads call it, all get the sum).
template <int NT>
__device__ int block_sum(int v, int *warp_tot) {
  constexpr int kWarps = NT / 32;
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

// T as a bitmap: min(K, nc) candidates, the first by (key desc, block asc)
// when PASSES = 4.  An MSB radix select over the top 8 * PASSES bits of the
// keys finds the bin b* holding the K-th largest key (per pass: the keys
// matching the prefix so far counted into a 256-bin shared histogram with
// plain shared atomics, the bin found by one warp and published through shared
// memory); T = the keys above b* and the first keys of b* in ascending block
// order, all of b* (one ballot per bitmap word) when it holds no more keys
// than are still needed, else through a block-wide prefix count.  With
// PASSES = 4 the bin is one key value and T is exact; with fewer passes T is
// exact up to the order inside the last bin (PASSES = 3: keys within 2^8 units
// in the last place of each other), which the certified selection accepts (it
// settles any K candidates).  bmT must be clear and hist[0] zero; all threads
// call it; the caller synchronises before reading bmT.
template <int PASSES, int NT>
__device__ void topk_bitmap(const uint32_t *keys, int nc, int K, uint32_t *bmT, uint32_t (*hist)[256],
                            SelScalars &sc) {
  constexpr int kThreads = NT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (nc <= K) {
    for (int b0 = warp * 32; b0 < nc; b0 += kThreads) {
      const unsigned m = __ballot_sync(0xFFFFFFFFu, b0 + lane < nc);
      if (lane == 0) bmT[b0 >> 5] = m;
    }
    return;
  }
  uint32_t prefix = 0u, pmask = 0u, bin_count = 0u;
  int remaining = K;
  for (int pass = 0; pass < PASSES; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t *h = hist[pass & 1];
    // four keys loaded before their atomics (independent loads in flight)
    for (int b0 = tid; b0 < nc; b0 += 4 * kThreads) {
      uint32_t k4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) k4[u] = b0 + u * kThreads < nc ? keys[b0 + u * kThreads] : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (b0 + u * kThreads < nc && (k4[u] & pmask) == prefix) atomicAdd(&h[(k4[u] >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // the bin of the remaining-th largest key; lane l owns bins 255-8l down to
      // 248-8l (two 16-byte loads per lane, consecutive lanes consecutive chunks)
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
      const uint32_t before = incl - sum, want = static_cast<uint32_t>(remaining);
      if (before < want && want <= incl) {  // exactly one lane
        uint32_t cum = before;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (cum < want && want <= cum + c[q]) {
            sc.digit = static_cast<uint32_t>(255 - 8 * lane - q);
            sc.remaining = static_cast<int>(want - cum);
            sc.dcount = c[q];
          }
          cum += c[q];
        }
      }
      // the other histogram is counted into next pass: clear it (its last
      // reader, this warp, finished a barrier ago)
      uint4 *nh = reinterpret_cast<uint4 *>(hist[(pass + 1) & 1]);
      nh[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
      nh[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    prefix |= sc.digit << shift;
    pmask |= 0xFFu << shift;
    remaining = sc.remaining;
    bin_count = sc.dcount;
  }
  const int need = remaining;  // keys of the last bin to take, lowest block id first
  if (static_cast<uint32_t>(need) == bin_count) {
    for (int b0 = warp * 32; b0 < nc; b0 += kThreads) {
      const int b = b0 + lane;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, b < nc && (keys[b] & pmask) >= prefix);
      if (lane == 0) bmT[b0 >> 5] = m;
    }
    return;
  }
  const int per = ceil_div(nc, kThreads);
  const int lo = min(nc, tid * per), hi = min(nc, lo + per);
  int ties = 0;
  for (int b = lo; b < hi; ++b) ties += (keys[b] & pmask) == prefix;
  int before = block_exclusive_scan<NT>(ties, sc.warp_tot);
  for (int b = lo; b < hi; ++b) {
    const uint32_t km = keys[b] & pmask;
    bool in = km > prefix;
    if (km == prefix) {
      in = before < need;
      ++before;
    }
    if (in) atomicOr(&bmT[b >> 5], 1u << (b & 31));
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
constexpr int kBatch = 4;  // blocks recomputed per pass

// Byte offsets of the certified kernel's extra shared memory, from the start
// of the dynamic allocation; one definition serves the kernel's pointers and
// the launcher's allocation size.
struct CertLayout {
  size_t stage, res, bmX, xl, rankE, end;
};
__host__ __device__ inline CertLayout cert_layout(size_t base_bytes, int Nb_max, int K, int CH, int Nq) {
  const size_t words = (static_cast<size_t>(Nb_max) + 31) / 32;
  const size_t Nq4 = (static_cast<size_t>(Nq) + 3) & ~static_cast<size_t>(3);
  CertLayout L;
  L.stage = (base_bytes + 15) & ~static_cast<size_t>(15);
  L.res = L.stage + 16 * static_cast<size_t>(kBatch) * (2 * CH + 1);      // uint4 [kBatch][2*CH + 1]
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

// CTA-wide min of each lo[k] and max of each hi[k] (NaN ignored), one
// barrier pair for all of them; every thread gets the results.
template <int N, int NT>
__device__ void block_minmax(float (&lo)[N], float (&hi)[N], float (*red)[kMaxWarps]) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < N; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo[k] = fminf(lo[k], __shfl_xor_sync(0xFFFFFFFFu, lo[k], o));
      hi[k] = fmaxf(hi[k], __shfl_xor_sync(0xFFFFFFFFu, hi[k], o));
    }
  }
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      red[2 * k][warp] = lo[k];
      red[2 * k + 1][warp] = hi[k];
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    for (int w = 0; w < kWarps; ++w) {
      lo[k] = fminf(lo[k], red[2 * k][w]);
      hi[k] = fmaxf(hi[k], red[2 * k + 1][w]);
    }
  }
}

// Fixed-order fp32 scores of the listed blocks (the oasis_score_blocks
// arithmetic: per query, sum over d ascending from +0 of q_d * (q_d >= 0 ?
// kmax_d : kmin_d), one rounding per term; max over the queries, NaN kept).
// Writes them to srow and their keys to keys and marks them in bmX (a
// recomputed score is exact: its radius counts as 0).  A thread takes one (block,
// query) pair at a time and reads the query from global memory (query j =
// draft j / G of head j % G: row qseg + ((j / G) * Hq + j % G) * D; a handful of
// blocks per segment are recomputed, so the reads stay in cache and the CTA
// keeps no copy of the queries).  The max over a block's queries is taken by
// one warp as the largest order key of the sums (+0 above -0), which does not
// depend on the order of the reduction.
template <int CH, int NT>
__device__ void recompute_blocks(const int32_t *xl, int n, const uint4 *gmin, const uint4 *gmax, int Nb_max,
                                 int Nq, const uint16_t *qseg, int G, int Hq, uint4 *stage, float *res, float *srow,
                                 uint32_t *keys, uint32_t *bmX, SelScalars &sc) {
  constexpr int ES = 2 * CH + 1;  // staged entry: kmin chunks, kmax chunks, one pad (bank spread)
  constexpr int kThreads = NT, kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Nq4 = (Nq + 3) & ~3;
  for (int e0 = 0; e0 < n; e0 += kBatch) {
    const int nb = min(kBatch, n - e0);
    for (int i = tid; i < nb * 2 * CH; i += kThreads) {
      const int e = i / (2 * CH), k = i % (2 * CH), c = k % CH;
      const int b = xl[e0 + e];
      stage[e * ES + k] = __ldg((k < CH ? gmin : gmax) + static_cast<int64_t>(c) * Nb_max + b);
    }
    __syncthreads();
    for (int i = tid; i < nb * Nq; i += kThreads) {
      const int e = i / Nq, j = i - e * Nq;
      const int jd = j / G;
      const uint4 *st = stage + e * ES;
      const uint4 *qj = reinterpret_cast<const uint4 *>(qseg + (static_cast<int64_t>(jd) * Hq + (j - jd * G)) * (8 * CH));
      float acc = 0.0f;
#pragma unroll 2
      for (int c = 0; c < CH; ++c) {
        const uint4 mn = st[c], mx = st[CH + c], qv = __ldg(qj + c);
        const uint32_t wn[4] = {mn.x, mn.y, mn.z, mn.w}, wx[4] = {mx.x, mx.y, mx.z, mx.w};
        const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float kn = (t & 1) ? bf16_hi(wn[t >> 1]) : bf16_lo(wn[t >> 1]);
          const float kx = (t & 1) ? bf16_hi(wx[t >> 1]) : bf16_lo(wx[t >> 1]);
          const float q = (t & 1) ? bf16_hi(wq[t >> 1]) : bf16_lo(wq[t >> 1]);
          acc = fmaf(q, q >= 0.0f ? kx : kn, acc);  // exact product, one rounding
        }
      }
      res[e * Nq4 + j] = acc;
    }
    __syncthreads();
    for (int e = warp; e < nb; e += kWarps) {
      uint32_t best = 0u;  // below the order key of every non-NaN float
      bool nan = false;
      for (int j = lane; j < Nq; j += 32) {
        const uint32_t u = __float_as_uint(res[e * Nq4 + j]);
        nan |= (u & 0x7FFFFFFFu) > 0x7F800000u;
        best = max(best, (u & 0x80000000u) ? ~u : (u | 0x80000000u));
      }
      best = __reduce_max_sync(0xFFFFFFFFu, best);
      nan = __any_sync(0xFFFFFFFFu, nan);
      if (lane == 0) {
        const float v = nan ? __uint_as_float(0x7FC00000u)
                            : __uint_as_float((best & 0x80000000u) ? (best & 0x7FFFFFFFu) : ~best);
        const int b = xl[e0 + e];
        srow[b] = v;
        bool isn = false;
        keys[b] = score_key(v, isn);
        if (isn) atomicOr(&sc.err, OASIS_STATUS_NAN_SCORE);
        atomicOr(&bmX[b >> 5], 1u << (b & 31));
      }
    }
    __syncthreads();
  }
}

// Rank of every entry of a list of distinct 64-bit keys: the number of larger
// (kDesc) or smaller entries.  One thread per entry reads the whole list; all
// threads of a warp read the same entry at a time (a broadcast), so a short list
// costs a few hundred cycles where a warp-wide ballot per entry costs thousands.
template <int NT, bool kDesc>
__device__ __forceinline__ void rank_list(const uint64_t *list, int n, int32_t *rank) {
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint64_t ci = list[i];
    int r = 0;
#pragma unroll 4
    for (int j = 0; j < n; ++j) r += kDesc ? (list[j] > ci) : (list[j] < ci);
    rank[i] = r;
  }
}

// interval of block b from its key and radius (a recomputed block has radius 0)
__device__ __forceinline__ void interval(const uint32_t *keys, const float *rrow, const uint32_t *bmX, int b,
                                         float &lo, float &hi) {
  const float v = key_score(keys[b]);
  const float r = bit(bmX, b) ? 0.0f : __ldg(rrow + b);
  lo = v - r;
  hi = v + r;
}

// CERTIFY = false: the selection on exact scores.  CERTIFY = true: `scores`
// holds estimates with radii (CertArgs); the decisions the estimates cannot
// settle are settled by recomputing fixed-order scores (see above).
template <bool CERTIFY, int CH, int NT>
__global__ void __launch_bounds__(NT) k_select(const float *scores, int Nb_max,
                                                     const int32_t *__restrict__ seq_len, int Hkv, int K, int W,
                                                     int cap, const int32_t *table_in, int32_t *table_out,
                                                     oasis_xfer_t *__restrict__ plan, int32_t *__restrict__ plan_count,
                                                     int32_t *status, CertArgs ca) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ SelScalars sc;
  __shared__ __align__(16) uint32_t hist[2][256];  // radix pass p counts into hist[p & 1]
  __shared__ float red[4][kMaxWarps];
  constexpr int kThreads = NT, kWarps = NT / 32;
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
  // certified selection only (laid out by cert_layout, which the launcher sizes with)
  constexpr int D = CH * 8;
  const int Nq = CERTIFY ? ca.G * ca.Nd : 0;
  const CertLayout cl = cert_layout(reinterpret_cast<unsigned char *>(fSorted + cap) - smraw, Nb_max, K, CH, Nq);
  uint4 *stage = reinterpret_cast<uint4 *>(smraw + cl.stage);      // staged summaries of recomputed blocks
  float *res = reinterpret_cast<float *>(smraw + cl.res);          // [kBatch][Nq4] per-query sums
  uint32_t *bmX = reinterpret_cast<uint32_t *>(smraw + cl.bmX);    // [words] recomputed blocks
  int32_t *xl = reinterpret_cast<int32_t *>(smraw + cl.xl);        // [Nb_max] blocks to recompute
  int32_t *rankE = reinterpret_cast<int32_t *>(smraw + cl.rankE);  // [K]
  float *srow_w = CERTIFY ? ca.scores + static_cast<int64_t>(s) * Nb_max : nullptr;
  // the segment's draft queries: [Nd][Hq][D] rows of sequence s / Hkv from head (s % Hkv) * G on
  const int Hq_c = CERTIFY ? Hkv * ca.G : 0;
  const uint16_t *qseg = CERTIFY ? ca.qdraft + (static_cast<int64_t>(s / Hkv) * ca.Nd * Hq_c + (s % Hkv) * ca.G) * D
                                 : nullptr;
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
  if constexpr (CERTIFY)
    for (int i = tid; i < words; i += kThreads) bmX[i] = 0u;
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
      topk_bitmap<3, NT>(keys, nc, K, bmT, hist, sc);
      __syncthreads();
      float lo_in[1] = {INFINITY}, hi_out[1] = {-INFINITY};
      for (int b = tid; b < nc; b += kThreads) {
        float lo, hi;
        interval(keys, rrow, bmX, b, lo, hi);
        if (lo != lo || hi != hi) continue;  // NaN estimate: recomputed below
        if (bit(bmT, b))
          lo_in[0] = fminf(lo_in[0], lo);
        else
          hi_out[0] = fmaxf(hi_out[0], hi);
      }
      if (tid == 0) nX = 0;  // read after the reduction's barriers
      block_minmax<1, NT>(lo_in, hi_out, red);
      for (int b = tid; b < nc; b += kThreads) {
        float lo, hi;
        interval(keys, rrow, bmX, b, lo, hi);
        if (!(lo > hi_out[0]) && !(hi < lo_in[0])) xl[atomicAdd(&nX, 1)] = b;  // NaN lands here too
      }
      __syncthreads();
      recompute_blocks<CH, NT>(xl, nX, gmin, gmax, Nb_max, Nq, qseg, ca.G, Hq_c, stage, res, srow_w, keys, bmX, sc);
      // T = the settled members of the estimated T, and as many of the recomputed
      // ones as the estimated T held, best first by the exact keys
      int need = 0;
      for (int i = tid; i < nX; i += kThreads) need += bit(bmT, xl[i]);
      need = block_sum<NT>(need, sc.warp_tot);
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
    topk_bitmap<4, NT>(keys, nc, K, bmT, hist, sc);
    __syncthreads();
  }
  if constexpr (CERTIFY) {
    if (nc <= K) {
      topk_bitmap<4, NT>(keys, nc, K, bmT, hist, sc);  // every candidate
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
      rank_list<NT, true>(listN, nN, rankN);   // rank by the estimates (larger first)
      rank_list<NT, false>(listE, nE, rankE);  // rank from the bottom (smaller first)
      __syncthreads();
      // lo[0]/hi[0]: min over A~ / max over N \ A~; lo[1]/hi[1]: min over the kept
      // of E / max over the evicted of E
      float lo_[2] = {INFINITY, INFINITY}, hi_[2] = {-INFINITY, -INFINITY};
      for (int i = tid; i < nN; i += kThreads) {
        float lo, hi;
        interval(keys, rrow, bmX, composite_block(listN[i]), lo, hi);
        if (rankN[i] < nA)
          lo_[0] = fminf(lo_[0], lo);
        else
          hi_[0] = fmaxf(hi_[0], hi);
      }
      for (int i = tid; i < nE; i += kThreads) {
        float lo, hi;
        interval(keys, rrow, bmX, composite_block(listE[i]), lo, hi);
        if (rankE[i] < nEvict)
          hi_[1] = fmaxf(hi_[1], hi);  // evicted by the estimates
        else
          lo_[1] = fminf(lo_[1], lo);  // kept by the estimates
      }
      if (tid == 0) nX = 0;  // read after the reduction's barriers
      block_minmax<2, NT>(lo_, hi_, red);
      const float a_lo = lo_[0], a_hi = hi_[0], e_lo = lo_[1], e_hi = hi_[1];
      for (int i = tid; i < nN && certA; i += kThreads) {
        const int b = composite_block(listN[i]);
        float lo, hi;
        interval(keys, rrow, bmX, b, lo, hi);
        if (!bit(bmX, b) && !(lo > a_hi) && !(hi < a_lo)) xl[atomicAdd(&nX, 1)] = b;
      }
      for (int i = tid; i < nE && certE; i += kThreads) {
        const int b = composite_block(listE[i]);
        float lo, hi;
        interval(keys, rrow, bmX, b, lo, hi);
        if (!bit(bmX, b) && !(lo > e_hi) && !(hi < e_lo)) xl[atomicAdd(&nX, 1)] = b;
      }
      __syncthreads();
      recompute_blocks<CH, NT>(xl, nX, gmin, gmax, Nb_max, Nq, qseg, ca.G, Hq_c, stage, res, srow_w, keys, bmX, sc);
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
  // Every rank is a count over a list of at most K entries (one thread per entry).
  rank_list<NT, true>(listN, nN, rankN);
  for (int i = tid; i < nE; i += kThreads) {
    const uint64_t ci = listE[i];
    int r = 0;
#pragma unroll 4
    for (int j = 0; j < nE; ++j) r += listE[j] < ci;
    if (r < nEvict) {
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
  for (int i = tid; i < nN; i += kThreads) {
    if (rankN[i] >= nA) continue;
    const int b = composite_block(listN[i]);
    int r = 0;
    for (int j = 0; j < nN; ++j) r += rankN[j] < nA && composite_block(listN[j]) < b;
    if (r < cap) aSorted[r] = b;
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


namespace {

// Threads per selection CTA: 512 while every segment's CTA can have an SM to
// itself, else 256, so that selection CTAs stay small enough to share SMs with
// the scoring and attention CTAs of other layers (measured on GB300: 512-thread
// CTAs cost the 256-segment decode step 13 us per layer-step; 256-thread CTAs
// cost the 64- and 128-segment steps 0.7 and 2.5 us).
int select_threads(int segments) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 0;
  }
  return segments <= sms ? 512 : 256;
}

template <int NT>
cudaError_t launch_exact(const float *scores, int Nb_max, const int32_t *seq_len, int S, int Hkv, int K, int W,
                         int cap, const int32_t *table_in, int32_t *table_out, oasis_xfer_t *plan,
                         int32_t *plan_count, int32_t *status, size_t smem, cudaStream_t st) {
  // static (histograms, scalars) + dynamic shared memory may pass the 48 KiB
  // default before the dynamic part alone does
  if (smem + kStaticSmemBound > 48 * 1024) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(k_select<false, 1, NT>), smem);
    if (e != cudaSuccess) return e;
  }
  LaunchCfg lc(dim3(S), dim3(NT), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_select<false, 1, NT>, scores, Nb_max, seq_len, Hkv, K, W, cap, table_in,
                            table_out, plan, plan_count, status, CertArgs{});
}

template <int CH, int NT>
cudaError_t launch_cert(const float *scores, int Nb_max, const int32_t *seq_len, int S, int Hkv, int K, int W,
                        int cap, const int32_t *table_in, int32_t *table_out, oasis_xfer_t *plan,
                        int32_t *plan_count, int32_t *status, const CertArgs &ca, size_t smem, cudaStream_t st) {
  if (smem + kStaticSmemBound > 48 * 1024) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(k_select<true, CH, NT>), smem);
    if (e != cudaSuccess) return e;
  }
  LaunchCfg lc(dim3(S), dim3(NT), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_select<true, CH, NT>, scores, Nb_max, seq_len, Hkv, K, W, cap, table_in,
                            table_out, plan, plan_count, status, ca);
}

}  // namespace

cudaError_t launch_select_topk_capped(const float *scores, int Nb_max, const int32_t *seq_len, int B, int Hkv,
                                      int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                                      oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, cudaStream_t st) {
  const size_t smem = select_smem_bytes(Nb_max, K, W, cap);
  const int S = B * Hkv;
  if (select_threads(S) == 512)
    return launch_exact<512>(scores, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                             status, smem, st);
  return launch_exact<256>(scores, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                           status, smem, st);
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
  const CertArgs ca{scores, radius, kmin, kmax, qdraft, G, Nd};
  const int S = B * Hkv;
  const float *sc = scores;
  const bool wide = select_threads(S) == 512;
  if (D == 128)
    return wide ? launch_cert<16, 512>(sc, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                                       status, ca, smem, st)
                : launch_cert<16, 256>(sc, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                                       status, ca, smem, st);
  return wide ? launch_cert<8, 512>(sc, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                                    status, ca, smem, st)
              : launch_cert<8, 256>(sc, Nb_max, seq_len, S, Hkv, K, W, cap, table_in, table_out, plan, plan_count,
                                    status, ca, smem, st);
}

}  // namespace oasis
