// Look-ahead block scores on the tensor cores, with a certified error radius
// per block (OasisKV paper review (xllm-io), §3 decode flow: the draft queries
// scan the compressed key summaries; §4 Fig. 7).
//
// The score of block b for query j is a dot product over 2*D terms,
//     s_jb = sum_d q+_jd * kmax_bd + sum_d q-_jd * kmin_bd,
// with q+ = q where q >= 0 (else +0) and q- = q where q < 0 (else +0): one of
// the two terms of each dim is an exact zero, so this is the Quest bound
// sum_d q_d * (q_d >= 0 ? kmax_d : kmin_d).  For a KV head it is a dense
// [blocks x 2D] x [2D x queries] product, run here as tcgen05 MMAs (M = 128
// blocks, N = the head's query columns, K = 2D, bf16 operands, fp32
// accumulation in tensor memory); the block score is the max over the columns.
//
// The tensor cores add in an order of their own, so the result s~ differs
// from the fixed-order fp32 sum s of oasis_score_blocks by rounding.  Every
// block gets a radius r with |s~ - s| <= r:
//     sum_d |term_jbd| <= |s~_b| + 2 C_b,   C_b = sum_d Q_d c_bd,
// where Q_d = max_j |q_jd| over the head's queries and c_bd is the magnitude of
// the summary values on the "wrong" side of zero (|kmax_bd| when kmax_bd < 0,
// plus kmin_bd when kmin_bd > 0; zero for the usual kmin <= 0 <= kmax).  Both the
// fixed-order sum of 128 terms (relative error below 2^-17 of the absolute
// sum) and any fp32 accumulation of the tensor cores (below 2^-17 even if each
// of the 16 MMA steps rounded or truncated) are far inside
//     r = 2^-12 (|s~_b| + 2 C_b) + 2^-110.
// A selection that compares such intervals and recomputes the fixed-order
// score of every block whose interval decides it (oasis_select_topk_capped_tc)
// is therefore identical to the selection on the fixed-order scores.
//
// Work split: the tiles (128 consecutive candidate blocks of one segment) of
// all segments form one range, split evenly over a persistent grid of one CTA
// per SM.  Roles in a CTA (warp-specialised, mbarrier hand-offs, every wait
// bounded):
//   warp 0, one lane  - bulk copies of a tile's 2*D/8 chunks (16 bytes per
//                       block per 8 dims, contiguous over the tile's blocks in
//                       the chunk-major summary layout) into a ring of stages;
//   warp 1, one lane  - the 2D/16 MMAs of a tile into one of two TMEM
//                       accumulators (the warp also owns the TMEM allocation);
//   warps 2-5         - per segment, the split query operand {q+, q-} in the
//                       no-swizzle K-major layout and Q_d (two buffers, built
//                       one segment ahead); per tile, C_b from the stage (each
//                       thread one block row), then the accumulator row from
//                       TMEM (tcgen05.ld), the max over the columns, the radius,
//                       and the stores.
// Shared-memory operands use the no-swizzle K-major layout of 8-row x 16-byte
// core matrices: the chunk-major summaries already are that layout (chunk c of
// 128 blocks = 16 core matrices at 128-byte steps), so a tile lands by plain
// bulk copies: LBO (next 8 K-elements) = 2048 bytes, SBO (next 8 rows) = 128.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kRows = 128;                    // blocks per tile (MMA M)
constexpr int kEpiWarps = 4;
constexpr int kThreadsTC = 32 * (2 + kEpiWarps);
constexpr uint32_t kChunkBytes = kRows * 16;  // one 8-dim chunk of a tile
constexpr uint32_t kWaitTriesTC = 1u << 22;   // bounded mbarrier polls (far beyond any real copy or MMA)
constexpr size_t kSmemCap = 227 * 1024;

// ---- tcgen05 / TMEM primitives (inline PTX, sm_100a family) -----------------
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // start address, leading (K) and stride (M/N) byte offsets in 16-byte units;
  // bit 46: descriptor version of this architecture; swizzle field 0 = none
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}
// instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24
template <int N>
__device__ __forceinline__ uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(kRows >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  // the registers are valid only after the wait: tie them to it
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory"); }

// Bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  for (uint32_t k = 0; k < kWaitTriesTC; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// bf16 sign of each half replicated over that half (0xFFFF where negative):
// prmt in its default mode, selector nibbles 9 and B = bytes 1 and 3 with the
// sign-replicate bit set
__device__ __forceinline__ uint32_t neg_halves(uint32_t x) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(r) : "r"(x));
  return r;
}

struct TileIter {
  // the CTA's tiles [t0, t1) in segment-major order; a tile is work when its
  // first block is a candidate of its segment
  int64_t t0, t1;
  int tps, Hkv, W, Nb_max;
  const int32_t *seq_len;
  __device__ int nc_of(int s) const {
    int L = __ldg(seq_len + s / Hkv);
    L = L < 0 ? 0 : (L > Nb_max * kBlockTokens ? Nb_max * kBlockTokens : L);
    return ceil_div(L, kBlockTokens) - W;
  }
  // first work tile at or after t (t1 if none); nc of its segment in *nc
  __device__ int64_t next(int64_t t, int *nc) const {
    while (t < t1) {
      const int s = static_cast<int>(t / tps);
      const int n = nc_of(s);
      const int64_t seg_end = std::min<int64_t>(t1, static_cast<int64_t>(s + 1) * tps);
      if (static_cast<int>(t - static_cast<int64_t>(s) * tps) * kRows < n) {
        *nc = n;
        return t;
      }
      t = seg_end;  // the remaining tiles of this segment are past its candidates
    }
    return t1;
  }
};

template <int N, int CH>
__global__ void __launch_bounds__(kThreadsTC, 1)
    k_score_tc(const uint16_t *__restrict__ kmin, const uint16_t *__restrict__ kmax, int Nb_max,
               const uint16_t *__restrict__ qdraft, int S, int Hkv, int G, int Nd,
               const int32_t *__restrict__ seq_len, int W, float *__restrict__ scores, float *__restrict__ radius,
               int32_t *status, int tps, int stages) {
  constexpr int D = CH * 8;
  constexpr int KS = 2 * D / 16;                       // MMAs per tile (K = 16 each)
  constexpr uint32_t kATile = 2u * CH * kChunkBytes;   // kmax chunks then kmin chunks
  constexpr uint32_t kBBytes = static_cast<uint32_t>(N) * 2 * D * 2;
  constexpr uint32_t kTmemCols = 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128);
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sA = smem;                                               // [stages][kATile]
  uint8_t *sB = sA + static_cast<size_t>(stages) * kATile;          // [2][kBBytes]
  float *sQ = reinterpret_cast<float *>(sB + 2 * kBBytes);          // [2][D]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sQ + 2 * D);        // full[st], empty[st], accF[2], accE[2], bq[2]
  uint64_t *full = bars, *empty = bars + stages, *accF = bars + 2 * stages, *accE = accF + 2, *bqF = accE + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bqF + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TileIter it;
  {
    const int64_t T = static_cast<int64_t>(S) * tps;
    it.t0 = T * blockIdx.x / gridDim.x;
    it.t1 = T * (blockIdx.x + 1) / gridDim.x;
    it.tps = tps;
    it.Hkv = Hkv;
    it.W = W;
    it.Nb_max = Nb_max;
    it.seq_len = seq_len;
  }
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + kEpiWarps);  // the MMAs' commit + each epilogue warp's scan
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accF[i], 1);
      mbar_init(&accE[i], kEpiWarps);
      mbar_init(&bqF[i], 32 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0 && blockIdx.x == 0) {
    for (int b = 0; b < S / Hkv; ++b) {  // report an out-of-range length once
      const int L = __ldg(seq_len + b);
      if (L < 0 || L > Nb_max * kBlockTokens) {
        report(status, OASIS_STATUS_SEQ_LEN);
        break;
      }
    }
  }

  if (warp == 0) {
    // ---------------- producer: bulk copies of the tiles into the stage ring
    if (lane == 0) {
      int64_t issued = 0;
      int nc = 0;
      for (int64_t t = it.next(it.t0, &nc); t < it.t1; t = it.next(t + 1, &nc)) {
        const int s = static_cast<int>(t / tps);
        const int base = static_cast<int>(t - static_cast<int64_t>(s) * tps) * kRows;
        const int rows = min(kRows, nc - base);
        const int st = static_cast<int>(issued % stages);
        if (issued >= stages &&
            !wait_or_abort(&empty[st], static_cast<uint32_t>((issued / stages) - 1) & 1u, abort_flag))
          break;
        const uint32_t bytes = static_cast<uint32_t>(rows) * 16u;
        mbar_arrive_expect_tx(&full[st], 2u * CH * bytes);
        uint8_t *dst = sA + static_cast<size_t>(st) * kATile;
        const uint4 *gx = reinterpret_cast<const uint4 *>(kmax) + static_cast<int64_t>(s) * CH * Nb_max + base;
        const uint4 *gn = reinterpret_cast<const uint4 *>(kmin) + static_cast<int64_t>(s) * CH * Nb_max + base;
#pragma unroll 4
        for (int c = 0; c < CH; ++c) {
          bulk_g2s(dst + c * kChunkBytes, gx + static_cast<int64_t>(c) * Nb_max, bytes, &full[st]);
          bulk_g2s(dst + (CH + c) * kChunkBytes, gn + static_cast<int64_t>(c) * Nb_max, bytes, &full[st]);
        }
        ++issued;
      }
      // never leave with copies in flight: wait for the last stages issued
      for (int64_t k = std::max<int64_t>(0, issued - stages); k < issued; ++k)
        mbar_wait_bounded(&full[k % stages], static_cast<uint32_t>(k / stages) & 1u, kWaitTriesTC);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16<N>();
      int64_t i = 0;
      int seg_prev = -1, nseg = 0, buf = 0;
      int nc = 0;
      bool ok = true;
      for (int64_t t = it.next(it.t0, &nc); t < it.t1 && ok; t = it.next(t + 1, &nc)) {
        const int s = static_cast<int>(t / tps);
        if (s != seg_prev) {  // the query operand of this segment
          buf = nseg & 1;
          ok = wait_or_abort(&bqF[buf], static_cast<uint32_t>(nseg >> 1) & 1u, abort_flag);
          ++nseg;
          seg_prev = s;
          if (!ok) break;
        }
        const int st = static_cast<int>(i % stages);
        const int acc = static_cast<int>(i & 1);
        ok = wait_or_abort(&full[st], static_cast<uint32_t>(i / stages) & 1u, abort_flag);
        if (ok && i >= 2) ok = wait_or_abort(&accE[acc], static_cast<uint32_t>((i >> 1) - 1) & 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = smem_addr(sA + static_cast<size_t>(st) * kATile);
        const uint32_t b0 = smem_addr(sB + static_cast<size_t>(buf) * kBBytes);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint64_t da = smem_desc(a0 + kk * 2 * kChunkBytes, kChunkBytes, 128);
          const uint64_t db = smem_desc(b0 + kk * 2 * (N * 16), N * 16, 128);
          tc_mma(tmem + static_cast<uint32_t>(acc * N), da, db, idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(&empty[st]);
        tc_commit(&accF[acc]);
        ++i;
      }
      // every MMA issued has completed before the accumulators are released:
      // the last commit arrives on accF of the last tile
      if (i > 0) mbar_wait_bounded(&accF[(i - 1) & 1], static_cast<uint32_t>((i - 1) >> 1) & 1u, kWaitTriesTC);
    }
  } else {
    // ---------------- epilogue warps: query operands, radii, TMEM -> scores
    const int et = tid - 64;                   // 0 .. 127
    const int quad = warp & 3;                 // the TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;          // the tile row (block) this thread owns
    const int Nq = G * Nd, Hq = Hkv * G;
    const int s_first = static_cast<int>(it.t0 / tps);
    const int s_last = it.t1 > it.t0 ? static_cast<int>((it.t1 - 1) / tps) : s_first - 1;
    int next_build = s_first, built = 0;
    // does segment s have a work tile in [t0, t1)?
    auto active = [&](int s) {
      const int64_t first = std::max<int64_t>(it.t0, static_cast<int64_t>(s) * tps);
      return static_cast<int>(first - static_cast<int64_t>(s) * tps) * kRows < it.nc_of(s);
    };
    // build {q+, q-} and Q of the next active segment into buffer built & 1
    auto build_next = [&]() {
      while (next_build <= s_last && !active(next_build)) ++next_build;
      if (next_build > s_last) return;
      const int s = next_build, bq = built & 1;
      const int bseq = s / Hkv, h = s % Hkv;
      uint8_t *B = sB + static_cast<size_t>(bq) * kBBytes;
      float *Q = sQ + bq * D;
      epi_barrier();  // every epilogue thread is done with this buffer's previous segment
      for (int d = et; d < D; d += 32 * kEpiWarps) Q[d] = 0.0f;
      epi_barrier();
      for (int item = et; item < N * CH; item += 32 * kEpiWarps) {
        const int n = item / CH, c = item % CH;
        const int j = min(n, Nq - 1), jd = j / G, g = j % G;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
            qdraft + ((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + g) * D + c * 8));
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t pos[4], neg[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t m = neg_halves(w4[e]);
          neg[e] = w4[e] & m;
          pos[e] = w4[e] & ~m;
          // Q_d = max over the queries of |q_d| (non-negative floats order as integers)
          atomicMax(reinterpret_cast<unsigned int *>(Q) + c * 8 + 2 * e, (w4[e] & 0x7FFFu) << 16);
          atomicMax(reinterpret_cast<unsigned int *>(Q) + c * 8 + 2 * e + 1, w4[e] & 0x7FFF0000u);
        }
        *reinterpret_cast<uint4 *>(B + c * (N * 16) + n * 16) = make_uint4(pos[0], pos[1], pos[2], pos[3]);
        *reinterpret_cast<uint4 *>(B + (CH + c) * (N * 16) + n * 16) = make_uint4(neg[0], neg[1], neg[2], neg[3]);
      }
      fence_proxy_async_smem();  // the tensor cores read B through the async proxy
      mbar_arrive(&bqF[bq]);
      epi_barrier();             // Q is complete for every epilogue thread
      ++next_build;
      ++built;
    };
    build_next();
    build_next();
    int64_t i = 0;
    int seg_prev = -1, used = 0, bq = 0;
    int nc = 0;
    const float gamma = 0x1p-12f, floor_r = 0x1p-110f;
    for (int64_t t = it.next(it.t0, &nc); t < it.t1; t = it.next(t + 1, &nc)) {
      const int s = static_cast<int>(t / tps);
      if (s != seg_prev) {
        if (seg_prev >= 0) build_next();  // the segment before is done: its buffer is free
        bq = used & 1;
        ++used;
        seg_prev = s;
      }
      const int base = static_cast<int>(t - static_cast<int64_t>(s) * tps) * kRows;
      const int rows = min(kRows, nc - base);
      const int st = static_cast<int>(i % stages);
      const int acc = static_cast<int>(i & 1);
      if (!wait_or_abort(&full[st], static_cast<uint32_t>(i / stages) & 1u, abort_flag)) break;
      // C_b: the summary values on the wrong side of zero, weighted by Q_d
      float C = 0.0f;
      if (row < rows) {
        const uint8_t *A = sA + static_cast<size_t>(st) * kATile + row * 16;
        const float *Q = sQ + bq * D;
#pragma unroll 4
        for (int c = 0; c < CH; ++c) {
          const uint4 x = *reinterpret_cast<const uint4 *>(A + c * kChunkBytes);
          const uint4 y = *reinterpret_cast<const uint4 *>(A + (CH + c) * kChunkBytes);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
          uint32_t any = 0, nw[4], pw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            nw[e] = xs[e] & neg_halves(xs[e]) & 0x7FFF7FFFu;  // |kmax| where kmax < 0
            pw[e] = ys[e] & ~neg_halves(ys[e]);               // kmin where kmin > 0
            any |= nw[e] | pw[e];
          }
          if (any) {
            const float *q = Q + c * 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              C = fmaf(q[2 * e], bf16_lo(nw[e]) + bf16_lo(pw[e]), C);
              C = fmaf(q[2 * e + 1], bf16_hi(nw[e]) + bf16_hi(pw[e]), C);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (!wait_or_abort(&accF[acc], static_cast<uint32_t>(i >> 1) & 1u, abort_flag)) break;
      tc_fence_after();
      float best = -FLT_MAX;
      bool nan = false;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * N);
#pragma unroll
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float v = __uint_as_float(r[k]);
          nan |= v != v;
          best = fmaxf(best, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accE[acc]);
      if (row < rows) {
        const float sc = nan ? __uint_as_float(0x7FC00000u) : best;
        const float rad = fmaf(gamma, fabsf(best) + 2.0f * C, floor_r);
        const int64_t o = static_cast<int64_t>(s) * Nb_max + base + row;
        scores[o] = sc;
        radius[o] = nan ? __uint_as_float(0x7F800000u) : rad;
      }
      ++i;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) report(status, OASIS_STATUS_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int N, int CH>
cudaError_t launch_tc(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                      int Hkv, int G, int Nd, const int32_t *seq_len, int W, float *scores, float *radius,
                      int32_t *status, cudaStream_t st) {
  constexpr int D = CH * 8;
  constexpr size_t kATile = 2u * CH * kChunkBytes;
  constexpr size_t kBBytes = static_cast<size_t>(N) * 2 * D * 2;
  const int S = B * Hkv;
  const int ncand = Nb_max - W;
  if (ncand <= 0) return cudaSuccess;  // no candidate can exist
  const int tps = (ncand + kRows - 1) / kRows;
  const size_t fixed = 2 * kBBytes + 2 * D * sizeof(float) + 16 * sizeof(uint64_t) + 64;
  const int stages = static_cast<int>(std::min<size_t>(4, (kSmemCap - fixed) / kATile));
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + stages * kATile + 1024;  // + alignment slack of the dynamic base
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_score_tc<N, CH>), kThreadsTC, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t T = static_cast<int64_t>(S) * tps;
  const int grid = static_cast<int>(std::min<int64_t>(sms, T));
  LaunchCfg lc(dim3(grid), dim3(kThreadsTC), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_score_tc<N, CH>, kmin, kmax, Nb_max, qdraft, S, Hkv, G, Nd, seq_len, W,
                            scores, radius, status, tps, stages);
}

template <int CH>
cudaError_t launch_tc_n(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                        int Hkv, int G, int Nd, const int32_t *seq_len, int W, float *scores, float *radius,
                        int32_t *status, cudaStream_t st) {
  const int Nq = G * Nd;
  if (Nq <= 16) return launch_tc<16, CH>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  if (Nq <= 32) return launch_tc<32, CH>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  if (Nq <= 48) return launch_tc<48, CH>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  if (Nq <= 64) return launch_tc<64, CH>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score_blocks_tc(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft,
                                   int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                                   float *scores, float *radius, int32_t *status, cudaStream_t st) {
  if (D == 128)
    return launch_tc_n<16>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  return launch_tc_n<8>(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
}

}  // namespace oasis
